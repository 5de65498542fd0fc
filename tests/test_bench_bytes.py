"""The byte counts the benchmark's roofline fractions divide by, for the 261888-token q8 workload
(16 layers, Hq 6 / Hkv 1, D 256, page 16) on a 152-SM plan: K and V codes of every logical
token, the used block-table entries, Q, the FP32 split state (max, sum, numerator) written by the
partial kernel and read back by the combine, and the FP16 output with its FP32 log-sum-exp.
Host-only: the plan is made for 152 SMs without a device."""
import pytest

from speculative_verify_paged_e4m3_gb300 import workload as W


@pytest.fixture(scope="module")
def B():
    from speculative_verify_paged_e4m3_gb300 import binding, build
    build.build()
    return binding


def plan_for(B, w):
    return B.dflash_verify_attn_plan(B.make_problem(
        w.batch, w.q_len, w.num_q_heads, w.num_kv_heads, w.head_dim, w.page_size,
        w.max_pages_per_seq, w.num_pages, w.max_ctx, device=-1))


def test_c3_step_bytes(B):
    from speculative_verify_paged_e4m3_gb300.runner import algorithmic_bytes
    w = W.config3()
    plan = plan_for(B, w)
    assert plan.num_splits == 152
    nb = algorithmic_bytes(w, plan)
    n, D, R = 261888, 256, 48
    assert nb["kv"] == 2 * n * D                    # one byte per code, K and V
    assert nb["bt"] == (n // 16) * 4                # 16368 int32 entries
    assert nb["q"] == 8 * 6 * D * 2                 # FP16
    # splits of roundup(ceil(n / 152), 128) = 1792 keys: 147 of them hold keys
    assert nb["active_splits"] == -(-n // 1792) == 147
    assert nb["state"] == 147 * R * (D + 2) * 4     # numerator row + (m, l), FP32
    assert nb["out"] == 8 * 6 * (D * 2 + 4)         # FP16 out + FP32 lse
    assert nb["partial"] == 141_458_496
    assert nb["combine"] == 7_306_560
    # the 70 % bar at step level against the measured 6782.4 GB/s copy peak
    step = 16 * (nb["partial"] + nb["combine"])
    assert step == 2_380_240_896
    assert round(step / (0.70 * 6782.4e9) * 1e6, 1) == 501.3
