"""Invariances of the attention that the CUDA path must keep on the GPU.

* Paging: where a logical page lives in the pool must not matter. Moving every physical page to
  another slot of the pool (its unused tail slots, filled with random codes, move along) and
  rewriting the block table to match must give the same out and lse, bit for bit, in every
  kernel mode ("[Perf] Reduce DFlash2 long-context verification decay", Implementation: the
  compact page map). The oracle pins the same property on the CPU.
* The causal tail: query token i of a q_len-token block sees keys 0 .. N - q_len + i, exactly
  what a single query token at the end of a context of N - q_len + i + 1 keys sees. So row i of
  a q8 call must match a q_len = 1 call over that shorter context, within the output tolerance
  (two kernel launches with different split boundaries: close, not the same bits).
"""
import numpy as np
import pytest
import torch

from gpu_helpers import MODES, gpu_forward, out_bound, to_device, to_np
from speculative_verify_paged_e4m3_gb300 import workload as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_verify_paged_e4m3_gb300 import build
    build.build()


def small(name, context, q_len=8, Hq=6, Hkv=1, P=16, seed=0, pool_factor=1.5):
    return W.Workload(name, layers=1, context=tuple(context), q_len=q_len, num_q_heads=Hq,
                      num_kv_heads=Hkv, page_size=P, pool_factor=pool_factor,
                      seed_base=95000 + seed)


def permute_pages(inp, seed):
    """The same logical cache with every physical page moved: page p goes to slot perm[p]."""
    num_pages = inp["k_pool"].shape[0]
    perm = np.random.default_rng(seed).permutation(num_pages)
    out = dict(inp)
    k = torch.empty_like(inp["k_pool"])
    v = torch.empty_like(inp["v_pool"])
    k[torch.from_numpy(perm)] = inp["k_pool"]
    v[torch.from_numpy(perm)] = inp["v_pool"]
    bt = inp["block_table"].clone()
    inside = (bt >= 0) & (bt < num_pages)
    bt[inside] = torch.from_numpy(perm)[bt[inside].long()].to(torch.int32)
    out.update(k_pool=k, v_pool=v, block_table=bt)
    return out


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("case", ["n4100_p16", "n9000_p64", "batch3_hkv2", "n300_p3296"])
def test_block_table_permutation_is_bitwise_invisible(mode, case):
    w = {"n4100_p16": small("perm_a", [4100], seed=1),
         "n9000_p64": small("perm_b", [9000], P=64, seed=2),
         "batch3_hkv2": small("perm_c", [3000, 517, 2048], Hq=12, Hkv=2, seed=3),
         "n300_p3296": small("perm_d", [300], P=3296, seed=4, pool_factor=3.0)}[case]
    inp = W.make_layer(w, 0, device="cpu")
    moved = permute_pages(inp, seed=11)
    assert not torch.equal(moved["block_table"], inp["block_table"])
    _, out_a, lse_a = gpu_forward(to_device(inp), kernel=mode)
    _, out_b, lse_b = gpu_forward(to_device(moved), kernel=mode)
    assert np.array_equal(to_np(out_a).view(np.uint16), to_np(out_b).view(np.uint16))
    assert np.array_equal(to_np(lse_a).view(np.uint32), to_np(lse_b).view(np.uint32))


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("n", [9, 1031, 4100, 70000])
def test_row_i_of_q8_is_a_q1_call_over_the_shorter_context(mode, n):
    q_len = 8
    w = small(f"tail{n}", [n], q_len=q_len, seed=20 + n % 97)
    inp = W.make_layer(w, 0, device="cpu")
    mpps = inp["block_table"].shape[1]
    max_ctx = mpps * w.page_size
    _, out8, lse8 = gpu_forward(to_device(inp), kernel=mode, max_context=max_ctx)
    out8, lse8 = to_np(out8).astype(np.float64), to_np(lse8).astype(np.float64)
    for i in range(q_len):
        one = dict(inp)
        one["q"] = inp["q"][:, i:i + 1].contiguous()
        one["context_lens"] = torch.tensor([n - q_len + i + 1], dtype=torch.int32)
        _, out1, lse1 = gpu_forward(to_device(one), kernel=mode, max_context=max_ctx)
        out1, lse1 = to_np(out1).astype(np.float64)[:, 0], to_np(lse1).astype(np.float64)[:, 0]
        assert np.all(np.abs(out8[:, i] - out1) <= out_bound(out1)), (i, np.abs(
            out8[:, i] - out1).max())
        assert np.all(np.abs(lse8[:, i] - lse1) <= 1e-5 * np.maximum(1.0, np.abs(lse1))), i
