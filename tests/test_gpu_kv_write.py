"""The drafted-token KV write (E4M3 quantise + scatter into the paged pools) against the oracle,
byte for byte over the whole pools, through the C ABI; then the attention over the written pools.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import compare, oracle_forward, to_np

pytestmark = pytest.mark.gpu

D = 256
# oracle flag bits -> status word bits
FLAG_MAP = {1: 0x2, 2: 0x4, 4: 0x1}


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_verify_paged_e4m3_gb300 import build
    build.build()


def make_case(seed, contexts, q_len=8, Hkv=1, P=16, max_context=None, pool_extra=4,
              bad_entries=(), scales=(0.0173, 0.0291), special=None, quantised_pools=False,
              sigma=(2.0, 3.0)):
    rng = np.random.default_rng(seed)
    B = len(contexts)
    max_context = max_context or max(contexts)
    max_pages = math.ceil(max(max(contexts), max_context) / P)
    num_pages = B * max_pages + pool_extra
    perm = rng.permutation(num_pages)
    bt = np.full((B, max_pages), -1, dtype=np.int32)
    for b in range(B):
        bt[b] = perm[b * max_pages:(b + 1) * max_pages]
    for b, lp, v in bad_entries:
        bt[b, lp] = v
    k_new = (rng.standard_normal((B, q_len, Hkv, D)) * sigma[0]).astype(np.float16)
    v_new = (rng.standard_normal((B, q_len, Hkv, D)) * sigma[1]).astype(np.float16)
    if quantised_pools:
        # what a quantised cache holds: codes of N(0, sigma) data at the layer scales (the
        # library float8 cast), the same spread as the drafted rows
        def codes(sigma, scale):
            x = rng.standard_normal((num_pages, P, Hkv, D)).astype(np.float32) * sigma / scale
            x = np.clip(x, -448, 448)  # the library cast does not saturate
            return torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        k_pool, v_pool = codes(sigma[0], scales[0]), codes(sigma[1], scales[1])
    else:
        k_pool = rng.integers(0, 256, size=(num_pages, P, Hkv, D), dtype=np.uint8)
        v_pool = rng.integers(0, 256, size=(num_pages, P, Hkv, D), dtype=np.uint8)
        # outliers past 448 * scale: saturate
        k_new.reshape(-1)[rng.integers(0, k_new.size, 64)] = np.float16(30.0)
        v_new.reshape(-1)[rng.integers(0, v_new.size, 64)] = np.float16(-40.0)
    if special is not None:
        k_new.reshape(-1)[:len(special)] = special
        v_new.reshape(-1)[:len(special)] = special
    return dict(k_new=k_new, v_new=v_new, bt=bt, ctx=np.array(contexts, dtype=np.int32),
                k_scale=np.float32(scales[0]), v_scale=np.float32(scales[1]), k_pool=k_pool,
                v_pool=v_pool, max_context=max_context, Hkv=Hkv, P=P, q_len=q_len)


def run_gpu(c):
    from speculative_verify_paged_e4m3_gb300 import binding as B
    B_, q_len, Hkv = c["k_new"].shape[0], c["q_len"], c["Hkv"]
    att = B.VerifyAttention(B_, q_len, 6 * Hkv, Hkv, D, c["P"], c["bt"].shape[1],
                            c["k_pool"].shape[0], c["max_context"], device=0)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    kp, vp = dev(c["k_pool"]), dev(c["v_pool"])
    att.kv_write(dev(c["k_new"]), dev(c["v_new"]), dev(c["bt"]), dev(c["ctx"]),
                 dev(np.array([c["k_scale"]])), dev(np.array([c["v_scale"]])), kp, vp)
    torch.cuda.synchronize()
    return att, kp.cpu().numpy(), vp.cpu().numpy(), att.workspace_views()[0].item()


def run_oracle(c):
    kp, vp, flags = oracle.load().kv_write(c["k_new"], c["v_new"], c["bt"], c["ctx"],
                                           c["k_scale"], c["v_scale"], c["k_pool"], c["v_pool"],
                                           c["max_context"])
    status = 0
    for bit, st in FLAG_MAP.items():
        if flags & bit:
            status |= st
    return kp, vp, status


def same_codes(got, want):
    """Byte equality, except that a NaN code may carry either sign."""
    nan = (want & 0x7F) == 0x7F
    assert np.array_equal(np.isin(got[nan] & 0x7F, [0x7F]), np.ones(nan.sum(), bool))
    diff = np.nonzero((got != want) & ~nan)
    assert diff[0].size == 0, f"{diff[0].size} bytes differ, first at {tuple(x[0] for x in diff)}"


@pytest.mark.parametrize("seed,contexts,Hkv,P", [
    (1, [100, 37, 9], 2, 16),
    (2, [4096], 1, 16),
    (3, [1000, 1001, 1002, 1003], 4, 64),
])
def test_kv_write_random(seed, contexts, Hkv, P):
    c = make_case(seed, contexts, Hkv=Hkv, P=P)
    _, kp, vp, status = run_gpu(c)
    ek, ev, est = run_oracle(c)
    same_codes(kp, ek)
    same_codes(vp, ev)
    assert status == est == 0


def test_kv_write_short_clamped_and_out_of_pool():
    # sequence 0 shorter than q_len (3 tokens have no slot), sequence 1 past max_context
    # (clamped), sequence 2 with one page entry outside the pool (its tokens are not written)
    c = make_case(4, [5, 200, 150], max_context=160, bad_entries=[(2, 9, 10 ** 6)])
    _, kp, vp, status = run_gpu(c)
    ek, ev, est = run_oracle(c)
    same_codes(kp, ek)
    same_codes(vp, ev)
    assert status == est == (0x1 | 0x2 | 0x4)


def test_kv_write_special_values_and_q1():
    special = np.array([np.nan, np.inf, -np.inf, -0.0, 0.0, 6e-8, -6e-8, 65504, -65504],
                       dtype=np.float16)
    for q_len in (1, 8):
        c = make_case(5, [33, 64], q_len=q_len, special=special)
        _, kp, vp, status = run_gpu(c)
        ek, ev, _ = run_oracle(c)
        same_codes(kp, ek)
        same_codes(vp, ev)


def test_kv_write_full_size_pool():
    # the 261888-token layout: 16368 pages of 16 tokens, one KV head; the whole pool is compared
    c = make_case(6, [261888], pool_extra=0)
    _, kp, vp, status = run_gpu(c)
    ek, ev, est = run_oracle(c)
    same_codes(kp, ek)
    same_codes(vp, ev)
    assert status == est == 0


def test_attention_over_written_tokens():
    """Write the drafted tokens, then verify over the pools: the attention of the GPU-written
    pools matches the oracle's attention over the oracle-written pools."""
    # the parity workloads' statistics: N(0, 1) keys and values, scale about amax / 448
    c = make_case(7, [700, 333], Hkv=2, quantised_pools=True, sigma=(1.0, 1.0),
                  scales=(5.0 / 448, 5.0 / 448))
    att, kp, vp, status = run_gpu(c)
    ek, ev, _ = run_oracle(c)
    same_codes(kp, ek)
    same_codes(vp, ev)
    rng = np.random.default_rng(8)
    q = rng.standard_normal((2, 8, 12, D)).astype(np.float16)
    inp = dict(q=torch.from_numpy(q), k_pool=torch.from_numpy(ek), v_pool=torch.from_numpy(ev),
               block_table=torch.from_numpy(c["bt"]), context_lens=torch.from_numpy(c["ctx"]),
               k_scale=torch.tensor([c["k_scale"]]), v_scale=torch.tensor([c["v_scale"]]))
    ref_out, ref_lse = oracle_forward(inp)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    out, lse = att(dev(q), dev(kp), dev(vp), dev(c["bt"]), dev(c["ctx"]),
                   dev(np.array([c["k_scale"]])), dev(np.array([c["v_scale"]])))
    torch.cuda.synchronize()
    compare(to_np(out), to_np(lse), ref_out, ref_lse, what="attention over written tokens")
