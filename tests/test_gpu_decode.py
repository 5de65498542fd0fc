"""E4M3 decode of the attention kernels, checked bit for bit through the attention itself.

The tensor-core kernel never decodes a K or V code in software: the codes go to the tensor core
(tcgen05.mma kind::f8f6f4) as they are. Its decode is therefore checked through problems whose
exact result exposes every code. One query token (q_len 1) sees one key (context length 1),
k_scale = v_scale = 1, and query head h is one-hot in dimension d_h with value 1:
  * the softmax over one key is exactly 1, so every head's output row is the decoded V row.
    FP16 holds every finite E4M3 value, so out[h][d] must equal dec(v_code[d]) exactly (the
    same bits, but for the sign of a zero);
  * the score of head h is dec(k_code[d_h]) / sqrt(256), and with one key the log-sum-exp is
    that score. Distinct E4M3 values differ by at least 2^-9, so their scores differ by at
    least 2^-13 = 1.2e-4, far more than the FP32 rounding of the score (a few 1e-7 relative,
    or absolute below 1): the LSE singles out the code.
Every finite code (254: S.1111.111 is NaN in E4M3FN) sits in the K and the V row, so a few calls
cover all of them. This is the check that the dequantised E4M3 values match exactly, on the path
that runs ("[Perf] Reduce DFlash2 attention cost and screen exact QK reuse", Test Result: exact
comparisons of complete FP32 score workspaces).
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import MODES, SIMT, kernel_args, to_np

pytestmark = pytest.mark.gpu

D = 256
P = 16


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_verify_paged_e4m3_gb300 import build
    build.build()


def finite_codes():
    return np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)


def one_key_problem(heads, k_row, v_row, dims, seed):
    """q [1, 1, heads, D] one-hot (head h in dims[h]); the key lives in slot 0 of physical page 1
    of a 2-page pool whose other bytes are random codes (NaN codes included); context length 1."""
    rng = np.random.default_rng(seed)
    k_pool = rng.integers(0, 256, size=(2, P, 1, D), dtype=np.uint8)
    v_pool = rng.integers(0, 256, size=(2, P, 1, D), dtype=np.uint8)
    k_pool[1, 0, 0] = k_row
    v_pool[1, 0, 0] = v_row
    q = np.zeros((1, 1, heads, D), dtype=np.float16)
    q[0, 0, np.arange(heads), dims] = 1.0
    return dict(q=torch.from_numpy(q), k_pool=torch.from_numpy(k_pool),
                v_pool=torch.from_numpy(v_pool),
                block_table=torch.tensor([[1]], dtype=torch.int32),
                context_lens=torch.tensor([1], dtype=torch.int32),
                k_scale=torch.tensor([1.0], dtype=torch.float32),
                v_scale=torch.tensor([1.0], dtype=torch.float32))


# 16 heads: the 16-row tensor-core instance; 48: the 48-row one (the pages' q8 shape carries 48
# rows per KV head); 256: six row blocks of 43 rows, every dimension in one call.
@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("heads", [16, 48, 256])
def test_decode_bit_exact_through_attention(mode, heads):
    from speculative_verify_paged_e4m3_gb300 import binding as B
    orc = oracle.load()
    codes = finite_codes()
    att = B.VerifyAttention(1, 1, heads, 1, D, P, 1, 2, P, **kernel_args(mode))
    if mode != SIMT:
        assert att.plan.kernel == B.DFLASH_KERNEL_TCGEN05
    seen_k, seen_v = set(), set()
    calls = -(-D // heads)
    # 254 finite codes in 256 slots (two repeats); the K row stays, so that the calls' one-hot
    # dimensions together read all of it; the V row changes order each call
    k_row = np.random.default_rng(499).permutation(np.concatenate([codes, codes[:2]]))
    for call in range(calls):
        rng = np.random.default_rng(500 + call)
        v_row = rng.permutation(np.concatenate([codes, codes[rng.integers(0, 254, 2)]]))
        dims = (call * heads + np.arange(heads)) % D
        inp = one_key_problem(heads, k_row, v_row, dims, seed=call)
        dev = {k: v.cuda() for k, v in inp.items()}
        out, lse = att(dev["q"], dev["k_pool"], dev["v_pool"], dev["block_table"],
                       dev["context_lens"], dev["k_scale"], dev["v_scale"])
        torch.cuda.synchronize()
        # V: every head's output row is the decoded V row, bit for bit (as FP16)
        v_dec = orc.e4m3_decode(v_row)
        want = v_dec.astype(np.float16)
        assert np.array_equal(want.astype(np.float64), v_dec)  # FP16 holds every E4M3 value
        # compared as values: equal values are equal bits, except that the code -0 may come out
        # as +0 (a sum of -0 and the +0 products of the masked keys is +0)
        got = to_np(out)[0, 0].astype(np.float64)
        for h in range(heads):
            assert np.array_equal(got[h], v_dec), (
                f"head {h}: V decode differs at dims {np.nonzero(got[h] != v_dec)[0][:8]}")
        seen_v.update(int(c) for c in v_row)
        # K: the LSE of head h is dec(k_code[d_h]) / 16, and names that code among all 254
        k_dec = orc.e4m3_decode(k_row[dims])
        lse_h = to_np(lse)[0, 0].astype(np.float64)
        err = np.abs(lse_h - k_dec / 16.0)
        assert np.all(err <= 2e-6 * np.maximum(1.0, np.abs(k_dec / 16.0))), err.max()
        values = orc.e4m3_decode(codes) / 16.0
        nearest = np.abs(lse_h[:, None] - values[None, :]).argmin(axis=1)
        assert np.array_equal(values[nearest], k_dec / 16.0)
        seen_k.update(int(c) for c in k_row[dims])
    assert seen_v == set(int(c) for c in codes)
    assert seen_k == set(int(c) for c in codes)


@pytest.mark.parametrize("mode", MODES)
def test_decode_with_power_of_two_scales(mode):
    """Power-of-two scales keep every product exact: out = dec(v) * v_scale bit for bit."""
    from speculative_verify_paged_e4m3_gb300 import binding as B
    orc = oracle.load()
    codes = finite_codes()
    heads = 48
    att = B.VerifyAttention(1, 1, heads, 1, D, P, 1, 2, P, **kernel_args(mode))
    rng = np.random.default_rng(77)
    k_row = rng.permutation(np.concatenate([codes, codes[:2]]))
    v_row = rng.permutation(np.concatenate([codes, codes[2:4]]))
    dims = np.arange(heads) * 5 % D
    for ks, vs in ((2.0, 0.25), (0.125, 8.0)):
        inp = one_key_problem(heads, k_row, v_row, dims, seed=9)
        inp["k_scale"] = torch.tensor([ks], dtype=torch.float32)
        inp["v_scale"] = torch.tensor([vs], dtype=torch.float32)
        dev = {k: v.cuda() for k, v in inp.items()}
        out, lse = att(dev["q"], dev["k_pool"], dev["v_pool"], dev["block_table"],
                       dev["context_lens"], dev["k_scale"], dev["v_scale"])
        torch.cuda.synchronize()
        want = orc.e4m3_decode(v_row) * vs  # exact, and an FP16 value
        assert np.array_equal(want.astype(np.float16).astype(np.float64), want)
        got = to_np(out)[0, 0].astype(np.float64)
        assert np.array_equal(got, np.broadcast_to(want, got.shape))
        k_dec = orc.e4m3_decode(k_row[dims]) * ks / 16.0
        lse_h = to_np(lse)[0, 0].astype(np.float64)
        assert np.all(np.abs(lse_h - k_dec) <= 2e-6 * np.maximum(1.0, np.abs(k_dec)))
