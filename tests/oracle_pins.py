"""Pins of the CPU oracle to things other than itself.

Each pin takes an oracle handle and raises AssertionError when the oracle disagrees with what the
pin knows independently: the OCP E4M3 table, torch's library float8 cast and float64
scaled-dot-product attention, closed forms of uniform and one-hot softmax, invariances of the
paged layout, split/merge agreement, and the q_len = 1 reduction. ``PINS`` lists them; the planted
mistake tests run all of them against mutated builds of the oracle and expect one to fail.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch
import torch.nn.functional as F

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------------------------------------
# small builders (layout only; no attention arithmetic)

def paged_case(rng, B=1, q_len=8, Hq=6, Hkv=1, D=256, P=16, contexts=(40,), pool_extra=3,
               k_codes=None, v_codes=None, q=None, ks=0.0123, vs=0.0457):
    """Random paged problem. Logical codes [sum(N), Hkv, D] are scattered into a shuffled pool."""
    total = sum(contexts)
    if k_codes is None:
        k_codes = rng.integers(0, 256, size=(total, Hkv, D), dtype=np.uint8)
        k_codes[(k_codes & 0x7F) == 0x7F] ^= 0x01  # no NaN codes inside the context
    if v_codes is None:
        v_codes = rng.integers(0, 256, size=(total, Hkv, D), dtype=np.uint8)
        v_codes[(v_codes & 0x7F) == 0x7F] ^= 0x01
    if q is None:
        q = rng.standard_normal((B, q_len, Hq, D)).astype(np.float16)
    max_pages = max(1, max(math.ceil(n / P) for n in contexts))
    used = sum(math.ceil(n / P) for n in contexts)
    num_pages = used + pool_extra
    k_pool = np.full((num_pages, P, Hkv, D), 0x7F, dtype=np.uint8)  # NaN outside the context
    v_pool = np.full((num_pages, P, Hkv, D), 0x7F, dtype=np.uint8)
    perm = rng.permutation(num_pages)
    bt = np.full((B, max_pages), -1, dtype=np.int32)
    t0 = 0
    u = 0
    for b, n in enumerate(contexts):
        for lp in range(math.ceil(n / P)):
            phys = perm[u]
            u += 1
            bt[b, lp] = phys
            cnt = min(P, n - lp * P)
            k_pool[phys, :cnt] = k_codes[t0 + lp * P:t0 + lp * P + cnt]
            v_pool[phys, :cnt] = v_codes[t0 + lp * P:t0 + lp * P + cnt]
        t0 += n
    bt[bt < 0] = 0  # never read: past the context
    return dict(q=q, k_pool=k_pool, v_pool=v_pool, block_table=bt,
                context_lens=np.array(contexts, dtype=np.int32), k_scale=ks, v_scale=vs)


def run(orc, case):
    return orc.verify_attn(case["q"], case["k_pool"], case["v_pool"], case["block_table"],
                           case["context_lens"], case["k_scale"], case["v_scale"])


def gather_logical(case, b):
    """Logical K and V codes [N, Hkv, D] of sequence b, read through the block table."""
    P = case["k_pool"].shape[1]
    n = int(case["context_lens"][b])
    j = np.arange(n)
    phys = case["block_table"][b, j // P]
    return case["k_pool"][phys, j % P], case["v_pool"][phys, j % P]


def torch_decode(codes):
    """Library decode: reinterpret as torch.float8_e4m3fn and widen to float64."""
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float64)


# ---------------------------------------------------------------------------------------------
# pins

def pin_e4m3_spec_points(orc):
    """Decode of the OCP table's printed points (tests/golden/e4m3_spec_points.txt)."""
    codes, vals = [], []
    with open(os.path.join(GOLDEN, "e4m3_spec_points.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            c, v = line.split()
            codes.append(int(c, 16))
            vals.append(float(v))
    got = orc.e4m3_decode(np.array(codes, dtype=np.uint8))
    for c, v, g in zip(codes, vals, got):
        if math.isnan(v):
            assert math.isnan(g), f"code {c:#04x}: expected NaN, got {g}"
        else:
            assert g == v and math.copysign(1, g) == math.copysign(1, v), (
                f"code {c:#04x}: expected {v}, got {g}")


def pin_e4m3_all_codes_vs_torch(orc):
    """All 256 codes against torch's float8_e4m3fn cast (a library routine)."""
    codes = np.arange(256, dtype=np.uint8)
    got = orc.e4m3_decode(codes)
    ref = torch_decode(codes).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def _sdpa_reference(case):
    """Dense float64 attention by torch's scaled_dot_product_attention with a causal-tail mask."""
    q = torch.from_numpy(case["q"].astype(np.float64))
    B, q_len, Hq, D = q.shape
    Hkv = case["k_pool"].shape[2]
    G = Hq // Hkv
    outs, lses = [], []
    for b in range(B):
        n = int(case["context_lens"][b])
        kc, vc = gather_logical(case, b)
        k = torch_decode(kc) * case["k_scale"]  # [N, Hkv, D]
        v = torch_decode(vc) * case["v_scale"]
        k = k.permute(1, 0, 2).repeat_interleave(G, dim=0)  # [Hq, N, D]
        v = v.permute(1, 0, 2).repeat_interleave(G, dim=0)
        qb = q[b].permute(1, 0, 2)  # [Hq, q_len, D]
        pos = n - q_len + torch.arange(q_len)
        mask = torch.arange(n)[None, :] <= pos[:, None]  # [q_len, N]
        o = F.scaled_dot_product_attention(qb, k, v, attn_mask=mask, scale=1.0 / math.sqrt(D))
        s = torch.matmul(qb, k.transpose(1, 2)) / math.sqrt(D)
        lse = torch.logsumexp(s.masked_fill(~mask, float("-inf")), dim=-1)  # [Hq, q_len]
        outs.append(o.permute(1, 0, 2).numpy())
        lses.append(lse.permute(1, 0).numpy())
    return np.stack(outs), np.stack(lses)


def pin_tiny_vs_torch_sdpa(orc):
    """Tiny cases (N <= 64) against torch's float64 SDPA on densely gathered K/V."""
    rng = np.random.default_rng(7)
    shapes = [
        dict(q_len=8, Hq=6, Hkv=1, D=256, P=16, contexts=(40,)),
        dict(q_len=1, Hq=6, Hkv=1, D=256, P=16, contexts=(17,)),
        dict(q_len=5, Hq=4, Hkv=2, D=16, P=3, contexts=(5, 23)),
        dict(q_len=3, Hq=2, Hkv=2, D=32, P=16, contexts=(64, 9, 33)),
        dict(q_len=8, Hq=6, Hkv=1, D=256, P=64, contexts=(8,)),
        dict(q_len=16, Hq=6, Hkv=1, D=256, P=16, contexts=(40,)),   # 96 rows per KV head
        dict(q_len=16, Hq=16, Hkv=1, D=32, P=16, contexts=(50, 16)),  # 256 rows per KV head
    ]
    for sh in shapes:
        case = paged_case(rng, B=len(sh["contexts"]), **sh)
        out, lse = run(orc, case)
        ref_out, ref_lse = _sdpa_reference(case)
        np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12, err_msg=str(sh))
        np.testing.assert_allclose(lse, ref_lse, rtol=1e-13, atol=1e-13, err_msg=str(sh))


def pin_uniform_closed_form(orc):
    """All-zero K codes: every visible score is 0, so lse = ln(visible count), out = mean of V."""
    rng = np.random.default_rng(11)
    N, q_len, Hq, Hkv, D = 37, 8, 6, 1, 256
    k_codes = np.zeros((N, Hkv, D), dtype=np.uint8)
    case = paged_case(rng, q_len=q_len, Hq=Hq, Hkv=Hkv, D=D, contexts=(N,), k_codes=k_codes)
    out, lse = run(orc, case)
    _, vc = gather_logical(case, 0)
    v = torch_decode(vc).numpy() * case["v_scale"]
    for i in range(q_len):
        n_vis = N - q_len + i + 1
        assert np.all(lse[0, i] == np.log(n_vis)), (i, lse[0, i], np.log(n_vis))
        mean = v[:n_vis, 0].mean(axis=0)
        np.testing.assert_allclose(out[0, i], np.broadcast_to(mean, (Hq, D)), rtol=0,
                                   atol=1e-14)


def pin_one_hot_closed_form(orc):
    """One key j* aligned with a one-hot Q: lse = ln(e^s* + n - 1), out weights in closed form.

    j* = N - q_len + 3 is visible to tokens i >= 3 only, which also pins the causal edge.
    """
    rng = np.random.default_rng(13)
    N, q_len, Hq, Hkv, D = 50, 8, 6, 1, 256
    ks = 0.01
    k_codes = np.zeros((N, Hkv, D), dtype=np.uint8)
    jstar = N - q_len + 3
    k_codes[jstar, 0, 0] = 0x7E  # 448
    q = np.zeros((1, q_len, Hq, D), dtype=np.float16)
    c = np.array([16.0, 8.0, 4.0, 2.0, 1.0, 0.5], dtype=np.float16)  # per query head
    q[0, :, :, 0] = c
    case = paged_case(rng, q_len=q_len, Hq=Hq, Hkv=Hkv, D=D, contexts=(N,), k_codes=k_codes,
                      q=q, ks=ks)
    out, lse = run(orc, case)
    _, vc = gather_logical(case, 0)
    v = torch_decode(vc).numpy()[:, 0] * case["v_scale"]
    for i in range(q_len):
        n_vis = N - q_len + i + 1
        for g in range(Hq):
            if i >= 3:
                sstar = float(c[g]) * 448.0 * ks / 16.0
                exp_lse = sstar + math.log1p((n_vis - 1) * math.exp(-sstar))
                w_star = 1.0 / (1.0 + (n_vis - 1) * math.exp(-sstar))
                w_rest = math.exp(-sstar) * w_star
                exp_out = w_star * v[jstar] + w_rest * (v[:n_vis].sum(axis=0) - v[jstar])
            else:
                exp_lse = math.log(n_vis)
                exp_out = v[:n_vis].mean(axis=0)
            assert abs(lse[0, i, g] - exp_lse) <= 1e-14 * max(1.0, abs(exp_lse)), (i, g)
            np.testing.assert_allclose(out[0, i, g], exp_out, rtol=0, atol=1e-14,
                                       err_msg=f"row {i},{g}")


def pin_block_table_permutation(orc):
    """Moving every page to another physical slot (and the table with it) changes no bit."""
    rng = np.random.default_rng(17)
    case = paged_case(rng, B=2, q_len=4, Hq=6, Hkv=1, D=64, P=16, contexts=(70, 33))
    out, lse = run(orc, case)
    num_pages = case["k_pool"].shape[0]
    perm = rng.permutation(num_pages)
    moved = dict(case)
    moved["k_pool"] = np.empty_like(case["k_pool"])
    moved["v_pool"] = np.empty_like(case["v_pool"])
    moved["k_pool"][perm] = case["k_pool"]
    moved["v_pool"][perm] = case["v_pool"]
    moved["block_table"] = perm[case["block_table"]].astype(np.int32)
    out2, lse2 = run(orc, moved)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def pin_page_size_invariance(orc):
    """The same logical K/V laid out with page sizes 16, 64, 48 and 1 gives identical bits."""
    rng = np.random.default_rng(19)
    N, q_len, Hq, Hkv, D = 97, 6, 6, 1, 32
    k_codes = rng.integers(0, 0x7E, size=(N, Hkv, D), dtype=np.uint8)
    v_codes = rng.integers(0, 0x7E, size=(N, Hkv, D), dtype=np.uint8) | (
        rng.integers(0, 2, size=(N, Hkv, D), dtype=np.uint8) << 7)
    q = rng.standard_normal((1, q_len, Hq, D)).astype(np.float16)
    res = []
    for P in (16, 64, 48, 1):
        case = paged_case(rng, q_len=q_len, Hq=Hq, Hkv=Hkv, D=D, P=P, contexts=(N,),
                          k_codes=k_codes, v_codes=v_codes, q=q)
        res.append(run(orc, case))
    for out, lse in res[1:]:
        assert np.array_equal(out, res[0][0]) and np.array_equal(lse, res[0][1])


def _merge(orc, case, bounds):
    import oracle as oracle_pkg
    B = len(case["context_lens"])
    sb = np.array([bounds] * B, dtype=np.int32)
    m, l, acc = orc.verify_attn_partials(case["q"], case["k_pool"], case["v_pool"],
                                         case["block_table"], case["context_lens"],
                                         case["k_scale"], case["v_scale"], sb)
    mt, lt, at = oracle_pkg.rows_view(m, l, acc)
    out, lse = orc.merge_partials(mt, lt, at)
    q_len, Hq = case["q"].shape[1], case["q"].shape[2]
    Hkv = case["k_pool"].shape[2]
    return (oracle_pkg.rows_to_bqh(out, B, q_len, Hq, Hkv),
            oracle_pkg.rows_to_bqh(lse, B, q_len, Hq, Hkv), m, l)


def pin_split_merge_agreement(orc):
    """Merging split state (with empty and fully masked splits) equals the unsplit result."""
    rng = np.random.default_rng(23)
    N, q_len = 60, 8
    case = paged_case(rng, q_len=q_len, Hq=6, Hkv=1, D=256, contexts=(N,))
    out, lse = run(orc, case)
    bounds = [0, 7, 7, 30, N - q_len + 1, N - 2, N]  # an empty split and tail-only splits
    mout, mlse, m, l = _merge(orc, case, bounds)
    np.testing.assert_allclose(mout, out, rtol=0, atol=1e-13)
    np.testing.assert_allclose(mlse, lse, rtol=1e-13, atol=0)
    # the empty split and, for token 0, the splits past its position carry no state
    assert np.all(m[0, 0, 1] == -np.inf) and np.all(l[0, 0, 1] == 0)
    assert np.all(m[0, 0, 4:, 0:6] == -np.inf)


def pin_split_merge_exact_integers(orc):
    """Integer-valued data (zero scores, integral V): merges of any split set agree bitwise."""
    rng = np.random.default_rng(29)
    N, q_len, D = 45, 8, 256
    k_codes = np.zeros((N, 1, D), dtype=np.uint8)
    v_codes = rng.choice(np.array([0x38, 0x40, 0x44, 0xB8, 0x00], dtype=np.uint8),
                         size=(N, 1, D))  # 1, 2, 3, -1, 0
    case = paged_case(rng, q_len=q_len, contexts=(N,), k_codes=k_codes, v_codes=v_codes,
                      ks=1.0, vs=1.0)
    one, one_lse, _, l1 = _merge(orc, case, [0, N])
    for bounds in ([0, 16, 32, N], [0, 1, 2, 3, 40, 40, N], [0, N - q_len + 1, N]):
        got, got_lse, _, l = _merge(orc, case, bounds)
        assert np.array_equal(got, one) and np.array_equal(got_lse, one_lse), bounds
    n_vis = N - q_len + np.arange(q_len) + 1
    assert np.array_equal(l1[0, 0, 0].reshape(q_len, 6)[:, 0], n_vis.astype(np.float64))


def pin_q1_reduction(orc, q_len=8, seed=31):
    """Token i of a q_len block equals a q_len = 1 call over the first N - q_len + i + 1 keys."""
    rng = np.random.default_rng(seed)
    N = 75
    case = paged_case(rng, q_len=q_len, Hq=6, Hkv=1, D=256, contexts=(N,))
    out, lse = run(orc, case)
    for i in range(q_len):
        one = dict(case)
        one["q"] = case["q"][:, i:i + 1]
        one["context_lens"] = np.array([N - q_len + i + 1], dtype=np.int32)
        o1, l1 = run(orc, one)
        assert np.array_equal(o1[:, 0], out[:, i]) and np.array_equal(l1[:, 0], lse[:, i]), i


def pin_q1_reduction_long_block(orc):
    """The same reduction for a 16-token block (more rows than one tensor-core CTA holds)."""
    pin_q1_reduction(orc, q_len=16, seed=32)


def _spec_points():
    """(code, value) pairs printed in the OCP table (tests/golden/e4m3_spec_points.txt)."""
    pts = []
    with open(os.path.join(GOLDEN, "e4m3_spec_points.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                c, v = line.split()
                pts.append((int(c, 16), float(v)))
    return pts


def pin_e4m3_encode_spec_points(orc):
    """Encode of the OCP table's printed finite values gives their codes (signed zero kept)."""
    pts = [(c, v) for c, v in _spec_points() if not math.isnan(v)]
    got = orc.e4m3_encode(np.array([v for _, v in pts]))
    for (c, v), g in zip(pts, got):
        assert g == c, f"value {v}: expected {c:#04x}, got {g:#04x}"


def pin_e4m3_encode_midpoints_ties_to_even(orc):
    """Halfway between two neighbouring finite codes (values from torch's float8 decode) the
    even code wins; a hair either side, the nearer one."""
    codes = np.arange(0x7F, dtype=np.uint8)  # 0x00 .. 0x7E, ascending values
    vals = torch_decode(codes).numpy()
    lo, hi = vals[:-1], vals[1:]
    mid = (lo + hi) / 2  # exact in float64
    got = orc.e4m3_encode(mid)
    even = np.where(codes[:-1] % 2 == 0, codes[:-1], codes[1:])
    assert np.array_equal(got, even), np.nonzero(got != even)
    gap = hi - lo
    assert np.array_equal(orc.e4m3_encode(mid - gap * 1e-6), codes[:-1])
    assert np.array_equal(orc.e4m3_encode(mid + gap * 1e-6), codes[1:])
    assert np.array_equal(orc.e4m3_encode(-mid), even | 0x80)


def pin_e4m3_encode_vs_torch_cast(orc):
    """Random FP32 values across the normal and subnormal range (|v| < 464, where the library
    cast needs no saturation) against torch's float8_e4m3fn cast."""
    rng = np.random.default_rng(7)
    mag = np.exp2(rng.uniform(-12, np.log2(460), size=20000)).astype(np.float32)
    v = (mag * rng.choice([-1, 1], size=mag.size)).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = orc.e4m3_encode(v.astype(np.float64))
    assert np.array_equal(got, ref), np.nonzero(got != ref)


def pin_e4m3_encode_saturation_nan_zero(orc):
    """Largest finite magnitude 448 (code S.1111.110) for everything at or beyond it, NaN to the
    NaN code, zeros keep their sign."""
    big = np.array([448.0, 449.0, 463.99, 464.0, 480.0, 1e30, np.inf])
    assert np.all(orc.e4m3_encode(big) == 0x7E)
    assert np.all(orc.e4m3_encode(-big) == 0xFE)
    assert orc.e4m3_encode(np.array([np.nan]))[0] & 0x7F == 0x7F
    assert list(orc.e4m3_encode(np.array([0.0, -0.0, 2.0 ** -11, -2.0 ** -11]))) == [
        0x00, 0x80, 0x00, 0x80]


def _kv_case():
    """Two sequences, three drafted tokens, two KV heads, D 8, page 4; pools filled with 0x55."""
    pts = dict((v, c) for c, v in _spec_points() if not math.isnan(v))
    vals = [1.0, 2.0, 0.5, -1.0, 448.0, 3.0, 256.0, 0.015625]
    scale, v_scale = 0.5, 0.25
    k_new = np.empty((2, 3, 2, 8), dtype=np.float16)
    v_new = np.empty_like(k_new)
    for b in range(2):
        for i in range(3):
            for h in range(2):
                rot = (b * 5 + i * 3 + h) % 8
                k_new[b, i, h] = [vals[(d + rot) % 8] * scale for d in range(8)]
                v_new[b, i, h] = [-vals[(d + rot + 1) % 8] * v_scale for d in range(8)]
    code = lambda x: pts[abs(x)] | (0x80 if x < 0 else 0)
    pool = np.full((5, 4, 2, 8), 0x55, dtype=np.uint8)
    return k_new, v_new, scale, v_scale, pool, code


def pin_kv_write_hand_placed(orc):
    """Drafted token i of a length-n sequence lands at position n - q_len + i (page via the block
    table, slot = position mod page size); nothing else in the pools changes; a token before the
    start is skipped and flagged."""
    k_new, v_new, scale, v_scale, pool, code = _kv_case()
    bt = np.array([[3, 0, -1], [4, -1, -1]], dtype=np.int32)
    ctx = np.array([6, 2], dtype=np.int32)
    kp, vp, flags = orc.kv_write(k_new, v_new, bt, ctx, scale, v_scale, pool, pool, 12)
    ek, ev = pool.copy(), pool.copy()
    # sequence 0: positions 3, 4, 5 -> (page 3, slot 3), (page 0, slot 0), (page 0, slot 1)
    # sequence 1: positions -1 (skipped), 0, 1 -> (page 4, slot 0), (page 4, slot 1)
    for b, i, page, slot in [(0, 0, 3, 3), (0, 1, 0, 0), (0, 2, 0, 1), (1, 1, 4, 0), (1, 2, 4, 1)]:
        for h in range(2):
            ek[page, slot, h] = [code(float(x) / scale) for x in k_new[b, i, h]]
            ev[page, slot, h] = [code(float(x) / v_scale) for x in v_new[b, i, h]]
    assert flags == 1, flags
    assert np.array_equal(kp, ek) and np.array_equal(vp, ev)


def pin_kv_write_clamps(orc):
    """An out-of-pool page entry skips its token (flag 2); a length beyond max_context is clamped
    to it (flag 4), so the tokens go to max_context - q_len + i."""
    k_new, v_new, scale, v_scale, pool, code = _kv_case()
    bt = np.array([[3, 7, 1], [2, 0, -1]], dtype=np.int32)
    ctx = np.array([6, 9], dtype=np.int32)
    kp, vp, flags = orc.kv_write(k_new, v_new, bt, ctx, scale, v_scale, pool, pool, 8)
    ek = pool.copy()
    # sequence 0: positions 3 (page 3, slot 3), 4 and 5 (page entry 7: out of the pool, skipped)
    # sequence 1: length 9 clamped to 8: positions 5, 6, 7 -> page 0, slots 1, 2, 3
    for b, i, page, slot in [(0, 0, 3, 3), (1, 0, 0, 1), (1, 1, 0, 2), (1, 2, 0, 3)]:
        for h in range(2):
            ek[page, slot, h] = [code(float(x) / scale) for x in k_new[b, i, h]]
    assert flags == 2 | 4, flags
    assert np.array_equal(kp, ek)


def pin_kv_write_fp32_quotient_decides(orc):
    """The byte is decided on the FP32 quotient: where x / scale in FP32 lands exactly on a
    midpoint between two codes while the exact quotient lies above it, the code is the even
    neighbour of the midpoint, not the upper one (found by search over FP32 scales)."""
    codes = np.arange(0x38, 0x40, dtype=np.uint8)  # 1.0 .. 1.875
    vals = torch_decode(codes).numpy()
    found = None
    # pairs whose lower code is even: there the FP32 tie gives the lower code, the exact
    # quotient the upper one
    for lo, hi in zip(vals[0:-1:2], vals[1::2]):
        m = (lo + hi) / 2
        for x in (1.0, 1.5, 3.0, 0.75, 1.25):
            s = np.float32(x / m)
            for cand in (s, np.nextafter(s, np.float32(0)), np.nextafter(s, np.float32(10))):
                q32 = np.float32(np.float32(x) / cand)
                exact = x / float(cand)  # float64: far closer than the FP32 ulp here
                if q32 == np.float32(m) and exact > m:
                    found = (x, cand, lo, hi)
                    break
            if found:
                break
        if found:
            break
    assert found is not None, "no FP32 midpoint case found"
    x, s, lo, hi = found
    k_new = np.full((1, 1, 1, 8), x, dtype=np.float16)
    pool = np.zeros((1, 4, 1, 8), dtype=np.uint8)
    kp, _, flags = orc.kv_write(k_new, k_new, np.array([[0]], np.int32), np.array([1], np.int32),
                                float(s), float(s), pool, pool, 4)
    want = orc.e4m3_encode(np.array([lo]))[0]
    assert want % 2 == 0
    assert flags == 0 and np.all(kp[0, 0, 0] == want), (kp[0, 0, 0], want, found)


PINS = [
    pin_e4m3_spec_points,
    pin_e4m3_all_codes_vs_torch,
    pin_tiny_vs_torch_sdpa,
    pin_uniform_closed_form,
    pin_one_hot_closed_form,
    pin_block_table_permutation,
    pin_page_size_invariance,
    pin_split_merge_agreement,
    pin_split_merge_exact_integers,
    pin_q1_reduction,
    pin_q1_reduction_long_block,
    pin_e4m3_encode_spec_points,
    pin_e4m3_encode_midpoints_ties_to_even,
    pin_e4m3_encode_vs_torch_cast,
    pin_e4m3_encode_saturation_nan_zero,
    pin_kv_write_hand_placed,
    pin_kv_write_clamps,
    pin_kv_write_fp32_quotient_decides,
]
