"""CUDA path against the oracle, element by element, through the C ABI (needs a GPU)."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (MODES, compare, gpu_forward, kernel_args, oracle_forward, to_device,
                         to_np)
from speculative_verify_paged_e4m3_gb300 import workload as W

pytestmark = pytest.mark.gpu

KERNELS = MODES  # CUDA-core; tensor-core + combine kernel; tensor-core fused forward


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_verify_paged_e4m3_gb300 import build
    build.build()


def small(name, context, q_len=8, Hq=6, Hkv=1, P=16, pool_factor=1.5, seed=0, boost=0.0,
          max_context=0):
    return W.Workload(name, layers=1, context=tuple(context), q_len=q_len, num_q_heads=Hq,
                      num_kv_heads=Hkv, page_size=P, pool_factor=pool_factor,
                      boost_frac=boost, boost_factor=4.0, seed_base=90000 + seed,
                      max_context=max_context)


def check(w, kernel, num_splits=0, layer=0):
    inp = W.make_layer(w, layer, device="cpu")
    dev = to_device(inp)
    att, out, lse = gpu_forward(dev, num_splits=num_splits, kernel=kernel)
    ref_out, ref_lse = oracle_forward(inp)
    compare(to_np(out), to_np(lse), ref_out, ref_lse, what=w.name)
    flags = att.workspace_views()[0].item()
    assert flags & 0x4 == 0, "a block-table entry inside the context was out of range?"
    return att, inp, dev, out, lse


@pytest.mark.parametrize("kernel", KERNELS)
def test_config0_full(kernel):
    check(W.config0(), kernel)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("q_len", range(1, 9))
@pytest.mark.parametrize("n", [1, 9, 100, 1031, 4100])
def test_tail_shapes_ragged_contexts(kernel, q_len, n):
    if n < q_len:
        n = q_len
    check(small(f"q{q_len}_n{n}", [n], q_len=q_len, seed=q_len * 7 + n), kernel)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("splits", [1, 2, 3, 7, 64, 500])
def test_forced_split_counts(kernel, splits):
    check(small(f"splits{splits}", [3000], seed=splits), kernel, num_splits=splits)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("tiles", range(1, 8))
@pytest.mark.parametrize("delta", [-1, 0, 1])
def test_single_split_tile_counts(kernel, tiles, delta):
    # one split of 1..7 whole 128-key tiles, one key short of them, or one key over: the copies'
    # start (three K tiles and two V stages at once), the order in which later stages are freed
    # and refilled, and a ragged last V stage, at every tile count where those phases meet
    n = max(8, 128 * tiles + delta)
    check(small(f"tiles{tiles}_{delta}", [n], seed=400 + 3 * tiles + delta), kernel, num_splits=1)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("splits,n,P", [(1, 20000, 16), (2, 33000, 64), (3, 26000, 32)])
def test_splits_longer_than_row_cache(kernel, splits, n, P):
    # more than 512 16-key chunks per split: chunks past the row cache come from the block table
    check(small(f"long{splits}", [n], P=P, seed=300 + splits), kernel, num_splits=splits)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("P,n", [(16, 777), (32, 1000), (48, 999), (64, 2049), (3296, 7000),
                                 (16, 128), (16, 129), (16, 255), (16, 256)])
def test_page_sizes(kernel, P, n):
    check(small(f"P{P}", [n], P=P, seed=P), kernel)


@pytest.mark.parametrize("kernel", KERNELS)
def test_whole_model_heads_ragged_batch(kernel):
    # Hq 24 / Hkv 4 (the four-way shard un-sharded): four KV-head units per sequence
    check(small("b2_hkv4", [1300, 700], Hq=24, Hkv=4, seed=41), kernel)


@pytest.mark.parametrize("kernel", KERNELS)
def test_batch_ragged_two_kv_heads(kernel):
    check(small("b3_hkv2", [1500, 17, 640], Hq=12, Hkv=2, seed=3), kernel)


@pytest.mark.parametrize("kernel", KERNELS + [0])
@pytest.mark.parametrize("q_len,Hq,Hkv,ctx", [
    (9, 6, 1, [1031]),          # 54 rows: two blocks of 27
    (10, 6, 1, [300]),          # one split per block pair, ragged tail tile
    (16, 6, 1, [4100]),         # 96 rows: two full blocks of 48 (CUDA-core: 48 as well)
    (8, 8, 1, [900]),           # 64 rows
    (16, 16, 1, [2000]),        # 256 rows, the most a plan takes
    (11, 6, 1, [11]),           # context exactly q_len
    (16, 12, 2, [1500, 17, 640]),  # ragged batch, two KV heads, 96 rows each
])
def test_row_blocks(kernel, q_len, Hq, Hkv, ctx):
    # more rows per KV head than one CTA carries: each split's rows are dealt to row blocks
    att, *_ = check(small(f"q{q_len}_g{Hq // Hkv}", ctx, q_len=q_len, Hq=Hq, Hkv=Hkv,
                          seed=q_len * 13 + Hq), kernel)
    R = q_len * Hq // Hkv
    cap = 64 if att.plan.kernel == 1 else 48
    assert att.plan.rows == R and att.plan.row_blocks == math.ceil(R / cap)
    if kernel == 0:
        assert att.plan.kernel == 2  # the tensor-core kernel whenever a block fits it


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("splits", [1, 3, 40])
def test_row_blocks_forced_splits(kernel, splits):
    check(small(f"q16_splits{splits}", [3000], q_len=16, seed=200 + splits), kernel,
          num_splits=splits)


@pytest.mark.parametrize("kernel", KERNELS)
def test_peaked_softmax(kernel):
    check(small("boost", [5000], P=64, seed=11, boost=0.05), kernel)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("q_len", [8, 16])
def test_workspace_state_matches_oracle_partials(kernel, q_len):
    w = small("partials", [2500], q_len=q_len, seed=21)
    att, inp, dev, out, lse = check(w, kernel, num_splits=5)
    from speculative_verify_paged_e4m3_gb300 import binding as B
    starts, active = B.dflash_verify_attn_split_bounds(att.plan, 2500)
    sb = np.array([starts], dtype=np.int32)
    m, l, acc = oracle.load().verify_attn_partials(
        to_np(inp["q"]), to_np(inp["k_pool"]), to_np(inp["v_pool"]), to_np(inp["block_table"]),
        to_np(inp["context_lens"]), inp["k_scale"].item(), inp["v_scale"].item(), sb)
    _, state, gacc = att.workspace_views()
    state = to_np(state).astype(np.float64)
    gacc = to_np(gacc).astype(np.float64)
    gm = state[..., 0] / math.log2(math.e)  # kernel keeps m in log2 units
    gl = state[..., 1]
    for s in range(active):
        for r in range(att.plan.rows):
            om, ol, oa = m[0, 0, s, r], l[0, 0, s, r], acc[0, 0, s, r]
            if om == -np.inf:
                assert gm[s, r] == -np.inf and gl[s, r] == 0
                continue
            # the state is defined up to its reference max: compare l * e^m, and the split's
            # own normalised output acc / l with the output tolerance
            scale = math.exp(gm[s, r] - om)
            assert abs(gl[s, r] * scale - ol) <= 1e-4 * ol, (s, r)
            np.testing.assert_allclose(gacc[s, r] / gl[s, r], oa / ol, rtol=0,
                                       atol=2e-3, err_msg=f"split {s} row {r}")


@pytest.mark.parametrize("kernel", KERNELS)
def test_context_shorter_than_q_len_and_empty(kernel):
    from speculative_verify_paged_e4m3_gb300 import binding as B
    w = small("short", [3, 0, 40], q_len=8, seed=31)
    inp = W.make_layer(w, 0, device="cpu")
    att, out, lse = gpu_forward(to_device(inp), kernel=kernel)
    ref_out, ref_lse = oracle_forward(inp)
    compare(to_np(out), to_np(lse), ref_out, ref_lse, what="short")
    assert np.all(np.isneginf(to_np(lse)[1]))
    assert np.all(to_np(out)[1] == 0)
    assert att.workspace_views()[0].item() & B.DFLASH_FLAG_CONTEXT_SHORT


@pytest.mark.parametrize("kernel", KERNELS)
def test_context_above_plan_is_clamped(kernel):
    from speculative_verify_paged_e4m3_gb300 import binding as B
    w = small("clamp", [1200], seed=41)
    inp = W.make_layer(w, 0, device="cpu")
    att, out, lse = gpu_forward(to_device(inp), kernel=kernel, max_context=1000)
    ref_out, ref_lse = oracle_forward(inp, context_override=[1000])
    compare(to_np(out), to_np(lse), ref_out, ref_lse, what="clamp")
    assert att.workspace_views()[0].item() & B.DFLASH_FLAG_CONTEXT_CLAMPED


@pytest.mark.parametrize("kernel", KERNELS)
def test_out_of_range_page_is_clamped_and_flagged(kernel):
    from speculative_verify_paged_e4m3_gb300 import binding as B
    w = small("badpage", [500], seed=51, pool_factor=1.0)
    inp = W.make_layer(w, 0, device="cpu")
    num_pages = inp["k_pool"].shape[0]
    inp["block_table"][0, 3] = num_pages + 100  # clamps to the last page
    inp["block_table"][0, 5] = -4               # clamps to page 0
    att, out, lse = gpu_forward(to_device(inp), kernel=kernel)
    fixed = dict(inp)
    fixed["block_table"] = inp["block_table"].clone()
    fixed["block_table"][0, 3] = num_pages - 1
    fixed["block_table"][0, 5] = 0
    ref_out, ref_lse = oracle_forward(fixed)
    compare(to_np(out), to_np(lse), ref_out, ref_lse, what="badpage")
    assert att.workspace_views()[0].item() & B.DFLASH_FLAG_PAGE_CLAMPED
    assert B.dflash_verify_attn_read_flags(att.workspace, clear=True) & 0x4
    assert B.dflash_verify_attn_read_flags(att.workspace) == 0


@pytest.mark.parametrize("kernel", KERNELS)
def test_deterministic_and_canaries_intact(kernel):
    from speculative_verify_paged_e4m3_gb300 import binding as B
    w = small("canary", [3333], seed=61)
    dev = to_device(W.make_layer(w, 0, device="cpu"))
    Bq, q_len, Hq, D = dev["q"].shape
    guard = 4096
    att = B.VerifyAttention(Bq, q_len, Hq, 1, D, 16, dev["block_table"].shape[1],
                            dev["k_pool"].shape[0], 3333, **kernel_args(kernel))
    ws_bytes = att.plan.workspace_bytes
    big_ws = torch.full((ws_bytes + 2 * guard,), 0xA5, dtype=torch.uint8, device="cuda")
    big_ws[guard:guard + 16].zero_()  # status word and grid-barrier words of the header
    att.workspace = big_ws[guard:guard + ws_bytes]
    n_out = Bq * q_len * Hq * D
    out_buf = torch.full((n_out + 2 * guard,), 7.0, dtype=torch.float16, device="cuda")
    lse_buf = torch.full((Bq * q_len * Hq + 2 * guard,), 7.0, dtype=torch.float32, device="cuda")
    outs = []
    for _ in range(2):
        out = out_buf[guard:guard + n_out].view(Bq, q_len, Hq, D)
        lse = lse_buf[guard:guard + Bq * q_len * Hq].view(Bq, q_len, Hq)
        att(dev["q"], dev["k_pool"], dev["v_pool"], dev["block_table"], dev["context_lens"],
            dev["k_scale"], dev["v_scale"], out=out, lse=lse)
        torch.cuda.synchronize()
        outs.append((out.clone(), lse.clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    for buf, val in ((out_buf, 7.0), (lse_buf, 7.0)):
        assert torch.all(buf[:guard] == val) and torch.all(buf[-guard:] == val)
    assert torch.all(big_ws[:guard] == 0xA5) and torch.all(big_ws[-guard:] == 0xA5)


def test_debug_dequant_bit_exact():
    from speculative_verify_paged_e4m3_gb300 import binding as B
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8).repeat(3).cuda()
    for sc in (1.0, 0.0123, 3.7e-3, 448.0 / 7.0):
        scale = torch.tensor([sc], dtype=torch.float32, device="cuda")
        dec = torch.empty(codes.shape, dtype=torch.float32, device="cuda")
        scd = torch.empty_like(dec)
        B.dflash_verify_attn_debug_dequant(codes, scale, dec, scd)
        torch.cuda.synchronize()
        ref = oracle.load().e4m3_decode(to_np(codes))
        g = to_np(dec).astype(np.float64)
        nan = np.isnan(ref)
        assert np.array_equal(np.isnan(g), nan)
        assert np.array_equal(g[~nan], ref[~nan])
        assert np.array_equal(np.signbit(g[~nan]), np.signbit(ref[~nan]))
        sc32 = np.float64(np.float32(sc))
        ref_scaled = (ref[~nan] * sc32).astype(np.float32)  # exact product, one rounding
        assert np.array_equal(to_np(scd)[~nan].view(np.uint32), ref_scaled.view(np.uint32))


@pytest.mark.parametrize("q_len", [8, 16])
def test_fused_and_separate_combine_agree_bitwise(q_len):
    """The fused forward runs the same merge arithmetic as the combine kernel: same bits."""
    from speculative_verify_paged_e4m3_gb300 import binding as B
    w = small("fused_vs_sep", [5000], q_len=q_len, seed=71)
    dev = to_device(W.make_layer(w, 0, device="cpu"))
    res = []
    for flags in (B.DFLASH_PROBLEM_FUSED_COMBINE, 0):
        att = B.VerifyAttention(1, q_len, 6, 1, 256, 16, dev["block_table"].shape[1],
                                dev["k_pool"].shape[0], 5000, num_splits=9,
                                kernel=B.DFLASH_KERNEL_TCGEN05, flags=flags)
        assert att.plan.combine_fused == (1 if flags else 0)
        out, lse = att(dev["q"], dev["k_pool"], dev["v_pool"], dev["block_table"],
                       dev["context_lens"], dev["k_scale"], dev["v_scale"])
        torch.cuda.synchronize()
        res.append((out.clone(), lse.clone()))
    assert torch.equal(res[0][0], res[1][0]) and torch.equal(res[0][1], res[1][1])


def test_fused_barrier_reused_across_grid_sizes():
    """One workspace, fused plans of different grid sizes back to back: the grid barrier resets
    itself, every result matches the oracle and no timeout is flagged."""
    from speculative_verify_paged_e4m3_gb300 import binding as B
    w = small("fused_reuse", [2600, 700], seed=81)
    inp = W.make_layer(w, 0, device="cpu")
    dev = to_device(inp)
    ref_out, ref_lse = oracle_forward(inp)
    ws = None
    for splits in (0, 37, 5, 76, 1, 0):
        att = B.VerifyAttention(2, 8, 6, 1, 256, 16, dev["block_table"].shape[1],
                                dev["k_pool"].shape[0], 2600, num_splits=splits,
                                kernel=B.DFLASH_KERNEL_TCGEN05,
                                flags=B.DFLASH_PROBLEM_FUSED_COMBINE)
        assert att.plan.combine_fused == 1
        if ws is None or ws.numel() < att.plan.workspace_bytes:
            big = torch.zeros(1 << 24, dtype=torch.uint8, device="cuda")
            ws = big
        att.workspace = ws
        out, lse = att(dev["q"], dev["k_pool"], dev["v_pool"], dev["block_table"],
                       dev["context_lens"], dev["k_scale"], dev["v_scale"])
        torch.cuda.synchronize()
        compare(to_np(out), to_np(lse), ref_out, ref_lse, what=f"fused splits={splits}")
        assert att.workspace_views()[0].item() == 0


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("batch", [33, 70])
def test_batch_beyond_one_warp_of_sequences(kernel, batch):
    # more sequences than a warp's lanes: the slot search runs over several 32-sequence chunks
    rng = np.random.default_rng(batch)
    lens = [int(x) for x in rng.integers(0, 700, size=batch)]
    lens[0], lens[batch // 2], lens[-1] = 0, 900, 17
    lens = [max(n, 8) if n else 0 for n in lens]  # a length below q_len is covered elsewhere
    att, *_ = check(small(f"b{batch}", lens, seed=batch), kernel)
    from speculative_verify_paged_e4m3_gb300 import binding as B
    start, per, act = B.dflash_verify_attn_split_slots(att.plan, lens)
    assert start[-1] <= att.plan.num_slots and sum(1 for a in act if a) == sum(1 for n in lens if n)


@pytest.mark.parametrize("lens,Hkv", [
    ([3000, 700, 0, 1600], 2),
    ([(37 * i) % 1500 for i in range(70)], 1),  # several 32-sequence chunks, some empty
])
def test_ragged_batch_slots_match_host_layout(lens, Hkv):
    """A ragged batch (some sequences empty): the partial kernel writes state into exactly the
    slots the host-side layout (dflash_verify_attn_split_slots) lists, and nothing else."""
    from speculative_verify_paged_e4m3_gb300 import binding as B
    w = small("slots", lens, Hq=6 * Hkv, Hkv=Hkv, seed=51)
    inp = W.make_layer(w, 0, device="cpu")
    dev = to_device(inp)
    q = dev["q"]
    att = B.VerifyAttention(q.shape[0], q.shape[1], q.shape[2], Hkv, 256, 16,
                            dev["block_table"].shape[1], dev["k_pool"].shape[0], w.max_ctx,
                            device=0)
    _, state, _ = att.workspace_views()
    state.fill_(float("nan"))
    B.dflash_verify_attn_run(att.plan, dev["q"], dev["k_pool"], dev["v_pool"],
                             dev["block_table"], dev["context_lens"], dev["k_scale"],
                             dev["v_scale"], att.workspace)
    torch.cuda.synchronize()
    start, per, act = B.dflash_verify_attn_split_slots(att.plan, w.context)
    written = ~torch.isnan(state[..., 1]).reshape(-1, att.plan.rows).all(dim=1).cpu().numpy()
    want = np.zeros(written.shape, dtype=bool)
    for u in range(len(act)):
        want[start[u]:start[u] + act[u]] = True
    assert np.array_equal(written, want), (np.nonzero(written != want), start, act)
