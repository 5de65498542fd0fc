"""The C ABI without a GPU: symbols, struct layout, planner results and error statuses."""
import ctypes
import math
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def B():
    from speculative_verify_paged_e4m3_gb300 import binding, build
    build.build()
    return binding


def declared_functions():
    names = set()
    for f in os.listdir(HEADER_DIR):
        if f.endswith(".h"):
            text = open(os.path.join(HEADER_DIR, f)).read()
            names |= set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(dflash_\w+)\s*\(", text,
                                    re.M))
    return sorted(names)


def test_every_declared_symbol_is_exported(B):
    names = declared_functions()
    assert len(names) >= 8
    lib = B.load_library()
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert set(B.EXPORTED) <= set(names)


def test_struct_layout_matches_c(B, tmp_path):
    prog = tmp_path / "sizes.c"
    prog.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "dflash_verify_attn.h"\n'
        "int main(void){printf(\"%zu %zu %zu %zu %zu\\n\", sizeof(dflash_verify_attn_problem),"
        " sizeof(dflash_verify_attn_plan_t), offsetof(dflash_verify_attn_plan_t, workspace_bytes),"
        " offsetof(dflash_verify_attn_plan_t, ws_acc_offset),"
        " offsetof(dflash_verify_attn_plan_t, problem)); return 0;}\n")
    exe = tmp_path / "sizes"
    subprocess.run(["gcc", "-I", HEADER_DIR, str(prog), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    assert got == [ctypes.sizeof(B.Problem), ctypes.sizeof(B.Plan),
                   B.Plan.workspace_bytes.offset, B.Plan.ws_acc_offset.offset,
                   B.Plan.problem.offset]


def problem(B, **kw):
    args = dict(batch=1, q_len=8, num_q_heads=6, num_kv_heads=1, head_dim=256, page_size=16,
                max_pages_per_seq=16384, num_pages=16384, max_context=262144, device=-1)
    args.update(kw)
    return B.make_problem(**args)


def test_plan_q8_capacity(B):
    plan = B.dflash_verify_attn_plan(problem(B))
    assert plan.rows == 48 and plan.num_splits >= 1
    assert plan.kernel == B.DFLASH_KERNEL_TCGEN05 and plan.tile_keys == 128
    assert plan.sm_count == 152
    assert plan.workspace_bytes >= plan.ws_acc_offset + plan.num_splits * 48 * 256 * 4
    assert plan.ws_state_offset % 256 == 0 and plan.ws_acc_offset % 256 == 0
    assert plan.ws_acc_offset >= plan.ws_state_offset + plan.num_splits * 48 * 8


@pytest.mark.parametrize("kw,status", [
    (dict(version=1), -1),
    (dict(batch=0), -1),
    (dict(q_len=0), -1),
    (dict(num_q_heads=5, num_kv_heads=2), -1),
    (dict(max_pages_per_seq=10), -1),
    (dict(max_context=0), -1),
    (dict(num_splits=-1), -1),
    (dict(kernel=7), -1),
    (dict(head_dim=128), -2),
    (dict(page_size=24, max_pages_per_seq=20000), -2),
    (dict(q_len=33, num_q_heads=8), -2),  # 264 rows per KV head: above 256
])
def test_plan_errors(B, kw, status):
    pr = problem(B, **{k: v for k, v in kw.items() if k != "version"})
    if "version" in kw:
        pr.version = kw["version"]
    assert B.dflash_verify_attn_plan_status(pr) == status


@pytest.mark.parametrize("q_len,hq,kernel,blocks,block_rows,threads_of", [
    (8, 6, 0, 1, 48, 48),     # the pages' shape: one CTA per split
    (9, 6, 0, 2, 27, 32),     # 54 rows: two blocks of 27 on the 32-row instance
    (10, 6, 0, 2, 30, 32),
    (16, 6, 0, 2, 48, 48),    # 96 rows
    (16, 16, 0, 6, 43, 48),   # 256 rows, the most a plan takes
    (8, 8, 2, 2, 32, 32),     # 64 rows forced onto the tensor-core kernel
    (16, 6, 1, 2, 48, None),  # CUDA-core kernel: 64 rows per block
    (8, 8, 1, 1, 64, None),
])
def test_plan_row_blocks(B, q_len, hq, kernel, blocks, block_rows, threads_of):
    plan = B.dflash_verify_attn_plan(problem(B, q_len=q_len, num_q_heads=hq, kernel=kernel))
    R = q_len * hq
    assert plan.rows == R and plan.row_blocks == blocks
    assert math.ceil(R / blocks) == block_rows and (blocks - 1) * block_rows < R
    if threads_of is not None:
        assert plan.kernel == B.DFLASH_KERNEL_TCGEN05
        ref = B.dflash_verify_attn_plan(problem(B, q_len=1, num_q_heads=threads_of))
        assert plan.threads == ref.threads and plan.smem_bytes == ref.smem_bytes
    else:
        assert plan.kernel == B.DFLASH_KERNEL_SIMT
    # one wave: every (split, row block) CTA of the single sequence and KV head fits the SMs
    cap = math.ceil(262144 / plan.min_split_keys)
    assert plan.num_splits == min(152 // blocks, cap)
    # the workspace holds every row of every slot, however the rows are blocked
    assert plan.workspace_bytes >= plan.ws_acc_offset + plan.num_splits * R * 256 * 4
    assert plan.ws_acc_offset >= plan.ws_state_offset + plan.num_splits * R * 8


def test_plan_row_blocks_fused(B):
    pr = problem(B, q_len=16, batch=4)
    pr.flags = B.DFLASH_PROBLEM_FUSED_COMBINE
    plan = B.dflash_verify_attn_plan(pr)
    assert plan.combine_fused == 1 and plan.row_blocks == 2
    assert 4 * plan.row_blocks * plan.num_splits <= 152


@pytest.mark.parametrize("batch,slots", [(1, 151), (1, 0), (4, 15), (4, 0)])
def test_plan_num_slots_tampered(B, batch, slots):
    # a single sequence's slots are Hkv * num_splits; a batch needs one per unit at least
    plan = B.dflash_verify_attn_plan(problem(B, batch=batch, num_q_heads=24, num_kv_heads=4))
    plan.num_slots = slots
    with pytest.raises(B.DflashError) as e:
        B.dflash_verify_attn_split_slots(plan, [1000] * batch)
    assert e.value.status == B.DFLASH_ERR_INVALID_ARGUMENT


@pytest.mark.parametrize("row_blocks", [0, -1, 1, 97])
def test_plan_row_blocks_tampered(B, row_blocks):
    # a plan whose row blocks do not cover R in blocks the kernel can hold is refused
    plan = B.dflash_verify_attn_plan(problem(B, q_len=16))
    plan.row_blocks = row_blocks
    lens = [262144]
    with pytest.raises(B.DflashError) as e:
        B.dflash_verify_attn_split_slots(plan, lens)
    assert e.value.status == B.DFLASH_ERR_INVALID_ARGUMENT


@pytest.mark.parametrize("kernel,tile,min_keys", [
    ("tc", 64, 256), ("tc", 256, 256), ("tc", 128, 200), ("simt", 128, 256), ("simt", 32, 48)])
def test_plan_tile_keys_tampered(B, kernel, tile, min_keys):
    # the kernels' tiles are compile-time constants (128 keys tensor-core, 32 CUDA-core): a plan
    # that says otherwise, or whose minimum split is not whole tiles, is refused
    kw = {} if kernel == "tc" else {"kernel": B.DFLASH_KERNEL_SIMT}
    plan = B.dflash_verify_attn_plan(problem(B, **kw))
    plan.tile_keys, plan.min_split_keys = tile, min_keys
    with pytest.raises(B.DflashError) as e:
        B.dflash_verify_attn_split_slots(plan, [1000])
    assert e.value.status == B.DFLASH_ERR_INVALID_ARGUMENT


@pytest.mark.parametrize("batch,hkv,q_len,splits,fused,slots", [
    (1, 1, 8, 0, False, 152),      # one sequence: Hkv * num_splits
    (1, 4, 8, 0, False, 152),
    (4, 4, 8, 0, False, 152),      # a batch: every SM (16 * 9 = 144 would leave 8 idle)
    (8, 4, 8, 0, False, 152),      # 32 * 4 = 128 would leave 24 idle
    (4, 4, 16, 0, False, 76),      # two row blocks: 76 slots x 2 CTAs
    (4, 4, 8, 0, True, 152),       # fused: still one CTA per SM
    (4, 4, 8, 5, False, 80),       # forced split count: units * S
    (200, 1, 8, 0, False, 200),    # more units than SMs: one slot each
])
def test_plan_num_slots(B, batch, hkv, q_len, splits, fused, slots):
    pr = problem(B, batch=batch, num_q_heads=6 * hkv, num_kv_heads=hkv, q_len=q_len,
                 num_splits=splits)
    if fused:
        pr.flags = B.DFLASH_PROBLEM_FUSED_COMBINE
    plan = B.dflash_verify_attn_plan(pr)
    assert plan.num_slots == slots
    assert plan.num_slots * plan.row_blocks <= max(152, batch * hkv * plan.row_blocks)
    R = plan.rows
    assert plan.workspace_bytes >= plan.ws_acc_offset + slots * R * 256 * 4
    assert plan.ws_acc_offset >= plan.ws_state_offset + slots * R * 8
    if batch == 1:
        assert slots == hkv * plan.num_splits


@pytest.mark.parametrize("n", [0, 1, 7, 8, 100, 1024, 32768, 131072, 261888, 262144, 300000])
def test_split_bounds_rule(B, n):
    plan = B.dflash_verify_attn_plan(problem(B))
    starts, active = B.dflash_verify_attn_split_bounds(plan, n)
    S = plan.num_splits
    nn = min(max(n, 0), 262144)
    assert len(starts) == S + 1 and starts[0] == 0 and starts[-1] == nn
    assert all(a <= b for a, b in zip(starts, starts[1:]))
    per = max(math.ceil(nn / S), plan.min_split_keys)
    per = math.ceil(per / plan.tile_keys) * plan.tile_keys
    assert active == (math.ceil(nn / per) if nn else 0)
    for s in range(S):
        assert starts[s] == min(nn, s * per)
        if s < active:
            assert starts[s + 1] > starts[s] and starts[s] % plan.tile_keys == 0
        else:
            assert starts[s + 1] == starts[s] == nn


def test_forced_split_count(B):
    plan = B.dflash_verify_attn_plan(problem(B, num_splits=300))
    assert plan.num_splits == 300
    starts, active = B.dflash_verify_attn_split_bounds(plan, 261888)
    assert active <= 300 and starts[active] == 261888


def test_run_rejects_bad_arguments_without_launching(B):
    plan = B.dflash_verify_attn_plan(problem(B))
    lib = B.load_library()
    # null pointers
    rc = lib.dflash_verify_attn_run(ctypes.byref(plan), None, None, None, None, None, None, None,
                                    None, 0, None)
    assert rc == B.DFLASH_ERR_INVALID_ARGUMENT
    # misaligned q (no device memory is touched: arguments are checked first)
    fake = 4096
    rc = lib.dflash_verify_attn_run(ctypes.byref(plan), fake + 2, fake, fake, fake, fake, fake,
                                    fake, fake, plan.workspace_bytes, None)
    assert rc == B.DFLASH_ERR_INVALID_ARGUMENT
    # workspace too small
    rc = lib.dflash_verify_attn_run(ctypes.byref(plan), fake, fake, fake, fake, fake, fake,
                                    fake, fake, plan.workspace_bytes - 1, None)
    assert rc == B.DFLASH_ERR_WORKSPACE_TOO_SMALL
    rc = lib.dflash_verify_attn_combine(ctypes.byref(plan), fake, plan.workspace_bytes - 1,
                                        fake, fake, fake, None)
    assert rc == B.DFLASH_ERR_WORKSPACE_TOO_SMALL
    bad = B.Plan()
    rc = lib.dflash_verify_attn_combine(ctypes.byref(bad), fake, 1 << 30, fake, fake, fake, None)
    assert rc == B.DFLASH_ERR_INVALID_ARGUMENT
    rc = lib.dflash_verify_attn_debug_dequant(None, -1, None, None, None, None)
    assert rc == B.DFLASH_ERR_INVALID_ARGUMENT


def test_status_strings(B):
    for s in (0, -1, -2, -3, -4):
        assert B.status_string(s)
    assert B.status_string(12345) == "unknown status"


def test_fused_combine_planning(B):
    """On request the tensor-core plan merges the splits in its own launch, when the whole grid
    fits on the GPU at once (one CTA per SM), and not otherwise; the default is two kernels."""
    F = B.DFLASH_PROBLEM_FUSED_COMBINE
    assert B.dflash_verify_attn_plan(problem(B)).combine_fused == 0
    plan = B.dflash_verify_attn_plan(problem(B, flags=F))
    assert plan.combine_fused == 1
    assert plan.num_splits * plan.problem.batch * plan.problem.num_kv_heads <= plan.sm_count
    simt = B.dflash_verify_attn_plan(problem(B, kernel=B.DFLASH_KERNEL_SIMT, flags=F))
    assert simt.combine_fused == 0
    forced = B.dflash_verify_attn_plan(problem(B, num_splits=300, flags=F))
    assert forced.combine_fused == 0
    forced_small = B.dflash_verify_attn_plan(problem(B, num_splits=100, flags=F))
    assert forced_small.combine_fused == 1 and forced_small.num_splits == 100
    many = B.dflash_verify_attn_plan(problem(B, batch=153, max_pages_per_seq=16, num_pages=4096,
                                             max_context=256, flags=F))
    assert many.combine_fused == 0
    # batch x KV heads units share the SMs: floor(152 / 3) splits each
    three = B.dflash_verify_attn_plan(problem(B, batch=3, flags=F))
    assert three.combine_fused == 1 and three.num_splits == 152 // 3


def test_fused_forward_rejects_bad_arguments_without_launching(B):
    plan = B.dflash_verify_attn_plan(problem(B, flags=B.DFLASH_PROBLEM_FUSED_COMBINE))
    assert plan.combine_fused == 1
    lib = B.load_library()
    fake = ctypes.c_void_p(1 << 20)
    args = [fake] * 8
    rc = lib.dflash_verify_attn_forward(ctypes.byref(plan), *args, ctypes.c_size_t(plan.workspace_bytes),
                                        None, fake, None)
    assert rc == B.DFLASH_ERR_INVALID_ARGUMENT  # no output
    rc = lib.dflash_verify_attn_forward(ctypes.byref(plan), *args,
                                        ctypes.c_size_t(plan.workspace_bytes - 1), fake, fake, None)
    assert rc == B.DFLASH_ERR_WORKSPACE_TOO_SMALL


def test_kv_write_rejects_bad_arguments_without_launching(B):
    plan = B.dflash_verify_attn_plan(problem(B))
    lib = B.load_library()
    fake = 4096
    ws = ctypes.c_size_t(plan.workspace_bytes)
    rc = lib.dflash_verify_attn_kv_write(ctypes.byref(plan), None, None, None, None, None, None,
                                         None, None, None, ctypes.c_size_t(0), None)
    assert rc == B.DFLASH_ERR_INVALID_ARGUMENT
    # k_new must allow FP16 pairs (4-byte aligned); no device memory is touched before this check
    rc = lib.dflash_verify_attn_kv_write(ctypes.byref(plan), fake + 2, fake, fake, fake, fake,
                                         fake, fake, fake, fake, ws, None)
    assert rc == B.DFLASH_ERR_INVALID_ARGUMENT
    rc = lib.dflash_verify_attn_kv_write(ctypes.byref(plan), fake, fake, fake, fake, fake, fake,
                                         fake, fake, fake, ctypes.c_size_t(plan.workspace_bytes - 1),
                                         None)
    assert rc == B.DFLASH_ERR_WORKSPACE_TOO_SMALL
    rc = lib.dflash_verify_attn_kv_write(ctypes.byref(B.Plan()), fake, fake, fake, fake, fake,
                                         fake, fake, fake, fake, ws, None)
    assert rc == B.DFLASH_ERR_INVALID_ARGUMENT


def test_default_split_count_fills_one_wave(B):
    """One CTA per SM: the default plan keeps batch x KV heads x splits within the SM count (a CTA
    past it would run in a second wave), and uses as many splits as fit."""
    for batch, hkv in [(1, 1), (3, 1), (1, 4), (4, 4), (5, 7), (200, 1)]:
        plan = B.dflash_verify_attn_plan(problem(B, batch=batch, num_q_heads=6 * hkv,
                                                 num_kv_heads=hkv))
        units = batch * hkv
        if units <= plan.sm_count:
            assert units * plan.num_splits <= plan.sm_count
            assert units * (plan.num_splits + 1) > plan.sm_count
        else:
            assert plan.num_splits == 1


def test_split_slots_layout(B):
    """Slots go to (sequence, KV head) units so that the busiest split is as short as possible:
    equal lengths here give num_splits slots each (the [batch, Hkv, S] layout), every non-empty
    unit gets at least one, an empty unit none, and they fit in the plan's num_slots."""
    plan = B.dflash_verify_attn_plan(problem(B, batch=4, num_q_heads=24, num_kv_heads=4,
                                             max_pages_per_seq=4096, num_pages=20000,
                                             max_context=65536))
    S, units = plan.num_splits, 16
    start, per, act = B.dflash_verify_attn_split_slots(plan, [65536] * 4)
    assert start == [u * S for u in range(units + 1)]
    ref_starts, ref_active = B.dflash_verify_attn_split_bounds(plan, 65536)
    assert all(a == ref_active for a in act) and all(p == ref_starts[1] for p in per)
    lens = [65536, 57344, 0, 40960]
    start, per, act = B.dflash_verify_attn_split_slots(plan, lens)
    cnt = [start[u + 1] - start[u] for u in range(units)]
    assert start[0] == 0 and start[-1] <= plan.num_slots and all(c >= 0 for c in cnt)
    for u in range(units):
        n = lens[u // 4]
        assert (cnt[u] == 0) == (n == 0) and (act[u] == 0) == (n == 0)
        if n:
            assert act[u] <= cnt[u] and per[u] * act[u] >= n > per[u] * (act[u] - 1)
    share = [cnt[u] / plan.num_slots for u in range(units)]
    total = 4 * sum(lens)
    for u in range(units):
        if lens[u // 4]:
            assert abs(share[u] - lens[u // 4] / total) * plan.num_slots <= 1.5
    # the longest split is no longer than about the average
    tiles = [math.ceil(p / 128) for p, a in zip(per, act) if a]
    assert max(tiles) <= math.ceil(sum(math.ceil(n / 128) for n in lens) * 4 / plan.num_slots) + 2


@pytest.mark.parametrize("lens", [
    [65536, 57344, 49152, 40960],      # the ragged whole-model-heads workload
    [262144, 1000, 300000, 77, 0, 5000, 131072, 4096],
    [128] * 3 + [262144],
    [1, 2, 3],
])
def test_split_slots_min_max_rule(B, lens):
    """The busiest slot holds the fewest tiles any split into contiguous, equal pieces per unit
    can give: brute force over T against the host rule."""
    Hkv = 4
    plan = B.dflash_verify_attn_plan(problem(B, batch=len(lens), num_q_heads=24, num_kv_heads=Hkv,
                                             max_pages_per_seq=16384, num_pages=20000))
    C = plan.num_slots
    w = [math.ceil(min(max(n, 0), 262144) / 128) for n in lens]
    T = next(t for t in range(1, max(w) + 1)
             if Hkv * sum(math.ceil(x / t) for x in w) <= C)
    start, per, act = B.dflash_verify_attn_split_slots(plan, lens)
    cnt = [start[u + 1] - start[u] for u in range(len(lens) * Hkv)]
    assert cnt == [math.ceil(x / T) for x in w for _ in range(Hkv)]
    assert start[-1] <= C
    tiles = [math.ceil(p / 128) for p, a in zip(per, act) if a]
    assert max(tiles) <= max(T, plan.min_split_keys // 128)
