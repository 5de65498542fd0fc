"""The forward entry point that allocates nothing (its split workspace is a device array built into
the library), for callers that may not call cudaMalloc: a plugin whose device memory belongs to a
host framework's allocator, a runtime that freezes its memory pool after start-up, a loop that
must never enter the allocator.

It is checked through the C ABI against the ordinary forward entry point (caller-owned
workspace) and against the oracle on consecutive calls that share the array: different inputs
and context lengths, every kernel mode, and fused-merge plans of different grid sizes back to
back (the fused merge keeps a grid-barrier counter in the array's header, which every call
clears). So a later call also shows that whatever an earlier one left in the shared array does
not leak into it. This file sorts last so that a run stopping at the first failure has run every
other test.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import MODES, TCGEN05_FUSED, compare, kernel_args, oracle_forward, out_bound
from gpu_helpers import to_device, to_np
from speculative_verify_paged_e4m3_gb300 import workload as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_verify_paged_e4m3_gb300 import binding, build
    build.build()
    return binding


def _close(a_out, a_lse, b_out, b_lse):
    a_out = to_np(a_out).astype(np.float64)
    b_out = to_np(b_out).astype(np.float64)
    assert np.all(np.abs(a_out - b_out) <= out_bound(b_out))
    a_lse, b_lse = to_np(a_lse).astype(np.float64), to_np(b_lse).astype(np.float64)
    assert np.array_equal(np.isneginf(a_lse), np.isneginf(b_lse))
    fin = ~np.isneginf(b_lse)
    assert np.all(np.abs(a_lse[fin] - b_lse[fin]) <= 1e-5 * np.maximum(1.0, np.abs(b_lse[fin])))


# (context length, forced split count; 0: the planner's) of consecutive calls. For the fused
# mode the forced counts give grids of 40, 100 and 152 CTAs in a row on the one shared counter.
CALLS = ((5000, 0), (777, 0), (6000, 40), (3000, 100), (7000, 0))


@pytest.mark.parametrize("mode", MODES)
def test_static_scratch_forward_matches_forward_on_consecutive_calls(B, mode):
    max_ctx = 8192
    grids = set()
    for call, (n, splits) in enumerate(CALLS):
        w = W.Workload(f"noalloc{mode}_{call}", layers=1, context=(n,), seed_base=70000 + call,
                       max_context=max_ctx)
        inp = W.make_layer(w, 0, device="cpu")
        dev = to_device(inp)
        att = B.VerifyAttention(1, 8, 6, 1, 256, 16, w.max_pages_per_seq,
                                dev["k_pool"].shape[0], max_ctx, num_splits=splits,
                                **kernel_args(mode))
        if mode == TCGEN05_FUSED:
            assert att.plan.combine_fused == 1
            grids.add(att.plan.num_splits)
        ref_out, ref_lse = att(dev["q"], dev["k_pool"], dev["v_pool"], dev["block_table"],
                               dev["context_lens"], dev["k_scale"], dev["v_scale"])
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        B.dflash_verify_attn_forward_static_scratch(
            att.plan, dev["q"], dev["k_pool"], dev["v_pool"], dev["block_table"],
            dev["context_lens"], dev["k_scale"], dev["v_scale"], out, lse)
        torch.cuda.synchronize()
        _close(out, lse, ref_out, ref_lse)
        exact_out, exact_lse = oracle_forward(inp)
        compare(to_np(out), to_np(lse), exact_out, exact_lse, what=f"call {call}")
    if mode == TCGEN05_FUSED:
        assert len(grids) >= 3


def test_static_scratch_rejects_plans_above_its_size(B):
    big = B.dflash_verify_attn_plan(B.make_problem(4, 8, 48, 8, 256, 16, 16384, 70000, 262144,
                                                   device=0, num_splits=600))
    assert big.workspace_bytes > 16 << 20
    rc = B.dflash_verify_attn_forward_static_scratch(big, 0, 0, 0, 0, 0, 0, 0, 0, 0,
                                                     check=False)
    assert rc == B.DFLASH_ERR_WORKSPACE_TOO_SMALL
