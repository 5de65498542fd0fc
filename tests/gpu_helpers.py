"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI, run the oracle on
the same inputs, and compare with the stated tolerances.

Tolerances (the acceptance bar for this operator, read as below):
  * out: |gpu - exact| <= max(2e-3, half an FP16 ulp of the exact value). The 2e-3 is the
    bound on FP16 outputs; only where the output format's own rounding exceeds it (|out| >= 8,
    where half an ulp is 2^-8 or more) does the bound become that half ulp, so that a correctly
    computed value rounded to FP16 is never called wrong.
  * lse: |gpu - exact| <= 1e-5 * max(1, |exact|); -inf must match exactly.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

OUT_ATOL = 2e-3
LSE_RTOL = 1e-5


def to_np(t):
    return t.detach().cpu().numpy()


def oracle_forward(inputs, context_override=None):
    orc = oracle.load()
    cl = to_np(inputs["context_lens"]) if context_override is None else np.asarray(
        context_override, dtype=np.int32)
    return orc.verify_attn(to_np(inputs["q"]), to_np(inputs["k_pool"]), to_np(inputs["v_pool"]),
                           to_np(inputs["block_table"]), cl, float(inputs["k_scale"].item()),
                           float(inputs["v_scale"].item()))


def fp16_half_ulp(x):
    a = np.abs(x).astype(np.float16)
    return 0.5 * np.spacing(a).astype(np.float64)


def out_bound(exact):
    """Largest accepted |gpu - exact| of each FP16 output element."""
    return np.maximum(OUT_ATOL, fp16_half_ulp(exact))


def compare(out_gpu, lse_gpu, out_ref, lse_ref, what=""):
    """Assert the tolerances; returns (max out error, max lse relative error)."""
    out_gpu = np.asarray(out_gpu, dtype=np.float64)
    lse_gpu = np.asarray(lse_gpu, dtype=np.float64)
    assert np.all(np.isfinite(out_gpu)), f"{what}: non-finite output"
    err = np.abs(out_gpu - out_ref)
    bound = out_bound(out_ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} outputs beyond tolerance, max err "
                           f"{err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}")
    inf_ref = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse_gpu), inf_ref), f"{what}: -inf lse mismatch"
    fin = ~inf_ref
    lerr = np.abs(lse_gpu[fin] - lse_ref[fin]) / np.maximum(1.0, np.abs(lse_ref[fin]))
    assert lerr.size == 0 or lerr.max() <= LSE_RTOL, f"{what}: lse rel err {lerr.max():.3e}"
    return float(err.max()) if err.size else 0.0, float(lerr.max()) if lerr.size else 0.0


def to_device(inputs, device="cuda"):
    return {k: v.to(device) for k, v in inputs.items()}


# Kernel modes of the parity tests: the CUDA-core kernel, the tensor-core kernel with the combine
# kernel (the default forward), and the tensor-core kernel with the splits merged inside the same
# cooperative launch.
SIMT, TCGEN05, TCGEN05_FUSED = 1, 2, 3
MODES = [SIMT, TCGEN05, TCGEN05_FUSED]


def kernel_args(mode):
    """VerifyAttention keyword arguments of a test mode."""
    from speculative_verify_paged_e4m3_gb300 import binding as B
    if mode == TCGEN05_FUSED:
        return dict(kernel=B.DFLASH_KERNEL_TCGEN05, flags=B.DFLASH_PROBLEM_FUSED_COMBINE)
    return dict(kernel=mode, flags=0)


def gpu_forward(inputs, num_splits=0, kernel=0, max_context=None, num_pages=None):
    """Plan for the inputs' shape and run partial + combine on the current stream (kernel: a
    test mode, see MODES, or 0 for the planner's choice)."""
    from speculative_verify_paged_e4m3_gb300 import binding as B
    q = inputs["q"]
    bq, q_len, Hq, D = q.shape
    num_pool_pages, P, Hkv, _ = inputs["k_pool"].shape
    mpps = inputs["block_table"].shape[1]
    if max_context is None:
        max_context = max(1, mpps * P)
    att = B.VerifyAttention(bq, q_len, Hq, Hkv, D, P, mpps,
                            num_pool_pages if num_pages is None else num_pages, max_context,
                            num_splits=num_splits, **kernel_args(kernel))
    out, lse = att(inputs["q"], inputs["k_pool"], inputs["v_pool"], inputs["block_table"],
                   inputs["context_lens"], inputs["k_scale"], inputs["v_scale"])
    torch.cuda.synchronize()
    return att, out, lse
