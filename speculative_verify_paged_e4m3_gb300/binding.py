"""Thin ctypes binding over libdflash_verify_attn.so (the C ABI in include/dflash_verify_attn.h).

Argument marshalling only: every step of the computation runs in the library's CUDA kernels.
Functions carry the C names; tensors are torch CUDA tensors whose data pointers are passed
through, and the stream is torch's current stream unless one is given. If the library has not
been built, every entry point raises (there is no fallback).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

DFLASH_VERIFY_ATTN_VERSION = 3
DFLASH_OK = 0
DFLASH_ERR_INVALID_ARGUMENT = -1
DFLASH_ERR_UNSUPPORTED = -2
DFLASH_ERR_WORKSPACE_TOO_SMALL = -3
DFLASH_ERR_CUDA = -4
DFLASH_FLAG_CONTEXT_CLAMPED = 0x1
DFLASH_FLAG_CONTEXT_SHORT = 0x2
DFLASH_FLAG_PAGE_CLAMPED = 0x4
DFLASH_FLAG_KERNEL_TIMEOUT = 0x8
DFLASH_PROBLEM_FUSED_COMBINE = 0x1
DFLASH_PROBLEM_PDL = 0x2
DFLASH_KERNEL_AUTO = 0
DFLASH_KERNEL_SIMT = 1
DFLASH_KERNEL_TCGEN05 = 2

EXPORTED = (
    "dflash_verify_attn_plan",
    "dflash_verify_attn_split_bounds",
    "dflash_verify_attn_split_slots",
    "dflash_verify_attn_run",
    "dflash_verify_attn_combine",
    "dflash_verify_attn_forward",
    "dflash_verify_attn_debug_dequant",
    "dflash_verify_attn_read_flags",
    "dflash_verify_attn_forward_static_scratch",
    "dflash_verify_attn_kv_write",
    "dflash_verify_attn_status_string",
)


class Problem(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "version", "batch", "q_len", "num_q_heads", "num_kv_heads", "head_dim", "page_size",
        "max_pages_per_seq", "num_pages", "max_context", "device", "num_splits", "kernel",
        "flags")]


class Plan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "version", "kernel", "num_splits", "tile_keys", "min_split_keys", "rows", "threads",
        "smem_bytes", "sm_count", "combine_fused", "row_blocks", "num_slots")] + [
        ("workspace_bytes", ctypes.c_size_t),
        ("ws_state_offset", ctypes.c_size_t),
        ("ws_acc_offset", ctypes.c_size_t),
        ("problem", Problem),
    ]


class DflashError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {status_string(status)} ({status})")
        self.status = status


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load_library() -> ctypes.CDLL:
    """Load the built library (raises if it is missing: build it with build.build())."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(f"CUDA library {path} is not built; run "
                                   "speculative_verify_paged_e4m3_gb300.build.build() first")
            lib = ctypes.CDLL(path)
            vp, sz, i32, i64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_int64
            pp = ctypes.POINTER(Plan)
            lib.dflash_verify_attn_plan.argtypes = [ctypes.POINTER(Problem), pp]
            lib.dflash_verify_attn_split_bounds.argtypes = [
                pp, i32, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]
            i32p = ctypes.POINTER(ctypes.c_int32)
            lib.dflash_verify_attn_split_slots.argtypes = [pp, i32p, i32p, i32p, i32p]
            lib.dflash_verify_attn_run.argtypes = [pp] + [vp] * 8 + [sz, vp]
            lib.dflash_verify_attn_combine.argtypes = [pp, vp, sz, vp, vp, vp, vp]
            lib.dflash_verify_attn_forward.argtypes = [pp] + [vp] * 8 + [sz, vp, vp, vp]
            lib.dflash_verify_attn_forward_static_scratch.argtypes = [pp] + [vp] * 10
            lib.dflash_verify_attn_kv_write.argtypes = [pp] + [vp] * 9 + [sz, vp]
            lib.dflash_verify_attn_debug_dequant.argtypes = [vp, i64, vp, vp, vp, vp]
            lib.dflash_verify_attn_read_flags.argtypes = [vp, ctypes.POINTER(ctypes.c_int32),
                                                          ctypes.c_int, vp]
            lib.dflash_verify_attn_status_string.argtypes = [ctypes.c_int]
            lib.dflash_verify_attn_status_string.restype = ctypes.c_char_p
            for name in EXPORTED[:-1]:
                getattr(lib, name).restype = ctypes.c_int
            _lib = lib
        return _lib


def status_string(status: int) -> str:
    return load_library().dflash_verify_attn_status_string(int(status)).decode()


dflash_verify_attn_status_string = status_string


def _check(fn: str, status: int):
    if status != DFLASH_OK:
        raise DflashError(fn, status)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_problem(batch, q_len, num_q_heads, num_kv_heads, head_dim, page_size,
                 max_pages_per_seq, num_pages, max_context, device=0, num_splits=0,
                 kernel=DFLASH_KERNEL_AUTO, flags=0) -> Problem:
    return Problem(DFLASH_VERIFY_ATTN_VERSION, batch, q_len, num_q_heads, num_kv_heads,
                   head_dim, page_size, max_pages_per_seq, num_pages, max_context, device,
                   num_splits, kernel, flags)


def dflash_verify_attn_plan(problem: Problem) -> Plan:
    plan = Plan()
    _check("dflash_verify_attn_plan",
           load_library().dflash_verify_attn_plan(ctypes.byref(problem), ctypes.byref(plan)))
    return plan


def dflash_verify_attn_plan_status(problem: Problem) -> int:
    """The raw status of planning (for tests of the error paths)."""
    plan = Plan()
    return load_library().dflash_verify_attn_plan(ctypes.byref(problem), ctypes.byref(plan))


def dflash_verify_attn_split_bounds(plan: Plan, n: int):
    starts = (ctypes.c_int32 * (plan.num_splits + 1))()
    active = ctypes.c_int32()
    _check("dflash_verify_attn_split_bounds",
           load_library().dflash_verify_attn_split_bounds(ctypes.byref(plan), int(n), starts,
                                                          ctypes.byref(active)))
    return list(starts), active.value


def dflash_verify_attn_split_slots(plan: Plan, context_lens):
    """(slot_start [units + 1], keys_per_split [units], active [units]) for the given host-side
    context lengths (units = batch * Hkv, unit u = b * Hkv + h)."""
    lens = list(int(x) for x in context_lens)
    units = plan.problem.batch * plan.problem.num_kv_heads
    if len(lens) != plan.problem.batch:
        raise ValueError("context_lens must have batch entries")
    cl = (ctypes.c_int32 * len(lens))(*lens)
    start = (ctypes.c_int32 * (units + 1))()
    per = (ctypes.c_int32 * units)()
    act = (ctypes.c_int32 * units)()
    _check("dflash_verify_attn_split_slots",
           load_library().dflash_verify_attn_split_slots(ctypes.byref(plan), cl, start, per, act))
    return list(start), list(per), list(act)


def dflash_verify_attn_run(plan: Plan, q, k_pool, v_pool, block_table, context_lens, k_scale,
                           v_scale, workspace, stream=None, check=True) -> int:
    rc = load_library().dflash_verify_attn_run(
        ctypes.byref(plan), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table),
        _ptr(context_lens), _ptr(k_scale), _ptr(v_scale), _ptr(workspace),
        workspace.numel() * workspace.element_size() if hasattr(workspace, "numel") else 0,
        _stream(stream))
    if check:
        _check("dflash_verify_attn_run", rc)
    return rc


def dflash_verify_attn_combine(plan: Plan, workspace, context_lens, out, lse, stream=None,
                               check=True) -> int:
    rc = load_library().dflash_verify_attn_combine(
        ctypes.byref(plan), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(context_lens), _ptr(out), _ptr(lse), _stream(stream))
    if check:
        _check("dflash_verify_attn_combine", rc)
    return rc


def dflash_verify_attn_forward(plan: Plan, q, k_pool, v_pool, block_table, context_lens,
                               k_scale, v_scale, workspace, out, lse, stream=None,
                               check=True) -> int:
    rc = load_library().dflash_verify_attn_forward(
        ctypes.byref(plan), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table),
        _ptr(context_lens), _ptr(k_scale), _ptr(v_scale), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(out), _ptr(lse), _stream(stream))
    if check:
        _check("dflash_verify_attn_forward", rc)
    return rc


def dflash_verify_attn_forward_static_scratch(plan: Plan, q, k_pool, v_pool, block_table,
                                              context_lens, k_scale, v_scale, out, lse,
                                              stream=None, check=True) -> int:
    """Forward pass using the library's built-in device scratch array (no workspace argument)."""
    rc = load_library().dflash_verify_attn_forward_static_scratch(
        ctypes.byref(plan), _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table),
        _ptr(context_lens), _ptr(k_scale), _ptr(v_scale), _ptr(out), _ptr(lse),
        _stream(stream))
    if check:
        _check("dflash_verify_attn_forward_static_scratch", rc)
    return rc


def dflash_verify_attn_kv_write(plan: Plan, k_new, v_new, block_table, context_lens, k_scale,
                                v_scale, k_pool, v_pool, workspace, stream=None,
                                check=True) -> int:
    rc = load_library().dflash_verify_attn_kv_write(
        ctypes.byref(plan), _ptr(k_new), _ptr(v_new), _ptr(block_table), _ptr(context_lens),
        _ptr(k_scale), _ptr(v_scale), _ptr(k_pool), _ptr(v_pool), _ptr(workspace),
        workspace.numel() * workspace.element_size() if hasattr(workspace, "numel") else 0,
        _stream(stream))
    if check:
        _check("dflash_verify_attn_kv_write", rc)
    return rc


def dflash_verify_attn_debug_dequant(codes, scale, decoded, scaled=None, stream=None):
    _check("dflash_verify_attn_debug_dequant",
           load_library().dflash_verify_attn_debug_dequant(
               _ptr(codes), codes.numel(), _ptr(scale), _ptr(decoded), _ptr(scaled),
               _stream(stream)))


def dflash_verify_attn_read_flags(workspace, clear=False, stream=None) -> int:
    v = ctypes.c_int32()
    _check("dflash_verify_attn_read_flags",
           load_library().dflash_verify_attn_read_flags(_ptr(workspace), ctypes.byref(v),
                                                        int(bool(clear)), _stream(stream)))
    return v.value


# ---------------------------------------------------------------------------------------------
# convenience layer (still marshalling only)

class VerifyAttention:
    """One layer shape: a plan plus its workspace; call() runs partial attention and combine."""

    def __init__(self, batch, q_len, num_q_heads, num_kv_heads, head_dim, page_size,
                 max_pages_per_seq, num_pages, max_context, device=None, num_splits=0,
                 kernel=DFLASH_KERNEL_AUTO, workspace=None, flags=0):
        dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
        self.device = dev
        self.problem = make_problem(batch, q_len, num_q_heads, num_kv_heads, head_dim,
                                    page_size, max_pages_per_seq, num_pages, max_context,
                                    dev.index, num_splits, kernel, flags)
        self.plan = dflash_verify_attn_plan(self.problem)
        if workspace is None:
            workspace = torch.zeros(self.plan.workspace_bytes, dtype=torch.uint8, device=dev)
        elif workspace.numel() * workspace.element_size() < self.plan.workspace_bytes:
            raise ValueError("workspace smaller than plan.workspace_bytes")
        self.workspace = workspace

    def workspace_views(self):
        """(status int32[1], state float32 [slots,R,2], acc float32 [slots,R,D]) views; for a
        single sequence slot h * num_splits + s is split s of KV head h."""
        pr, pl = self.problem, self.plan
        shape = (pl.num_slots, pl.rows)
        ws = self.workspace
        n_state = pl.num_slots * pl.rows * 2
        state = ws[pl.ws_state_offset:pl.ws_state_offset + 4 * n_state].view(torch.float32)
        n_acc = n_state // 2 * pr.head_dim
        acc = ws[pl.ws_acc_offset:pl.ws_acc_offset + 4 * n_acc].view(torch.float32)
        return (ws[:4].view(torch.int32), state.view(shape + (2,)),
                acc.view(shape + (pr.head_dim,)))

    def __call__(self, q, k_pool, v_pool, block_table, context_lens, k_scale, v_scale,
                 out=None, lse=None, stream=None):
        pr = self.problem
        if out is None:
            out = torch.empty((pr.batch, pr.q_len, pr.num_q_heads, pr.head_dim),
                              dtype=torch.float16, device=self.device)
        if lse is None:
            lse = torch.empty((pr.batch, pr.q_len, pr.num_q_heads), dtype=torch.float32,
                              device=self.device)
        dflash_verify_attn_forward(self.plan, q, k_pool, v_pool, block_table, context_lens,
                                   k_scale, v_scale, self.workspace, out, lse, stream)
        return out, lse

    def kv_write(self, k_new, v_new, block_table, context_lens, k_scale, v_scale, k_pool,
                 v_pool, stream=None):
        """Write the drafted tokens' K/V rows ([B, q_len, Hkv, D] FP16) into the pools."""
        dflash_verify_attn_kv_write(self.plan, k_new, v_new, block_table, context_lens, k_scale,
                                    v_scale, k_pool, v_pool, self.workspace, stream)
