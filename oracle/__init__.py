"""FP64 CPU oracle for DFlash2 speculative-verification attention (paged E4M3 KV cache).

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. It shares no code with the CUDA path; the product never
imports it.

The arithmetic lives in ``verify_attn_oracle.c`` (plain C, FP64, OpenMP over query rows); this
module compiles it with gcc on first use and marshals NumPy arrays through ctypes. See the C
file's header for the definition it implements and the passages it follows.

Pins (tests/test_oracle_pins.py): E4M3 decode against the OCP format's printed values and the
library cast ``torch.float8_e4m3fn``; E4M3 encode by round trip over every code, midpoints
(ties to even), saturation and the library cast; the KV write on hand-placed tokens; tiny cases against torch's float64 scaled-dot-product
attention (a library routine); uniform- and one-hot-softmax closed forms; block-table permutation
and page-size invariance; split/merge agreement; the q_len = 1 reduction; planted mistakes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "verify_attn_oracle.c")
BUILD_DIR = os.path.join(_HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libverify_attn_oracle.so")

_lock = threading.Lock()
_default = None

_dp = ctypes.POINTER(ctypes.c_double)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_i32p = ctypes.POINTER(ctypes.c_int32)


def compile_oracle(source: str = SOURCE, out_path: str = LIB_PATH) -> str:
    """Compile the C oracle into a shared library (gcc, -O2, OpenMP) and return its path."""
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    tmp = out_path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", tmp, source, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(tmp, out_path)
    return out_path


def _ptr(a: np.ndarray, t):
    return a.ctypes.data_as(t)


class Oracle:
    """ctypes handle on one build of the C oracle."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        lib.oracle_e4m3_decode.argtypes = [_u8p, ctypes.c_int64, _dp]
        lib.oracle_e4m3_decode.restype = None
        common = [ctypes.c_int] * 8 + [_dp, _u8p, _u8p, _i32p, _i32p, ctypes.c_double,
                                       ctypes.c_double]
        lib.oracle_verify_attn.argtypes = common + [_dp, _dp]
        lib.oracle_verify_attn.restype = ctypes.c_int
        lib.oracle_verify_attn_partials.argtypes = common + [ctypes.c_int, _i32p, _dp, _dp, _dp]
        lib.oracle_verify_attn_partials.restype = ctypes.c_int
        lib.oracle_merge_partials.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int, _dp,
                                              _dp, _dp, _dp, _dp]
        lib.oracle_merge_partials.restype = None
        lib.oracle_e4m3_encode_array.argtypes = [_dp, ctypes.c_int64, _u8p]
        lib.oracle_e4m3_encode_array.restype = None
        _fp = ctypes.POINTER(ctypes.c_float)
        lib.oracle_kv_write.argtypes = [ctypes.c_int] * 8 + [_fp, _fp, _i32p, _i32p,
                                                               ctypes.c_float, ctypes.c_float,
                                                               _u8p, _u8p]
        lib.oracle_kv_write.restype = ctypes.c_int
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = ctypes.c_int
        self.lib = lib
        self.path = lib_path

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def e4m3_decode(self, codes) -> np.ndarray:
        codes = np.ascontiguousarray(codes, dtype=np.uint8)
        out = np.empty(codes.shape, dtype=np.float64)
        self.lib.oracle_e4m3_decode(_ptr(codes, _u8p), codes.size, _ptr(out, _dp))
        return out

    def e4m3_encode(self, values) -> np.ndarray:
        """E4M3FN codes of real values (nearest, ties to even, saturated to +-448)."""
        v = np.ascontiguousarray(values, dtype=np.float64)
        out = np.empty(v.shape, dtype=np.uint8)
        self.lib.oracle_e4m3_encode_array(_ptr(v, _dp), v.size, _ptr(out, _u8p))
        return out

    def kv_write(self, k_new, v_new, block_table, context_lens, k_scale, v_scale, k_pool, v_pool,
                 max_context):
        """Write the drafted tokens' K/V rows into copies of the pools.

        k_new, v_new: FP16 values [B, q_len, Hkv, D]; pools uint8 [num_pages, P, Hkv, D].
        Returns (k_pool, v_pool, flags) with flags as oracle_kv_write returns them.
        """
        fp = ctypes.POINTER(ctypes.c_float)
        k_new = np.ascontiguousarray(np.asarray(k_new).astype(np.float32))
        v_new = np.ascontiguousarray(np.asarray(v_new).astype(np.float32))
        k_pool = np.array(k_pool, dtype=np.uint8, copy=True, order="C")
        v_pool = np.array(v_pool, dtype=np.uint8, copy=True, order="C")
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        B, q_len, Hkv, D = k_new.shape
        num_pages, P, Hkv_p, D_p = k_pool.shape
        if (Hkv_p, D_p) != (Hkv, D) or v_new.shape != k_new.shape or v_pool.shape != k_pool.shape:
            raise ValueError("kv_write: shapes disagree")
        if bt.ndim != 2 or bt.shape[0] != B or cl.shape != (B,):
            raise ValueError("kv_write: block_table must be [B, max_pages] and context_lens [B]")
        flags = self.lib.oracle_kv_write(B, q_len, Hkv, D, P, bt.shape[1], num_pages,
                                         int(max_context), k_new.ctypes.data_as(fp),
                                         v_new.ctypes.data_as(fp), _ptr(bt, _i32p),
                                         _ptr(cl, _i32p), float(k_scale), float(v_scale),
                                         _ptr(k_pool, _u8p), _ptr(v_pool, _u8p))
        return k_pool, v_pool, int(flags)

    @staticmethod
    def _common(q, k_pool, v_pool, block_table, context_lens, k_scale, v_scale):
        q = np.asarray(q)
        if q.dtype == np.float16:
            q = q.astype(np.float64)  # exact: every FP16 value is a double
        q = np.ascontiguousarray(q, dtype=np.float64)
        k_pool = np.ascontiguousarray(k_pool, dtype=np.uint8)
        v_pool = np.ascontiguousarray(v_pool, dtype=np.uint8)
        block_table = np.ascontiguousarray(block_table, dtype=np.int32)
        context_lens = np.ascontiguousarray(context_lens, dtype=np.int32)
        B, q_len, Hq, D = q.shape
        num_pages, P, Hkv, Dk = k_pool.shape
        if Dk != D or v_pool.shape != k_pool.shape:
            raise ValueError("q / k_pool / v_pool shapes disagree")
        if block_table.ndim != 2 or block_table.shape[0] != B or context_lens.shape != (B,):
            raise ValueError("block_table must be [B, max_pages] and context_lens [B]")
        dims = (B, q_len, Hq, Hkv, D, P, block_table.shape[1], num_pages)
        args = (q, k_pool, v_pool, block_table, context_lens)
        return dims, args, float(k_scale), float(v_scale)

    def verify_attn(self, q, k_pool, v_pool, block_table, context_lens, k_scale, v_scale):
        """Unsplit causal attention. Returns (out float64 [B,q,Hq,D], lse float64 [B,q,Hq])."""
        dims, (q, k, v, bt, cl), ks, vs = self._common(q, k_pool, v_pool, block_table,
                                                       context_lens, k_scale, v_scale)
        B, q_len, Hq, Hkv, D = dims[:5]
        out = np.empty((B, q_len, Hq, D), dtype=np.float64)
        lse = np.empty((B, q_len, Hq), dtype=np.float64)
        rc = self.lib.oracle_verify_attn(*dims, _ptr(q, _dp), _ptr(k, _u8p), _ptr(v, _u8p),
                                         _ptr(bt, _i32p), _ptr(cl, _i32p), ks, vs,
                                         _ptr(out, _dp), _ptr(lse, _dp))
        if rc != 0:
            raise ValueError(f"oracle_verify_attn failed with status {rc}")
        return out, lse

    def verify_attn_partials(self, q, k_pool, v_pool, block_table, context_lens, k_scale,
                             v_scale, split_bounds):
        """Per-split state. split_bounds is int [B, S+1]. Returns m, l [B,Hkv,S,R], acc [..,D]."""
        dims, (q, k, v, bt, cl), ks, vs = self._common(q, k_pool, v_pool, block_table,
                                                       context_lens, k_scale, v_scale)
        B, q_len, Hq, Hkv, D = dims[:5]
        sb = np.ascontiguousarray(split_bounds, dtype=np.int32)
        if sb.ndim != 2 or sb.shape[0] != B:
            raise ValueError("split_bounds must be [B, S+1]")
        S = sb.shape[1] - 1
        R = q_len * (Hq // Hkv)
        m = np.empty((B, Hkv, S, R), dtype=np.float64)
        l = np.empty_like(m)
        acc = np.empty((B, Hkv, S, R, D), dtype=np.float64)
        rc = self.lib.oracle_verify_attn_partials(*dims, _ptr(q, _dp), _ptr(k, _u8p),
                                                  _ptr(v, _u8p), _ptr(bt, _i32p),
                                                  _ptr(cl, _i32p), ks, vs, S, _ptr(sb, _i32p),
                                                  _ptr(m, _dp), _ptr(l, _dp), _ptr(acc, _dp))
        if rc != 0:
            raise ValueError(f"oracle_verify_attn_partials failed with status {rc}")
        return m, l, acc

    def merge_partials(self, m, l, acc):
        """Combine split state. m, l [rows, S]; acc [rows, S, D] -> out [rows, D], lse [rows]."""
        m = np.ascontiguousarray(m, dtype=np.float64)
        l = np.ascontiguousarray(l, dtype=np.float64)
        acc = np.ascontiguousarray(acc, dtype=np.float64)
        rows, S = m.shape
        D = acc.shape[-1]
        if l.shape != m.shape or acc.shape != (rows, S, D):
            raise ValueError("merge_partials: m, l [rows,S] and acc [rows,S,D] expected")
        out = np.empty((rows, D), dtype=np.float64)
        lse = np.empty((rows,), dtype=np.float64)
        self.lib.oracle_merge_partials(rows, S, D, _ptr(m, _dp), _ptr(l, _dp), _ptr(acc, _dp),
                                       _ptr(out, _dp), _ptr(lse, _dp))
        return out, lse


def load(rebuild: bool = False) -> Oracle:
    """The oracle built from this directory's C source (compiled on first use)."""
    global _default
    with _lock:
        if _default is None or rebuild:
            stale = (not os.path.exists(LIB_PATH)
                     or os.path.getmtime(LIB_PATH) < os.path.getmtime(SOURCE))
            if rebuild or stale:
                compile_oracle()
            _default = Oracle(LIB_PATH)
        return _default


def rows_view(m, l, acc):
    """Reshape [B,Hkv,S,R](,D) split state into the [rows,S](,D) form merge_partials takes."""
    B, Hkv, S, R = m.shape
    D = acc.shape[-1]
    mt = np.moveaxis(m, 2, 3).reshape(B * Hkv * R, S)
    lt = np.moveaxis(l, 2, 3).reshape(B * Hkv * R, S)
    at = np.moveaxis(acc, 2, 3).reshape(B * Hkv * R, S, D)
    return mt, lt, at


def rows_to_bqh(x, B, q_len, Hq, Hkv):
    """Map per-(b, h, r) rows (r = i*G + g) back to [B, q_len, Hq, ...] order."""
    G = Hq // Hkv
    tail = x.shape[1:]
    y = x.reshape((B, Hkv, q_len, G) + tail)
    y = np.moveaxis(y, 1, 2)  # [B, q_len, Hkv, G, ...]
    return y.reshape((B, q_len, Hq) + tail)
