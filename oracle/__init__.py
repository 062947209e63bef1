"""fp64 CPU oracle for split-K paged decode attention -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The library (``split_paged_decode_gb300``)
never imports it and shares no code with it: the oracle is plain C
(``oracle.c``) compiled with gcc into ``liboracle.so`` next to this file.

Functions take numpy arrays; bf16 tensors are passed as their uint16 bit
patterns (``t.view(torch.int16).numpy().view(np.uint16)``).

What is computed is documented in ``oracle.c``: the plain softmax-attention
definition (``decode``) and the same result through an explicit partition of
the key axis and the log-sum-exp merge of the fa4_splitk_combine_write page
(``partitioned``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


class _Shape(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int),
        ("num_q", ctypes.c_int),
        ("num_q_heads", ctypes.c_int),
        ("num_kv_heads", ctypes.c_int),
        ("qk_depth", ctypes.c_int),
        ("ov_depth", ctypes.c_int),
        ("page_size", ctypes.c_int),
        ("max_pages_per_seq", ctypes.c_int),
        ("num_pages", ctypes.c_int),
        ("v_in_k", ctypes.c_int),
    ]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc -O3, no fast-math)."""
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "oracle.h")))
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O3", "-std=c11", "-Wall", "-shared", "-fPIC", "-o", tmp, _SRC,
               "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # SPD_ORACLE_LIB points the tests at a deliberately broken build of
            # oracle.c (the mutation test); normally the in-tree build is used.
            path = os.environ.get("SPD_ORACLE_LIB")
            if not path:
                path = build()
            lib = ctypes.CDLL(path)
            p = ctypes.c_void_p
            lib.oracle_decode.argtypes = [ctypes.POINTER(_Shape), ctypes.c_double, p, p, p, p, p,
                                          p, ctypes.c_int64, p, p, ctypes.c_int]
            lib.oracle_decode.restype = ctypes.c_int
            lib.oracle_partitioned.argtypes = [ctypes.POINTER(_Shape), ctypes.c_double, p, p, p,
                                               p, p, p, ctypes.c_int, p, p, p, p, ctypes.c_int]
            lib.oracle_partitioned.restype = ctypes.c_int
            lib.oracle_decode_fp8.argtypes = [ctypes.POINTER(_Shape), ctypes.c_int, ctypes.c_double, p, p, p, p,
                                              p, p, p, p, ctypes.c_int64, p, p, ctypes.c_int]
            lib.oracle_decode_fp8.restype = ctypes.c_int
            lib.oracle_e4m3_value.argtypes = [ctypes.c_int]
            lib.oracle_e4m3_value.restype = ctypes.c_double
            lib.oracle_hardware_threads.argtypes = []
            lib.oracle_hardware_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def hardware_threads() -> int:
    return int(_load().oracle_hardware_threads())


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected uint16 bf16 bit patterns, got {a.dtype}")
    return a


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def decode(q, k_pages, v_pages, page_table, seq_lens, scale: float, *, ov_depth: int | None = None,
           rows=None, threads: int = 1):
    """Plain-definition attention in fp64.

    q [B,T,Hq,Dk], k_pages [NP,Hkv,PS,Dk], v_pages [NP,Hkv,PS,Dv] (uint16 bf16 bits);
    v_pages None means the MLA latent layout, V = first ``ov_depth`` columns of K.
    rows: optional int array [n,3] of (b, t, h) to evaluate only those rows.
    Returns (out float64 [B,T,Hq,Dv] or [n,Dv], lse float64 [B,T,Hq] or [n]).
    """
    lib = _load()
    q = _u16(q)
    k_pages = _u16(k_pages)
    page_table = _i32(page_table)
    seq_lens = _i32(seq_lens)
    B, T, Hq, Dk = q.shape
    NP, Hkv, PS, _ = k_pages.shape
    if v_pages is None:
        if ov_depth is None:
            raise ValueError("ov_depth is required for the latent layout")
        Dv, v_in_k, vp = int(ov_depth), 1, None
    else:
        v_pages = _u16(v_pages)
        Dv, v_in_k, vp = v_pages.shape[3], 0, v_pages
        if v_pages.shape[:3] != k_pages.shape[:3]:
            raise ValueError("v_pages and k_pages disagree on pages / heads / page_size")
    shape = _Shape(B, T, Hq, Hkv, Dk, Dv, PS, page_table.shape[1], NP, v_in_k)
    if rows is None:
        out = np.zeros((B, T, Hq, Dv), np.float64)
        lse = np.zeros((B, T, Hq), np.float64)
        rows_arr, n = None, 0
    else:
        rows_arr = _i32(rows).reshape(-1, 3)
        n = rows_arr.shape[0]
        out = np.zeros((n, Dv), np.float64)
        lse = np.zeros((n,), np.float64)
    rc = lib.oracle_decode(ctypes.byref(shape), float(scale), _ptr(q), _ptr(k_pages), _ptr(vp),
                           _ptr(page_table), _ptr(seq_lens), _ptr(rows_arr), n, _ptr(out),
                           _ptr(lse), int(threads))
    if rc != 0:
        raise ValueError("oracle_decode rejected its arguments (bad page id, length or shape)")
    return out, lse


def partitioned(q, k_pages, v_pages, page_table, seq_lens, scale: float, bounds, *,
                ov_depth: int | None = None, threads: int = 1, return_parts: bool = False):
    """Split-K path in fp64: per-partition (max, sum, O_p) then the LSE merge.

    bounds: int array [B, P+1] of key positions; partition p of sequence b is
    keys [bounds[b,p], bounds[b,p+1]). Returns (out, lse) and, with
    return_parts, also (part_max, part_sum) of shape [B,T,Hq,P].
    """
    lib = _load()
    q = _u16(q)
    k_pages = _u16(k_pages)
    page_table = _i32(page_table)
    seq_lens = _i32(seq_lens)
    bounds = _i32(bounds)
    B, T, Hq, Dk = q.shape
    NP, Hkv, PS, _ = k_pages.shape
    if v_pages is None:
        if ov_depth is None:
            raise ValueError("ov_depth is required for the latent layout")
        Dv, v_in_k, vp = int(ov_depth), 1, None
    else:
        v_pages = _u16(v_pages)
        Dv, v_in_k, vp = v_pages.shape[3], 0, v_pages
    P = bounds.shape[1] - 1
    if bounds.shape[0] != B or P < 1:
        raise ValueError("bounds must be [batch, P+1]")
    shape = _Shape(B, T, Hq, Hkv, Dk, Dv, PS, page_table.shape[1], NP, v_in_k)
    out = np.zeros((B, T, Hq, Dv), np.float64)
    lse = np.zeros((B, T, Hq), np.float64)
    pmax = np.zeros((B, T, Hq, P), np.float64)
    psum = np.zeros((B, T, Hq, P), np.float64)
    rc = lib.oracle_partitioned(ctypes.byref(shape), float(scale), _ptr(q), _ptr(k_pages),
                                _ptr(vp), _ptr(page_table), _ptr(seq_lens), _ptr(bounds), P,
                                _ptr(out), _ptr(lse), _ptr(pmax), _ptr(psum), int(threads))
    if rc != 0:
        raise ValueError("oracle_partitioned rejected its arguments")
    if return_parts:
        return out, lse, pmax, psum
    return out, lse


def e4m3_value(code: int) -> float:
    """The value the fp8 oracle reads for one OCP FP8 E4M3 code (0..255)."""
    return float(_load().oracle_e4m3_value(int(code)))


def decode_fp8(q, k8, v8, page_table, seq_lens, scale: float, *, k_rope=None, k_scale=None,
               ov_depth: int | None = None, rows=None, threads: int = 1):
    """Plain-definition attention in fp64 over an fp8 (E4M3) cache.

    q [B,T,Hq,Dk] (uint16 bf16 bits), k8 [NP,Hkv,PS,Dk-R] (uint8 E4M3 codes),
    v8 [NP,Hkv,PS,Dv] (uint8) or None for the latent layout (V = the first
    ``ov_depth`` dequantized values of the fp8 part of the key row),
    k_rope [NP,Hkv,PS,R] (uint16 bf16 bits) or None (R = 0), k_scale
    [NP,Hkv,PS] float32 per-token K scale or None (ones). Returns (out, lse)
    as ``decode`` does.
    """
    lib = _load()
    q = _u16(q)
    k8 = np.ascontiguousarray(k8)
    if k8.dtype != np.uint8:
        raise TypeError(f"expected uint8 E4M3 codes, got {k8.dtype}")
    page_table = _i32(page_table)
    seq_lens = _i32(seq_lens)
    B, T, Hq, Dk = q.shape
    NP, Hkv, PS, D8 = k8.shape
    R = 0
    if k_rope is not None:
        k_rope = _u16(k_rope)
        R = k_rope.shape[3]
        if k_rope.shape[:3] != k8.shape[:3]:
            raise ValueError("k_rope and k8 disagree on pages / heads / page_size")
    if D8 + R != Dk:
        raise ValueError(f"q depth {Dk} != fp8 part {D8} + rope part {R}")
    if k_scale is not None:
        k_scale = np.ascontiguousarray(k_scale, dtype=np.float32)
        if k_scale.shape != k8.shape[:3]:
            raise ValueError("k_scale must be [num_pages, num_kv_heads, page_size]")
    if v8 is None:
        if ov_depth is None:
            raise ValueError("ov_depth is required for the latent layout")
        Dv, v_in_k = int(ov_depth), 1
    else:
        v8 = np.ascontiguousarray(v8)
        if v8.dtype != np.uint8:
            raise TypeError(f"expected uint8 E4M3 codes, got {v8.dtype}")
        Dv, v_in_k = v8.shape[3], 0
    shape = _Shape(B, T, Hq, Hkv, Dk, Dv, PS, page_table.shape[1], NP, v_in_k)
    if rows is None:
        out = np.zeros((B, T, Hq, Dv), np.float64)
        lse = np.zeros((B, T, Hq), np.float64)
        rows_arr, n = None, 0
    else:
        rows_arr = _i32(rows).reshape(-1, 3)
        n = rows_arr.shape[0]
        out = np.zeros((n, Dv), np.float64)
        lse = np.zeros((n,), np.float64)
    rc = lib.oracle_decode_fp8(ctypes.byref(shape), R, float(scale), _ptr(q), _ptr(k8), _ptr(v8), _ptr(k_rope),
                               _ptr(k_scale), _ptr(page_table), _ptr(seq_lens), _ptr(rows_arr), n, _ptr(out),
                               _ptr(lse), int(threads))
    if rc != 0:
        raise ValueError("oracle_decode_fp8 rejected its arguments (bad page id, length or shape)")
    return out, lse
