"""Thin ctypes binding of libfa_decode.so (include/fa_decode.h).

Argument marshalling only: every step of the decode runs in the library's
CUDA kernels. Functions keep the C names; tensors may be passed as torch
tensors (their data pointers are taken) or as integer addresses. There is no
fallback: if the library is missing, loading it raises.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfa_decode.so")

FA_OK = 0
FA_ERR_INVALID_ARG = -1
FA_ERR_UNSUPPORTED = -2
FA_ERR_CUDA = -3
FA_ERR_DEVICE = -4
FA_STATUS_TIMEOUT = 1
FA_STATUS_BAD_PAGE = 2
FA_DEBUG_SKIP_LOADS = 1
FA_DEBUG_FORCE_SIMT = 2
FA_DEBUG_TWO_CLUSTERS = 4
FA_DEBUG_NO_STREAM_K = 8
FA_TRACE_WORDS_PER_CTA = 64
FA_NOALLOC_STATUS_SLOTS = 64
FA_KV_BF16 = 0
FA_KV_E4M3 = 1

# Every symbol include/fa_decode.h declares.
EXPORTED = ("fa_decode_create", "fa_decode_run", "fa_decode_create_kv", "fa_decode_run_kv", "fa_decode_check",
            "fa_decode_set_debug",
            "fa_decode_set_trace", "fa_decode_describe", "fa_decode_run_noalloc", "fa_decode_destroy",
            "fa_decode_last_error")


class FaDecodeError(RuntimeError):
    """A failed call: `code` is the FA_ERR_* return value; `status` holds the
    device's FA_STATUS_* bits when the call reported them (else None)."""

    def __init__(self, code: int, message: str, status: int | None = None):
        super().__init__(f"{message} (code {code})")
        self.code = code
        self.status = status


_lib = None


def load_library(path: str | None = None):
    """Load libfa_decode.so (built by split_paged_decode_gb300.build); raise if absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise FileNotFoundError(
            f"{p} is missing: build it with `python -m split_paged_decode_gb300.build` "
            "(or __graft_entry__.build()); there is no fallback path")
    lib = ctypes.CDLL(p)
    vp, i32, i64, u32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint32
    lib.fa_decode_create.argtypes = [ctypes.POINTER(vp), i32, i32, i32, i32, i32, i32, i32, i32]
    lib.fa_decode_create.restype = i32
    lib.fa_decode_run.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, i32, i32, i32]
    lib.fa_decode_run.restype = i32
    lib.fa_decode_create_kv.argtypes = [ctypes.POINTER(vp), i32, i32, i32, i32, i32, i32, i32, i32, i32, i32]
    lib.fa_decode_create_kv.restype = i32
    lib.fa_decode_run_kv.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, i32, i32, i32]
    lib.fa_decode_run_kv.restype = i32
    lib.fa_decode_check.argtypes = [vp, vp, ctypes.POINTER(u32)]
    lib.fa_decode_check.restype = i32
    lib.fa_decode_set_debug.argtypes = [vp, u32, i64]
    lib.fa_decode_set_debug.restype = i32
    lib.fa_decode_set_trace.argtypes = [vp, vp, i64]
    lib.fa_decode_set_trace.restype = i32
    lib.fa_decode_describe.argtypes = [vp, ctypes.c_char_p, i32]
    lib.fa_decode_describe.restype = i32
    lib.fa_decode_run_noalloc.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp,
                                          ctypes.c_float, vp, vp, vp, i32, i32, i32, i32, ctypes.POINTER(u32)]
    lib.fa_decode_run_noalloc.restype = i32
    lib.fa_decode_destroy.argtypes = [vp]
    lib.fa_decode_destroy.restype = i32
    lib.fa_decode_last_error.argtypes = []
    lib.fa_decode_last_error.restype = ctypes.c_char_p
    if path is None:
        _lib = lib
    return lib


def fa_decode_last_error() -> str:
    return load_library().fa_decode_last_error().decode()


def _check(rc: int):
    if rc != FA_OK:
        raise FaDecodeError(rc, fa_decode_last_error())


def _addr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(stream) -> int | None:
    if stream is None:
        import torch

        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def fa_decode_create(num_q_heads: int, num_kv_heads: int, qk_depth: int, nope_depth: int, ov_depth: int,
                     page_size: int, num_q: int, splitk: int) -> int:
    """Create a plan; returns the handle (an integer address). Raises FaDecodeError."""
    h = ctypes.c_void_p()
    _check(load_library().fa_decode_create(ctypes.byref(h), num_q_heads, num_kv_heads, qk_depth, nope_depth,
                                           ov_depth, page_size, num_q, splitk))
    return int(h.value)


def fa_decode_run(h: int, q, k_pages, v_pages, page_table, seq_lens, scale: float, out, lse, stream=None,
                  batch: int | None = None, max_pages_per_seq: int | None = None,
                  num_pages: int | None = None) -> None:
    """Enqueue one decode forward. Sizes default to the torch tensors' shapes.

    Runs of one handle must not overlap on the GPU (one stream at a time, or
    ordered by events): the handle's stream-K scratch is shared by its runs.
    """
    if batch is None:
        batch = int(q.shape[0])
    if max_pages_per_seq is None:
        max_pages_per_seq = int(page_table.shape[1])
    if num_pages is None:
        num_pages = int(k_pages.shape[0])
    _check(load_library().fa_decode_run(h, _addr(q), _addr(k_pages), _addr(v_pages), _addr(page_table),
                                        _addr(seq_lens), float(scale), _addr(out), _addr(lse), _stream(stream),
                                        batch, max_pages_per_seq, num_pages))


def fa_decode_create_kv(num_q_heads: int, num_kv_heads: int, qk_depth: int, nope_depth: int, ov_depth: int,
                        page_size: int, num_q: int, splitk: int, kv_format: int, rope_depth: int = 0) -> int:
    """Create a plan for a cache of format kv_format (FA_KV_BF16 / FA_KV_E4M3)."""
    h = ctypes.c_void_p()
    _check(load_library().fa_decode_create_kv(ctypes.byref(h), num_q_heads, num_kv_heads, qk_depth, nope_depth,
                                              ov_depth, page_size, num_q, splitk, kv_format, rope_depth))
    return int(h.value)


def fa_decode_run_kv(h: int, q, k_pages, v_pages, k_rope_pages, k_scale, page_table, seq_lens, scale: float, out,
                     lse, stream=None, batch: int | None = None, max_pages_per_seq: int | None = None,
                     num_pages: int | None = None) -> None:
    """Enqueue one decode forward over the handle's cache format (E4M3 codes
    as uint8 tensors, per-token K scales as an fp32 tensor or None)."""
    if batch is None:
        batch = int(q.shape[0])
    if max_pages_per_seq is None:
        max_pages_per_seq = int(page_table.shape[1])
    if num_pages is None:
        num_pages = int(k_pages.shape[0])
    _check(load_library().fa_decode_run_kv(h, _addr(q), _addr(k_pages), _addr(v_pages), _addr(k_rope_pages),
                                           _addr(k_scale), _addr(page_table), _addr(seq_lens), float(scale),
                                           _addr(out), _addr(lse), _stream(stream), batch, max_pages_per_seq,
                                           num_pages))


def fa_decode_check(h: int, stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status bits."""
    st = ctypes.c_uint32(0)
    rc = load_library().fa_decode_check(h, _stream(stream), ctypes.byref(st))
    if rc not in (FA_OK, FA_ERR_DEVICE):
        _check(rc)
    return int(st.value)


def fa_decode_set_debug(h: int, flags: int, wait_limit_ns: int = 0) -> None:
    _check(load_library().fa_decode_set_debug(h, flags, wait_limit_ns))


def fa_decode_set_trace(h: int, buf=None) -> None:
    """Record a per-CTA timeline into `buf` (a device int64 tensor, zeroed by the
    caller; FA_TRACE_WORDS_PER_CTA words per CTA) on later runs; None stops it."""
    if buf is None:
        _check(load_library().fa_decode_set_trace(h, None, 0))
    else:
        _check(load_library().fa_decode_set_trace(h, _addr(buf), buf.numel()))


def fa_decode_describe(h: int) -> str:
    buf = ctypes.create_string_buffer(512)
    _check(load_library().fa_decode_describe(h, buf, len(buf)))
    return buf.value.decode()


def fa_decode_run_noalloc(num_q_heads: int, num_kv_heads: int, qk_depth: int, nope_depth: int, ov_depth: int,
                          page_size: int, num_q: int, splitk: int, q, k_pages, v_pages, page_table, seq_lens,
                          scale: float, out, lse, stream=None, batch: int | None = None,
                          max_pages_per_seq: int | None = None, num_pages: int | None = None,
                          status_slot: int = 0, wait: bool = True) -> int | None:
    """One decode forward without any device allocation (see include/fa_decode.h).

    For callers that cannot allocate device memory. With wait=True the call
    synchronises the stream and returns the status bits (raising FaDecodeError
    with code FA_ERR_DEVICE and those bits in `.status` if any is set); with
    wait=False it only enqueues and returns None.
    """
    if batch is None:
        batch = int(q.shape[0])
    if max_pages_per_seq is None:
        max_pages_per_seq = int(page_table.shape[1])
    if num_pages is None:
        num_pages = int(k_pages.shape[0])
    st = ctypes.c_uint32(0)
    rc = load_library().fa_decode_run_noalloc(
        num_q_heads, num_kv_heads, qk_depth, nope_depth, ov_depth, page_size, num_q, splitk, _addr(q),
        _addr(k_pages), _addr(v_pages), _addr(page_table), _addr(seq_lens), float(scale), _addr(out), _addr(lse),
        _stream(stream), batch, max_pages_per_seq, num_pages, status_slot, ctypes.byref(st) if wait else None)
    if rc == FA_ERR_DEVICE:
        raise FaDecodeError(rc, fa_decode_last_error(), status=int(st.value))
    _check(rc)
    return int(st.value) if wait else None


def fa_decode_destroy(h: int) -> None:
    _check(load_library().fa_decode_destroy(h))
