"""GB300-native split-K paged decode attention.

The compute path is libfa_decode.so (hand-written sm_103a CUDA behind the C
ABI of include/fa_decode.h); this package holds its ctypes binding, its build
script and the seeded synthetic workloads used to test and measure it.
"""
from .binding import (EXPORTED, FA_DEBUG_FORCE_SIMT, FA_DEBUG_SKIP_LOADS, FA_DEBUG_TWO_CLUSTERS, FA_DEBUG_NO_STREAM_K, FA_TRACE_WORDS_PER_CTA, FA_ERR_CUDA, FA_NOALLOC_STATUS_SLOTS, FA_ERR_DEVICE, FA_ERR_INVALID_ARG,
                      FA_ERR_UNSUPPORTED, FA_KV_BF16, FA_KV_E4M3, FA_OK, FA_STATUS_BAD_PAGE, FA_STATUS_TIMEOUT, FaDecodeError,
                      fa_decode_check, fa_decode_create, fa_decode_create_kv, fa_decode_describe, fa_decode_destroy,
                      fa_decode_last_error, fa_decode_run, fa_decode_run_kv, fa_decode_run_noalloc, fa_decode_set_debug,
                      fa_decode_set_trace,
                      load_library)

__all__ = [
    "EXPORTED", "FA_DEBUG_FORCE_SIMT", "FA_DEBUG_SKIP_LOADS", "FA_DEBUG_TWO_CLUSTERS", "FA_DEBUG_NO_STREAM_K", "FA_TRACE_WORDS_PER_CTA", "FA_ERR_CUDA", "FA_NOALLOC_STATUS_SLOTS", "FA_ERR_DEVICE", "FA_ERR_INVALID_ARG",
    "FA_ERR_UNSUPPORTED", "FA_KV_BF16", "FA_KV_E4M3", "FA_OK", "FA_STATUS_BAD_PAGE", "FA_STATUS_TIMEOUT", "FaDecodeError",
    "fa_decode_check", "fa_decode_create", "fa_decode_create_kv", "fa_decode_describe", "fa_decode_destroy",
    "fa_decode_last_error", "fa_decode_run", "fa_decode_run_kv", "fa_decode_run_noalloc", "fa_decode_set_debug", "fa_decode_set_trace", "load_library",
]
