"""The C ABI on the CPU: the library loads, exports what the header declares,
and rejects bad arguments on the host (no GPU needed, no compute calls)."""
import ctypes
import os
import re

import pytest

import split_paged_decode_gb300 as spd
from split_paged_decode_gb300 import build as spd_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    spd_build.build_library()
    return spd.load_library()


def declared_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if not f.endswith(".h"):
            continue
        text = open(os.path.join(inc, f)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(fa_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert set(spd.EXPORTED) <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_binding_names_match_header():
    assert set(declared_functions()) == set(spd.EXPORTED)


def declared_constants():
    consts = {}
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            for name, val in re.findall(r"^#define\s+(FA_\w+)\s+\(?(-?\d+)u?\)?", open(os.path.join(inc, f)).read(),
                                        flags=re.M):
                consts[name] = int(val)
    return consts


def test_binding_constants_match_header():
    """Every status, error, debug and size constant the header defines has the
    same value in the binding (the tests and callers use the binding's)."""
    consts = declared_constants()
    assert {"FA_OK", "FA_STATUS_TIMEOUT", "FA_DEBUG_NO_STREAM_K", "FA_TRACE_WORDS_PER_CTA"} <= set(consts)
    for name, val in consts.items():
        assert getattr(spd, name, None) == val, f"{name}: header {val}, binding {getattr(spd, name, None)}"


def _create(lib, *args):
    h = ctypes.c_void_p()
    rc = lib.fa_decode_create(ctypes.byref(h), *args)
    return rc, h


@pytest.mark.parametrize("args", [
    (0, 1, 128, -1, 128, 128, 1, 1),      # no heads
    (32, 6, 128, -1, 128, 128, 1, 1),     # heads not divisible
    (32, 8, 128, 200, 128, 128, 1, 1),    # nope > qk
    (32, 8, 128, -1, 128, 0, 1, 1),       # page size
    (32, 8, 128, -1, 128, 128, 0, 1),     # num_q
    (32, 8, 128, -1, 128, 128, 1, 3),     # splitk not a power of two
    (32, 8, 128, -1, 128, 128, 1, 32),    # splitk too large
])
def test_create_rejects_invalid_arguments(lib, args):
    rc, h = _create(lib, *args)
    assert rc == spd.FA_ERR_INVALID_ARG
    assert not h.value
    assert lib.fa_decode_last_error().decode()


@pytest.mark.parametrize("args", [
    (32, 8, 96, -1, 96, 128, 1, 1),       # depth pair not built
    (32, 8, 128, -1, 128, 20, 1, 1),      # page size not a multiple of 8
    (32, 8, 128, -1, 128, 96, 1, 1),      # page size and tile do not divide
    (4, 1, 64, -1, 64, 64, 1, 16),        # 64 / 16 = 4-column bands
    (40, 2, 128, -1, 128, 64, 1, 1),      # 20 rows, group not a multiple of 16
    (32, 8, 128, -1, 128, 64, 8, 1),      # 32 rows with num_q > 1
])
def test_create_rejects_unsupported_shapes(lib, args):
    rc, h = _create(lib, *args)
    assert rc == spd.FA_ERR_UNSUPPORTED, lib.fa_decode_last_error()
    assert not h.value


def test_null_handle_calls_fail_cleanly(lib):
    assert lib.fa_decode_run(None, None, None, None, None, None, 1.0, None, None, None, 1, 1, 1) \
        == spd.FA_ERR_INVALID_ARG
    assert lib.fa_decode_check(None, None, None) == spd.FA_ERR_INVALID_ARG
    assert lib.fa_decode_set_debug(None, 0, 0) == spd.FA_ERR_INVALID_ARG
    assert lib.fa_decode_describe(None, None, 0) == spd.FA_ERR_INVALID_ARG
    assert lib.fa_decode_destroy(None) == spd.FA_OK


def test_valid_create_without_gpu_reports_cuda_error(lib):
    """On a machine without a GB300 a valid shape fails at the device query."""
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rc, h = _create(lib, 32, 8, 128, -1, 128, 128, 1, 4)
    assert rc in (spd.FA_ERR_CUDA, spd.FA_ERR_UNSUPPORTED)
    assert not h.value


def test_trace_hook_rejects_null_handle(lib):
    """The trace hook (a profiling aid) validates on the host like every call."""
    assert lib.fa_decode_set_trace(None, None, 0) == spd.FA_ERR_INVALID_ARG
    with pytest.raises(spd.FaDecodeError):
        spd.fa_decode_set_trace(0, None)


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(FileNotFoundError):
        spd.load_library(str(tmp_path / "libfa_decode.so"))


def _create_kv(lib, *args):
    h = ctypes.c_void_p()
    rc = lib.fa_decode_create_kv(ctypes.byref(h), *args)
    return rc, h


@pytest.mark.parametrize("args, code", [
    ((32, 8, 128, -1, 128, 128, 1, 4, 2, 0), "FA_ERR_INVALID_ARG"),                  # unknown cache format
    ((32, 8, 128, -1, 128, 128, 1, 4, spd.FA_KV_BF16, 16), "FA_ERR_INVALID_ARG"),    # rope apart on a bf16 cache
    ((32, 8, 128, -1, 128, 128, 1, 4, spd.FA_KV_E4M3, 128), "FA_ERR_INVALID_ARG"),   # rope as wide as the row
    ((32, 8, 64, -1, 64, 64, 1, 2, spd.FA_KV_E4M3, 0), "FA_ERR_UNSUPPORTED"),        # E4M3 head dim 64
    ((128, 1, 576, 512, 512, 64, 1, 2, spd.FA_KV_E4M3, 32), "FA_ERR_UNSUPPORTED"),   # latent rope of 32
    ((8, 1, 576, 512, 512, 64, 1, 2, spd.FA_KV_E4M3, 64), "FA_ERR_UNSUPPORTED"),     # 8 heads: neither MLA kernel
])
def test_create_kv_rejects_on_the_host(lib, args, code):
    """Cache-format arguments and E4M3 shapes without a kernel are refused
    before any device query."""
    rc, h = _create_kv(lib, *args)
    assert rc == getattr(spd, code), lib.fa_decode_last_error()
    assert not h.value


@pytest.mark.parametrize("args", [
    (32, 8, 128, -1, 128, 128, 1, 4, spd.FA_KV_E4M3, 0),      # the GQA tcgen05 kernel
    (128, 1, 576, 512, 512, 64, 1, 2, spd.FA_KV_E4M3, 64),    # the MLA tcgen05 kernel, E4M3 mode
    (32, 1, 576, 512, 512, 64, 1, 2, spd.FA_KV_E4M3, 64),     # the FMA kernel, E4M3 latent mode
])
def test_create_kv_planned_shapes_reach_the_device_query(lib, args):
    """Shapes with an E4M3 kernel pass the host checks; without a GB300 the
    plan then fails at the device query."""
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rc, h = _create_kv(lib, *args)
    assert rc in (spd.FA_ERR_CUDA, spd.FA_ERR_UNSUPPORTED)
    assert "compute capability" in lib.fa_decode_last_error().decode() or rc == spd.FA_ERR_CUDA
    assert not h.value
