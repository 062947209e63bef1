"""The source hash that ties a stored ncu traffic figure to its kernel: each
kernel family hashes its own translation units and the local headers they
include, so a change to one kernel leaves the other kernels' figures valid,
and a comment edit leaves every hash unchanged."""
import os
import sys

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, REPO)

import bench  # noqa: E402


def test_kernel_names_map_to_their_translation_units():
    assert bench.kernel_units("void mla_tc_decode_kernel<1>(DecodeParams)") == ("kernel_mla_tc.cu",)
    assert bench.kernel_units("void tc_decode_kernel<6, 4, 0, 0>(DecodeParams)") == ("kernel_tc.cu",
                                                                                      "kernel_tc_fp8.cu")
    assert bench.kernel_units("simt_decode_kernel<64, 64, 64, 4, 4, false, false, 0>") == ("kernel_simt.cu",)
    assert bench.kernel_units("at::FillFunctor") is None


def test_each_family_hashes_its_own_include_closure():
    tc = bench.kernel_source_files(("kernel_tc.cu", "kernel_tc_fp8.cu"))
    mla = bench.kernel_source_files(("kernel_mla_tc.cu",))
    assert {"kernel_tc.cu", "kernel_tc_fp8.cu", "kernel_tc.cuh", "fa_decode_internal.h", "fa_decode.h"} <= set(tc)
    assert "kernel_mla_tc.cu" not in tc and "kernel_simt.cu" not in tc
    assert {"kernel_mla_tc.cu", "tcgen05.cuh", "fp8.cuh", "device_common.cuh"} <= set(mla)
    assert "kernel_tc.cuh" not in mla and "fa_decode_host.cu" not in mla
    assert bench.kernel_source_hash(("kernel_tc.cu", "kernel_tc_fp8.cu")) != bench.kernel_source_hash(
        ("kernel_mla_tc.cu",))


def test_comments_and_whitespace_do_not_count():
    a = "int x = 1; // one\n/* two */ int y = 2;\n"
    b = "int x = 1;\n\n   int y = 2; // other\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only('const char* s = "// not a comment";') != bench._code_only("const char* s = ;")
