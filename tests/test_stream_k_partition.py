"""The stream-K partition's arithmetic (fa_decode_internal.h, stream_k_plan.h),
checked on the host: a small C++ program built against the same headers the
kernels and the planner include (see tests/stream_k_partition.cpp for the
properties)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA_INCLUDE = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")


def test_stream_k_partition(tmp_path):
    cxx = shutil.which("g++")
    if cxx is None or not os.path.exists(os.path.join(CUDA_INCLUDE, "cuda.h")):
        pytest.skip("g++ or the CUDA headers are missing")
    exe = str(tmp_path / "stream_k_partition")
    subprocess.run([cxx, "-std=c++17", "-O2", "-I", os.path.join(ROOT, "include"), "-I",
                    os.path.join(ROOT, "split_paged_decode_gb300", "csrc"), "-I", CUDA_INCLUDE,
                    os.path.join(ROOT, "tests", "stream_k_partition.cpp"), "-o", exe], check=True)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0 and out.stdout.startswith("ok "), out.stdout + out.stderr
