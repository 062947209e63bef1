"""The allocation-free entry point (fa_decode_run_noalloc), on the GPU.

Some callers cannot call cudaMalloc: their device memory all comes from
their own pool or arena, or they run on a path that cannot afford an
allocation's implicit synchronisation. fa_decode_run_noalloc serves them by
reporting device status into a fixed, statically declared device array
instead of a per-handle allocation. This file checks, through the C ABI,
that two calls in a row give the same output as the regular
fa_decode_create / fa_decode_run path within the library's tolerance, and
that a status slot beyond the array is refused. It is named so that pytest
collects it last, and it works alone in a fresh process as well as after the
other tests (the static array keeps the previous call's contents, which the
entry point clears).
"""
import numpy as np
import pytest
import torch

import split_paged_decode_gb300 as spd
from split_paged_decode_gb300.workloads import DecodeWorkload, generate

from helpers import OUT_ATOL, OUT_RTOL, LSE_ATOL, DeviceCall

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from split_paged_decode_gb300 import build

    build.build_library()
    spd.load_library()


def _close(a, b):
    a = a.float().cpu().numpy().astype(np.float64)
    b = b.float().cpu().numpy().astype(np.float64)
    return np.all(np.abs(a - b) <= OUT_ATOL + OUT_RTOL * np.abs(b))


@pytest.mark.parametrize("kw", [
    dict(qk_depth=128, ov_depth=128, splitk=4),                  # tensor-core kernel, cluster of 4
    dict(qk_depth=64, ov_depth=64, splitk=2),                    # FMA kernel
    dict(qk_depth=128, ov_depth=128, splitk=0, num_q=2),         # per-sequence split, causal rows
])
def test_noalloc_matches_regular_entry_point_twice(kw):
    base = dict(name="noalloc", batch=4, num_q=1, num_q_heads=8, num_kv_heads=2, page_size=64,
                seq_len_lo=1, seq_len_hi=3000, seed=321)
    base.update(kw)
    w = DecodeWorkload(**base)
    inp = generate(w)
    with DeviceCall(inp) as ref:
        ref.run()
        assert ref.status() == 0
        args = (w.num_q_heads, w.num_kv_heads, w.qk_depth, w.nope_depth, w.ov_depth, w.page_size, w.num_q,
                w.splitk)
        for call in range(2):  # two calls in a row share (and reuse) the static status word
            out = torch.full_like(ref.out, float("nan"))
            lse = torch.full_like(ref.lse, float("nan"))
            st = spd.fa_decode_run_noalloc(*args, ref.q, ref.k, ref.v, ref.pt, ref.lens, inp.scale, out, lse,
                                           status_slot=call)
            assert st == 0
            assert _close(out, ref.out), f"call {call}: output differs from fa_decode_run"
            fin = torch.isfinite(ref.lse)
            assert torch.equal(torch.isfinite(lse), fin)
            assert torch.all((lse[fin] - ref.lse[fin]).abs() <= LSE_ATOL)


def test_noalloc_rejects_slot_beyond_array():
    inp = generate(DecodeWorkload(name="noalloc_slot", batch=1, num_q=1, num_q_heads=4, num_kv_heads=1,
                                  qk_depth=128, ov_depth=128, page_size=64, splitk=1, seq_len=64, seed=5))
    with DeviceCall(inp) as ref:
        w = inp.workload
        with pytest.raises(spd.FaDecodeError) as e:
            spd.fa_decode_run_noalloc(w.num_q_heads, w.num_kv_heads, 128, -1, 128, 64, 1, 1, ref.q, ref.k, ref.v,
                                      ref.pt, ref.lens, inp.scale, ref.out, ref.lse,
                                      status_slot=spd.FA_NOALLOC_STATUS_SLOTS)
        assert e.value.code == spd.FA_ERR_INVALID_ARG
