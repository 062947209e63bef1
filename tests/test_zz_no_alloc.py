"""The allocation-free entry point (fa_decode_run_noalloc), on the GPU.

Some callers cannot call cudaMalloc: their device memory all comes from
their own pool or arena, or they run on a path that cannot afford an
allocation's implicit synchronisation. fa_decode_run_noalloc serves them by
reporting device status into a fixed, statically declared device array
instead of a per-handle allocation. This file checks, through the C ABI:
two calls in a row against the fp64 oracle and against the regular
fa_decode_create / fa_decode_run path, within the library's tolerance; one
status slot reused by three calls (a fault reported, then a clean call that
must not see the old bits, then a call that only enqueues); and that a slot
beyond the array is refused. It is named so that pytest collects it last,
and it works alone in a fresh process as well as after the other tests (the
static array keeps the previous call's contents, which the entry point
clears before each launch).
"""
import numpy as np
import pytest
import torch

import split_paged_decode_gb300 as spd
from split_paged_decode_gb300.workloads import DecodeWorkload, generate

from helpers import LSE_ATOL, OUT_ATOL, OUT_RTOL, DeviceCall, check_against_oracle

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


class _NoAllocCall:
    """Output buffers for one fa_decode_run_noalloc call on the inputs of `ref`."""

    def __init__(self, ref: DeviceCall):
        self.inp = ref.inp
        self.out = torch.full_like(ref.out, float("nan"))
        self.lse = torch.full_like(ref.lse, float("nan"))


def _args(w):
    return (w.num_q_heads, w.num_kv_heads, w.qk_depth, w.nope_depth, w.ov_depth, w.page_size, w.num_q, w.splitk)


@pytest.mark.parametrize("kw", [
    dict(qk_depth=128, ov_depth=128, splitk=4),                  # tensor-core kernel, cluster of 4
    dict(qk_depth=64, ov_depth=64, splitk=2),                    # FMA kernel
    dict(qk_depth=128, ov_depth=128, splitk=0, num_q=2),         # per-sequence split, causal rows
])
def test_noalloc_matches_oracle_and_regular_entry_point_twice(kw):
    base = dict(name="noalloc", batch=4, num_q=1, num_q_heads=8, num_kv_heads=2, page_size=64,
                seq_len_lo=1, seq_len_hi=3000, seed=321)
    base.update(kw)
    w = DecodeWorkload(**base)
    inp = generate(w)
    with DeviceCall(inp) as ref:
        ref.run()
        assert ref.status() == 0
        for call in range(2):  # two calls in a row on the same status word
            c = _NoAllocCall(ref)
            st = spd.fa_decode_run_noalloc(*_args(w), ref.q, ref.k, ref.v, ref.pt, ref.lens, inp.scale, c.out,
                                           c.lse, status_slot=7)
            assert st == 0
            check_against_oracle(c, what=f"noalloc call {call}")
            assert _close(c.out, ref.out), f"call {call}: output differs from fa_decode_run"
            fin = torch.isfinite(ref.lse)
            assert torch.equal(torch.isfinite(c.lse), fin)
            assert torch.all((c.lse[fin] - ref.lse[fin]).abs() <= LSE_ATOL)


def test_noalloc_one_slot_fault_then_clean_then_enqueue_only():
    """The status word of a slot keeps what the previous call left; each call
    clears it first, so a clean call after a reported fault reports nothing."""
    w = DecodeWorkload(name="noalloc_slot", batch=3, num_q=1, num_q_heads=8, num_kv_heads=2, qk_depth=128,
                       ov_depth=128, page_size=64, splitk=2, seq_len_lo=1, seq_len_hi=700, seed=80)
    inp = generate(w)
    slot = 11
    with DeviceCall(inp) as ref:
        # 1. an out-of-range page id: read as zeros, flagged, never a fault
        bad = inp.page_table.clone()
        bad[1, 0] = inp.num_pages + 1000
        c = _NoAllocCall(ref)
        with pytest.raises(spd.FaDecodeError) as e:
            spd.fa_decode_run_noalloc(*_args(w), ref.q, ref.k, ref.v, bad.cuda(), ref.lens, inp.scale, c.out,
                                      c.lse, status_slot=slot)
        assert e.value.code == spd.FA_ERR_DEVICE
        assert e.value.status & spd.FA_STATUS_BAD_PAGE
        rows = [(b, 0, h) for b in (0, 2) for h in range(8)]  # untouched sequences stay right
        check_against_oracle(c, rows=rows, what="noalloc bad page neighbours")
        # 2. a clean call on the same slot reports nothing
        c = _NoAllocCall(ref)
        assert spd.fa_decode_run_noalloc(*_args(w), ref.q, ref.k, ref.v, ref.pt, ref.lens, inp.scale, c.out,
                                         c.lse, status_slot=slot) == 0
        check_against_oracle(c, what="noalloc after a fault")
        # 3. enqueue only (no status read), on a side stream, then synchronise
        c = _NoAllocCall(ref)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        assert spd.fa_decode_run_noalloc(*_args(w), ref.q, ref.k, ref.v, ref.pt, ref.lens, inp.scale, c.out,
                                         c.lse, stream=s, status_slot=slot, wait=False) is None
        s.synchronize()
        check_against_oracle(c, what="noalloc enqueue only")


def test_noalloc_rejects_slot_beyond_array():
    inp = generate(DecodeWorkload(name="noalloc_slot", batch=1, num_q=1, num_q_heads=4, num_kv_heads=1,
                                  qk_depth=128, ov_depth=128, page_size=64, splitk=1, seq_len=64, seed=5))
    with DeviceCall(inp) as ref:
        w = inp.workload
        for slot in (-1, spd.FA_NOALLOC_STATUS_SLOTS):
            with pytest.raises(spd.FaDecodeError) as e:
                spd.fa_decode_run_noalloc(w.num_q_heads, w.num_kv_heads, 128, -1, 128, 64, 1, 1, ref.q, ref.k,
                                          ref.v, ref.pt, ref.lens, inp.scale, ref.out, ref.lse, status_slot=slot)
            assert e.value.code == spd.FA_ERR_INVALID_ARG
