"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Bound: |out - ref| <= 1e-2 + 1e-2 |ref| element-wise on the bf16 output and
|lse - ref| <= 1e-3 on the fp32 log-sum-exp; the single-key case and page
permutations are checked bit for bit here, page gathering on every path in
test_gather_bit_exact.py.
"""
import numpy as np
import pytest
import torch

import split_paged_decode_gb300 as spd
from split_paged_decode_gb300.workloads import WORKLOADS, DecodeWorkload, generate

from helpers import DeviceCall, check_against_oracle, compare, ramp_keys, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from split_paged_decode_gb300 import build

    build.build_library()
    spd.load_library()


def wl(**kw):
    base = dict(name="case", batch=3, num_q=1, num_q_heads=8, num_kv_heads=2, qk_depth=128, ov_depth=128,
                page_size=64, splitk=2, seq_len_lo=1, seq_len_hi=700, seed=100)
    base.update(kw)
    return DecodeWorkload(**base)


def run_and_check(w, seq_lens=None, rows=None, what=None, path="auto"):
    inp = generate(w, seq_lens=seq_lens)
    with DeviceCall(inp, path=path) as call:
        call.run()
        assert call.status() == 0
        check_against_oracle(call, rows=rows, what=what or w.name)
        return call.out.cpu(), call.lse.cpu()


# --- small shapes: several tiles, ragged tails, empty partitions -----------------------

PATHS = ["auto", "simt"]  # auto takes the tcgen05 kernel for head dim 128 and <= 16 rows


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("P", [1, 2, 4, 8, 16])
def test_gqa_d128_splits(P, path):
    run_and_check(wl(splitk=P, seed=10 + P), what=f"d128 P{P} {path}", path=path)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("ps", [8, 16, 32, 64, 128, 256])
def test_page_sizes(ps, path):
    run_and_check(wl(page_size=ps, splitk=4, seed=20), what=f"ps{ps} {path}", path=path)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("g,T", [(1, 1), (2, 1), (4, 1), (8, 1), (16, 1), (4, 2), (4, 4), (2, 8), (1, 16)])
def test_rows_per_cta(g, T, path):
    run_and_check(wl(num_q_heads=2 * g, num_kv_heads=2, num_q=T, seed=30 + g * T), what=f"g{g} T{T} {path}",
                  path=path)


def test_tensor_core_path_is_selected():
    inp = generate(wl(seed=9))
    with DeviceCall(inp) as call:
        assert call.describe().startswith("path=tcgen05"), call.describe()
    with DeviceCall(generate(wl(qk_depth=64, ov_depth=64, seed=9))) as call:
        assert call.describe().startswith("path=simt"), call.describe()


@pytest.mark.parametrize("P", [1, 2, 4, 8])
def test_d64(P):
    run_and_check(wl(qk_depth=64, ov_depth=64, splitk=P, seed=40 + P), what=f"d64 P{P}")


@pytest.mark.parametrize("P", [1, 2, 4])
def test_latent_small(P):
    w = wl(num_q_heads=32, num_kv_heads=1, qk_depth=576, nope_depth=512, ov_depth=512, latent=True,
           splitk=P, batch=2, seq_len_hi=300, scale=1.0 / np.sqrt(192.0), seed=50 + P)
    run_and_check(w, what=f"latent P{P}")


def mla_wl(**kw):
    base = dict(num_q_heads=128, num_kv_heads=1, qk_depth=576, nope_depth=512, ov_depth=512, latent=True,
                splitk=2, batch=3, page_size=64, seq_len_lo=1, seq_len_hi=700, scale=1.0 / np.sqrt(192.0), seed=150)
    base.update(kw)
    return wl(**base)


def test_mla_tensor_core_path_is_selected():
    with DeviceCall(generate(mla_wl())) as call:
        d = call.describe()
        assert d.startswith("path=tcgen05") and "mla_tc" in d, d


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("P", [1, 2, 4, 8, 16])
def test_mla_splits(P, path):
    """MLA latent layout, 128 heads (two 64-head blocks), ragged lengths across tiles."""
    run_and_check(mla_wl(splitk=P, seed=150 + P), seq_lens=[700, 129, 2000], what=f"mla P{P} {path}", path=path)


@pytest.mark.parametrize("Hq,ps", [(64, 64), (256, 128), (128, 32), (128, 256)])
def test_mla_heads_and_pages(Hq, ps):
    run_and_check(mla_wl(num_q_heads=Hq, page_size=ps, seed=160 + Hq + ps), seq_lens=[1, 300, 1000],
                  what=f"mla Hq{Hq} ps{ps}")


def test_mla_short_and_empty():
    """Lengths 0 and 1, shorter than a tile and at tile edges; ranks without tiles."""
    run_and_check(mla_wl(batch=6, splitk=4, seed=170), seq_lens=[0, 1, 127, 128, 129, 255], what="mla short")


def test_mla_nonfinite_rows_past_the_sequence_do_not_leak():
    w = mla_wl(batch=3, splitk=2, seed=171)
    lens = [70, 200, 129]
    inp = generate(w, seq_lens=lens)
    for b, L in enumerate(lens):
        last = int(inp.page_table[b, (L - 1) // 64])
        inp.k_pages[last, :, L % 64:, :] = float("nan")
    with DeviceCall(inp) as call:
        call.run()
        assert call.status() == 0
        check_against_oracle(call, what="mla non-finite tails")


def test_latent_explicit_v_cache():
    """(576, 512) with a separate V cache uses the separate-V kernel."""
    w = wl(num_q_heads=16, num_kv_heads=1, qk_depth=576, nope_depth=512, ov_depth=512, latent=False,
           splitk=2, batch=2, seq_len_hi=200, seed=55)
    run_and_check(w, what="576/512 explicit V")


def test_v_equal_k_pointer_means_v_is_k_prefix():
    w = wl(splitk=2, seed=56)
    inp = generate(w)
    with DeviceCall(inp) as call:
        call.v = call.k  # same pointer: V rows are the K rows
        call.run()
        assert call.status() == 0
        inp.v_pages = None  # the oracle's latent layout with ov == qk
        check_against_oracle(call, what="v is k")


@pytest.mark.parametrize("path", PATHS)
def test_causal_short_sequences_and_empty(path):
    """Lengths 0, 1, below num_q and at tile edges; rows with no visible key give 0 / -inf."""
    w = wl(num_q=4, num_q_heads=8, num_kv_heads=2, batch=10, splitk=4, seed=60)
    run_and_check(w, seq_lens=[0, 1, 2, 3, 4, 63, 64, 65, 127, 129], what=f"short/empty {path}", path=path)


@pytest.mark.parametrize("path", PATHS)
def test_ragged_auto_split(path):
    w = wl(batch=12, num_q=4, splitk=0, seq_len_lo=1, seq_len_hi=9000, page_size=64, seed=61)
    run_and_check(w, seq_lens=[1, 5, 1024, 1025, 4096, 4097, 8192, 9000, 64, 65, 2000, 3000],
                  what=f"auto split {path}", path=path)


@pytest.mark.parametrize("path", PATHS)
def test_more_tiles_than_ranks_and_fewer(path):
    w = wl(batch=4, splitk=8, seed=62)
    run_and_check(w, seq_lens=[64, 65, 128 * 8 + 1, 128 * 17 - 3], what=f"tiles vs ranks {path}", path=path)


@pytest.mark.parametrize("path", PATHS)
def test_nonfinite_rows_past_the_sequence_do_not_leak(path):
    """Rows past L_b in a sequence's last page may hold anything (here NaN / inf):
    they must not reach the output."""
    w = wl(batch=3, splitk=2, page_size=64, seed=63)
    inp = generate(w, seq_lens=[70, 200, 129])
    for b, L in enumerate([70, 200, 129]):
        last = int(inp.page_table[b, (L - 1) // 64])
        inp.k_pages[last, :, L % 64:, :] = float("nan")
        inp.v_pages[last, :, L % 64:, :] = float("inf")
    with DeviceCall(inp, path=path) as call:
        call.run()
        assert call.status() == 0
        check_against_oracle(call, what=f"non-finite tails {path}")


# --- several (sequence, kv head) units per cluster ----------------------------------------

@pytest.mark.parametrize("P", [1, 2, 4, 8, 16])
def test_multi_unit_schedule(P):
    """Two clusters work through 2 x 7 units each, with empty sequences, sequences
    shorter than one tile per rank (ranks without tiles) and tails of every kind."""
    w = wl(batch=7, num_kv_heads=2, num_q_heads=8, splitk=P, page_size=64, seed=90 + P)
    lens = [0, 1, 130, 700, 129, 2000, 64]
    run_and_check(w, seq_lens=lens, what=f"multi-unit P{P}", path="two_clusters")


@pytest.mark.parametrize("g,T", [(1, 1), (4, 1), (8, 1), (4, 4), (16, 1)])
def test_multi_unit_rows(g, T):
    w = wl(batch=5, num_kv_heads=3, num_q_heads=3 * g, num_q=T, splitk=4, seed=95 + g * T)
    run_and_check(w, what=f"multi-unit g{g} T{T}", path="two_clusters")


def test_multi_unit_matches_one_unit_per_cluster_bitwise():
    """A unit's arithmetic does not depend on which cluster takes it."""
    inp = generate(wl(batch=6, splitk=4, seed=97))
    with DeviceCall(inp, path="no_stream_k") as one, DeviceCall(inp, path="two_clusters") as many:
        one.run()
        many.run()
        assert one.status() == 0 and many.status() == 0
        assert torch.equal(one.out, many.out)
        assert torch.equal(one.lse, many.lse)


def test_many_units_default_grid():
    """More units than resident clusters without any debug flag (the batched shape)."""
    w = wl(batch=40, num_kv_heads=8, num_q_heads=32, splitk=4, page_size=128, seq_len_lo=1, seq_len_hi=3000,
           seed=98)
    run_and_check(w, what="many units")


# --- stream-K partition: fewer units than resident clusters ----------------------------
# With a fixed split and fewer (sequence, kv head) units than clusters fit on
# the device, the units' key ranges (a full page-table row each) are laid end
# to end and cut into one equal range per resident cluster; a unit shared by
# several clusters is merged by the last of them through the handle's scratch.

@pytest.mark.parametrize("P", [1, 2, 4, 8])
def test_stream_k_long(P):
    w = wl(batch=1, splitk=P, seq_len=P * 4 * 128 * 6 + 77, seed=110 + P)  # 2 units over ~12 clusters
    run_and_check(w, what=f"stream-K P{P}")


def test_stream_k_empty_and_short():
    """Sequences of length 0 and 1 next to a long one: most of their clusters see no key."""
    w = wl(batch=3, num_kv_heads=1, num_q_heads=4, splitk=2, seq_len_lo=1, seq_len_hi=5000, seed=115)
    run_and_check(w, seq_lens=[0, 1, 5000], what="stream-K short")


def test_stream_k_sixteen():
    """One unit over 65541 keys: shared by the most clusters (16), a ragged last tile."""
    w = wl(batch=1, num_kv_heads=1, num_q_heads=4, splitk=4, page_size=128, seq_len=65541, seed=116)
    run_and_check(w, what="stream-K 16")


@pytest.mark.parametrize("g,T", [(4, 4), (16, 1), (8, 1)])
def test_stream_k_rows(g, T):
    w = wl(batch=2, num_kv_heads=1, num_q_heads=g, num_q=T, splitk=2, seq_len_lo=2000, seq_len_hi=6000,
           seed=117 + g)
    run_and_check(w, what=f"stream-K g{g} T{T}")


def test_stream_k_two_clusters():
    """Two clusters, one unit: each takes half of its range."""
    w = wl(batch=1, num_kv_heads=1, num_q_heads=4, splitk=4, seq_len=9000, seed=118)
    run_and_check(w, what="stream-K two clusters", path="two_clusters")


def test_stream_k_more_units_than_clusters():
    """Three units over two clusters (whole-unit rounds would be 2 against an
    equal share of 1.5): each range holds one whole unit and half of the
    middle one, which the two clusters merge through the scratch."""
    w = wl(batch=3, num_kv_heads=1, num_q_heads=4, splitk=4, seq_len_lo=3000, seq_len_hi=9000, seed=123)
    run_and_check(w, seq_lens=[9000, 8500, 9000], what="stream-K more units than clusters", path="two_clusters")
    run_and_check(w, seq_lens=[9000, 1, 4000], what="stream-K more units, short middle unit", path="two_clusters")


def test_stream_k_ranges_across_units():
    """Three units of unequal length over ~26 clusters: ranges that end in one
    unit and start in the next, and ranges past a short sequence's end."""
    w = wl(batch=3, num_kv_heads=1, num_q_heads=4, splitk=2, seq_len_lo=3000, seq_len_hi=9000, seed=121)
    run_and_check(w, seq_lens=[9000, 3000, 6001], what="stream-K across units")


def test_stream_k_repeat_bitwise():
    """The counts reset themselves and the chunk merge order is fixed: repeated
    runs give the same bits; one cluster per unit agrees within tolerance."""
    inp = generate(wl(batch=2, splitk=4, seq_len=20000, seed=119))
    with DeviceCall(inp) as call, DeviceCall(inp, path="no_stream_k") as one:
        call.run()
        assert call.status() == 0
        out0, lse0 = call.out.clone(), call.lse.clone()
        for _ in range(3):
            call.out.fill_(float("nan"))
            call.run()
            assert call.status() == 0
            assert torch.equal(call.out, out0) and torch.equal(call.lse, lse0)
        check_against_oracle(call, what="stream-K repeat")
        one.run()
        assert one.status() == 0
        assert torch.allclose(one.out.float(), out0.float(), atol=1e-2, rtol=1e-2)
        assert torch.allclose(one.lse, lse0, atol=1e-4)


def test_stream_k_after_timeout():
    """A stream-K launch that gives up leaves no count behind once checked."""
    inp = generate(wl(batch=1, splitk=2, seq_len=12000, seed=120))
    with DeviceCall(inp) as call:
        spd.fa_decode_set_debug(call.h, spd.FA_DEBUG_SKIP_LOADS, 20_000_000)  # 20 ms
        call.run()
        assert spd.fa_decode_check(call.h) & spd.FA_STATUS_TIMEOUT
        spd.fa_decode_set_debug(call.h, 0, 0)
        call.run()
        assert call.status() == 0
        check_against_oracle(call, what="stream-K after timeout")


# --- the five workloads at full size -----------------------------------------------------

@pytest.mark.parametrize("name", ["tiny", "batched_gqa", "long_context", "ragged_speculative", "mla"])
def test_workload_full_size(name):
    """Each workload at full size in the launch configuration the benchmark
    times, every output row compared with the oracle."""
    run_and_check(WORKLOADS[name], what=name)


@pytest.mark.parametrize("name", ["batched_gqa", "long_context", "ragged_speculative"])
def test_workload_full_size_simt(name):
    run_and_check(WORKLOADS[name], what=f"{name} simt", path="simt")


# --- bit-exact properties ----------------------------------------------------------------

def test_single_key_is_bit_exact():
    """One visible key: weight exp2(0) / 1 = 1, so out is that key's V row exactly."""
    w = wl(batch=4, splitk=2, seed=70)
    inp = generate(w, seq_lens=[1, 1, 1, 1])
    with DeviceCall(inp) as call:
        call.run()
        assert call.status() == 0
        out = call.out.cpu()
        for b in range(4):
            page = int(inp.page_table[b, 0])
            for h in range(8):
                assert torch.equal(out[b, 0, h], inp.v_pages[page, h // 4, 0]), (b, h)
        ref_out, ref_lse = run_oracle(inp)
        compare(out.float().numpy(), call.lse.cpu().numpy(), ref_out, ref_lse, "single key")


def test_page_permutation_is_bitwise_invariant():
    w = wl(batch=3, splitk=4, seed=71)
    inp = generate(w)
    with DeviceCall(inp) as call:
        call.run()
        out1, lse1 = call.out.clone(), call.lse.clone()
        perm = torch.randperm(inp.num_pages, generator=torch.Generator().manual_seed(5))
        k2 = torch.empty_like(inp.k_pages)
        v2 = torch.empty_like(inp.v_pages)
        k2[perm] = inp.k_pages
        v2[perm] = inp.v_pages
        pt = inp.page_table.clone()
        pt[pt >= 0] = perm[pt[pt >= 0].long()].to(torch.int32)
        call.k, call.v, call.pt = k2.cuda(), v2.cuda(), pt.cuda()
        call.run()
        assert call.status() == 0
        assert torch.equal(call.out, out1)
        assert torch.equal(call.lse, lse1)


def test_repeated_runs_are_deterministic():
    inp = generate(wl(splitk=4, seed=72))
    with DeviceCall(inp) as call:
        call.run()
        a = call.out.clone()
        call.run()
        assert torch.equal(call.out, a)


def test_side_stream():
    inp = generate(wl(splitk=2, seed=73))
    s = torch.cuda.Stream()
    with DeviceCall(inp) as call:
        with torch.cuda.stream(s):
            call.run(stream=s)
        s.synchronize()
        assert spd.fa_decode_check(call.h, s) == 0
        check_against_oracle(call, what="side stream")


# --- failure reporting without a fault ---------------------------------------------------

def test_bad_page_id_is_reported_not_faulted():
    w = wl(batch=3, splitk=2, seed=80)
    inp = generate(w)
    bad = inp.page_table.clone()
    bad[1, 0] = inp.num_pages + 1000  # out of range: read as zeros, flagged
    with DeviceCall(inp) as call:
        call.pt = bad.cuda()
        call.run()
        st = spd.fa_decode_check(call.h)
        assert st & spd.FA_STATUS_BAD_PAGE
        rows = [(b, 0, h) for b in (0, 2) for h in range(8)]  # untouched sequences stay right
        check_against_oracle(call, rows=rows, what="bad page neighbours")


def test_bounded_wait_times_out_and_context_survives():
    """With loads suppressed, every CTA's first wait runs out after the short
    limit and the kernel returns with FA_STATUS_TIMEOUT; the next run is normal."""
    inp = generate(wl(batch=2, splitk=2, seed=81))
    with DeviceCall(inp) as call:
        spd.fa_decode_set_debug(call.h, spd.FA_DEBUG_SKIP_LOADS, 20_000_000)  # 20 ms
        call.run()
        st = spd.fa_decode_check(call.h)
        assert st & spd.FA_STATUS_TIMEOUT
        spd.fa_decode_set_debug(call.h, 0, 0)
        call.run()
        assert call.status() == 0
        check_against_oracle(call, what="after timeout")


@pytest.mark.parametrize("P", [2, 4])
def test_mla_bounded_wait_times_out_and_context_survives(P):
    """The MLA kernel with loads suppressed: the first waits run out, a CTA
    that has given up announces nothing to its peers and their waits for it
    (ready, pushed partials) give up too; the status says timeout, and the next
    run on the same handle matches the oracle."""
    inp = generate(mla_wl(splitk=P, seed=180 + P))
    with DeviceCall(inp) as call:
        assert "mla_tc" in call.describe()
        spd.fa_decode_set_debug(call.h, spd.FA_DEBUG_SKIP_LOADS, 20_000_000)  # 20 ms
        call.run()
        st = spd.fa_decode_check(call.h)
        assert st & spd.FA_STATUS_TIMEOUT
        spd.fa_decode_set_debug(call.h, 0, 0)
        call.run()
        assert call.status() == 0
        check_against_oracle(call, what=f"mla P{P} after timeout")


def test_run_rejects_misaligned_pointer():
    inp = generate(wl(seed=82))
    with DeviceCall(inp) as call:
        with pytest.raises(spd.FaDecodeError) as e:
            spd.fa_decode_run(call.h, call.q.data_ptr() + 2, call.k, call.v, call.pt, call.lens, inp.scale,
                              call.out, call.lse, batch=3, max_pages_per_seq=call.pt.shape[1],
                              num_pages=call.k.shape[0])
        assert e.value.code == spd.FA_ERR_INVALID_ARG


# --- the per-sequence split in one launch, and programmatic dependent launch -------------

def _split_of(L):
    return 1 if L <= 1024 else (2 if L <= 4096 else 4)


@pytest.mark.parametrize("hkv,lens", [
    (1, [5000, 2000, 3000, 4000, 10, 20, 30, 40, 50]),        # 1 unit of split 4, 3 of 2, 5 of 1: idle CTAs
    (3, [100, 2500, 9000, 1024, 1025, 4096, 4097, 1]),        # odd kv heads
    (2, [1, 2, 3, 4, 5, 6, 7]),                               # split 1 only
    (2, [8000, 6000, 5000]),                                  # split 4 only
    (2, [0, 3000, 0, 700, 0]),                                # empty sequences between
])
def test_per_sequence_split_one_launch(hkv, lens):
    """4-CTA clusters serving one unit of split 4, two of split 2 or four of
    split 1, chosen on the device; groups that run out of units leave CTAs idle."""
    w = wl(batch=len(lens), num_q=4, num_q_heads=4 * hkv, num_kv_heads=hkv, splitk=0, seq_len_lo=1,
           seq_len_hi=9000, seed=190 + hkv)
    inp = generate(w, seq_lens=lens)
    with DeviceCall(inp) as call:
        assert "one launch" in call.describe(), call.describe()
        call.run()
        assert call.status() == 0
        check_against_oracle(call, what=f"one-launch split hkv{hkv}")


def test_one_launch_split_is_one_kernel():
    """The per-sequence split on the tensor-core path is one launch: the
    per-CTA trace (which holds the last launch of a call) shows an entry for
    exactly the 4 CTAs of every group of units, and no other."""
    lens = [5000, 2000, 3000, 10, 20, 30, 4097, 1025, 700]
    w = wl(batch=len(lens), num_q=4, num_q_heads=8, num_kv_heads=2, splitk=0, seq_len_lo=1, seq_len_hi=9000,
           seed=195)
    inp = generate(w, seq_lens=lens)
    H = w.num_kv_heads
    n = {P: sum(1 for L in lens if _split_of(L) == P) * H for P in (1, 2, 4)}
    groups = n[4] + (n[2] + 1) // 2 + (n[1] + 3) // 4
    with DeviceCall(inp) as call:
        ctas = 4 * w.batch * H
        buf = torch.zeros(ctas * spd.FA_TRACE_WORDS_PER_CTA, dtype=torch.int64, device="cuda")
        spd.fa_decode_set_trace(call.h, buf)
        call.run()
        assert call.status() == 0
        entered = int((buf.view(ctas, -1)[:, 0] > 0).sum())
        assert entered == 4 * groups, (entered, groups)
        spd.fa_decode_set_trace(call.h, None)
        check_against_oracle(call, what="one-launch split, traced")


@pytest.mark.parametrize("splitk", [4, 0])
def test_chained_launches_read_the_previous_output(splitk):
    """Programmatic dependent launch: a decode whose queries are the previous
    decode's output, enqueued back to back on one stream, reads that output
    only once it is complete."""
    w = wl(batch=6, num_q=1, num_q_heads=8, num_kv_heads=2, splitk=splitk, seq_len_lo=500, seq_len_hi=9000,
           seed=196 + splitk)
    inp = generate(w)
    with DeviceCall(inp) as a, DeviceCall(inp) as b:
        b.q = a.out  # [B, T, Hq, 128]: the first decode's output is the second's queries
        for _ in range(3):
            a.out.fill_(float("nan"))
            b.out.fill_(float("nan"))
            a.run()
            b.run()
            torch.cuda.synchronize()
            assert a.status() == 0 and b.status() == 0
            check_against_oracle(a, what="chain first")
            chained = generate(w)
            chained.q = a.out.cpu()
            b.inp = chained
            check_against_oracle(b, what="chain second")


RAMP_CASES = {
    # two softmax warpgroups, 4 rows, one unit per cluster
    "deep_4rows": (dict(batch=2, splitk=4, seq_len_lo=1500, seq_len_hi=2600, seed=130), "auto"),
    # 8 rows under the stream-K partition (2 units, fewer than the resident clusters)
    "stream_k_8rows": (dict(batch=1, num_q_heads=16, splitk=8, seq_len_lo=9000, seq_len_hi=9000, seed=131), "auto"),
    # two clusters, each working through several units in turn
    "multi_unit": (dict(batch=5, splitk=2, seq_len_lo=300, seq_len_hi=2600, seed=132), "two_clusters"),
    # 16 rows (4 tokens x group 4, causal) on the shallow ring, the per-sequence split in one launch
    "shallow_16rows": (dict(batch=4, num_q=4, splitk=0, seq_len_lo=100, seq_len_hi=3000, seed=133), "auto"),
}


@pytest.mark.parametrize("case", sorted(RAMP_CASES))
def test_running_max_moves_every_tile(case):
    """Scores that rise along the keys move every row's running max on nearly
    every tile, so the in-place rescale of the TMEM O fragment (after the
    fragment's previous product) runs on most tiles, against the oracle."""
    kw, path = RAMP_CASES[case]
    inp = ramp_keys(generate(wl(**kw)))
    with DeviceCall(inp, path=path) as call:
        call.run()
        assert call.status() == 0
        check_against_oracle(call, what=f"ramp {case}")
