"""The fp8 (OCP E4M3) cache on the GPU, through the C ABI, against the fp64
fp8 oracle (oracle_decode_fp8).

The kernel reads E4M3 K and V tiles and an optional per-token K scale; its
arithmetic error is bounded like the bf16 path's (Q and P are carried as two
E4M3 operands each, ~8 bits), so the bound is the same:
|out - ref| <= 1e-2 + 1e-2 |ref| and |lse - ref| <= 1e-3. Page gathering is
checked bit for bit with dominant keys (see dominant.py).
"""
import pytest
import torch

import split_paged_decode_gb300 as spd
from split_paged_decode_gb300.workloads import WORKLOADS, DecodeWorkload, generate

import dominant
from helpers import DeviceCall, check_against_oracle, ramp_keys

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from split_paged_decode_gb300 import build

    build.build_library()
    spd.load_library()


def wl(**kw):
    base = dict(name="fp8", batch=3, num_q=1, num_q_heads=8, num_kv_heads=2, qk_depth=128, ov_depth=128,
                page_size=64, splitk=2, seq_len_lo=1, seq_len_hi=700, seed=900, kv_dtype="e4m3", k_scale=True)
    base.update(kw)
    return DecodeWorkload(**base)


def run_and_check(w, seq_lens=None, path="auto", what=""):
    inp = generate(w, seq_lens=seq_lens)
    with DeviceCall(inp, path=path) as call:
        assert "e4m3" in call.describe(), call.describe()
        call.run()
        assert call.status() == 0
        check_against_oracle(call, what=what or w.name)


@pytest.mark.parametrize("scaled", [True, False])
@pytest.mark.parametrize("P", [1, 2, 4, 8, 16])
def test_splits(P, scaled):
    run_and_check(wl(splitk=P, k_scale=scaled, seed=900 + P), what=f"fp8 P{P} scale {scaled}")


@pytest.mark.parametrize("ps", [8, 16, 32, 128, 256])
def test_page_sizes(ps):
    run_and_check(wl(page_size=ps, splitk=4, seed=910 + ps), what=f"fp8 ps{ps}")


@pytest.mark.parametrize("g,T", [(1, 1), (4, 1), (8, 1), (16, 1), (4, 4), (2, 8)])
def test_rows_per_cta(g, T):
    run_and_check(wl(num_q_heads=2 * g, num_q=T, splitk=4, seed=920 + g * T), what=f"fp8 g{g} T{T}")


def test_causal_short_and_empty():
    w = wl(num_q=4, batch=10, splitk=4, seed=930)
    run_and_check(w, seq_lens=[0, 1, 2, 3, 4, 63, 64, 65, 127, 129], what="fp8 short/empty")


@pytest.mark.parametrize("P", [2, 4, 16])
def test_multi_unit_schedule(P):
    w = wl(batch=7, splitk=P, seed=940 + P)
    run_and_check(w, seq_lens=[0, 1, 130, 700, 129, 2000, 64], path="two_clusters", what=f"fp8 multi-unit P{P}")


@pytest.mark.parametrize("P", [1, 4, 8])
def test_stream_k(P):
    w = wl(batch=2, num_kv_heads=1, num_q_heads=4, splitk=P, seq_len_lo=9000, seq_len_hi=20000, seed=950 + P)
    run_and_check(w, what=f"fp8 stream-K P{P}")


def test_per_sequence_split():
    w = wl(batch=12, num_q=4, splitk=0, seed=960)
    run_and_check(w, seq_lens=[1, 5, 1024, 1025, 4096, 4097, 8192, 9000, 64, 65, 2000, 3000], what="fp8 auto split")


def test_nonfinite_codes_and_scales_past_the_sequence_do_not_leak():
    w = wl(batch=3, splitk=2, seed=970)
    lens = [70, 200, 129]
    inp = generate(w, seq_lens=lens)
    for b, L in enumerate(lens):
        last = int(inp.page_table[b, (L - 1) // 64])
        inp.k_pages[last, :, L % 64:, :] = 0x7F   # NaN code
        inp.v_pages[last, :, L % 64:, :] = 0xFF
        inp.k_scale[last, :, L % 64:] = float("nan")
    with DeviceCall(inp) as call:
        call.run()
        assert call.status() == 0
        check_against_oracle(call, what="fp8 non-finite tails")


def test_bad_page_id_is_reported_not_faulted():
    inp = generate(wl(batch=3, splitk=2, seed=980))
    bad = inp.page_table.clone()
    bad[1, 0] = inp.num_pages + 1000
    with DeviceCall(inp) as call:
        call.pt = bad.cuda()
        call.run()
        assert spd.fa_decode_check(call.h) & spd.FA_STATUS_BAD_PAGE
        rows = [(b, 0, h) for b in (0, 2) for h in range(8)]
        check_against_oracle(call, rows=rows, what="fp8 bad page neighbours")


def test_timeout_and_recovery():
    inp = generate(wl(batch=2, splitk=2, seed=981))
    with DeviceCall(inp) as call:
        spd.fa_decode_set_debug(call.h, spd.FA_DEBUG_SKIP_LOADS, 20_000_000)
        call.run()
        assert spd.fa_decode_check(call.h) & spd.FA_STATUS_TIMEOUT
        spd.fa_decode_set_debug(call.h, 0, 0)
        call.run()
        assert call.status() == 0
        check_against_oracle(call, what="fp8 after timeout")


def test_bf16_entry_point_refuses_an_e4m3_handle():
    inp = generate(wl(seed=982))
    with DeviceCall(inp) as call:
        with pytest.raises(spd.FaDecodeError) as e:
            spd.fa_decode_run(call.h, call.q, call.k, call.v, call.pt, call.lens, inp.scale, call.out, call.lse)
        assert e.value.code == spd.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("scaled", [True, False])
@pytest.mark.parametrize("P,ps,path", [(1, 64, "auto"), (4, 16, "auto"), (8, 128, "auto"), (16, 256, "auto"),
                                       (4, 64, "two_clusters")])
def test_gather_bit_exact(P, ps, path, scaled):
    w = wl(batch=6, splitk=P, page_size=ps, seq_len_lo=1, seq_len_hi=3000, k_scale=scaled, seed=990 + P + ps)
    inp = generate(w, seq_lens=[1, 130, 700, 2000, 129, 4097])
    pos = dominant.choose_positions(w, inp.seq_lens.tolist(), salt=P + ps)
    dominant.plant(inp, pos)
    dominant.check_margin(inp, pos)
    with DeviceCall(inp, path=path) as call:
        call.run()
        assert call.status() == 0
        dominant.check_bit_exact(call.out, inp, pos, what=f"fp8 gather P{P} ps{ps} {path}")
        check_against_oracle(call, what=f"fp8 gather P{P} ps{ps} oracle")


@pytest.mark.parametrize("name", ["batched_gqa", "long_context", "ragged_speculative"])
def test_workload_full_size(name):
    """The head-dim-128 workloads with an E4M3 cache and per-token K scales."""
    w = WORKLOADS[name].with_(kv_dtype="e4m3", k_scale=True)
    run_and_check(w, what=f"{name} e4m3")


@pytest.mark.parametrize("case, kw, path", [
    ("deep_4rows", dict(batch=2, splitk=4, seq_len_lo=1500, seq_len_hi=2600, seed=980), "auto"),
    ("multi_unit", dict(batch=7, splitk=2, seq_len_lo=300, seq_len_hi=2600, seed=981), "two_clusters"),
    ("stream_k_8rows", dict(batch=1, num_q_heads=16, splitk=8, seq_len_lo=9000, seq_len_hi=9000, seed=982), "auto"),
    ("shallow_16rows", dict(batch=4, num_q=4, splitk=0, seq_len_lo=100, seq_len_hi=3000, seed=983), "auto"),
])
def test_running_max_moves_every_tile(case, kw, path):
    """The fp8 kernel's rescale path on most tiles (threshold 2^4): scores rising
    along the keys, against the fp8 oracle."""
    inp = ramp_keys(generate(wl(**kw)))
    with DeviceCall(inp, path=path) as call:
        assert "e4m3" in call.describe(), call.describe()
        call.run()
        assert call.status() == 0
        check_against_oracle(call, what=f"fp8 ramp {case}")


# --- the MLA latent layout over an E4M3 cache with a bf16 rope cache ---------
# K_j = [k_scale_j * e4m3(k8_j[0:512]), bf16 rope_j[0:64]] and V_j =
# k_scale_j * e4m3(k8_j[0:512]): the FA4Config page's separate rope dtype and
# per-token K scale. A multiple of 64 heads per kv head takes the tcgen05 MLA
# kernel (64 heads per CTA), fewer the FMA kernel (16 heads per CTA).

def mla_wl(**kw):
    base = dict(name="fp8_mla", batch=3, num_q=1, num_q_heads=64, num_kv_heads=1, qk_depth=576, nope_depth=512,
                ov_depth=512, page_size=64, splitk=2, seq_len_lo=1, seq_len_hi=700, latent=True,
                scale=1.0 / 24.0, seed=1100, kv_dtype="e4m3", k_scale=True, rope_depth=64)
    base.update(kw)
    return DecodeWorkload(**base)


def expect_kernel(call, heads_per_kv, path="auto"):
    """The description names the default kernel; a forced FMA run needs its latent kernel."""
    d = call.describe()
    if path == "simt":
        assert "latent_kernel=simt_e4m3" in d, d
    else:
        assert ("kernel=mla_tc_e4m3" in d) == (heads_per_kv % 64 == 0), d


@pytest.mark.parametrize("heads", [32, 64, 128])
@pytest.mark.parametrize("scaled", [True, False])
@pytest.mark.parametrize("P", [1, 2, 4, 16])
def test_mla_latent_rope_splits(P, scaled, heads):
    w = mla_wl(splitk=P, k_scale=scaled, num_q_heads=heads, seed=1100 + P + heads)
    inp = generate(w, seq_lens=[1, 333, 700])
    with DeviceCall(inp) as call:
        expect_kernel(call, heads)
        call.run()
        assert call.status() == 0
        check_against_oracle(call, what=f"fp8 mla P{P} scale {scaled} heads {heads}")


@pytest.mark.parametrize("path", ["auto", "simt"])
@pytest.mark.parametrize("ps", [8, 32, 128])
def test_mla_latent_rope_page_sizes(ps, path):
    inp = generate(mla_wl(page_size=ps, splitk=4, seed=1120 + ps), seq_lens=[65, 1000, 257])
    with DeviceCall(inp, path=path) as call:
        expect_kernel(call, 64, path)
        call.run()
        assert call.status() == 0
        check_against_oracle(call, what=f"fp8 mla ps{ps} {path}")


@pytest.mark.parametrize("heads", [16, 64])
def test_mla_latent_rope_per_sequence_split_and_short(heads):
    w = mla_wl(batch=8, num_q_heads=heads, splitk=0, seed=1130 + heads)
    run_and_check(w, seq_lens=[0, 1, 31, 32, 33, 1100, 4097, 9000], what=f"fp8 mla auto split heads {heads}")


@pytest.mark.parametrize("heads", [32, 64])
def test_mla_latent_rope_nonfinite_tails_do_not_leak(heads):
    w = mla_wl(batch=3, splitk=2, num_q_heads=heads, seed=1140 + heads)
    lens = [70, 200, 129]
    inp = generate(w, seq_lens=lens)
    for b, L in enumerate(lens):
        last = int(inp.page_table[b, (L - 1) // 64])
        inp.k_pages[last, :, L % 64:, :] = 0x7F   # NaN code
        inp.k_rope[last, :, L % 64:, :] = float("nan")
        inp.k_scale[last, :, L % 64:] = float("nan")
    with DeviceCall(inp) as call:
        call.run()
        assert call.status() == 0
        check_against_oracle(call, what=f"fp8 mla non-finite tails heads {heads}")


@pytest.mark.parametrize("P", [1, 4])
def test_mla_latent_rope_scale_bound_moves(P):
    """K scales that change along the sequence (x2 every 128 keys, up to x32,
    then back to x1) with the codes divided by the same factor, so the keys
    keep their magnitudes: the tcgen05 kernel moves its bound on the scales
    folded into P up and down mid-sequence and corrects O, against the oracle."""
    w = mla_wl(batch=2, splitk=P, seed=1160 + P)
    lens = [1500, 2300]
    inp = generate(w, seq_lens=lens)
    ps = w.page_size
    for b, L in enumerate(lens):
        for key in range(L):
            page, row = int(inp.page_table[b, key // ps]), key % ps
            f = float(2 ** ((key // 128) % 6))
            inp.k_scale[page, :, row] *= f
            codes = inp.k_pages[page, :, row, :].view(torch.float8_e4m3fn).float() / f
            inp.k_pages[page, :, row, :] = codes.to(torch.float8_e4m3fn).view(torch.uint8)
    with DeviceCall(inp) as call:
        expect_kernel(call, 64)
        call.run()
        assert call.status() == 0
        check_against_oracle(call, what=f"fp8 mla changing scales P{P}")


@pytest.mark.parametrize("P", [2, 4])
def test_mla_latent_rope_running_max_moves_every_tile(P):
    """Scores rising along the keys: the rescale path (threshold 2^4 for the
    E4M3 P split) on most tiles."""
    inp = ramp_keys(generate(mla_wl(batch=2, splitk=P, seed=1170 + P), seq_lens=[1800, 2600]))
    with DeviceCall(inp) as call:
        expect_kernel(call, 64)
        call.run()
        assert call.status() == 0
        check_against_oracle(call, what=f"fp8 mla ramp P{P}")


@pytest.mark.parametrize("path", ["auto", "simt"])
def test_mla_latent_rope_full_size(path):
    """The mla workload (32 seqs x 128 heads, L8192, split 2) over the E4M3 latent cache."""
    w = WORKLOADS["mla"].with_(kv_dtype="e4m3", k_scale=True, rope_depth=64)
    inp = generate(w)
    with DeviceCall(inp, path=path) as call:
        expect_kernel(call, 128, path)
        call.run()
        assert call.status() == 0
        check_against_oracle(call, what=f"mla e4m3 {path}")


@pytest.mark.parametrize("heads,P,ps,path", [(64, 1, 64, "auto"), (64, 2, 16, "auto"), (128, 4, 128, "auto"),
                                         (64, 16, 64, "auto"), (64, 4, 32, "simt"), (32, 2, 64, "auto")])
def test_mla_latent_rope_gather_bit_exact(heads, P, ps, path):
    """Dominant keys (the bf16 rope part of the chosen row, K scale 0.25):
    every output row that sees its key equals 0.25 * codes[:512] of that row
    bit for bit, on the tcgen05 E4M3 mode and on the FMA kernel."""
    w = mla_wl(batch=6, splitk=P, page_size=ps, num_q_heads=heads, seed=1180 + P + ps + heads)
    inp = generate(w, seq_lens=[1, 130, 700, 2000, 129, 4097])
    pos = dominant.choose_positions(w, inp.seq_lens.tolist(), salt=P + ps)
    dominant.plant(inp, pos)
    dominant.check_margin(inp, pos)
    with DeviceCall(inp, path=path) as call:
        expect_kernel(call, heads, path)
        call.run()
        assert call.status() == 0
        n = dominant.check_bit_exact(call.out, inp, pos, what=f"fp8 mla gather heads {heads} P{P} ps{ps} {path}")
        assert n > 0
        check_against_oracle(call, what=f"fp8 mla gather heads {heads} P{P} ps{ps} {path} oracle")


def test_mla_latent_rope_argument_checks():
    inp = generate(mla_wl(seed=1150))
    with DeviceCall(inp) as call:
        # no rope cache; a separate V cache (a copy: the same pointer would read as the latent layout)
        for rope, v, code in [(None, None, spd.FA_ERR_INVALID_ARG), (call.rope, call.k.clone(), spd.FA_ERR_UNSUPPORTED)]:
            with pytest.raises(spd.FaDecodeError) as e:
                spd.fa_decode_run_kv(call.h, call.q, call.k, v, rope, call.ks, call.pt, call.lens, inp.scale,
                                     call.out, call.lse)
            assert e.value.code == code, e.value
