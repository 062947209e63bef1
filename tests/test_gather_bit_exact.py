"""Page gathering is bit-exact on every kernel path (GPU, through the C ABI).

Each (sequence, kv head) gets one dominant key (see dominant.py): every other
key's softmax weight underflows to exactly zero, so the output row of every
query that sees it must equal that key's V row bit for bit. The chosen keys
sit at key 0, at page ends and starts, at the sequence's last key in a partial
page, in every split rank's share of the tiles and at arbitrary in-page
offsets of later pages; every output is also compared with the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import split_paged_decode_gb300 as spd
from split_paged_decode_gb300.workloads import WORKLOADS, DecodeWorkload, generate

import dominant
from helpers import DeviceCall, check_against_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def library():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from split_paged_decode_gb300 import build

    build.build_library()
    spd.load_library()


def wl(**kw):
    base = dict(name="dominant", batch=6, num_q=1, num_q_heads=8, num_kv_heads=2, qk_depth=128, ov_depth=128,
                page_size=64, splitk=2, seq_len_lo=1, seq_len_hi=3000, seed=700)
    base.update(kw)
    return DecodeWorkload(**base)


def run_dominant(w, seq_lens=None, path="auto", splitk_of=None, salt=0, oracle_rows="all", expect_kernel=None):
    inp = generate(w, seq_lens=seq_lens)
    pos = dominant.choose_positions(w, inp.seq_lens.tolist(), splitk_of=splitk_of, salt=salt)
    dominant.plant(inp, pos)
    dominant.check_margin(inp, pos)
    with DeviceCall(inp, path=path) as call:
        if expect_kernel is not None:
            assert expect_kernel in call.describe(), call.describe()
        call.run()
        assert call.status() == 0
        n = dominant.check_bit_exact(call.out, inp, pos, what=f"{w.name} {path}")
        assert n > 0
        if oracle_rows == "all":
            check_against_oracle(call, what=f"{w.name} {path} oracle")
        elif oracle_rows == "dominant":
            check_against_oracle(call, rows=dominant.expected_rows(inp, pos), what=f"{w.name} {path} oracle")
    return n


LENS = [1, 130, 700, 2000, 129, 4097]


# --- head dim 128, GQA: the tcgen05 kernel (deep ring, fixed split) and the FMA kernel ------

@pytest.mark.parametrize("P", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("ps", [16, 64, 128, 256])
def test_tc_deep_ring(P, ps):
    run_dominant(wl(splitk=P, page_size=ps, seed=700 + P + ps), seq_lens=LENS, salt=P + ps)


@pytest.mark.parametrize("P", [2, 4])
@pytest.mark.parametrize("salt", [0, 3])
def test_tc_multi_unit_schedule(P, salt):
    """Two clusters, each working through many units in turn."""
    run_dominant(wl(batch=7, splitk=P, seed=710 + P), seq_lens=[0, 1, 130, 700, 129, 2000, 64], path="two_clusters",
                 salt=salt)


@pytest.mark.parametrize("P", [1, 2, 4, 8])
@pytest.mark.parametrize("ps", [32, 128])
def test_simt_d128(P, ps):
    run_dominant(wl(splitk=P, page_size=ps, seed=720 + P), seq_lens=LENS, path="simt", salt=P)


@pytest.mark.parametrize("g,T", [(4, 4), (16, 1), (1, 1), (8, 2)])
def test_rows_per_cta(g, T):
    run_dominant(wl(num_q_heads=2 * g, num_q=T, splitk=4, seed=730 + g * T), seq_lens=LENS, salt=g + T)


@pytest.mark.parametrize("frac", [0.0, 0.13, 0.5, 0.77, 0.999])
def test_stream_k(frac):
    """One or two long units cut over many clusters: the chosen key lands in
    clusters at different places of the units' key ranges."""
    w = wl(batch=2, num_kv_heads=1, num_q_heads=4, splitk=4, page_size=128, seed=740)
    lens = [20000, 9000]
    inp = generate(w, seq_lens=lens)
    pos = {(b, 0): int(frac * (L - 1)) for b, L in enumerate(lens)}
    dominant.plant(inp, pos)
    dominant.check_margin(inp, pos)
    with DeviceCall(inp) as call:
        call.run()
        assert call.status() == 0
        dominant.check_bit_exact(call.out, inp, pos, what=f"stream-K {frac}")
        check_against_oracle(call, what=f"stream-K {frac} oracle")


@pytest.mark.parametrize("path", ["auto", "simt"])
def test_per_sequence_split_causal(path):
    """splitk 0 (one cluster size per sequence, 16 causal rows per CTA)."""
    w = wl(batch=12, num_q=4, splitk=0, page_size=64, seed=750)
    lens = [1, 5, 1024, 1025, 4096, 4097, 8192, 9000, 64, 65, 2000, 3000]

    def split_of(L):
        return 1 if L <= 1024 else (2 if L <= 4096 else 4)

    run_dominant(w, seq_lens=lens, path=path, splitk_of=split_of)


@pytest.mark.parametrize("P", [1, 2])
def test_simt_d64(P):
    run_dominant(wl(qk_depth=64, ov_depth=64, num_q_heads=4, num_kv_heads=1, splitk=P, seed=760 + P),
                 seq_lens=LENS, salt=P)


# --- the MLA latent layout: V is the first 512 columns of the same row --------------------

def mla(**kw):
    base = dict(num_q_heads=128, num_kv_heads=1, qk_depth=576, nope_depth=512, ov_depth=512, latent=True,
                splitk=2, batch=4, page_size=64, scale=1.0 / np.sqrt(192.0), seed=770)
    base.update(kw)
    return wl(**base)


@pytest.mark.parametrize("P", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("ps", [32, 64, 128])
def test_mla_tensor_core(P, ps):
    run_dominant(mla(splitk=P, page_size=ps, seed=770 + P + ps), seq_lens=[700, 129, 2000, 1], salt=P + ps,
                 expect_kernel="mla_tc")


@pytest.mark.parametrize("P", [1, 2])
def test_mla_simt(P):
    run_dominant(mla(splitk=P, seed=780 + P), seq_lens=[700, 129, 300, 1], path="simt", salt=P)


def test_latent_simt_32_heads():
    """The latent layout with fewer heads than the MLA tensor-core kernel takes."""
    run_dominant(mla(num_q_heads=32, batch=3, splitk=2, seed=790), seq_lens=[300, 1, 129])


# --- the five workloads at full size, in the configuration the benchmark times -------------

@pytest.mark.parametrize("name", ["tiny", "batched_gqa", "long_context", "ragged_speculative", "mla"])
def test_workload_full_size(name):
    w = WORKLOADS[name]
    split_of = (lambda L: 1 if L <= 1024 else (2 if L <= 4096 else 4)) if w.splitk == 0 else None
    n = run_dominant(w, splitk_of=split_of, oracle_rows="dominant")
    assert n >= w.num_q_heads
