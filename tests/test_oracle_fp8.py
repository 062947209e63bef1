"""Pins of the fp8-cache oracle (oracle_decode_fp8) against facts it does not
compute itself (CPU only).

The fp8 cache (FA4Config page: struct parameters qkv_dtype, rope_dtype_,
scale_dtype_) stores OCP FP8 E4M3 codes, an optional per-token fp32 K scale
and, for the latent layout, a rope part kept in bf16 in its own cache. The
pins: the code table against torch's float8_e4m3fn; reduction to the pinned
bf16 oracle wherever the fp8 cache is exactly a bf16 cache (unit scales, and
every E4M3 value is a bf16 value); a power-of-two scale equals a scaled
softmax; an independent NumPy / SciPy brute force with varying scales, the
rope part, the latent V, causal rows and small pages; masked rows never read.
"""
import math

import numpy as np
import pytest
import torch
from scipy.special import logsumexp, softmax

import oracle
from split_paged_decode_gb300.workloads import DecodeWorkload, bf16_bits, generate

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def fp8(**kw):
    base = dict(name="pin8", batch=3, num_q=1, num_q_heads=8, num_kv_heads=2, qk_depth=32, ov_depth=32,
                page_size=16, splitk=1, seq_len_lo=1, seq_len_hi=100, seed=31, kv_dtype="e4m3")
    base.update(kw)
    return DecodeWorkload(**base)


def latent(**kw):
    base = dict(num_q_heads=8, num_kv_heads=1, qk_depth=40, nope_depth=32, ov_depth=32, latent=True,
                rope_depth=8, k_scale=True, scale=0.2)
    base.update(kw)
    return fp8(**base)


def run_fp8(inp, **kw):
    w = inp.workload
    return oracle.decode_fp8(bf16_bits(inp.q), inp.k_pages.numpy(),
                             None if inp.v_pages is None else inp.v_pages.numpy(), inp.page_table.numpy(),
                             inp.seq_lens.numpy(), inp.scale,
                             k_rope=None if inp.k_rope is None else bf16_bits(inp.k_rope),
                             k_scale=None if inp.k_scale is None else inp.k_scale.numpy(), ov_depth=w.ov_depth,
                             **kw)


def e4m3_f64(codes: torch.Tensor) -> np.ndarray:
    """E4M3 codes widened by torch's own float8 type (a library routine)."""
    return codes.contiguous().view(torch.float8_e4m3fn).to(torch.float64).numpy()


def brute_force(inp):
    """Dense gather in NumPy of the dequantized rows, SciPy softmax per query."""
    w = inp.workload
    q = inp.q.to(torch.float64).numpy()
    K8 = e4m3_f64(inp.k_pages)
    ks = np.ones(K8.shape[:3]) if inp.k_scale is None else inp.k_scale.to(torch.float64).numpy()
    Kf = K8 * ks[..., None]
    K = Kf if inp.k_rope is None else np.concatenate([Kf, inp.k_rope.to(torch.float64).numpy()], axis=3)
    V = Kf[..., : w.ov_depth] if inp.v_pages is None else e4m3_f64(inp.v_pages)
    pt = inp.page_table.numpy()
    B, T, Hq, _ = q.shape
    g = w.num_q_heads // w.num_kv_heads
    out = np.zeros((B, T, Hq, w.ov_depth))
    lse = np.full((B, T, Hq), -np.inf)
    for b in range(B):
        L = int(inp.seq_lens[b])
        j = np.arange(L)
        phys = pt[b, j // w.page_size]
        for h in range(Hq):
            kv = h // g
            Kd = K[phys, kv, j % w.page_size]
            Vd = V[phys, kv, j % w.page_size]
            for t in range(T):
                n = L - T + t + 1
                if n <= 0:
                    continue
                s = inp.scale * (Kd[:n] @ q[b, t, h])
                out[b, t, h] = softmax(s) @ Vd[:n]
                lse[b, t, h] = logsumexp(s)
    return out, lse


def close(a, b, tol=1e-12):
    fin = np.isfinite(b)
    assert np.array_equal(np.isfinite(a), fin)
    assert np.all(a[~fin] == b[~fin])
    np.testing.assert_allclose(a[fin], b[fin], rtol=tol, atol=tol)


def test_code_table_matches_torch_float8():
    for code in range(256):
        ref = float(e4m3_f64(torch.tensor([code], dtype=torch.uint8))[0])
        got = oracle.e4m3_value(code)
        if math.isnan(ref):
            assert math.isnan(got), code
        else:
            assert got == ref, (code, got, ref)
    # the format's landmarks: 1.0, the largest finite value, the smallest subnormal, NaN
    assert oracle.e4m3_value(0x38) == 1.0 and oracle.e4m3_value(0x7E) == 448.0
    assert oracle.e4m3_value(0x01) == 2.0 ** -9 and oracle.e4m3_value(0x81) == -(2.0 ** -9)
    assert math.isnan(oracle.e4m3_value(0x7F)) and math.isnan(oracle.e4m3_value(0xFF))


def _as_bf16_cache(inp):
    """The same cache with every E4M3 code widened to bf16 (exact)."""
    k = inp.k_pages.view(torch.float8_e4m3fn).to(torch.bfloat16)
    v = None if inp.v_pages is None else inp.v_pages.view(torch.float8_e4m3fn).to(torch.bfloat16)
    if inp.k_rope is not None:
        k = torch.cat([k, inp.k_rope], dim=3)
    return k, v


@pytest.mark.parametrize("kw", [dict(), dict(num_q=4), dict(num_q_heads=2, num_kv_heads=2, page_size=8)])
def test_unit_scale_reduces_to_the_bf16_oracle_bitwise(kw):
    inp = generate(fp8(**kw))
    k, v = _as_bf16_cache(inp)
    ref = oracle.decode(bf16_bits(inp.q), bf16_bits(k), bf16_bits(v), inp.page_table.numpy(),
                        inp.seq_lens.numpy(), inp.scale)
    got = run_fp8(inp)
    assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])


def test_latent_rope_with_unit_scale_reduces_to_the_bf16_latent_oracle_bitwise():
    inp = generate(latent(k_scale=False))
    k, _ = _as_bf16_cache(inp)
    ref = oracle.decode(bf16_bits(inp.q), bf16_bits(k), None, inp.page_table.numpy(), inp.seq_lens.numpy(),
                        inp.scale, ov_depth=32)
    got = run_fp8(inp)
    assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])


@pytest.mark.parametrize("c", [0.25, 4.0])
def test_constant_power_of_two_scale_is_a_scaled_softmax(c):
    """K_j = c * e4m3(k8_j) for every j: s_j = (scale * c) q.e4m3(k8_j), exactly."""
    inp = generate(fp8(seed=33))
    base = run_fp8(inp)
    inp.k_scale = torch.full(inp.k_pages.shape[:3], c, dtype=torch.float32)
    got = run_fp8(inp)
    inp.k_scale = None
    inp.scale = inp.scale * c
    ref = run_fp8(inp)
    assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])
    assert not np.array_equal(got[0], base[0])


@pytest.mark.parametrize("w", [
    fp8(k_scale=True, seed=34),
    fp8(k_scale=True, num_q=4, seq_len_lo=1, seq_len_hi=60, seed=35),
    fp8(k_scale=True, num_q_heads=4, num_kv_heads=4, page_size=8, qk_depth=16, ov_depth=24, seed=36),
    latent(seed=37),
    latent(num_q=2, k_scale=False, seed=38),
    latent(page_size=8, num_q_heads=4, seed=39),
])
def test_brute_force(w):
    inp = generate(w)
    got = run_fp8(inp)
    ref = brute_force(inp)
    close(got[0], ref[0])
    close(got[1], ref[1])


def test_masked_rows_are_never_read():
    """Rows past L_b and spare pages may hold NaN codes and NaN scales."""
    inp = generate(fp8(k_scale=True, seed=40))
    clean = run_fp8(inp)
    ps = inp.workload.page_size
    for b, L in enumerate(inp.seq_lens.tolist()):
        last = int(inp.page_table[b, (L - 1) // ps])
        if L % ps:
            inp.k_pages[last, :, L % ps:, :] = 0x7F
            inp.v_pages[last, :, L % ps:, :] = 0xFF
            inp.k_scale[last, :, L % ps:] = float("nan")
    got = run_fp8(inp)
    assert np.array_equal(got[0], clean[0]) and np.array_equal(got[1], clean[1])


def test_single_key_returns_its_dequantized_value_row():
    inp = generate(latent(batch=2, seed=41), seq_lens=[1, 1])
    out, lse = run_fp8(inp)
    for b in range(2):
        page = int(inp.page_table[b, 0])
        v = e4m3_f64(inp.k_pages[page, 0, 0, :32]) * float(inp.k_scale[page, 0, 0])
        for h in range(8):
            assert np.array_equal(out[b, 0, h], v)
    inp2 = generate(fp8(batch=2, k_scale=True, seed=42), seq_lens=[1, 1])
    out2, _ = run_fp8(inp2)
    for b in range(2):
        page = int(inp2.page_table[b, 0])
        for h in range(8):
            v = e4m3_f64(inp2.v_pages[page, h // 4, 0])  # V carries no scale
            assert np.array_equal(out2[b, 0, h], v)


def test_rejects_bad_arguments():
    inp = generate(latent(seed=43))
    with pytest.raises(ValueError):  # rope part missing: depths do not add up
        oracle.decode_fp8(bf16_bits(inp.q), inp.k_pages.numpy(), None, inp.page_table.numpy(),
                          inp.seq_lens.numpy(), inp.scale, ov_depth=32)
    bad = inp.page_table.clone()
    bad[0, 0] = inp.k_pages.shape[0] + 5
    with pytest.raises(ValueError):
        oracle.decode_fp8(bf16_bits(inp.q), inp.k_pages.numpy(), None, bad.numpy(), inp.seq_lens.numpy(),
                          inp.scale, k_rope=bf16_bits(inp.k_rope), k_scale=inp.k_scale.numpy(), ov_depth=32)
