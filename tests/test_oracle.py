"""Pins of the fp64 oracle against facts fixed by the mathematics (CPU only).

Nothing here calls the CUDA library. Each test compares the oracle with a
value it does not compute itself: a closed form, an identity of softmax
attention, an independent NumPy/SciPy brute force on a dense gather, or the
oracle's own plain definition reached by a different route (the split-K
log-sum-exp merge of the fa4_splitk_combine_write page).
"""
import math

import numpy as np
import pytest
import torch
from scipy.special import logsumexp, softmax

import oracle
from split_paged_decode_gb300.workloads import DecodeWorkload, bf16_bits, generate

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def small(**kw):
    base = dict(name="pin", batch=3, num_q=1, num_q_heads=8, num_kv_heads=2, qk_depth=32,
                ov_depth=32, page_size=16, splitk=1, seq_len_lo=1, seq_len_hi=100, seed=11)
    base.update(kw)
    return DecodeWorkload(**base)


def as_np(inp):
    q = bf16_bits(inp.q)
    k = bf16_bits(inp.k_pages)
    v = None if inp.v_pages is None else bf16_bits(inp.v_pages)
    return q, k, v, inp.page_table.numpy(), inp.seq_lens.numpy()


def run_oracle(inp, **kw):
    q, k, v, pt, lens = as_np(inp)
    return oracle.decode(q, k, v, pt, lens, inp.scale, ov_depth=inp.workload.ov_depth, **kw)


def widen(t):
    return t.to(torch.float64).numpy()


def brute_force(inp):
    """Dense gather in NumPy, then SciPy softmax / logsumexp per query row."""
    w = inp.workload
    q = widen(inp.q)
    K = widen(inp.k_pages)
    V = K[..., : w.ov_depth] if inp.v_pages is None else widen(inp.v_pages)
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
            kh = h // g
            Kd = K[phys, kh, j % w.page_size]          # [L, Dk]
            Vd = V[phys, kh, j % w.page_size]          # [L, Dv]
            for t in range(T):
                n = L - T + t + 1
                if n <= 0:
                    continue
                s = inp.scale * (Kd[:n] @ q[b, t, h])
                out[b, t, h] = softmax(s) @ Vd[:n]
                lse[b, t, h] = logsumexp(s)
    return out, lse


def assert_close(a, b, rtol=1e-12, atol=1e-12):
    np.testing.assert_allclose(a, b, rtol=rtol, atol=atol)


def assert_lse_close(a, b, tol=1e-12):
    fin = np.isfinite(b)
    assert np.array_equal(np.isfinite(a), fin)
    assert np.all(a[~fin] == b[~fin])
    np.testing.assert_allclose(a[fin], b[fin], rtol=tol, atol=tol)


# --- brute force on tiny inputs -------------------------------------------------

@pytest.mark.parametrize("kw", [
    dict(),                                             # GQA, ragged, random pages
    dict(num_q=4, seq_len_lo=1, seq_len_hi=40),          # causal tail, some rows empty
    dict(num_q_heads=4, num_kv_heads=4),                 # MHA
    dict(num_kv_heads=1, qk_depth=48, ov_depth=32, latent=True, nope_depth=32),  # latent
    dict(qk_depth=32, ov_depth=16, page_size=8),          # ov != qk, small pages
])
def test_brute_force(kw):
    inp = generate(small(**kw))
    out, lse = run_oracle(inp, threads=2)
    ref, ref_lse = brute_force(inp)
    assert_close(out, ref)
    assert_lse_close(lse, ref_lse)


def test_row_subset_matches_full():
    inp = generate(small(num_q=2))
    out, lse = run_oracle(inp)
    rng = np.random.default_rng(0)
    rows = np.stack([rng.integers(0, 3, 20), rng.integers(0, 2, 20), rng.integers(0, 8, 20)], 1)
    sub, sub_lse = run_oracle(inp, rows=rows)
    for i, (b, t, h) in enumerate(rows):
        assert np.array_equal(sub[i], out[b, t, h])
        assert sub_lse[i] == lse[b, t, h] or (np.isinf(sub_lse[i]) and np.isinf(lse[b, t, h]))


# --- split-K combine identity ------------------------------------------------------

@pytest.mark.parametrize("P", [1, 2, 3, 8, 16])
@pytest.mark.parametrize("num_q", [1, 4])
def test_partitioned_equals_plain(P, num_q):
    inp = generate(small(num_q=num_q, seq_len_lo=1, seq_len_hi=120, seed=20 + P))
    q, k, v, pt, lens = as_np(inp)
    rng = np.random.default_rng(P)
    bounds = []
    for L in lens:
        cuts = np.sort(rng.integers(0, int(L) + 1, P - 1))  # repeats give empty partitions
        bounds.append(np.concatenate([[0], cuts, [int(L)]]))
    bounds = np.array(bounds, np.int32)
    out, lse = oracle.partitioned(q, k, v, pt, lens, inp.scale, bounds, ov_depth=32)
    ref, ref_lse = run_oracle(inp)
    assert_close(out, ref, rtol=1e-12, atol=1e-13)
    assert_lse_close(lse, ref_lse)


def test_partition_with_all_keys_in_one_part_and_rest_empty():
    inp = generate(small(seed=5))
    q, k, v, pt, lens = as_np(inp)
    P = 4
    bounds = np.array([[0, 0, int(L), int(L), int(L)] for L in lens], np.int32)
    out, lse, pmax, psum = oracle.partitioned(q, k, v, pt, lens, inp.scale, bounds,
                                              ov_depth=32, return_parts=True)
    ref, ref_lse = run_oracle(inp)
    assert_close(out, ref)
    assert_lse_close(lse, ref_lse)
    # empty partitions report (-inf, 0); the populated one carries the whole sum
    assert np.all(np.isneginf(pmax[..., [0, 2, 3]])) and np.all(psum[..., [0, 2, 3]] == 0)
    assert np.all(psum[..., 1] >= 1.0)  # its own max contributes exp2(0) = 1


def test_partition_sums_are_exp2_of_raw_scores():
    """Per-partition state is (raw max, sum of exp2((s_raw - max) * scale * log2 e))."""
    inp = generate(small(batch=1, seq_len_lo=30, seq_len_hi=30, seed=3))
    q, k, v, pt, lens = as_np(inp)
    bounds = np.array([[0, 10, 30]], np.int32)
    _, _, pmax, psum = oracle.partitioned(q, k, v, pt, lens, inp.scale, bounds, ov_depth=32,
                                          return_parts=True)
    qd, K = widen(inp.q), widen(inp.k_pages)
    j = np.arange(30)
    phys = inp.page_table.numpy()[0, j // 16]
    for h in range(8):
        raw = K[phys, h // 4, j % 16] @ qd[0, 0, h]
        for p, (lo, hi) in enumerate([(0, 10), (10, 30)]):
            m = raw[lo:hi].max()
            assert pmax[0, 0, h, p] == pytest.approx(m, rel=1e-13)
            s = np.sum(np.exp(inp.scale * (raw[lo:hi] - m)))
            assert psum[0, 0, h, p] == pytest.approx(s, rel=1e-12)


# --- closed forms ----------------------------------------------------------------

def hand_inputs(K_rows, V_rows, q_row, scale, page_size=4):
    """One sequence, one head, pages in identity order, from explicit fp values."""
    K_rows = np.asarray(K_rows, np.float32)
    V_rows = np.asarray(V_rows, np.float32)
    L, Dk = K_rows.shape
    Dv = V_rows.shape[1]
    n_pages = (L + page_size - 1) // page_size + 1
    k = torch.zeros((n_pages, 1, page_size, Dk), dtype=torch.bfloat16)
    v = torch.zeros((n_pages, 1, page_size, Dv), dtype=torch.bfloat16)
    for j in range(L):
        k[j // page_size, 0, j % page_size] = torch.from_numpy(K_rows[j]).to(torch.bfloat16)
        v[j // page_size, 0, j % page_size] = torch.from_numpy(V_rows[j]).to(torch.bfloat16)
    q = torch.from_numpy(np.asarray(q_row, np.float32)).to(torch.bfloat16).reshape(1, 1, 1, Dk)
    pt = np.arange(n_pages - 1, dtype=np.int32).reshape(1, -1)
    out, lse = oracle.decode(bf16_bits(q), bf16_bits(k), bf16_bits(v), pt,
                             np.array([L], np.int32), scale)
    return out[0, 0, 0], lse[0, 0, 0], k, v, q


def test_two_keys_hand_example():
    # s0 = scale * 2, s1 = 0 with scale = ln(3)/2: weights 3/4 and 1/4, lse = ln 4.
    out, lse, *_ = hand_inputs([[2, 0], [0, 0]], [[1, 0], [0, 1]], [1, 0], math.log(3) / 2)
    assert_close(out, [0.75, 0.25], rtol=1e-15, atol=1e-15)
    assert lse == pytest.approx(math.log(4), rel=1e-15)


def test_two_keys_sigmoid():
    rng = np.random.default_rng(7)
    K = rng.standard_normal((2, 16)).astype(np.float32)
    V = rng.standard_normal((2, 8)).astype(np.float32)
    qv = rng.standard_normal(16).astype(np.float32)
    out, lse, k, v, q = hand_inputs(K, V, qv, 0.3)
    Kb, Vb, qb = widen(k[0, 0, :2]), widen(v[0, 0, :2]), widen(q.reshape(-1))
    s0, s1 = 0.3 * Kb[0] @ qb, 0.3 * Kb[1] @ qb
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    assert_close(out, w0 * Vb[0] + (1 - w0) * Vb[1])
    assert lse == pytest.approx(max(s0, s1) + math.log1p(math.exp(-abs(s0 - s1))), rel=1e-14)


def test_single_key_returns_its_value_row():
    inp = generate(small(seq_len_lo=1, seq_len_hi=1, seed=9))
    out, lse = run_oracle(inp)
    V = widen(inp.v_pages)
    K = widen(inp.k_pages)
    q = widen(inp.q)
    for b in range(3):
        phys = int(inp.page_table[b, 0])
        for h in range(8):
            assert np.array_equal(out[b, 0, h], V[phys, h // 4, 0])
            assert lse[b, 0, h] == pytest.approx(inp.scale * K[phys, h // 4, 0] @ q[b, 0, h],
                                                 rel=1e-14, abs=1e-14)


def test_identical_keys_give_mean_of_values():
    inp = generate(small(batch=2, seq_len_lo=37, seq_len_hi=37, seed=4))
    # every key row of a kv head equal to that head's first row
    k = inp.k_pages.clone()
    for b in range(2):
        row0 = k[int(inp.page_table[b, 0]), :, 0].clone()
        for j in range(37):
            k[int(inp.page_table[b, j // 16]), :, j % 16] = row0
    inp.k_pages = k
    out, lse = run_oracle(inp)
    V, K, q = widen(inp.v_pages), widen(k), widen(inp.q)
    for b in range(2):
        j = np.arange(37)
        phys = inp.page_table.numpy()[b, j // 16]
        for h in range(8):
            mean = V[phys, h // 4, j % 16].mean(axis=0)
            assert_close(out[b, 0, h], mean, rtol=1e-13, atol=1e-14)
            s = inp.scale * K[phys[0], h // 4, 0] @ q[b, 0, h]
            assert lse[b, 0, h] == pytest.approx(s + math.log(37), rel=1e-13, abs=1e-13)


def test_zero_scale_gives_mean_and_log_count():
    inp = generate(small(num_q=3, seed=6))
    inp.scale = 0.0
    out, lse = run_oracle(inp)
    V = widen(inp.v_pages)
    pt = inp.page_table.numpy()
    for b in range(3):
        L = int(inp.seq_lens[b])
        for t in range(3):
            n = L - 3 + t + 1
            if n <= 0:
                assert np.all(out[b, t] == 0) and np.all(np.isneginf(lse[b, t]))
                continue
            j = np.arange(n)
            for h in range(8):
                mean = V[pt[b, j // 16], h // 4, j % 16].mean(axis=0)
                assert_close(out[b, t, h], mean, rtol=1e-13, atol=1e-14)
                assert lse[b, t, h] == pytest.approx(math.log(n), rel=1e-14)


# --- invariances -------------------------------------------------------------------

def test_page_permutation_invariance():
    inp = generate(small(seed=8))
    out, lse = run_oracle(inp)
    rng = np.random.default_rng(1)
    n_pages = inp.num_pages
    perm = rng.permutation(n_pages)            # new slot of old page i is perm[i]
    k2 = torch.empty_like(inp.k_pages)
    v2 = torch.empty_like(inp.v_pages)
    k2[torch.from_numpy(perm)] = inp.k_pages
    v2[torch.from_numpy(perm)] = inp.v_pages
    pt = inp.page_table.numpy()
    pt2 = np.where(pt >= 0, perm[np.maximum(pt, 0)], -1).astype(np.int32)
    out2, lse2 = oracle.decode(bf16_bits(inp.q), bf16_bits(k2), bf16_bits(v2), pt2,
                               inp.seq_lens.numpy(), inp.scale)
    assert_close(out2, out, rtol=1e-15, atol=1e-15)
    assert_lse_close(lse2, lse, tol=1e-15)


def test_causal_rows_equal_single_token_calls():
    T = 4
    inp = generate(small(num_q=T, seq_len_lo=10, seq_len_hi=70, seed=12))
    out, lse = run_oracle(inp)
    q, k, v, pt, lens = as_np(inp)
    for t in range(T):
        lens_t = (lens - T + t + 1).astype(np.int32)
        o1, l1 = oracle.decode(np.ascontiguousarray(q[:, t:t + 1]), k, v, pt, lens_t, inp.scale)
        assert_close(out[:, t], o1[:, 0], rtol=1e-15, atol=1e-15)
        assert_lse_close(lse[:, t], l1[:, 0], tol=1e-15)


def test_gqa_equals_mha_with_repeated_kv():
    w = small(seed=13)
    inp = generate(w)
    out, lse = run_oracle(inp)
    g = w.group
    k_rep = inp.k_pages.repeat_interleave(g, dim=1)
    v_rep = inp.v_pages.repeat_interleave(g, dim=1)
    out2, lse2 = oracle.decode(bf16_bits(inp.q), bf16_bits(k_rep), bf16_bits(v_rep),
                               inp.page_table.numpy(), inp.seq_lens.numpy(), inp.scale)
    assert_close(out2, out, rtol=1e-15, atol=1e-15)
    assert_lse_close(lse2, lse, tol=1e-15)


def test_latent_value_is_key_prefix():
    """Latent layout equals an explicit V cache holding the first ov columns of K."""
    w = small(num_kv_heads=1, qk_depth=48, ov_depth=32, latent=True, nope_depth=32, seed=14)
    inp = generate(w)
    out, lse = run_oracle(inp)
    v = inp.k_pages[..., :32].contiguous()
    out2, lse2 = oracle.decode(bf16_bits(inp.q), bf16_bits(inp.k_pages), bf16_bits(v),
                               inp.page_table.numpy(), inp.seq_lens.numpy(), inp.scale)
    assert_close(out2, out, rtol=0, atol=0)
    assert_lse_close(lse2, lse, tol=0)


def test_garbage_rows_are_never_read():
    """Changing every masked row (page tails, spare pages) leaves the result bit-identical."""
    inp = generate(small(num_q=2, seed=15))
    out, lse = run_oracle(inp)
    k, v = inp.k_pages.clone(), inp.v_pages.clone()
    ps = 16
    live = np.zeros((inp.num_pages, ps), bool)
    for b in range(3):
        L = int(inp.seq_lens[b])
        for j in range(L):
            live[int(inp.page_table[b, j // ps]), j % ps] = True
    dead = torch.from_numpy(~live)[:, None, :, None]  # [NP, 1, PS, 1]
    k = torch.where(dead, torch.tensor(float("nan"), dtype=torch.bfloat16), k)
    v = torch.where(dead, torch.tensor(float("nan"), dtype=torch.bfloat16), v)
    out2, lse2 = oracle.decode(bf16_bits(inp.q), bf16_bits(k), bf16_bits(v),
                               inp.page_table.numpy(), inp.seq_lens.numpy(), inp.scale)
    assert np.array_equal(out2, out)
    assert np.array_equal(lse2, lse)


def test_rejects_bad_page_id():
    inp = generate(small(seed=16))
    q, k, v, pt, lens = as_np(inp)
    pt = pt.copy()
    pt[0, 0] = inp.num_pages  # out of range
    with pytest.raises(ValueError):
        oracle.decode(q, k, v, pt, lens, inp.scale)


def test_tiny_regression_fixture():
    """The oracle still reproduces its committed output on the tiny workload."""
    import json
    import os

    from split_paged_decode_gb300.workloads import WORKLOADS

    path = os.path.join(os.path.dirname(__file__), "golden", "tiny_oracle.json")
    doc = json.load(open(path))
    inp = generate(WORKLOADS["tiny"])
    out, lse = run_oracle(inp)
    assert_close(out.reshape(4, 64), np.array(doc["out"]), rtol=1e-13, atol=1e-15)
    assert_close(lse.reshape(4), np.array(doc["lse"]), rtol=1e-13, atol=1e-15)
