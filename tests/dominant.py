"""Dominant-key inputs: a check of page gathering that is exact at any size.

For every (sequence b, kv head k) one key position j is chosen. The columns
`dom_cols` of every query row are made positive (|q| + 1) and the same
columns of key row j are set to `alpha`; the other columns of K_j and all
other key rows keep their random values. Key j then scores so far above
every other visible key that the other keys' softmax weights
exp2((s_i - s_j) * scale * log2 e) underflow to exactly 0 in fp32 (the
margin is checked below, in fp64, on the actual inputs). The weight of key j
is exp2(0) = 1 and its sum is 1, so the split-K merge and every rescale give
back V_j unchanged: the output row of every query that sees j must equal
V_j bit for bit (V_j = K_j[:ov_depth] in the latent layout, whose non-
dominant columns stay random). A wrong K row, in-page offset or page slot
moves or loses the winner, and a wrong V row returns different bits, so a
gather slip cannot hide inside the rounding tolerance.

Test-side arithmetic only (numpy / torch on the CPU); nothing here is shared
with the library or the oracle.
"""
from __future__ import annotations

import math

import numpy as np
import torch

# exp2 of anything below -126 is flushed to zero by the kernels' ex2.approx.ftz;
# ask for a wide margin beyond that.
MIN_MARGIN_EXP2 = 160.0


def dom_cols(w) -> slice:
    """Query / key columns that carry the dominance: the rope part of the latent
    layout (the columns past ov_depth), else the upper half of the row."""
    if w.latent and w.ov_depth < w.qk_depth:
        return slice(w.ov_depth, w.qk_depth)
    return slice(w.qk_depth // 2, w.qk_depth)


def choose_positions(w, lens, splitk_of=None, salt: int = 0) -> dict:
    """One key position per (b, kv head), cycling through the places a gather
    can go wrong: key 0, the last row of the first page, the first row of the
    second page, the sequence's last key (in its partial last page), a key in
    each split rank's share of the tiles (128-key tiles, even split, remainder
    to the low ranks) and an arbitrary in-page offset of a later page."""
    ps = w.page_size
    pos = {}
    n = 0
    for b, L in enumerate(int(x) for x in lens):
        for k in range(w.num_kv_heads):
            n += 1
            if L <= 0:
                continue
            P = splitk_of(L) if splitk_of else max(1, w.splitk)
            kind = (n + salt) % 7
            if kind == 0:
                j = 0
            elif kind == 1:
                j = ps - 1
            elif kind == 2:
                j = ps
            elif kind == 3:
                j = L - 1
            elif kind in (4, 5):
                tiles = (L + 127) // 128
                r = (n * 3 + salt) % P
                base, rem = divmod(tiles, P)
                t0 = r * base + min(r, rem)
                cnt = base + (1 if r < rem else 0)
                j = (t0 + (cnt // 2 if cnt else 0)) * 128 + (37 * n + 11) % 128
            else:
                page = ((n * 5 + salt) % max(1, (L + ps - 1) // ps))
                j = page * ps + (29 * n + 3) % ps
            pos[(b, k)] = int(min(max(j, 0), L - 1))
    return pos


def plant(inp, positions: dict, alpha: float = 64.0):
    """Modify `inp` in place (q and the K cache) so that each chosen key dominates.
    An E4M3 cache gets the code of 448 in the dominant columns and, with
    per-token scales, the scale 0.25 (key value 112) for the chosen row; an
    E4M3 latent cache with a bf16 rope cache gets `alpha` in the chosen row's
    rope values (the dominant columns) and the scale 0.25."""
    w = inp.workload
    cols = dom_cols(w)
    q = inp.q.float()
    q[..., cols] = q[..., cols].abs() + 1.0
    inp.q = q.to(torch.bfloat16)
    ps = w.page_size
    for (b, k), j in positions.items():
        page = int(inp.page_table[b, j // ps])
        if w.kv_dtype == "e4m3" and inp.k_rope is not None:
            # latent E4M3 cache: the dominant columns are the bf16 rope part
            inp.k_rope[page, k, j % ps, :] = alpha
            if inp.k_scale is not None:
                inp.k_scale[page, k, j % ps] = 0.25
        elif w.kv_dtype == "e4m3":
            inp.k_pages[page, k, j % ps, cols] = 0x7E
            if inp.k_scale is not None:
                inp.k_scale[page, k, j % ps] = 0.25
        else:
            inp.k_pages[page, k, j % ps, cols] = alpha
    return inp


def _e4m3(codes: torch.Tensor, dtype) -> torch.Tensor:
    return codes.contiguous().view(torch.float8_e4m3fn).to(dtype)


def value_row(inp, b: int, k: int, j: int) -> torch.Tensor:
    """V_j as bf16 (an E4M3 value row widened exactly; in the latent layout
    the K scale times the row's first ov_depth codes, exact for the planted
    scale 0.25)."""
    w = inp.workload
    ps = w.page_size
    page = int(inp.page_table[b, j // ps])
    if w.kv_dtype == "e4m3" and inp.v_pages is None:
        v = _e4m3(inp.k_pages[page, k, j % ps, :w.ov_depth], torch.float64)
        if inp.k_scale is not None:
            v = v * float(inp.k_scale[page, k, j % ps])
        vb = v.to(torch.bfloat16)
        assert bool((vb.double() == v).all()), "planted V row is not exact in bf16"
        return vb
    if w.kv_dtype == "e4m3":
        return _e4m3(inp.v_pages[page, k, j % ps, :], torch.bfloat16)
    if inp.v_pages is None:
        return inp.k_pages[page, k, j % ps, :w.ov_depth]
    return inp.v_pages[page, k, j % ps, :]


def _gather_keys(inp, b: int, k: int, L: int) -> torch.Tensor:
    w = inp.workload
    ps = w.page_size
    j = torch.arange(L)
    pages = inp.page_table[b, (j // ps)].long()
    if w.kv_dtype == "e4m3":
        kk = _e4m3(inp.k_pages[pages, k, j % ps, :], torch.float64)
        if inp.k_scale is not None:
            kk = kk * inp.k_scale[pages, k, j % ps].double().unsqueeze(1)
        if inp.k_rope is not None:
            kk = torch.cat([kk, inp.k_rope[pages, k, j % ps, :].double()], dim=1)
        return kk
    return inp.k_pages[pages, k, j % ps, :].double()


def check_margin(inp, positions: dict):
    """fp64 check of the premise: for every query row that sees its kv head's
    chosen key, that key beats every other visible key by more than
    MIN_MARGIN_EXP2 in exp2 units."""
    w = inp.workload
    c = inp.scale / math.log(2.0)
    g = w.num_q_heads // w.num_kv_heads
    worst = math.inf
    for (b, k), j in positions.items():
        L = int(inp.seq_lens[b])
        kg = _gather_keys(inp, b, k, L)
        qs = inp.q[b, :, k * g:(k + 1) * g, :].double().reshape(-1, w.qk_depth)
        s = qs @ kg.T  # [T*g, L] raw scores
        for t in range(w.num_q):
            n_vis = L - w.num_q + t + 1
            if j >= n_vis:
                continue
            rows = s[t * g:(t + 1) * g, :n_vis].clone()
            sj = rows[:, j].clone()
            rows[:, j] = -math.inf
            if n_vis > 1:
                worst = min(worst, float(((sj - rows.max(dim=1).values) * c).min()))
    assert worst > MIN_MARGIN_EXP2, f"dominant-key margin only {worst:.1f} exp2 units"
    return worst


def check_bit_exact(out: torch.Tensor, inp, positions: dict, what: str = "") -> int:
    """Every output row of a query that sees its chosen key equals V_j exactly:
    the same value in every column (bf16 values compared exactly; +0 and -0
    count as equal, since sum_j p_j V_j turns an E4M3 -0 into +0). Returns the
    number of rows checked."""
    w = inp.workload
    g = w.num_q_heads // w.num_kv_heads
    out = out.cpu()
    checked = 0
    bad = []
    for (b, k), j in positions.items():
        L = int(inp.seq_lens[b])
        v = value_row(inp, b, k, j)
        for t in range(w.num_q):
            if j >= L - w.num_q + t + 1:
                continue
            got = out[b, t, k * g:(k + 1) * g, :]
            same = (got.float() == v.float().unsqueeze(0)).all(dim=1)
            checked += g
            if not bool(same.all()):
                h = int(torch.nonzero(~same)[0, 0]) + k * g
                bad.append((b, t, h, j))
    assert not bad, f"{what}: {len(bad)} rows differ from V_j, first (b, t, h, j) = {bad[0]}"
    return checked


def expected_rows(inp, positions: dict) -> np.ndarray:
    """(b, t, h) of every row that sees its chosen key."""
    w = inp.workload
    g = w.num_q_heads // w.num_kv_heads
    rows = []
    for (b, k), j in positions.items():
        L = int(inp.seq_lens[b])
        for t in range(w.num_q):
            if j < L - w.num_q + t + 1:
                rows += [(b, t, h) for h in range(k * g, (k + 1) * g)]
    return np.asarray(rows, np.int32).reshape(-1, 3)
