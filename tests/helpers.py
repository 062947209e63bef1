"""Shared test helpers: run the library on a seeded workload, run the oracle on
the same inputs, and compare element by element with the stated tolerance."""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
import split_paged_decode_gb300 as spd
from split_paged_decode_gb300.workloads import DecodeInputs, bf16_bits

# Tolerances of the decode output (bf16) and of the fp32 log-sum-exp.
OUT_ATOL = 1e-2
OUT_RTOL = 1e-2
LSE_ATOL = 1e-3


def oracle_threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def run_oracle(inp: DecodeInputs, rows=None):
    w = inp.workload
    if w.kv_dtype == "e4m3":
        return oracle.decode_fp8(bf16_bits(inp.q), inp.k_pages.numpy(),
                                 None if inp.v_pages is None else inp.v_pages.numpy(), inp.page_table.numpy(),
                                 inp.seq_lens.numpy(), inp.scale,
                                 k_rope=None if inp.k_rope is None else bf16_bits(inp.k_rope),
                                 k_scale=None if inp.k_scale is None else inp.k_scale.numpy(),
                                 ov_depth=w.ov_depth, rows=rows, threads=oracle_threads())
    v = None if inp.v_pages is None else bf16_bits(inp.v_pages)
    return oracle.decode(bf16_bits(inp.q), bf16_bits(inp.k_pages), v, inp.page_table.numpy(),
                         inp.seq_lens.numpy(), inp.scale, ov_depth=w.ov_depth, rows=rows,
                         threads=oracle_threads())


class DeviceCall:
    """Device copies of one input set plus a handle, for repeated runs."""

    def __init__(self, inp: DecodeInputs, splitk: int | None = None, device="cuda", path: str = "auto"):
        w = inp.workload
        self.inp = inp
        self.q = inp.q.to(device)
        self.k = inp.k_pages.to(device)
        self.v = None if inp.v_pages is None else inp.v_pages.to(device)
        self.pt = inp.page_table.to(device)
        self.lens = inp.seq_lens.to(device)
        self.out = torch.full((w.batch, w.num_q, w.num_q_heads, w.ov_depth), float("nan"),
                              dtype=torch.bfloat16, device=device)
        self.lse = torch.full((w.batch, w.num_q, w.num_q_heads), float("nan"), dtype=torch.float32,
                              device=device)
        P = w.splitk if splitk is None else splitk
        self.e4m3 = w.kv_dtype == "e4m3"
        self.ks = None if inp.k_scale is None else inp.k_scale.to(device)
        self.rope = None if inp.k_rope is None else inp.k_rope.to(device)
        if self.e4m3:
            self.h = spd.fa_decode_create_kv(w.num_q_heads, w.num_kv_heads, w.qk_depth, w.nope_depth,
                                             w.ov_depth, w.page_size, w.num_q, P, spd.FA_KV_E4M3, w.rope_depth)
        else:
            self.h = spd.fa_decode_create(w.num_q_heads, w.num_kv_heads, w.qk_depth, w.nope_depth,
                                          w.ov_depth, w.page_size, w.num_q, P)
        if path == "simt":
            spd.fa_decode_set_debug(self.h, spd.FA_DEBUG_FORCE_SIMT, 0)
        elif path == "two_clusters":  # each cluster works through many units in turn
            spd.fa_decode_set_debug(self.h, spd.FA_DEBUG_TWO_CLUSTERS, 0)
        elif path == "no_stream_k":  # every unit's key range on one cluster
            spd.fa_decode_set_debug(self.h, spd.FA_DEBUG_NO_STREAM_K, 0)

    def describe(self) -> str:
        return spd.fa_decode_describe(self.h)

    def run(self, stream=None):
        if self.e4m3:
            spd.fa_decode_run_kv(self.h, self.q, self.k, self.v, self.rope, self.ks, self.pt, self.lens,
                                 self.inp.scale, self.out, self.lse, stream=stream)
        else:
            spd.fa_decode_run(self.h, self.q, self.k, self.v, self.pt, self.lens, self.inp.scale, self.out,
                              self.lse, stream=stream)

    def status(self) -> int:
        return spd.fa_decode_check(self.h)

    def close(self):
        if self.h:
            spd.fa_decode_destroy(self.h)
            self.h = 0

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()


def compare(out, lse, ref_out, ref_lse, what=""):
    """Element-wise bound |out-ref| <= atol + rtol*|ref|, |lse-ref| <= 1e-3 (-inf must match)."""
    out = np.asarray(out, np.float64)
    lse = np.asarray(lse, np.float64)
    assert np.all(np.isfinite(out)), f"{what}: non-finite outputs"
    err = np.abs(out - ref_out)
    bound = OUT_ATOL + OUT_RTOL * np.abs(ref_out)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outputs out of tolerance; "
                           f"worst excess {np.max(err - bound):.3e} at {np.unravel_index(np.argmax(err - bound), err.shape)}")
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin), f"{what}: lse finiteness differs"
    assert np.all(lse[~fin] == ref_lse[~fin]), f"{what}: lse of rows without keys must be -inf"
    lerr = np.abs(lse[fin] - ref_lse[fin])
    assert lerr.size == 0 or lerr.max() <= LSE_ATOL, f"{what}: lse error {lerr.max():.3e}"


def check_against_oracle(call: DeviceCall, rows=None, what=""):
    """Compare the device result with the oracle on all rows, or on rows [(b,t,h), ...]."""
    out = call.out.float().cpu().numpy()
    lse = call.lse.cpu().numpy()
    if rows is None:
        ref_out, ref_lse = run_oracle(call.inp)
        compare(out, lse, ref_out, ref_lse, what)
    else:
        rows = np.asarray(rows, np.int32).reshape(-1, 3)
        ref_out, ref_lse = run_oracle(call.inp, rows=rows)
        compare(out[rows[:, 0], rows[:, 1], rows[:, 2]], lse[rows[:, 0], rows[:, 1], rows[:, 2]],
                ref_out, ref_lse, what)


def ramp_keys(inp, alpha: float = 0.01):
    """Make the running max move on nearly every tile: key j of every sequence
    becomes alpha * (j + 1) in every component (E4M3 caches: codes of those
    values with a unit per-token scale) and every query row becomes all ones,
    so a row's scores rise by 128 * alpha per key, about 20 exp2 units per
    128-key tile at scale 1/sqrt(128): above both rescale thresholds (2^8,
    2^4). Rows past a sequence's end keep their garbage (they must stay
    masked). Returns inp, modified in place."""
    w = inp.workload
    ps = w.page_size
    e4m3 = w.kv_dtype == "e4m3"
    for b, L in enumerate(inp.seq_lens.tolist()):
        for pi in range((int(L) + ps - 1) // ps):
            page = int(inp.page_table[b, pi])
            n = min(ps, int(L) - pi * ps)
            vals = alpha * (torch.arange(pi * ps, pi * ps + n, dtype=torch.float32) + 1.0)
            block = vals[:, None].expand(n, inp.k_pages.shape[3])
            if e4m3:
                codes = block.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
                inp.k_pages[page, :, :n, :] = codes
                if inp.k_scale is not None:
                    inp.k_scale[page, :, :n] = 1.0
            else:
                inp.k_pages[page, :, :n, :] = block.to(inp.k_pages.dtype)
    inp.q.fill_(1.0)
    return inp
