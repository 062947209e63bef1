"""Seeded synthetic decode workloads: shapes and input generation only.

This module is shared by the tests, the benchmark and the smoke check, and is
the only code the CUDA path and the fp64 oracle have in common. It holds no
attention arithmetic: it draws random caches, page permutations and lengths.

Draw recipe (all on a CPU ``torch.Generator`` seeded with the workload seed):
  1. per-sequence KV lengths (fixed, or uniform in [lo, hi] for ragged runs);
  2. Q, K, V as fp32 N(0, 1) rounded to bf16 (round-to-nearest-even);
  3. a permutation of the physical page pool (identity for ``page_order ==
     "identity"``);
  4. garbage: key rows past L_b inside the last page of every sequence and all
     spare pages are overwritten with +-1e4 (random sign), finite but large,
     so that any read of a masked row shows up as a large error.
The pool holds exactly the pages the sequences need plus ``ceil(1 %)`` (at
least one) spare pages that no page table entry names. Unused page-table
entries are -1.

fp8 caches (``kv_dtype == "e4m3"``), same generator, in this order:
  1. lengths as above;
  2. Q as above (bf16); K as fp32 N(0, 1) over the fp8 part of the row
     (qk_depth - rope_depth columns); the rope part (``rope_depth`` columns)
     as bf16 N(0, 1) in its own cache; V as fp32 N(0, 1) (separate-V layout);
  3. the page permutation;
  4. quantisation to OCP FP8 E4M3 codes by torch's float8_e4m3fn cast
     (round to nearest even): with ``k_scale`` every key row gets the fp32
     scale max|K_row| / 448 and stores K_row / scale (clamped to +-448),
     otherwise K and V are cast as drawn;
  5. garbage past L_b and in spare pages: codes of +-448, scale 1e4, rope
     +-1e4.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    batch: int
    num_q: int
    num_q_heads: int
    num_kv_heads: int
    qk_depth: int
    ov_depth: int
    page_size: int
    splitk: int                 # 1, 2, 4, 8 (16 non-portable); 0 = chosen per sequence
    seq_len: int = 0            # fixed KV length (includes the num_q new tokens)
    seq_len_lo: int = 0         # ragged: lengths uniform in [lo, hi] when hi > 0
    seq_len_hi: int = 0
    nope_depth: int = -1        # -1: equal to qk_depth (no rope part)
    latent: bool = False        # MLA: V is the first ov_depth columns of the K row
    page_order: str = "random"  # "random" or "identity"
    scale: float = 0.0          # 0.0 means 1 / sqrt(qk_depth)
    seed: int = 0
    kv_dtype: str = "bf16"      # "bf16" or "e4m3" (OCP FP8 E4M3 codes)
    k_scale: bool = False       # e4m3: a per-token fp32 K scale
    rope_depth: int = 0         # e4m3: trailing key columns kept in bf16 in their own cache

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale > 0.0 else 1.0 / math.sqrt(self.qk_depth)

    def with_(self, **kw) -> "DecodeWorkload":
        return dataclasses.replace(self, **kw)


# The five decode workloads the library is built and measured on.
WORKLOADS = {
    "tiny": DecodeWorkload(
        "tiny", batch=1, num_q=1, num_q_heads=4, num_kv_heads=1, qk_depth=64, ov_depth=64,
        page_size=64, splitk=2, seq_len=256, page_order="identity", scale=1.0 / 8.0, seed=0),
    "batched_gqa": DecodeWorkload(
        "batched_gqa", batch=16, num_q=1, num_q_heads=32, num_kv_heads=8, qk_depth=128,
        ov_depth=128, page_size=128, splitk=4, seq_len=4096, seed=1),
    "long_context": DecodeWorkload(
        "long_context", batch=1, num_q=1, num_q_heads=64, num_kv_heads=8, qk_depth=128,
        ov_depth=128, page_size=128, splitk=8, seq_len=131072, seed=2),
    "ragged_speculative": DecodeWorkload(
        "ragged_speculative", batch=64, num_q=4, num_q_heads=32, num_kv_heads=8, qk_depth=128,
        ov_depth=128, page_size=64, splitk=0, seq_len_lo=1, seq_len_hi=8192, seed=3),
    "mla": DecodeWorkload(
        "mla", batch=32, num_q=1, num_q_heads=128, num_kv_heads=1, qk_depth=576, nope_depth=512,
        ov_depth=512, page_size=64, splitk=2, seq_len=8192, latent=True,
        scale=1.0 / math.sqrt(192.0), seed=4),
}


@dataclass
class DecodeInputs:
    """CPU tensors of one decode call (bf16 caches, int32 tables)."""
    workload: DecodeWorkload
    q: torch.Tensor            # [B, T, Hq, Dk] bf16
    k_pages: torch.Tensor      # [NP, Hkv, PS, Dk] bf16
    v_pages: torch.Tensor | None  # [NP, Hkv, PS, Dv] bf16, None for the latent layout
    page_table: torch.Tensor   # [B, max_pages_per_seq] int32, -1 where unused
    seq_lens: torch.Tensor     # [B] int32
    scale: float
    # e4m3 caches: k_pages / v_pages hold uint8 codes [NP, Hkv, PS, D]; the
    # rope part of the key row and the per-token K scale live apart.
    k_rope: torch.Tensor | None = None   # [NP, Hkv, PS, rope_depth] bf16
    k_scale: torch.Tensor | None = None  # [NP, Hkv, PS] fp32

    @property
    def num_pages(self) -> int:
        return int(self.k_pages.shape[0])

    @property
    def max_pages_per_seq(self) -> int:
        return int(self.page_table.shape[1])


def _randn_bf16(shape, gen: torch.Generator) -> torch.Tensor:
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def draw_lengths(w: DecodeWorkload, gen: torch.Generator) -> torch.Tensor:
    if w.seq_len_hi > 0:
        return torch.randint(w.seq_len_lo, w.seq_len_hi + 1, (w.batch,), generator=gen,
                             dtype=torch.int64).to(torch.int32)
    return torch.full((w.batch,), w.seq_len, dtype=torch.int32)


def generate(w: DecodeWorkload, seq_lens=None) -> DecodeInputs:
    """Draw one seeded input set for workload ``w`` (see the module docstring).

    ``seq_lens`` overrides step 1 with explicit lengths (a list or tensor).
    """
    if w.kv_dtype == "e4m3":
        return _generate_e4m3(w, seq_lens)
    if w.kv_dtype != "bf16":
        raise ValueError(f"kv_dtype {w.kv_dtype!r}: bf16 or e4m3")
    gen = torch.Generator().manual_seed(w.seed)
    if seq_lens is None:
        lens = draw_lengths(w, gen)
    else:
        lens = torch.as_tensor(seq_lens, dtype=torch.int32).reshape(w.batch)
    ps = w.page_size
    pages_per_seq = [(int(L) + ps - 1) // ps for L in lens.tolist()]
    used = sum(pages_per_seq)
    spare = max(1, math.ceil(used / 100))
    num_pages = used + spare
    max_pages = max(1, max(pages_per_seq) if pages_per_seq else 1)

    q = _randn_bf16((w.batch, w.num_q, w.num_q_heads, w.qk_depth), gen)
    k_pages = _randn_bf16((num_pages, w.num_kv_heads, ps, w.qk_depth), gen)
    v_pages = None if w.latent else _randn_bf16((num_pages, w.num_kv_heads, ps, w.ov_depth), gen)

    if w.page_order == "identity":
        perm = torch.arange(num_pages, dtype=torch.int64)
    else:
        perm = torch.randperm(num_pages, generator=gen)
    page_table = torch.full((w.batch, max_pages), -1, dtype=torch.int32)
    cursor = 0
    for b, n in enumerate(pages_per_seq):
        page_table[b, :n] = perm[cursor:cursor + n].to(torch.int32)
        cursor += n
    spare_ids = perm[used:]

    def garbage(shape):
        sign = torch.randint(0, 2, shape, generator=gen, dtype=torch.int8).to(torch.float32)
        return ((sign * 2.0 - 1.0) * 1.0e4).to(torch.bfloat16)

    caches = [k_pages] if v_pages is None else [k_pages, v_pages]
    for b, L in enumerate(lens.tolist()):
        n = pages_per_seq[b]
        tail = n * ps - int(L)
        if n == 0 or tail == 0:
            continue
        last = int(page_table[b, n - 1])
        for c in caches:
            c[last, :, ps - tail:, :] = garbage((c.shape[1], tail, c.shape[3]))
    for pid in spare_ids.tolist():
        for c in caches:
            c[pid] = garbage(tuple(c.shape[1:]))

    return DecodeInputs(w, q, k_pages, v_pages, page_table, lens, float(w.softmax_scale))


def _pool(w: DecodeWorkload, lens: torch.Tensor):
    ps = w.page_size
    pages_per_seq = [(int(L) + ps - 1) // ps for L in lens.tolist()]
    used = sum(pages_per_seq)
    return pages_per_seq, used, used + max(1, math.ceil(used / 100)), max(1, max(pages_per_seq) if pages_per_seq else 1)


def _generate_e4m3(w: DecodeWorkload, seq_lens=None) -> DecodeInputs:
    gen = torch.Generator().manual_seed(w.seed)
    lens = draw_lengths(w, gen) if seq_lens is None else torch.as_tensor(seq_lens, dtype=torch.int32).reshape(w.batch)
    ps = w.page_size
    pages_per_seq, used, num_pages, max_pages = _pool(w, lens)
    d8 = w.qk_depth - w.rope_depth
    q = _randn_bf16((w.batch, w.num_q, w.num_q_heads, w.qk_depth), gen)
    k = torch.randn((num_pages, w.num_kv_heads, ps, d8), generator=gen, dtype=torch.float32)
    k_rope = _randn_bf16((num_pages, w.num_kv_heads, ps, w.rope_depth), gen) if w.rope_depth else None
    v = None if w.latent else torch.randn((num_pages, w.num_kv_heads, ps, w.ov_depth), generator=gen,
                                          dtype=torch.float32)
    perm = torch.arange(num_pages, dtype=torch.int64) if w.page_order == "identity" else \
        torch.randperm(num_pages, generator=gen)
    page_table = torch.full((w.batch, max_pages), -1, dtype=torch.int32)
    cursor = 0
    for b, n in enumerate(pages_per_seq):
        page_table[b, :n] = perm[cursor:cursor + n].to(torch.int32)
        cursor += n

    def e4m3(x):
        return x.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)

    k_scale = None
    if w.k_scale:
        k_scale = k.abs().amax(dim=3) / 448.0
        k8 = e4m3(k / k_scale.unsqueeze(3))
    else:
        k8 = e4m3(k)
    v8 = None if v is None else e4m3(v)

    def garbage_codes(shape):
        sign = torch.randint(0, 2, shape, generator=gen, dtype=torch.uint8)
        return (sign << 7) | 0x7E  # +-448

    def garbage_bf16(shape):
        sign = torch.randint(0, 2, shape, generator=gen, dtype=torch.int8).to(torch.float32)
        return ((sign * 2.0 - 1.0) * 1.0e4).to(torch.bfloat16)

    def spoil(sel_page, rows):
        for c in [k8] + ([v8] if v8 is not None else []):
            c[sel_page, :, rows, :] = garbage_codes((c.shape[1], rows.stop - rows.start, c.shape[3]))
        if k_rope is not None:
            k_rope[sel_page, :, rows, :] = garbage_bf16((k_rope.shape[1], rows.stop - rows.start, k_rope.shape[3]))
        if k_scale is not None:
            k_scale[sel_page, :, rows] = 1.0e4

    for b, L in enumerate(lens.tolist()):
        n = pages_per_seq[b]
        tail = n * ps - int(L)
        if n and tail:
            spoil(int(page_table[b, n - 1]), slice(ps - tail, ps))
    for pid in perm[used:].tolist():
        spoil(pid, slice(0, ps))
    return DecodeInputs(w, q, k8, v8, page_table, lens, float(w.softmax_scale), k_rope=k_rope, k_scale=k_scale)


def bf16_bits(t: torch.Tensor):
    """uint16 numpy view of a CPU bf16 tensor (the form the oracle takes)."""
    import numpy as np

    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
