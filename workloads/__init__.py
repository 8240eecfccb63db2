"""Seeded synthetic inputs for the paged split-KV append + decode attention path.

This module is shared by the tests, the benchmark and the oracle comparisons. It
builds inputs only: sequence lengths, a page allocation (block tables and slot
mappings, the page-table bookkeeping a serving engine does before it calls the
append), query rows and the raw key/value tokens. It holds none of the method's
arithmetic: no rounding to the cache format, no scores, no softmax, no merge.

Workloads (each one of the configurations the paged decode read is measured on):

- ``tiny``: 2 sequences of 37 and 100 positions, 1 query row, 4 query heads over
  2 KV heads, head dim 64, 16-position pages, fp32 queries / keys / values.
- ``single_row``: 32 sequences, lengths uniform on [512, 8192], 1 query row,
  32 query heads over 8 KV heads, head dim 128, 16-position pages, bf16 pool and
  bf16 queries, pages scattered by one global permutation.
- ``verify``: 4 streams, 16 query rows at the tail of a 32768-position context
  (causal inside the window), 24 query heads over 4 KV heads, head dim 256,
  64-position pages, bf16.
- ``prefill``: 1 sequence, 128 causal query rows at positions 32640..32767 over
  32768 keys, 24 / 4 heads, head dim 256, 64-position pages, fp8-e4m3 pool with
  one fp32 scale per tensor (amax / 448), bf16 queries.
- ``ragged``: 64 sequences, lengths log-uniform on [1, 131072], 1 query row,
  32 / 8 heads, head dim 128, 16-position pages, bf16 pool, pages of all
  sequences interleaved by one global permutation.

Every workload also has a ``*_small`` variant with the same head layout, page
size and formats but lengths short enough for the float64 oracle to compute every
output in seconds (several tiles, several splits and a ragged tail).

A decode step appends the newest ``rows`` positions of every sequence (the query
rows' own keys and values) and then attends: the pool is prefilled with the first
``len - rows`` positions and the step's append writes the rest.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np
import torch

DTYPES = ("f32", "bf16", "e4m3")
E4M3_MAX = 448.0  # largest finite OCP E4M3 value: the per-tensor scale maps amax onto it


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    batch: int
    rows: int
    h_q: int
    h_kv: int
    d: int
    page_tokens: int
    pool_dtype: str          # "f32" | "bf16" | "e4m3"
    q_dtype: str             # "f32" | "bf16"
    seed: int
    lens: tuple              # ("fixed", (l0, l1, ...)) | ("uniform", lo, hi) | ("loguniform", lo, hi)

    @property
    def group(self) -> int:
        return self.h_q // self.h_kv


CONFIGS = {
    "tiny": Config("tiny", 2, 1, 4, 2, 64, 16, "f32", "f32", 0, ("fixed", (37, 100))),
    "single_row": Config("single_row", 32, 1, 32, 8, 128, 16, "bf16", "bf16", 1, ("uniform", 512, 8192)),
    "verify": Config("verify", 4, 16, 24, 4, 256, 64, "bf16", "bf16", 2, ("fixed", (32768,) * 4)),
    "prefill": Config("prefill", 1, 128, 24, 4, 256, 64, "e4m3", "bf16", 3, ("fixed", (32768,))),
    "ragged": Config("ragged", 64, 1, 32, 8, 128, 16, "bf16", "bf16", 4, ("loguniform", 1, 131072)),
    # oracle-sized variants: same heads, pages and formats, short lengths
    "single_row_small": Config("single_row_small", 6, 1, 32, 8, 128, 16, "bf16", "bf16", 11, ("uniform", 1, 1500)),
    "verify_small": Config("verify_small", 2, 16, 24, 4, 256, 64, "bf16", "bf16", 12, ("uniform", 700, 2300)),
    "prefill_small": Config("prefill_small", 1, 128, 24, 4, 256, 64, "e4m3", "bf16", 13, ("fixed", (1500,))),
    "ragged_small": Config("ragged_small", 16, 1, 32, 8, 128, 16, "bf16", "bf16", 14, ("loguniform", 1, 20000)),
}

FULL_CONFIGS = ("tiny", "single_row", "verify", "prefill", "ragged")


def draw_lens(cfg: Config, rng: np.random.Generator) -> np.ndarray:
    """Sequence lengths (positions each sequence holds after the step's append).

    Bounds are inclusive. Log-uniform lengths are round(exp(U(0, ln hi))) clamped
    to [lo, hi]."""
    kind = cfg.lens[0]
    if kind == "fixed":
        vals = np.asarray(cfg.lens[1], dtype=np.int64)
        assert vals.size == cfg.batch
    elif kind == "uniform":
        lo, hi = cfg.lens[1], cfg.lens[2]
        vals = rng.integers(lo, hi, size=cfg.batch, endpoint=True)
    elif kind == "loguniform":
        lo, hi = cfg.lens[1], cfg.lens[2]
        vals = np.rint(np.exp(rng.uniform(0.0, math.log(hi), size=cfg.batch)))
        vals = np.clip(vals, lo, hi).astype(np.int64)
    else:
        raise ValueError(kind)
    return vals.astype(np.int32)


def allocate_pages(lens: np.ndarray, page_tokens: int, rng: np.random.Generator, spare_pages: int = 0):
    """Grant every sequence ceil(len / page_tokens) pages, with page ids drawn from
    one global permutation, so the pages of all sequences are interleaved in the
    pool. Returns (block_table [B, max_pages] int32 padded with -1, num_pages)."""
    pages = [(int(l) + page_tokens - 1) // page_tokens for l in lens]
    total = sum(pages)
    num_pages = total + spare_pages
    perm = rng.permutation(num_pages)[:total].astype(np.int32)
    max_pages = max(1, max(pages) if pages else 1)
    bt = np.full((len(lens), max_pages), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(pages):
        bt[b, :n] = perm[off:off + n]
        off += n
    return bt, max(num_pages, 1)


def slots_for(block_table: np.ndarray, page_tokens: int, b: int, positions: np.ndarray) -> np.ndarray:
    """The slot of each position of sequence b: page id * page_tokens + position in page."""
    pages = block_table[b, positions // page_tokens].astype(np.int64)
    return (pages * page_tokens + positions % page_tokens).astype(np.int32)


TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclasses.dataclass
class Case:
    cfg: Config
    lens: np.ndarray             # [B] int32, host
    block_table: np.ndarray      # [B, max_pages] int32, host, -1 padded
    num_pages: int
    tok_offset: np.ndarray       # [B+1] int64: sequence b's raw tokens are k_raw[tok_offset[b]:tok_offset[b+1]]
    k_raw: torch.Tensor          # [sum(lens), h_kv, d] fp32 (the values written into the pool)
    v_raw: torch.Tensor
    q: torch.Tensor              # [B, rows, h_q, d] in q_dtype
    scale: float                 # softmax scale 1/sqrt(d)
    k_scale: float               # dequant scale of the pool (1.0 unless e4m3)
    v_scale: float
    n_new: np.ndarray            # [B] positions the step appends per sequence (min(rows, len))

    @property
    def max_seq_len(self) -> int:
        return int(self.lens.max()) if self.lens.size else 0

    def prefill_index(self):
        """(token rows into k_raw, slots) of the positions the pool holds before the step."""
        idx, slots = [], []
        for b in range(self.cfg.batch):
            n_pre = int(self.lens[b]) - int(self.n_new[b])
            pos = np.arange(n_pre, dtype=np.int64)
            idx.append(self.tok_offset[b] + pos)
            slots.append(slots_for(self.block_table, self.cfg.page_tokens, b, pos))
        return np.concatenate(idx).astype(np.int64), np.concatenate(slots).astype(np.int32)

    def step_index(self):
        """(token rows into k_raw, slots) of the positions the step appends."""
        idx, slots = [], []
        for b in range(self.cfg.batch):
            L = int(self.lens[b])
            pos = np.arange(L - int(self.n_new[b]), L, dtype=np.int64)
            idx.append(self.tok_offset[b] + pos)
            slots.append(slots_for(self.block_table, self.cfg.page_tokens, b, pos))
        return np.concatenate(idx).astype(np.int64), np.concatenate(slots).astype(np.int32)

    def all_index(self):
        i0, s0 = self.prefill_index()
        i1, s1 = self.step_index()
        return np.concatenate([i0, i1]), np.concatenate([s0, s1])

    def kv_bytes(self) -> int:
        """Bytes of K and V one decode pass reads: every held position of every KV head."""
        elt = {"f32": 4, "bf16": 2, "e4m3": 1}[self.cfg.pool_dtype]
        return int(self.lens.astype(np.int64).sum()) * self.cfg.h_kv * self.cfg.d * elt * 2


def make_case(cfg: Config | str, device: str | torch.device = "cpu", seed: Optional[int] = None,
              lens: Optional[Sequence[int]] = None, spare_pages: int = 0) -> Case:
    """Build one seeded synthetic case. Host metadata comes from numpy's PCG64 and
    the tensors from a torch generator seeded the same way on ``device`` (values
    drawn on the CPU and on a GPU differ; every comparison hands both sides the
    same tensors)."""
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    seed = cfg.seed if seed is None else seed
    rng = np.random.default_rng(seed)
    if lens is None:
        lens_arr = draw_lens(cfg, rng)
    else:
        lens_arr = np.asarray(lens, dtype=np.int32)
        cfg = dataclasses.replace(cfg, batch=int(lens_arr.size))
    bt, num_pages = allocate_pages(lens_arr, cfg.page_tokens, rng, spare_pages)
    tok_offset = np.zeros(cfg.batch + 1, dtype=np.int64)
    tok_offset[1:] = np.cumsum(lens_arr.astype(np.int64))
    n_tok = int(tok_offset[-1])

    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    k_raw = torch.randn((n_tok, cfg.h_kv, cfg.d), generator=gen, device=device, dtype=torch.float32)
    v_raw = torch.randn((n_tok, cfg.h_kv, cfg.d), generator=gen, device=device, dtype=torch.float32)
    q = torch.randn((cfg.batch, cfg.rows, cfg.h_q, cfg.d), generator=gen, device=device,
                    dtype=torch.float32).to(TORCH_DTYPE[cfg.q_dtype])
    if cfg.pool_dtype == "e4m3":
        k_scale = float((k_raw.abs().max() / E4M3_MAX).item()) if n_tok else 1.0
        v_scale = float((v_raw.abs().max() / E4M3_MAX).item()) if n_tok else 1.0
    else:
        k_scale = v_scale = 1.0
    n_new = np.minimum(lens_arr, cfg.rows).astype(np.int32)
    return Case(cfg=cfg, lens=lens_arr, block_table=bt, num_pages=num_pages, tok_offset=tok_offset,
                k_raw=k_raw, v_raw=v_raw, q=q, scale=1.0 / math.sqrt(cfg.d),
                k_scale=k_scale, v_scale=v_scale, n_new=n_new)


def permute_pages(case: Case, seed: int) -> tuple[np.ndarray, np.ndarray]:
    """A relabelling of physical page ids: returns (perm, new_block_table) with
    new id = perm[old id]. Writing the same tokens through the new table moves the
    data with its pages."""
    rng = np.random.default_rng(seed)
    perm = rng.permutation(case.num_pages).astype(np.int32)
    bt = case.block_table.copy()
    mask = bt >= 0
    bt[mask] = perm[bt[mask]]
    return perm, bt


def slots_with_table(case: Case, block_table: np.ndarray, index: str = "all"):
    """Slots of the case's tokens under another block table (same token order as the index functions)."""
    out = []
    for b in range(case.cfg.batch):
        L = int(case.lens[b])
        n_new = int(case.n_new[b])
        if index == "prefill":
            pos = np.arange(L - n_new, dtype=np.int64)
        elif index == "step":
            pos = np.arange(L - n_new, L, dtype=np.int64)
        else:
            pos = None
        if pos is not None:
            out.append(slots_for(block_table, case.cfg.page_tokens, b, pos))
    if index == "all":
        return np.concatenate([slots_with_table(case, block_table, "prefill"),
                               slots_with_table(case, block_table, "step")])
    return np.concatenate(out).astype(np.int32)
