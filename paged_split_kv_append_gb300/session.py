"""Device state for one paged decode workload, and its decode step.

A ``PagedDecodeSession`` owns the device buffers a serving loop keeps resident: the K
and V pools, the block table and lengths, the step's queries and new tokens, the
decode workspace, the output and the status word. ``step()`` is one pass of the hot
path through the C ABI: ``nbx_paged_kv_append`` writes the step's new positions into
the pools, then ``nbx_paged_decode_attn`` computes attention for every query row.
Nothing here computes: torch provides memory and streams only.
"""

from __future__ import annotations

from typing import Optional

import torch

from . import (NBX_BF16, NBX_E4M3, NBX_F32, nbx_paged_decode_attn, nbx_paged_decode_workspace_bytes_for,
               nbx_paged_kv_append)

POOL_TORCH = {"f32": torch.float32, "bf16": torch.bfloat16, "e4m3": torch.uint8}


def new_pool(num_pages: int, h_kv: int, page_tokens: int, d: int, dtype: str, device, fill_nan: bool = True):
    """A pool [num_pages, h_kv, page_tokens, d]; e4m3 pools are held as uint8 codes. With
    ``fill_nan`` every position starts as NaN (0x7F for e4m3), so a read of a position the
    pool does not hold shows up in the output."""
    shape = (num_pages, h_kv, page_tokens, d)
    if dtype == "e4m3":
        return torch.full(shape, 0x7F if fill_nan else 0, dtype=torch.uint8, device=device)
    return torch.full(shape, float("nan") if fill_nan else 0.0, dtype=POOL_TORCH[dtype], device=device)


class PagedDecodeSession:
    def __init__(self, *, num_pages: int, h_kv: int, page_tokens: int, d: int, pool_dtype: str, batch: int,
                 rows: int, h_q: int, max_seq_len: int, device, fill_nan: bool = True, q_dtype: str = "bf16"):
        self.device = torch.device(device)
        self.num_pages, self.h_kv, self.page_tokens, self.d = num_pages, h_kv, page_tokens, d
        self.pool_dtype = pool_dtype
        self.batch, self.rows, self.h_q, self.max_seq_len = batch, rows, h_q, max_seq_len
        self.k_pool = new_pool(num_pages, h_kv, page_tokens, d, pool_dtype, self.device, fill_nan)
        self.v_pool = new_pool(num_pages, h_kv, page_tokens, d, pool_dtype, self.device, fill_nan)
        codes = {"f32": NBX_F32, "bf16": NBX_BF16, "e4m3": NBX_E4M3}
        ws = nbx_paged_decode_workspace_bytes_for(codes[q_dtype], codes[pool_dtype], batch, rows, h_q, h_kv, d,
                                                  max_seq_len, page_tokens)
        if ws == 0 and batch > 0:
            raise ValueError("invalid decode sizes")
        self.workspace = torch.empty(max(ws, 256), dtype=torch.uint8, device=self.device)
        self.out = torch.empty((batch, rows, h_q, d), dtype=torch.float32, device=self.device)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.q = self.block_table = self.seq_lens = None
        self.new_k = self.new_v = self.new_slots = None
        self.scale, self.k_scale, self.v_scale = 1.0, 1.0, 1.0

    # ---------------------------------------------------------------- state
    def append(self, new_k: torch.Tensor, new_v: torch.Tensor, slots: torch.Tensor, stream=None) -> None:
        nbx_paged_kv_append(new_k, new_v, self.k_pool, self.v_pool, slots, self.k_scale, self.v_scale,
                            status=self.status, stream=stream)

    def prefill(self, k_raw: torch.Tensor, v_raw: torch.Tensor, index, slots, chunk_tokens: int = 1 << 18) -> None:
        """Append the tokens k_raw[index] at the given slots, in chunks (index/slots on the host)."""
        import numpy as np
        index = np.asarray(index)
        slots = np.asarray(slots, dtype=np.int32)
        for lo in range(0, index.size, chunk_tokens):
            hi = min(index.size, lo + chunk_tokens)
            ii = torch.from_numpy(index[lo:hi]).to(k_raw.device)
            kk = k_raw.index_select(0, ii).to(self.device)
            vv = v_raw.index_select(0, ii).to(self.device)
            ss = torch.from_numpy(slots[lo:hi]).to(self.device)
            self.append(kk, vv, ss)

    def set_inputs(self, q: torch.Tensor, block_table, seq_lens, new_k: Optional[torch.Tensor],
                   new_v: Optional[torch.Tensor], new_slots, scale: float, k_scale: float = 1.0,
                   v_scale: float = 1.0) -> None:
        """The step's inputs; host arrays are copied to the device once."""
        def dev(x, dtype=None):
            t = x if isinstance(x, torch.Tensor) else torch.as_tensor(x)
            if dtype is not None:
                t = t.to(dtype)
            return t.to(self.device).contiguous()
        self.q = dev(q)
        self.block_table = dev(block_table, torch.int32)
        self.seq_lens = dev(seq_lens, torch.int32)
        self.new_k = None if new_k is None else dev(new_k)
        self.new_v = None if new_v is None else dev(new_v)
        self.new_slots = None if new_slots is None else dev(new_slots, torch.int32)
        self.scale, self.k_scale, self.v_scale = float(scale), float(k_scale), float(v_scale)

    # ---------------------------------------------------------------- the step
    def decode(self, stream=None) -> torch.Tensor:
        return nbx_paged_decode_attn(self.q, self.k_pool, self.v_pool, self.block_table, self.seq_lens,
                                     self.max_seq_len, self.scale, self.k_scale, self.v_scale, out=self.out,
                                     workspace=self.workspace, status=self.status, stream=stream)

    def step(self, stream=None) -> torch.Tensor:
        """Append the step's new positions, then decode: one pass of the hot path."""
        if self.new_k is not None and self.new_k.shape[0] > 0:
            self.append(self.new_k, self.new_v, self.new_slots, stream=stream)
        return self.decode(stream=stream)

    def status_bits(self) -> int:
        return int(self.status.item())
