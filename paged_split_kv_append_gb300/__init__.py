"""Python binding of libnbx: paged KV append and split-KV decode attention on GB300.

Argument marshalling only: every function takes torch tensors, checks their dtypes,
shapes and devices, and calls the C entry point of the same name in libnbx.so with
raw device pointers and the current CUDA stream. All computation runs in the
library's CUDA kernels; there is no other code path. If libnbx.so is missing the
first call raises ``NbxLibraryMissing`` (build it with ``build()``).

The C ABI is declared in ``include/nbx.h``.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import _build

__all__ = [
    "NBX_F32", "NBX_BF16", "NBX_E4M3", "NbxError", "NbxLibraryMissing", "build", "lib", "library_path",
    "nbx_paged_kv_append", "nbx_paged_decode_workspace_bytes", "nbx_paged_decode_attn",
    "nbx_paged_decode_merge", "nbx_set_decode_grid_limit", "nbx_set_decode_wait_test", "nbx_status_string",
    "nbx_paged_decode_bounds", "nbx_paged_decode_attn_fixed_shift", "nbx_decode_fixed_shift_gate",
    "dtype_code",
    "DEV_BAD_SLOT", "DEV_BAD_PAGE", "DEV_BAD_LEN", "DEV_TIMEOUT",
]

NBX_F32, NBX_BF16, NBX_E4M3 = 0, 1, 2
DEV_BAD_SLOT, DEV_BAD_PAGE, DEV_BAD_LEN, DEV_TIMEOUT = 0x1, 0x2, 0x4, 0x8
PARTIAL_SIMT, PARTIAL_TCGEN05, PARTIAL_TCGEN05_FP8 = 0, 1, 2

_lib = None
_lock = threading.Lock()


class NbxError(RuntimeError):
    def __init__(self, func: str, status: int):
        super().__init__(f"{func}: {nbx_status_string(status)} (status {status})")
        self.status = status


class NbxLibraryMissing(RuntimeError):
    pass


def library_path() -> str:
    return _build.LIB


def build(force: bool = False) -> str:
    """Compile libnbx.so for sm_103a in-tree (nvcc) and return its path."""
    return _build.build(force=force)


def _declare(l):
    vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    l.nbx_paged_kv_append.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, i32, i32, i32, vp, f32, f32, vp, vp]
    l.nbx_paged_kv_append.restype = i32
    l.nbx_paged_decode_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
    l.nbx_paged_decode_workspace_bytes.restype = sz
    l.nbx_paged_decode_workspace_bytes_for.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, i32]
    l.nbx_paged_decode_workspace_bytes_for.restype = sz
    l.nbx_paged_decode_attn.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, i32, i32, i32, i32, vp, i32, vp, i32,
                                        f32, f32, f32, vp, vp, sz, vp, vp]
    l.nbx_paged_decode_attn.restype = i32
    l.nbx_paged_decode_step.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, i32, vp, vp, i32, i32, i32, i32, vp, i32,
                                        vp, i32, f32, f32, f32, vp, vp, sz, vp, vp]
    l.nbx_paged_decode_step.restype = i32
    l.nbx_decode_attn_contiguous.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, i32, i32, i32, vp, i32, f32, f32, f32,
                                             vp, vp, sz, vp, vp]
    l.nbx_decode_attn_contiguous.restype = i32
    l.nbx_paged_decode_merge.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp]
    l.nbx_paged_decode_merge.restype = i32
    l.nbx_paged_decode_partial_kernel.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32]
    l.nbx_paged_decode_partial_kernel.restype = i32
    l.nbx_set_decode_grid_limit.argtypes = [i32]
    l.nbx_set_decode_grid_limit.restype = None
    l.nbx_set_decode_wait_test.argtypes = [ctypes.c_ulonglong, ctypes.c_ulonglong]
    l.nbx_set_decode_wait_test.restype = None
    l.nbx_paged_decode_bounds.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, i32, i32, i32, i32, vp, i32, vp, i32,
                                          f32, f32, vp, vp, vp, vp]
    l.nbx_paged_decode_bounds.restype = i32
    l.nbx_paged_decode_attn_fixed_shift.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, i32, i32, i32, i32, vp, i32,
                                                    vp, i32, f32, f32, f32, vp, vp, sz, vp, vp, vp, vp]
    l.nbx_paged_decode_attn_fixed_shift.restype = i32
    l.nbx_decode_fixed_shift_gate.argtypes = [i32, ctypes.c_double, ctypes.POINTER(i32), ctypes.POINTER(i32)]
    l.nbx_decode_fixed_shift_gate.restype = i32
    l.nbx_status_string.argtypes = [i32]
    l.nbx_status_string.restype = ctypes.c_char_p
    l.nbx_abi_version.argtypes = []
    l.nbx_abi_version.restype = i32


def lib() -> ctypes.CDLL:
    """The loaded libnbx.so (loaded once, on first use)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path):
                raise NbxLibraryMissing(f"libnbx.so not found at {path}: run paged_split_kv_append_gb300.build()")
            l = ctypes.CDLL(path)
            _declare(l)
            _lib = l
    return _lib


_DTYPES = {torch.float32: NBX_F32, torch.bfloat16: NBX_BF16, torch.float8_e4m3fn: NBX_E4M3, torch.uint8: NBX_E4M3}


def dtype_code(t: torch.Tensor) -> int:
    try:
        return _DTYPES[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}") from None


def nbx_status_string(status: int) -> str:
    return lib().nbx_status_string(int(status)).decode()


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(func: str, status: int):
    if status != 0:
        raise NbxError(func, status)


def _cuda_contig(name: str, t: torch.Tensor):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def nbx_paged_kv_append(new_k: torch.Tensor, new_v: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                        slot_mapping: torch.Tensor, k_scale: float = 1.0, v_scale: float = 1.0,
                        status: Optional[torch.Tensor] = None, stream=None) -> None:
    """new_k / new_v [n_tok, h_kv, d] (fp32 or bf16) into the pools [num_pages, h_kv, page_tokens, d]
    (fp32, bf16 or e4m3) at slot_mapping [n_tok] int32; cast on store."""
    for n, t in (("new_k", new_k), ("new_v", new_v), ("k_pool", k_pool), ("v_pool", v_pool),
                 ("slot_mapping", slot_mapping)):
        _cuda_contig(n, t)
    if slot_mapping.dtype != torch.int32:
        raise ValueError("slot_mapping must be int32")
    if new_k.shape != new_v.shape or k_pool.shape != v_pool.shape or k_pool.dtype != v_pool.dtype:
        raise ValueError("K and V must have the same shapes and dtypes")
    n_tok, h_kv, d = new_k.shape
    num_pages, h_kv_p, page_tokens, d_p = k_pool.shape
    if (h_kv_p, d_p) != (h_kv, d) or slot_mapping.numel() != n_tok:
        raise ValueError(f"new {list(new_k.shape)} does not fit the pool {list(k_pool.shape)}")
    st = lib().nbx_paged_kv_append(_ptr(new_k), _ptr(new_v), dtype_code(new_k), n_tok, h_kv, d, _ptr(k_pool),
                                   _ptr(v_pool), dtype_code(k_pool), num_pages, page_tokens, _ptr(slot_mapping),
                                   float(k_scale), float(v_scale), _ptr(status), _stream(stream))
    _check("nbx_paged_kv_append", st)


def nbx_paged_decode_workspace_bytes(batch: int, rows: int, h_q: int, h_kv: int, d: int, max_seq_len: int) -> int:
    return int(lib().nbx_paged_decode_workspace_bytes(batch, rows, h_q, h_kv, d, max_seq_len))


def nbx_paged_decode_workspace_bytes_for(q_dtype: int, pool_dtype: int, batch: int, rows: int, h_q: int, h_kv: int,
                                         d: int, max_seq_len: int, page_tokens: int) -> int:
    return int(lib().nbx_paged_decode_workspace_bytes_for(q_dtype, pool_dtype, batch, rows, h_q, h_kv, d,
                                                          max_seq_len, page_tokens))


def nbx_paged_decode_attn(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor, block_table: torch.Tensor,
                          seq_lens: torch.Tensor, max_seq_len: int, scale: float, k_scale: float = 1.0,
                          v_scale: float = 1.0, out: Optional[torch.Tensor] = None,
                          workspace: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                          stream=None) -> torch.Tensor:
    """q [batch, rows, h_q, d] (fp32 or bf16), pools [num_pages, h_kv, page_tokens, d], block_table
    [batch, max_pages] int32 (-1 padded), seq_lens [batch] int32 -> out [batch, rows, h_q, d] fp32."""
    for n, t in (("q", q), ("k_pool", k_pool), ("v_pool", v_pool), ("block_table", block_table),
                 ("seq_lens", seq_lens)):
        _cuda_contig(n, t)
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise ValueError("block_table and seq_lens must be int32")
    if k_pool.shape != v_pool.shape or k_pool.dtype != v_pool.dtype:
        raise ValueError("k_pool and v_pool must match")
    batch, rows, h_q, d = q.shape
    num_pages, h_kv, page_tokens, d_p = k_pool.shape
    if d_p != d or block_table.dim() != 2 or block_table.shape[0] != batch or seq_lens.numel() != batch:
        raise ValueError(f"q {list(q.shape)}, pool {list(k_pool.shape)}, block_table {list(block_table.shape)}, "
                         f"seq_lens {list(seq_lens.shape)} do not fit")
    max_pages = block_table.shape[1]
    if out is None:
        out = torch.empty((batch, rows, h_q, d), dtype=torch.float32, device=q.device)
    _cuda_contig("out", out)
    need = nbx_paged_decode_workspace_bytes_for(dtype_code(q), dtype_code(k_pool), batch, rows, h_q, h_kv, d,
                                                max_seq_len, page_tokens)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    st = lib().nbx_paged_decode_attn(_ptr(q), dtype_code(q), batch, rows, h_q, d, _ptr(k_pool), _ptr(v_pool),
                                     dtype_code(k_pool), num_pages, h_kv, page_tokens, _ptr(block_table), max_pages,
                                     _ptr(seq_lens), int(max_seq_len), float(scale), float(k_scale),
                                     float(v_scale), _ptr(out), _ptr(workspace), workspace.numel(),
                                     _ptr(status), _stream(stream))
    _check("nbx_paged_decode_attn", st)
    return out


def nbx_paged_decode_step(q: torch.Tensor, new_k: torch.Tensor, new_v: torch.Tensor, k_pool: torch.Tensor,
                          v_pool: torch.Tensor, block_table: torch.Tensor, lens: torch.Tensor, max_seq_len: int,
                          scale: float, k_scale: float = 1.0, v_scale: float = 1.0, out: Optional[torch.Tensor] = None,
                          workspace: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                          stream=None) -> torch.Tensor:
    """One decode step: new_k/new_v [batch, rows, h_kv, d] (fp32 or bf16) are written at positions
    lens[b] .. lens[b] + rows - 1, the rows of q [batch, rows, h_q, d] attend, and lens [batch] int32
    advances by rows, all on the stream. Returns out [batch, rows, h_q, d] fp32."""
    for n, t in (("q", q), ("new_k", new_k), ("new_v", new_v), ("k_pool", k_pool), ("v_pool", v_pool),
                 ("block_table", block_table), ("lens", lens)):
        _cuda_contig(n, t)
    if block_table.dtype != torch.int32 or lens.dtype != torch.int32:
        raise ValueError("block_table and lens must be int32")
    if k_pool.shape != v_pool.shape or k_pool.dtype != v_pool.dtype or new_k.shape != new_v.shape or \
            new_k.dtype != new_v.dtype:
        raise ValueError("k/v tensors must match")
    batch, rows, h_q, d = q.shape
    num_pages, h_kv, page_tokens, d_p = k_pool.shape
    if d_p != d or tuple(new_k.shape) != (batch, rows, h_kv, d) or block_table.dim() != 2 or \
            block_table.shape[0] != batch or lens.numel() != batch:
        raise ValueError(f"q {list(q.shape)}, new_k {list(new_k.shape)}, pool {list(k_pool.shape)}, "
                         f"block_table {list(block_table.shape)}, lens {list(lens.shape)} do not fit")
    if out is None:
        out = torch.empty((batch, rows, h_q, d), dtype=torch.float32, device=q.device)
    _cuda_contig("out", out)
    need = nbx_paged_decode_workspace_bytes_for(dtype_code(q), dtype_code(k_pool), batch, rows, h_q, h_kv, d,
                                                max_seq_len, page_tokens)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    st = lib().nbx_paged_decode_step(_ptr(q), dtype_code(q), batch, rows, h_q, d, _ptr(new_k), _ptr(new_v),
                                     dtype_code(new_k), _ptr(k_pool), _ptr(v_pool), dtype_code(k_pool), num_pages,
                                     h_kv, page_tokens, _ptr(block_table), block_table.shape[1], _ptr(lens),
                                     int(max_seq_len), float(scale), float(k_scale), float(v_scale), _ptr(out),
                                     _ptr(workspace), workspace.numel(), _ptr(status), _stream(stream))
    _check("nbx_paged_decode_step", st)
    return out


def nbx_decode_attn_contiguous(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, seq_lens: torch.Tensor,
                               max_seq_len: int, scale: float, k_scale: float = 1.0, v_scale: float = 1.0,
                               out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                               status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """q [batch, rows, h_q, d], caches [batch, h_kv, capacity, d] (no page table), seq_lens [batch]
    int32 -> out [batch, rows, h_q, d] fp32."""
    for n, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("seq_lens", seq_lens)):
        _cuda_contig(n, t)
    if seq_lens.dtype != torch.int32:
        raise ValueError("seq_lens must be int32")
    if k_cache.shape != v_cache.shape or k_cache.dtype != v_cache.dtype:
        raise ValueError("k_cache and v_cache must match")
    batch, rows, h_q, d = q.shape
    b_c, h_kv, capacity, d_c = k_cache.shape
    if b_c != batch or d_c != d or seq_lens.numel() != batch:
        raise ValueError(f"q {list(q.shape)}, cache {list(k_cache.shape)}, seq_lens {list(seq_lens.shape)} do not fit")
    if out is None:
        out = torch.empty((batch, rows, h_q, d), dtype=torch.float32, device=q.device)
    _cuda_contig("out", out)
    need = nbx_paged_decode_workspace_bytes_for(dtype_code(q), dtype_code(k_cache), batch, rows, h_q, h_kv, d,
                                                max_seq_len, capacity)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    st = lib().nbx_decode_attn_contiguous(_ptr(q), dtype_code(q), batch, rows, h_q, d, _ptr(k_cache), _ptr(v_cache),
                                          dtype_code(k_cache), h_kv, capacity, _ptr(seq_lens), int(max_seq_len),
                                          float(scale), float(k_scale), float(v_scale), _ptr(out), _ptr(workspace),
                                          workspace.numel(), _ptr(status), _stream(stream))
    _check("nbx_decode_attn_contiguous", st)
    return out


def nbx_paged_decode_merge(acc_part: torch.Tensor, m_part: torch.Tensor, l_part: torch.Tensor,
                           out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """acc_part [n_rows, splits, d], m_part / l_part [n_rows, splits] fp32 (m in natural-log units)
    -> out [n_rows, d] fp32."""
    for n, t in (("acc_part", acc_part), ("m_part", m_part), ("l_part", l_part)):
        _cuda_contig(n, t)
        if t.dtype != torch.float32:
            raise ValueError(f"{n} must be fp32")
    n_rows, splits, d = acc_part.shape
    if out is None:
        out = torch.empty((n_rows, d), dtype=torch.float32, device=acc_part.device)
    st = lib().nbx_paged_decode_merge(_ptr(acc_part), _ptr(m_part), _ptr(l_part), n_rows, splits, d, _ptr(out),
                                      _stream(stream))
    _check("nbx_paged_decode_merge", st)
    return out


def nbx_paged_decode_partial_kernel(q_dtype: int, pool_dtype: int, rows: int, h_q: int, h_kv: int, d: int,
                                    num_pages: int, page_tokens: int) -> int:
    """PARTIAL_SIMT or PARTIAL_TCGEN05: the split-partial kernel a decode with these sizes runs."""
    k = lib().nbx_paged_decode_partial_kernel(q_dtype, pool_dtype, rows, h_q, h_kv, d, num_pages, page_tokens)
    _check("nbx_paged_decode_partial_kernel", k if k < 0 else 0)
    return k


def nbx_set_decode_grid_limit(max_ctas: int) -> None:
    lib().nbx_set_decode_grid_limit(int(max_ctas))


def nbx_set_decode_wait_test(wait_limit_ns: int = 0, producer_delay_ns: int = 0) -> None:
    """Tests of the timeout path only: the SIMT partial kernel's wait bound (0 = the default 2 s) and
    a delay before its producer warps start (0 = none)."""
    lib().nbx_set_decode_wait_test(int(wait_limit_ns), int(producer_delay_ns))


def _decode_shapes(q, k_pool, v_pool, block_table, seq_lens):
    for n, t in (("q", q), ("k_pool", k_pool), ("v_pool", v_pool), ("block_table", block_table),
                 ("seq_lens", seq_lens)):
        _cuda_contig(n, t)
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise ValueError("block_table and seq_lens must be int32")
    if k_pool.shape != v_pool.shape or k_pool.dtype != v_pool.dtype:
        raise ValueError("k_pool and v_pool must match")
    batch, rows, h_q, d = q.shape
    num_pages, h_kv, page_tokens, d_p = k_pool.shape
    if d_p != d or block_table.dim() != 2 or block_table.shape[0] != batch or seq_lens.numel() != batch:
        raise ValueError(f"q {list(q.shape)}, pool {list(k_pool.shape)}, block_table {list(block_table.shape)}, "
                         f"seq_lens {list(seq_lens.shape)} do not fit")
    return batch, rows, h_q, d, num_pages, h_kv, page_tokens, block_table.shape[1]


def nbx_paged_decode_bounds(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor, block_table: torch.Tensor,
                            seq_lens: torch.Tensor, max_seq_len: int, k_scale: float = 1.0, v_scale: float = 1.0,
                            status: Optional[torch.Tensor] = None, stream=None):
    """The fixed-shift softmax's score bounds: (q_norm [batch, rows, h_q], kv_max [batch, h_kv, 2]) fp32."""
    batch, rows, h_q, d, num_pages, h_kv, page_tokens, max_pages = _decode_shapes(q, k_pool, v_pool, block_table,
                                                                                  seq_lens)
    q_norm = torch.empty((batch, rows, h_q), dtype=torch.float32, device=q.device)
    kv_max = torch.empty((batch, h_kv, 2), dtype=torch.float32, device=q.device)
    st = lib().nbx_paged_decode_bounds(_ptr(q), dtype_code(q), batch, rows, h_q, d, _ptr(k_pool), _ptr(v_pool),
                                       dtype_code(k_pool), num_pages, h_kv, page_tokens, _ptr(block_table), max_pages,
                                       _ptr(seq_lens), int(max_seq_len), float(k_scale), float(v_scale), _ptr(q_norm),
                                       _ptr(kv_max), _ptr(status), _stream(stream))
    _check("nbx_paged_decode_bounds", st)
    return q_norm, kv_max


def nbx_paged_decode_attn_fixed_shift(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                                      block_table: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                                      scale: float, q_norm: torch.Tensor, kv_max: torch.Tensor, k_scale: float = 1.0,
                                      v_scale: float = 1.0, out: Optional[torch.Tensor] = None,
                                      workspace: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                                      stream=None) -> torch.Tensor:
    """nbx_paged_decode_attn with the fixed-shift softmax where the bounds pass the gate."""
    batch, rows, h_q, d, num_pages, h_kv, page_tokens, max_pages = _decode_shapes(q, k_pool, v_pool, block_table,
                                                                                  seq_lens)
    _cuda_contig("q_norm", q_norm)
    _cuda_contig("kv_max", kv_max)
    if q_norm.dtype != torch.float32 or kv_max.dtype != torch.float32 or q_norm.numel() != batch * rows * h_q or \
            kv_max.numel() != batch * h_kv * 2:
        raise ValueError("q_norm [batch, rows, h_q] and kv_max [batch, h_kv, 2] must be fp32")
    if out is None:
        out = torch.empty((batch, rows, h_q, d), dtype=torch.float32, device=q.device)
    _cuda_contig("out", out)
    need = nbx_paged_decode_workspace_bytes_for(dtype_code(q), dtype_code(k_pool), batch, rows, h_q, h_kv, d,
                                                max_seq_len, page_tokens)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    st = lib().nbx_paged_decode_attn_fixed_shift(_ptr(q), dtype_code(q), batch, rows, h_q, d, _ptr(k_pool),
                                                 _ptr(v_pool), dtype_code(k_pool), num_pages, h_kv, page_tokens,
                                                 _ptr(block_table), max_pages, _ptr(seq_lens), int(max_seq_len),
                                                 float(scale), float(k_scale), float(v_scale), _ptr(out),
                                                 _ptr(workspace), workspace.numel(), _ptr(q_norm), _ptr(kv_max),
                                                 _ptr(status), _stream(stream))
    _check("nbx_paged_decode_attn_fixed_shift", st)
    return out


def nbx_decode_fixed_shift_gate(n_keys: int, v_max_bound: float = 256.0):
    """(C, gate) of the fixed-shift softmax for n_keys keys and a value bound (host-only)."""
    c, g = ctypes.c_int(), ctypes.c_int()
    st = lib().nbx_decode_fixed_shift_gate(int(n_keys), float(v_max_bound), ctypes.byref(c), ctypes.byref(g))
    _check("nbx_decode_fixed_shift_gate", st)
    return c.value, g.value
