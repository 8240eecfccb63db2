"""Paged KV append and decode attention, float64 (oracle; test infrastructure only).

The plain definition of what the GPU path computes. No tiling, no online
softmax, no fusion: each function is the formula of the passage it cites, in
float64, over the keys and values the pool holds (read through the block table,
decoded from the pool's format and multiplied by the pool's scale).

Notation: B sequences, R query rows per sequence, Hq query heads, Hkv KV heads,
G = Hq / Hkv, head dim D, P positions per page, len_b the positions sequence b
holds (the step's appended positions included).
"""

from __future__ import annotations

import math

import numpy as np

from . import formats

SPLIT_POSITIONS = 256     # positions per split (nbxtensor/ops/paged_decode_attn.py, PAGED_DECODE_SPLIT_POSITIONS)
MAX_SPLITS = 64           # most splits a sequence is cut into (same file, PAGED_DECODE_MAX_SPLITS)


def new_pool(num_pages: int, h_kv: int, page_tokens: int, d: int, dtype: str, fill=None) -> np.ndarray:
    """A pool [num_pages, Hkv, P, D] of codes (nbxtensor/ops/paged_decode_attn.py, module
    docstring: one pool per layer and per K / V, laid out [num_pages, kv_heads, page_tokens, D])."""
    pool = np.zeros((num_pages, h_kv, page_tokens, d), dtype=formats.CODE_DTYPE[dtype])
    if fill is not None:
        pool[...] = fill
    return pool


def append(pool: np.ndarray, new: np.ndarray, slots: np.ndarray, page_tokens: int, dtype: str,
           scale: float = 1.0) -> np.ndarray:
    """Write new positions into the pool through the slot mapping, cast on store.

    nbxtensor/ops/attention_wrappers.py, ``paged_kv_append`` and
    nbxtensor/ops/paged_decode_attn.py, ``paged_kv_append_kernel``: for token t and
    KV head h, page = slot // P, pos = slot % P, pool[page, h, pos, :] = cast(new[t, h, :]).
    With a pool scale (fp8 cache), the stored value is cast(fp32(new) * fp32(1 / scale)),
    the reciprocal taken once in fp32; scale 1 leaves the values unchanged.

    Slots outside [0, num_pages * P) are skipped. Returns the boolean mask of the
    skipped tokens. ``new`` is float32 [N, Hkv, D]; the pool is updated in place.
    """
    new = np.asarray(new, dtype=np.float32)
    slots = np.asarray(slots, dtype=np.int64)
    num_pages = pool.shape[0]
    bad = (slots < 0) | (slots >= num_pages * page_tokens)
    inv = np.float32(1.0) / np.float32(scale)
    vals = (new * inv).astype(np.float32)                      # one IEEE fp32 multiply per element
    codes = formats.encode(vals, dtype)
    ok = ~bad
    pages = slots[ok] // page_tokens
    pos = slots[ok] % page_tokens
    pool[pages, :, pos, :] = codes[ok]
    return bad


def read_sequence(pool: np.ndarray, dtype: str, scale: float, block_row: np.ndarray, length: int,
                  h_kv: int, page_tokens: int) -> np.ndarray:
    """Positions 0..length-1 of one KV head of one sequence, read through its block table.

    nbxtensor/ops/paged_decode_attn.py, ``paged_decode_attn_split_kernel``: position j
    lives in page block_table[b, j // P] at row j % P. Values are decoded to float64
    and multiplied by the pool scale. Returns [length, D]."""
    n_pages = (length + page_tokens - 1) // page_tokens
    pages = np.asarray(block_row[:n_pages], dtype=np.int64)
    if np.any(pages < 0) or np.any(pages >= pool.shape[0]):
        raise ValueError("block table entry outside the pool inside the sequence")
    vals = formats.decode(pool[pages, h_kv], dtype)               # [n_pages, P, D]
    return vals.reshape(-1, pool.shape[-1])[:length] * float(scale)


def query_position(length: int, rows: int, r: int) -> int:
    """Query row r of a sequence holding `length` positions sits at length - rows + r
    (the rows are the newest positions) and sees keys 0..that position."""
    return length - rows + r


def attend(q: np.ndarray, keys: np.ndarray, values: np.ndarray, scale: float) -> np.ndarray:
    """softmax(scale * q . k_j) over j, applied to the values: the definition, in float64.

    nbxtensor/ops/paged_decode_attn.py, ``paged_decode_attn_split_kernel``: s_j = scale *
    sum_d q_d k_jd, weights exp(s_j - max s) / sum, output sum_j w_j v_j. No keys -> 0
    (the fully masked row of nbxtensor/ops/attention_wrappers.py, ``_math_attention``)."""
    if keys.shape[0] == 0:
        return np.zeros(values.shape[-1], dtype=np.float64)
    s = scale * (keys @ np.asarray(q, dtype=np.float64))
    w = np.exp(s - s.max())
    return (w @ values) / w.sum()


def kv_head(h: int, h_q: int, h_kv: int) -> int:
    """The KV head query head h reads: consecutive query heads share one
    (nbxtensor/ops/paged_decode_attn.py, ``paged_decode_attn_split_kernel``:
    h_kv = (pid % H_Q) // GQA_GROUPS, GQA_GROUPS = H_q // H_kv)."""
    return h // (h_q // h_kv)


def decode_attention(q: np.ndarray, k_pool: np.ndarray, v_pool: np.ndarray, dtype: str,
                     block_table: np.ndarray, seq_lens: np.ndarray, page_tokens: int,
                     scale: float, k_scale: float = 1.0, v_scale: float = 1.0,
                     heads=None) -> np.ndarray:
    """Paged decode attention for every (sequence, row, query head), float64.

    q [B, R, Hq, D] (any float dtype, read exactly), pools [num_pages, Hkv, P, D] of codes,
    block_table [B, max_pages] int32 (-1 past each sequence), seq_lens [B].
    Query head h reads KV head ``kv_head(h)``; row r attends keys 0..len-R+r.
    ``heads``: optional iterable of (b, r, h) to compute; the others stay 0.
    Returns [B, R, Hq, D] float64."""
    q = np.asarray(q, dtype=np.float64)
    B, R, Hq, D = q.shape
    h_kv_n = k_pool.shape[1]
    out = np.zeros((B, R, Hq, D), dtype=np.float64)
    wanted = None if heads is None else set(tuple(x) for x in heads)
    for b in range(B):
        L = int(seq_lens[b])
        if L <= 0:
            continue
        kv = {}
        for r in range(R):
            pos = query_position(L, R, r)
            for h in range(Hq):
                if wanted is not None and (b, r, h) not in wanted:
                    continue
                hk = kv_head(h, Hq, h_kv_n)
                if hk not in kv:
                    kv[hk] = (read_sequence(k_pool, dtype, k_scale, block_table[b], L, hk, page_tokens),
                              read_sequence(v_pool, dtype, v_scale, block_table[b], L, hk, page_tokens))
                K, V = kv[hk]
                out[b, r, h] = attend(q[b, r, h], K[:pos + 1], V[:pos + 1], scale) if pos >= 0 else 0.0
    return out


def split_plan(length: int, page_tokens: int) -> tuple[int, int]:
    """(splits, positions per split) of one sequence.

    nbxtensor/ops/paged_decode_attn.py, ``paged_decode_splits``: splits =
    max(1, min(ceil(len / 256), 64)). The positions per split are ceil(len / splits)
    rounded up to a multiple of the alignment A (the same file,
    ``paged_decode_attn_split_kernel``: seg_len = ceil(ceil(len / splits) / ALIGN) * ALIGN).
    A is the page when a page holds at most 256 positions, so no split starts inside a page,
    and 256 for larger pages (a contiguous cache read as one page per sequence), where a
    256-aligned start is still a tile start. Split s covers [s*seg, min((s+1)*seg, len));
    the last splits may be empty."""
    splits = max(1, min(-(-max(int(length), 1) // SPLIT_POSITIONS), MAX_SPLITS))
    align = page_tokens if page_tokens <= SPLIT_POSITIONS else SPLIT_POSITIONS
    seg = -(-int(length) // splits)
    seg = -(-seg // align) * align
    return splits, seg


def split_bounds(length: int, page_tokens: int) -> list[int]:
    """Boundaries c_0 = 0 <= c_1 <= ... <= c_S = len of the split plan."""
    splits, seg = split_plan(length, page_tokens)
    return [min(s * seg, int(length)) for s in range(splits)] + [int(length)]


def split_partial(q: np.ndarray, keys: np.ndarray, values: np.ndarray, scale: float, lo: int, hi: int,
                  last_visible: int):
    """One split's unnormalised partial (m, l, acc) over keys [lo, hi) ∩ [0, last_visible].

    nbxtensor/ops/paged_decode_attn.py, ``paged_decode_attn_split_kernel``: the split
    stores its running max m, its sum of exp l and its unnormalised accumulator acc.
    Here they are computed directly: m = max s_j, l = sum exp(s_j - m),
    acc = sum exp(s_j - m) v_j. An empty split gives (-inf, 0, 0)."""
    hi = min(hi, last_visible + 1)
    D = values.shape[-1]
    if hi <= lo:
        return -np.inf, 0.0, np.zeros(D, dtype=np.float64)
    s = scale * (keys[lo:hi] @ np.asarray(q, dtype=np.float64))
    m = s.max()
    w = np.exp(s - m)
    return float(m), float(w.sum()), w @ values[lo:hi]


def merge(m: np.ndarray, l: np.ndarray, acc: np.ndarray) -> np.ndarray:
    """Fixed-order merge of split partials into the output.

    nbxtensor/ops/attention_wrappers.py, ``decode_reduce`` (the fixed-order combine of a
    split decode), with TensorFold PR #1219 "Gotchas" on which splits to skip: here only a
    split with m = -inf (no visible key) is skipped, so a NaN still reaches the output.
    M = max_s m_s; L = sum_s l_s exp(m_s - M); out = (sum_s acc_s exp(m_s - M)) / L,
    s ascending. m, l: [S]; acc: [S, D]. No non-empty split -> 0."""
    m = np.asarray(m, dtype=np.float64)
    l = np.asarray(l, dtype=np.float64)
    acc = np.asarray(acc, dtype=np.float64)
    live = m != -np.inf
    if not np.any(live):
        return np.zeros(acc.shape[-1], dtype=np.float64)
    M = m[live].max()
    L = 0.0
    num = np.zeros(acc.shape[-1], dtype=np.float64)
    for s in range(m.shape[0]):
        if not live[s]:
            continue
        w = math.exp(m[s] - M)
        L += l[s] * w
        num += acc[s] * w
    return num / L


def decode_attention_split(q, k_pool, v_pool, dtype, block_table, seq_lens, page_tokens, scale,
                           k_scale=1.0, v_scale=1.0, bounds_fn=None):
    """The same output computed split by split and merged (for the merge invariant and
    for partials the GPU merge is checked on). ``bounds_fn(b, length)`` returns split
    boundaries; the default is the split rule. Returns (out [B,R,Hq,D], partials) with
    partials[(b, r, h)] = (m [S], l [S], acc [S, D])."""
    q = np.asarray(q, dtype=np.float64)
    B, R, Hq, D = q.shape
    h_kv_n = k_pool.shape[1]
    out = np.zeros((B, R, Hq, D), dtype=np.float64)
    parts = {}
    for b in range(B):
        L = int(seq_lens[b])
        bounds = bounds_fn(b, L) if bounds_fn is not None else split_bounds(L, page_tokens)
        S = len(bounds) - 1
        kv = {}
        for r in range(R):
            pos = query_position(L, R, r)
            for h in range(Hq):
                hk = kv_head(h, Hq, h_kv_n)
                if hk not in kv:
                    kv[hk] = ((read_sequence(k_pool, dtype, k_scale, block_table[b], L, hk, page_tokens),
                               read_sequence(v_pool, dtype, v_scale, block_table[b], L, hk, page_tokens))
                              if L > 0 else (np.zeros((0, D)), np.zeros((0, D))))
                K, V = kv[hk]
                ms = np.full(S, -np.inf)
                ls = np.zeros(S)
                accs = np.zeros((S, D))
                for s in range(S):
                    ms[s], ls[s], accs[s] = split_partial(q[b, r, h], K, V, scale, bounds[s], bounds[s + 1], pos)
                parts[(b, r, h)] = (ms, ls, accs)
                out[b, r, h] = merge(ms, ls, accs)
    return out, parts
