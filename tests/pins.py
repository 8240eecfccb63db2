"""Pins of the oracle: checks against something other than the oracle itself.

Each function returns an error measure; the tests assert it is small, and the
planted-mistake tests assert it becomes large when a mistake is planted in the
oracle. Independent sides used here: torch-CPU library casts, torch's float64
scaled_dot_product_attention on contiguous (non-paged) tensors, closed forms.
"""

from __future__ import annotations

import numpy as np
import torch
import torch.nn.functional as F

import oracle.formats as fm
import oracle.paged as op
import workloads as wl


def oracle_pools(case: wl.Case):
    """The oracle's own pools: every position of every sequence appended through the slots."""
    cfg = case.cfg
    idx, slots = case.all_index()
    kp = op.new_pool(case.num_pages, cfg.h_kv, cfg.page_tokens, cfg.d, cfg.pool_dtype)
    vp = op.new_pool(case.num_pages, cfg.h_kv, cfg.page_tokens, cfg.d, cfg.pool_dtype)
    k = case.k_raw.cpu().numpy()[idx]
    v = case.v_raw.cpu().numpy()[idx]
    op.append(kp, k, slots, cfg.page_tokens, cfg.pool_dtype, case.k_scale)
    op.append(vp, v, slots, cfg.page_tokens, cfg.pool_dtype, case.v_scale)
    return kp, vp


def oracle_output(case: wl.Case, pools=None, block_table=None) -> np.ndarray:
    kp, vp = pools if pools is not None else oracle_pools(case)
    bt = case.block_table if block_table is None else block_table
    return op.decode_attention(case.q.float().cpu().numpy(), kp, vp, case.cfg.pool_dtype, bt, case.lens,
                               case.cfg.page_tokens, case.scale, case.k_scale, case.v_scale)


def torch_cast_values(raw: torch.Tensor, dtype: str, scale: float) -> torch.Tensor:
    """What the cache holds for raw fp32 values, by torch's own casts, as float64."""
    raw = raw.float()
    if dtype == "f32":
        return raw.double()
    if dtype == "bf16":
        return raw.to(torch.bfloat16).double()
    inv = torch.tensor(1.0, dtype=torch.float32) / torch.tensor(scale, dtype=torch.float32)
    return (raw * inv).to(torch.float8_e4m3fn).double() * scale


def brute_force(case: wl.Case) -> np.ndarray:
    """softmax(scale * Q K^T + causal) V per sequence on contiguous float64 tensors,
    built from the raw tokens in position order (no pages, no block table), by torch's
    scaled_dot_product_attention."""
    cfg = case.cfg
    out = np.zeros((cfg.batch, cfg.rows, cfg.h_q, cfg.d), dtype=np.float64)
    G = cfg.group
    for b in range(cfg.batch):
        L = int(case.lens[b])
        if L == 0:
            continue
        sl = slice(int(case.tok_offset[b]), int(case.tok_offset[b + 1]))
        K = torch_cast_values(case.k_raw[sl].cpu(), cfg.pool_dtype, case.k_scale)   # [L, Hkv, D]
        V = torch_cast_values(case.v_raw[sl].cpu(), cfg.pool_dtype, case.v_scale)
        K = K.permute(1, 0, 2).repeat_interleave(G, dim=0)      # [Hq, L, D]
        V = V.permute(1, 0, 2).repeat_interleave(G, dim=0)
        Q = case.q[b].cpu().double().permute(1, 0, 2)           # [Hq, R, D]
        pos = L - cfg.rows + torch.arange(cfg.rows)
        mask = torch.arange(L)[None, :] <= pos[:, None]         # [R, L]
        o = F.scaled_dot_product_attention(Q[None], K[None], V[None], attn_mask=mask[None, None],
                                           scale=case.scale)[0]  # [Hq, R, D]
        o[:, ~mask.any(dim=1)] = 0.0                            # rows with no visible key (a NaN input stays NaN)
        out[b] = o.permute(1, 0, 2).numpy()
    return out


def pin_brute_force(case: wl.Case) -> float:
    return float(np.max(np.abs(oracle_output(case) - brute_force(case))))


def pin_merge_partitions(case: wl.Case, seed: int = 0) -> float:
    """Merge of random partitions (empty splits included) against the one-pass result."""
    kp, vp = oracle_pools(case)
    cfg = case.cfg
    rng = np.random.default_rng(seed)
    one = op.decode_attention(case.q.float().numpy(), kp, vp, cfg.pool_dtype, case.block_table, case.lens,
                              cfg.page_tokens, case.scale, case.k_scale, case.v_scale)

    def bounds(b, L):
        n = int(rng.integers(1, 9))
        cuts = np.sort(rng.integers(0, L + 1, size=n - 1)) if n > 1 else np.array([], dtype=np.int64)
        return [0] + [int(c) for c in cuts] + [L]

    split, _ = op.decode_attention_split(case.q.float().numpy(), kp, vp, cfg.pool_dtype, case.block_table,
                                         case.lens, cfg.page_tokens, case.scale, case.k_scale, case.v_scale,
                                         bounds_fn=bounds)
    rule, _ = op.decode_attention_split(case.q.float().numpy(), kp, vp, cfg.pool_dtype, case.block_table,
                                        case.lens, cfg.page_tokens, case.scale, case.k_scale, case.v_scale)
    return float(max(np.max(np.abs(split - one)), np.max(np.abs(rule - one))))


def nan_aware_error(got: np.ndarray, want: np.ndarray) -> float:
    """Max |got - want| over the outputs that are finite in both; inf when the two are not NaN at
    exactly the same outputs."""
    gn, wn = np.isnan(got), np.isnan(want)
    if not np.array_equal(gn, wn):
        return float("inf")
    ok = ~gn
    return float(np.max(np.abs(got[ok] - want[ok]))) if np.any(ok) else 0.0


def pin_split_vs_brute_force(case: wl.Case, seed: int = 0) -> float:
    """The split path (per-split partials, then the fixed-order merge) against brute force, under the
    split rule and under random partitions (empty splits included): NaN at exactly the outputs where
    torch's float64 attention gives NaN, 0 where a row sees no key, the rest equal to ~1e-12. This pins
    the merge's skip rule on non-finite and empty inputs, which finite partitions never reach."""
    kp, vp = oracle_pools(case)
    cfg = case.cfg
    rng = np.random.default_rng(seed)
    want = brute_force(case)

    def bounds(b, L):
        n = int(rng.integers(1, 9))
        cuts = np.sort(rng.integers(0, L + 1, size=n - 1)) if n > 1 else np.array([], dtype=np.int64)
        return [0] + [int(c) for c in cuts] + [L]

    err = 0.0
    for fn in (None, bounds):
        got, _ = op.decode_attention_split(case.q.float().numpy(), kp, vp, cfg.pool_dtype, case.block_table,
                                           case.lens, cfg.page_tokens, case.scale, case.k_scale, case.v_scale,
                                           bounds_fn=fn)
        err = max(err, nan_aware_error(got, want))
    return err


def nan_case() -> wl.Case:
    """A multi-row case whose outputs reach both unusual branches of the merge: a sequence shorter
    than the window (its first rows see no key: every split is empty), a NaN key that every row of
    its sequence sees, and a NaN in one element of one value."""
    cfg = wl.CONFIGS["verify_small"]
    cfg = type(cfg)(**{**cfg.__dict__, "rows": 4, "h_q": 6, "h_kv": 2, "d": 64, "page_tokens": 16})
    case = wl.make_case(cfg, lens=[3, 50, 130, 600])
    case.k_raw[int(case.tok_offset[1]) + 5, 0, 7] = float("nan")      # sequence 1, KV head 0, position 5
    case.v_raw[int(case.tok_offset[3]) + 300, 1, 11] = float("nan")   # sequence 3, KV head 1, position 300
    return case


def pin_bf16_vs_torch(x: np.ndarray) -> int:
    """Number of bf16 codes that differ from torch's cast (NaNs compared as NaN-ness)."""
    x = np.asarray(x, dtype=np.float32)
    ours = fm.bf16_encode(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    ours_nan = ((ours & 0x7F80) == 0x7F80) & ((ours & 0x7F) != 0)
    return int(np.sum((ours != ref) & ~nan) + np.sum(nan & ~ours_nan))


def pin_e4m3_vs_torch(x: np.ndarray) -> int:
    """Number of E4M3 codes that differ from torch's cast, on magnitudes below 464
    (torch does not saturate: from 464 up it returns NaN where the format's
    saturating conversion returns 448)."""
    x = np.asarray(x, dtype=np.float32)
    assert np.all(np.abs(x) < 464.0)
    ours = fm.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return int(np.sum(ours != ref))
