"""Planted controls: a mistake planted in the oracle (on the CPU) must make its pins fail.

Each test patches one step of the oracle with a plausible slip and checks that the
pin guarding that step goes red. Nothing here touches the GPU.
"""

import numpy as np
import pytest

import oracle.formats as fm
import oracle.paged as op
import workloads as wl
from tests import pins

TOL = 1e-12


@pytest.fixture
def multi_row_case():
    cfg = wl.CONFIGS["verify_small"]
    cfg = type(cfg)(**{**cfg.__dict__, "rows": 4, "h_q": 6, "h_kv": 2, "d": 64, "page_tokens": 16})
    return wl.make_case(cfg, lens=[50, 130])


@pytest.fixture
def fp8_case():
    return wl.make_case("prefill_small", lens=[200])


def test_control_clean(multi_row_case, fp8_case):
    assert pins.pin_brute_force(multi_row_case) < TOL
    assert pins.pin_brute_force(fp8_case) < TOL


def test_control_wrong_gqa_head_map(monkeypatch, multi_row_case):
    monkeypatch.setattr(op, "kv_head", lambda h, h_q, h_kv: h % h_kv)
    assert pins.pin_brute_force(multi_row_case) > 1e-3


def test_control_causal_off_by_one(monkeypatch, multi_row_case):
    monkeypatch.setattr(op, "query_position", lambda length, rows, r: length - rows + r + 1)
    assert pins.pin_brute_force(multi_row_case) > 1e-3


def test_control_causal_off_by_one_low(monkeypatch, multi_row_case):
    monkeypatch.setattr(op, "query_position", lambda length, rows, r: length - rows + r - 1)
    assert pins.pin_brute_force(multi_row_case) > 1e-3


def test_control_scale_dropped(monkeypatch, multi_row_case):
    orig = op.attend
    monkeypatch.setattr(op, "attend", lambda q, k, v, scale: orig(q, k, v, 1.0))
    assert pins.pin_brute_force(multi_row_case) > 1e-3


def test_control_keys_and_values_swapped(monkeypatch, multi_row_case):
    orig = op.attend
    monkeypatch.setattr(op, "attend", lambda q, k, v, scale: orig(q, v, k, scale))
    assert pins.pin_brute_force(multi_row_case) > 1e-3


def test_control_page_index_off_by_one(monkeypatch, multi_row_case):
    orig = op.read_sequence

    def shifted(pool, dtype, scale, block_row, length, h_kv, page_tokens):
        row = np.concatenate([block_row[1:], block_row[:1]])
        return orig(pool, dtype, scale, np.where(row < 0, block_row[0], row), length, h_kv, page_tokens)
    monkeypatch.setattr(op, "read_sequence", shifted)
    assert pins.pin_brute_force(multi_row_case) > 1e-3


def test_control_fp8_scale_not_inverted(monkeypatch, fp8_case):
    orig = op.append
    monkeypatch.setattr(op, "append", lambda pool, new, slots, P, dtype, scale=1.0:
                        orig(pool, np.asarray(new, np.float32) * np.float32(scale) * np.float32(scale),
                             slots, P, dtype, scale))
    assert pins.pin_brute_force(fp8_case) > 1e-3


def test_control_merge_drops_last_split(monkeypatch):
    case = wl.make_case("verify_small", lens=[900, 1300])
    orig = op.merge

    def drop_last(m, l, acc):
        m = np.array(m, dtype=np.float64)
        live = np.nonzero(m != -np.inf)[0]
        if live.size > 1:
            m[live[-1]] = -np.inf
        return orig(m, l, acc)
    monkeypatch.setattr(op, "merge", drop_last)
    assert pins.pin_merge_partitions(case) > 1e-3


def test_control_merge_without_rescale(monkeypatch):
    case = wl.make_case("ragged_small", lens=[700, 2100])

    def no_rescale(m, l, acc):
        m = np.asarray(m)
        live = m != -np.inf
        return np.asarray(acc)[live].sum(axis=0) / np.asarray(l)[live].sum()
    monkeypatch.setattr(op, "merge", no_rescale)
    assert pins.pin_merge_partitions(case) > 1e-3


def test_control_bf16_truncation(monkeypatch):
    def truncate(x):
        return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)
    monkeypatch.setattr(fm, "bf16_encode", truncate)
    x = np.random.default_rng(0).standard_normal(1000).astype(np.float32)
    assert pins.pin_bf16_vs_torch(x) > 100


class _HalfUpNumpy:
    """numpy, except that rint rounds halves up instead of to even."""
    def __getattr__(self, name):
        return getattr(np, name)

    @staticmethod
    def rint(v):
        return np.floor(np.asarray(v) + 0.5)


def test_control_e4m3_ties_away_from_zero(monkeypatch):
    grid = np.unique(fm.e4m3_decode(np.arange(256, dtype=np.uint8)))
    grid = grid[np.isfinite(grid) & (grid >= 0)]
    mids = ((grid[:-1] + grid[1:]) / 2).astype(np.float32)
    assert pins.pin_e4m3_vs_torch(mids) == 0
    monkeypatch.setattr(fm, "np", _HalfUpNumpy())
    assert pins.pin_e4m3_vs_torch(mids) > 10


def test_control_split_rule_without_page_alignment(monkeypatch):
    def unaligned(length, page_tokens):
        splits = max(1, min(-(-max(int(length), 1) // 256), 64))
        return splits, -(-int(length) // splits)
    monkeypatch.setattr(op, "split_plan", unaligned)
    starts = [x for L in (300, 1000, 5000) for x in op.split_bounds(L, 16)[:-1] if x < L]
    assert any(x % 16 for x in starts)


def test_control_merge_skips_unless_sum_positive(monkeypatch):
    # the rule of TensorFold PR #1219 ("Gotchas"): a chunk takes part only when its sum of weights is
    # positive. A split holding a NaN key has a NaN sum, so the rule drops it and hides the NaN.
    orig = op.merge

    def positive_sum_only(m, l, acc):
        m = np.array(m, dtype=np.float64)
        m[~(np.asarray(l, dtype=np.float64) > 0)] = -np.inf
        return orig(m, l, acc)
    case = pins.nan_case()
    assert pins.pin_split_vs_brute_force(case) < TOL
    monkeypatch.setattr(op, "merge", positive_sum_only)
    assert pins.pin_split_vs_brute_force(case) > 1e-3


def test_control_merge_of_no_live_split_is_nan(monkeypatch):
    # a merge that takes M over every split: with no visible key M = -inf and exp(m - M) = NaN

    def max_over_all(m, l, acc):
        m = np.asarray(m, dtype=np.float64)
        with np.errstate(invalid="ignore"):
            w = np.exp(m - m.max())
        return (w[:, None] * np.asarray(acc)).sum(axis=0) / (w * np.asarray(l)).sum()
    case = pins.nan_case()
    monkeypatch.setattr(op, "merge", max_over_all)
    assert pins.pin_split_vs_brute_force(case) > 1e-3
