"""Pins of the oracle's attention, split rule and merge (no GPU)."""

import json
import os

import numpy as np
import pytest
import torch

import oracle.formats as fm
import oracle.paged as op
import workloads as wl
from tests import pins

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

SMALL = ["tiny", "single_row_small", "verify_small", "prefill_small", "ragged_small"]


@pytest.mark.parametrize("name", ["tiny", "single_row_small", "verify_small", "prefill_small"])
def test_oracle_matches_brute_force_sdpa(name):
    cfg = wl.CONFIGS[name]
    case = wl.make_case(cfg, lens=(wl.draw_lens(cfg, np.random.default_rng(cfg.seed))[:2]
                                   if cfg.batch > 2 else None))
    assert pins.pin_brute_force(case) < 1e-12


def test_oracle_matches_brute_force_multi_row_short_sequences():
    # rows > length: the first rows see no key (output 0); lengths that end mid-page
    cfg = wl.CONFIGS["verify_small"]
    cfg = type(cfg)(**{**cfg.__dict__, "rows": 5, "h_q": 6, "h_kv": 2, "d": 64, "page_tokens": 16})
    case = wl.make_case(cfg, lens=[3, 17, 1, 0, 40])
    assert pins.pin_brute_force(case) < 1e-12
    out = pins.oracle_output(case)
    assert np.all(out[2, :4] == 0.0) and np.all(out[3] == 0.0)


def test_single_key_returns_its_value():
    cfg = wl.CONFIGS["single_row_small"]
    case = wl.make_case(cfg, lens=[1, 1, 1])
    kp, vp = pins.oracle_pools(case)
    out = pins.oracle_output(case, (kp, vp))
    for b in range(3):
        page = case.block_table[b, 0]
        for h in range(cfg.h_q):
            v0 = fm.decode(vp[page, h // cfg.group, 0], cfg.pool_dtype) * case.v_scale
            assert np.array_equal(out[b, 0, h], v0)


def test_identical_keys_return_mean_of_values():
    cfg = wl.CONFIGS["prefill_small"]
    case = wl.make_case(cfg, lens=[300])
    case.k_raw[:] = case.k_raw[7]          # every position has the same key
    kp, vp = pins.oracle_pools(case)
    out = pins.oracle_output(case, (kp, vp))
    for r in (0, 60, 127):
        pos = 300 - cfg.rows + r
        for h in (0, 5, 23):
            V = op.read_sequence(vp, cfg.pool_dtype, case.v_scale, case.block_table[0], 300, h // cfg.group,
                                 cfg.page_tokens)
            assert np.max(np.abs(out[0, r, h] - V[:pos + 1].mean(axis=0))) < 1e-13


def test_two_keys_worked_example():
    with open(os.path.join(GOLDEN, "two_keys.json")) as f:
        g = json.load(f)
    D, P = g["head_dim"], g["page_tokens"]
    kp = op.new_pool(1, 1, P, D, "f32")
    vp = op.new_pool(1, 1, P, D, "f32")
    op.append(kp, np.array(g["k"], dtype=np.float32)[:, None, :], np.array([0, 1]), P, "f32")
    op.append(vp, np.array(g["v"], dtype=np.float32)[:, None, :], np.array([0, 1]), P, "f32")
    q = np.array(g["q"], dtype=np.float32).reshape(1, 1, 1, D)
    out = op.decode_attention(q, kp, vp, "f32", np.array([[0]], dtype=np.int32), np.array([2]), P, g["scale"])
    assert np.max(np.abs(out[0, 0, 0] - np.array(g["expected"]))) < g["tolerance"]


@pytest.mark.parametrize("name", ["tiny", "verify_small", "ragged_small"])
def test_merge_of_any_partition_equals_one_pass(name):
    cfg = wl.CONFIGS[name]
    lens = None
    if name == "verify_small":
        lens = [900, 1300]
    if name == "ragged_small":
        lens = [1, 5, 300, 2100]
    case = wl.make_case(cfg, lens=lens)
    assert pins.pin_merge_partitions(case) < 1e-12


def test_split_rule():
    for P in (16, 64):
        for L in list(range(0, 700)) + [16128, 16129, 16385, 20000, 32768, 65537, 131072]:
            S, seg = op.split_plan(L, P)
            assert S == max(1, min(-(-max(L, 1) // 256), 64))
            assert seg % P == 0
            b = op.split_bounds(L, P)
            assert b[0] == 0 and b[-1] == L and all(x <= y for x, y in zip(b, b[1:]))
            assert all(x % P == 0 for x in b[:-1] if x < L)   # no non-empty split starts inside a page
            assert S * seg >= L
    assert op.split_plan(256, 16) == (1, 256)
    assert op.split_plan(257, 16) == (2, 144)
    assert op.split_plan(131072, 16) == (64, 2048)
    assert op.split_plan(32768, 64) == (64, 512)
    # a page larger than a split (a contiguous cache: one page per sequence) keeps 256-aligned splits
    for P in (1024, 4096, 1 << 17):
        for L in (1, 255, 256, 257, 4000, 32768, 131072):
            if L > P:
                continue
            S, seg = op.split_plan(L, P)
            assert S == max(1, min(-(-max(L, 1) // 256), 64)) and seg % 256 == 0 and S * seg >= L
    assert op.split_plan(4000, 4096) == (16, 256)
    assert op.split_plan(32768, 1 << 17) == (64, 512)
    # empty trailing splits exist when rounding to whole pages overshoots
    b = op.split_bounds(16385, 64)
    assert b[-2] == b[-1] == 16385


def test_page_permutation_leaves_output_identical():
    case = wl.make_case("ragged_small", lens=[1, 33, 700, 64])
    base = pins.oracle_output(case)
    perm, bt2 = wl.permute_pages(case, seed=5)
    cfg = case.cfg
    idx, _ = case.all_index()
    slots2 = wl.slots_with_table(case, bt2, "all")
    kp = op.new_pool(case.num_pages, cfg.h_kv, cfg.page_tokens, cfg.d, cfg.pool_dtype)
    vp = op.new_pool(case.num_pages, cfg.h_kv, cfg.page_tokens, cfg.d, cfg.pool_dtype)
    op.append(kp, case.k_raw.numpy()[idx], slots2, cfg.page_tokens, cfg.pool_dtype)
    op.append(vp, case.v_raw.numpy()[idx], slots2, cfg.page_tokens, cfg.pool_dtype)
    moved = pins.oracle_output(case, (kp, vp), bt2)
    assert np.array_equal(base, moved)


def test_gqa_equals_duplicated_kv_heads():
    case = wl.make_case("single_row_small", lens=[50, 333])
    cfg = case.cfg
    G = cfg.group
    base = pins.oracle_output(case)
    kp, vp = pins.oracle_pools(case)
    kp1 = np.repeat(kp, G, axis=1)     # KV head h // G copied to every query head h
    vp1 = np.repeat(vp, G, axis=1)
    out1 = op.decode_attention(case.q.float().numpy(), kp1, vp1, cfg.pool_dtype, case.block_table, case.lens,
                               cfg.page_tokens, case.scale)
    assert np.array_equal(base, out1)


def test_append_skips_out_of_range_slots():
    kp = op.new_pool(2, 1, 16, 8, "bf16", fill=0xFFFF)
    new = np.ones((4, 1, 8), dtype=np.float32)
    bad = op.append(kp, new, np.array([0, -1, 32, 31]), 16, "bf16")
    assert list(bad) == [False, True, True, False]
    assert np.all(kp[0, 0, 0] == 0x3F80) and np.all(kp[1, 0, 15] == 0x3F80)
    assert np.sum(kp != 0xFFFF) == 16


def test_append_applies_the_scale_in_fp32():
    x = np.array([[[1.0, -3.0, 100.0, 0.3]]], dtype=np.float32)
    kp = op.new_pool(1, 1, 16, 4, "e4m3")
    op.append(kp, x, np.array([5]), 16, "e4m3", scale=0.25)
    inv = np.float32(1.0) / np.float32(0.25)
    assert np.array_equal(kp[0, 0, 5], fm.e4m3_encode(x[0, 0] * inv))
    # by hand: 4 -> E=9,M=0; -12 -> E=10,M=4; 400 = 12.5 * 32 -> tie to even 12 -> 384, E=15,M=4; 1.2 -> 1.25, E=7,M=2
    assert list(kp[0, 0, 5]) == [0x48, 0xD4, 0x7C, 0x3A]


def test_workload_inputs_are_seeded():
    a = wl.make_case("ragged_small")
    b = wl.make_case("ragged_small")
    assert np.array_equal(a.lens, b.lens) and np.array_equal(a.block_table, b.block_table)
    assert torch.equal(a.k_raw, b.k_raw) and torch.equal(a.q, b.q)
    ids = a.block_table[a.block_table >= 0]
    assert len(np.unique(ids)) == ids.size and ids.max() < a.num_pages


def test_split_path_matches_brute_force_with_nan_and_empty_rows():
    case = pins.nan_case()
    want = pins.brute_force(case)
    G = case.cfg.group
    # the brute force itself shows both branches: NaN outputs and rows with no key
    assert np.all(np.isnan(want[1, :, :G])) and not np.any(np.isnan(want[1, :, G:]))
    assert np.all(np.isnan(want[3, :, G:, 11])) and not np.any(np.isnan(np.delete(want[3, :, G:], 11, axis=-1)))
    assert np.all(want[0, 0] == 0.0)
    assert pins.pin_split_vs_brute_force(case) < 1e-12
    # the one-pass oracle agrees with the brute force on the same outputs
    assert pins.nan_aware_error(pins.oracle_output(case), want) < 1e-12
