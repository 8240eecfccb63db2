"""Pins of the oracle's cache formats: torch-CPU casts and decode tables, closed-form points."""

import json
import os

import numpy as np
import torch

import oracle.formats as fm
from tests import pins

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _interesting_f32(rng, n=200_000):
    x = rng.standard_normal(n).astype(np.float32) * np.float32(2.0) ** rng.integers(-140, 128, n).astype(np.float32)
    edge = np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, np.nan, 1e-45, -1e-45, 3.4028235e38, -3.4028235e38,
                     1.17549435e-38, 1.0 + 2.0 ** -8, 1.0 + 2.0 ** -9, 1.0 + 3 * 2.0 ** -9],
                    dtype=np.float32)
    return np.concatenate([x, edge])


def test_bf16_encode_matches_torch_cast():
    rng = np.random.default_rng(0)
    x = _interesting_f32(rng)
    assert pins.pin_bf16_vs_torch(x) == 0


def test_bf16_ties_round_to_even():
    # bit patterns with the dropped half exactly 0x8000: ties go to the even upper half
    uppers = np.arange(0x3F80, 0x3F90, dtype=np.uint32)
    x = ((uppers << 16) | 0x8000).view(np.float32)
    got = fm.bf16_encode(x)
    want = np.where(uppers % 2 == 0, uppers, uppers + 1).astype(np.uint16)
    assert np.array_equal(got, want)
    assert pins.pin_bf16_vs_torch(x) == 0


def test_bf16_decode_every_code():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = fm.bf16_decode(codes)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).double().numpy()
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()


def test_e4m3_decode_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ours = fm.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()
    # closed-form points of the format definition
    assert np.nanmax(ours) == 448.0 and np.nanmin(ours) == -448.0
    assert ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6 and ours[0x38] == 1.0
    assert np.isnan(ours[0x7F]) and np.isnan(ours[0xFF]) and np.sum(np.isnan(ours)) == 2


def test_e4m3_encode_matches_torch_cast_in_range():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(200_000) * 2.0 ** rng.uniform(-12, 8.7, 200_000)).astype(np.float32)
    x = x[np.abs(x) < 464.0]
    # every grid value, every midpoint between neighbours (ties), and points just off the midpoints
    grid = np.unique(fm.e4m3_decode(np.arange(256, dtype=np.uint8)))
    grid = grid[np.isfinite(grid)]
    mids = (grid[:-1] + grid[1:]) / 2
    extra = np.concatenate([grid, mids, np.nextafter(mids.astype(np.float32), np.float32(np.inf)),
                            np.nextafter(mids.astype(np.float32), np.float32(-np.inf)), [460.0, -460.0]])
    x = np.concatenate([x, extra.astype(np.float32)])
    assert pins.pin_e4m3_vs_torch(x) == 0


def test_e4m3_saturates_and_keeps_nan():
    x = np.array([464.0, 480.0, 1e6, np.inf, -464.0, -np.inf, np.nan], dtype=np.float32)
    got = fm.e4m3_encode(x)
    assert list(got[:4]) == [0x7E] * 4
    assert list(got[4:6]) == [0xFE] * 2
    assert np.isnan(fm.e4m3_decode(got[6:]))[0]


def test_e4m3_round_trip_every_finite_code():
    codes = np.arange(256, dtype=np.uint8)
    vals = fm.e4m3_decode(codes)
    fin = np.isfinite(vals)
    back = fm.e4m3_encode(vals[fin].astype(np.float32))
    assert np.array_equal(back, codes[fin])


def test_e4m3_worked_points():
    """Points derived by hand from the format definition (tests/golden/e4m3_points.json)."""
    with open(os.path.join(GOLDEN, "e4m3_points.json")) as f:
        g = json.load(f)
    for p in g["points"]:
        got = int(fm.e4m3_encode(np.array([p["x"]], dtype=np.float32))[0])
        assert got == int(p["code"], 16), p
        if p.get("value") is not None:
            assert fm.e4m3_decode(np.array([got], dtype=np.uint8))[0] == p["value"], p
