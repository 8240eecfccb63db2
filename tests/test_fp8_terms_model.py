"""CPU pins of the error bounds the tensor-core kernel's fp8 path rests on (E4M3 pools multiplied
as stored): a query vector and the softmax weights enter the E4M3 products as two E4M3 terms each,
hi = x rounded to 4 significant bits (Veltkamp's split in binary32) and lo = the rest, each stored
as an E4M3 code. These tests model that split in numpy binary32, store the terms with the oracle's
E4M3 rounding (itself pinned against torch and hand-worked points), and check the bounds the
kernel's tolerance is derived from:

- a query term pair is exact for every bf16 element of at least 2^-9 of its vector's largest
  (the vector scaled so that the largest lies in [128, 256)), and off by at most 2^-16 of the
  largest otherwise;
- a weight p in (0, 2^8.75] is off by at most 2^-9 p, plus 2^-9 when p < 2^-1.
"""

import numpy as np

from oracle import formats as fm

F32 = np.float32


def split4(x: np.ndarray):
    """Veltkamp's split with the factor 2^20 + 1 on binary32: hi has at most 4 significant bits,
    hi + lo == x exactly."""
    x = x.astype(F32)
    c = (x * F32(1048577.0)).astype(F32)
    hi = (c - (c - x).astype(F32)).astype(F32)
    lo = (x - hi).astype(F32)
    return hi, lo


def terms_value(x: np.ndarray) -> np.ndarray:
    """The value the two E4M3 terms of x carry, in float64."""
    hi, lo = split4(x)
    return fm.e4m3_decode(fm.e4m3_encode(hi)) + fm.e4m3_decode(fm.e4m3_encode(lo))


def test_split_is_exact_and_hi_has_four_bits():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(200_000) * np.exp2(rng.uniform(-12, 8, 200_000))).astype(F32)
    hi, lo = split4(x)
    assert np.array_equal(hi.astype(np.float64) + lo.astype(np.float64), x.astype(np.float64))
    m, _ = np.frexp(hi[hi != 0].astype(np.float64))
    assert np.array_equal(m * 16, np.round(m * 16))       # 4 significant bits


def bf16_vectors(rng, n, d, spread):
    v = rng.standard_normal((n, d)) * np.exp2(rng.uniform(-spread, 0, (n, d)))
    return fm.bf16_decode(fm.bf16_encode(v.astype(F32))).astype(F32)


def test_query_terms_exact_near_the_vectors_largest():
    rng = np.random.default_rng(1)
    for spread in (0, 4, 12, 24):
        q = bf16_vectors(rng, 2000, 256, spread)
        amax = np.max(np.abs(q), axis=1, keepdims=True)
        # the kernel's power of two: the largest |element| into [128, 256)
        e = 7 - (np.frexp(amax)[1] - 1)
        x = (q * np.exp2(e)).astype(F32)                    # exact: a power of two
        xm = np.max(np.abs(x), axis=1, keepdims=True)
        assert np.all((xm >= 128) & (xm < 256))
        got = terms_value(x)
        big = np.abs(x) >= xm * 2.0 ** -9
        assert np.array_equal(got[big], x[big].astype(np.float64)), spread
        assert np.all(np.abs(got - x) <= xm * 2.0 ** -16), spread


def test_weight_terms_error_bound():
    rng = np.random.default_rng(2)
    p = np.exp2(rng.uniform(-24, 8.75, 400_000)).astype(F32)
    # ties of the 4-bit rounding and of the E4M3 grid, around every binade the weights reach
    k = np.arange(-24, 9)
    grid = np.concatenate([np.ldexp(1.0 + j / 16.0, k) for j in range(16)] + [np.ldexp(1.5, k - 9)])
    p = np.concatenate([p, grid[(grid > 0) & (grid <= 2.0 ** 8.75)].astype(F32)])
    got = terms_value(p)
    err = np.abs(got - p.astype(np.float64))
    bound = 2.0 ** -9 * p + np.where(p < 0.5, 2.0 ** -9, 0.0)
    assert np.all(err <= bound)
    # and no code saturates: the largest weight the running max allows stays below 448
    hi, _ = split4(np.array([2.0 ** 8.75], dtype=F32))
    assert fm.e4m3_decode(fm.e4m3_encode(hi))[0] == hi[0] < 448


def test_floor_budget_bound_of_a_tile():
    # the worst tile the kernel accepts without moving its running max: as many weights below
    # 2^-1 as its largest weight allows; each is off by at most 2^-9, so the tile's weights are
    # off by at most 2^-8 of their sum
    rng = np.random.default_rng(3)
    for _ in range(2000):
        pmax = np.exp2(rng.uniform(0, 8.75))
        n_small = min(63, int(np.floor(pmax)))
        small = np.exp2(rng.uniform(-20, -1, n_small))
        rest = np.exp2(rng.uniform(-1, np.log2(pmax), 63 - n_small))
        p = np.concatenate([[pmax], small, rest]).astype(F32)
        err = np.sum(np.abs(terms_value(p) - p.astype(np.float64)))
        assert err <= 2.0 ** -8 * np.sum(p.astype(np.float64))
