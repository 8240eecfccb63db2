"""Cache formats, written from their definitions (oracle; test infrastructure only).

The paged pool stores keys and values in the pool's dtype, cast on store
(nbxtensor/ops/paged_decode_attn.py, ``paged_kv_append_kernel``: the D values of
a new position are stored converted to the pool's element type). The pool dtypes
are fp32, bf16 and fp8 E4M3 with one fp32 scale per tensor (the fp8 cache of
TensorFold PR #1219, "Checks": partial and merge checked on bf16 and fp8 caches).

Codes are held in integer arrays of the format's width: fp32 pools as float32,
bf16 as uint16 bit patterns, E4M3 as uint8 bit patterns.

bf16: the upper 16 bits of an IEEE binary32 (1 sign, 8 exponent, 7 fraction
bits). Conversion from fp32 rounds to nearest, ties to even, on the dropped 16
bits; a NaN stays a (quiet) NaN.

E4M3 (OCP 8-bit floating point, the "FN" variant): 1 sign, 4 exponent bits with
bias 7, 3 mantissa bits. Exponent field 0 holds subnormals M/8 * 2^-6; fields
1..15 hold (1 + M/8) * 2^(E-7), except E=15, M=7 which is NaN. There is no
infinity; the largest finite magnitude is 1.75 * 2^8 = 448 and the smallest
subnormal 2^-9. Conversion rounds to nearest, ties to even, and saturates: any
magnitude above 448 (infinity included) becomes 448 with its sign; NaN stays NaN.
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E4M3_NAN = 0x7F
BF16_QNAN = 0x7FC0

CODE_DTYPE = {"f32": np.float32, "bf16": np.uint16, "e4m3": np.uint8}
ELT_BYTES = {"f32": 4, "bf16": 2, "e4m3": 1}


def bf16_encode(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even on the 16 dropped bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32).astype(np.uint64)
    upper = bits >> 16
    lower = bits & 0xFFFF
    round_up = (lower > 0x8000) | ((lower == 0x8000) & ((upper & 1) == 1))
    out = upper + round_up.astype(np.uint64)   # a carry moves into the exponent: the next binade, or infinity
    is_nan = np.isnan(x)
    out = np.where(is_nan, (upper & 0x8000) | BF16_QNAN, out)
    return out.astype(np.uint16)


def bf16_decode(codes: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 (exact): the pattern is the top half of a binary32."""
    codes = np.ascontiguousarray(codes, dtype=np.uint16)
    return (codes.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """fp32 -> E4M3 bit patterns: round to nearest even on the E4M3 grid, saturate
    magnitudes above 448 to 448, NaN -> 0x7F."""
    x = np.asarray(x, dtype=np.float32)
    a = np.abs(x.astype(np.float64))
    sign = np.signbit(x).astype(np.uint8) << 7
    finite = np.isfinite(a)
    a_f = np.where(finite, a, 0.0)
    # spacing of the grid around a: 2^-9 below 2^-6 (subnormals), else 2^(e-3) in [2^e, 2^(e+1))
    _, k = np.frexp(a_f)                       # a = f * 2^k with f in [0.5, 1)
    e = np.maximum(k - 1, -6)
    quantum = np.ldexp(1.0, e - 3)
    n = a_f / quantum                          # exact: division by a power of two
    v = np.rint(n) * quantum                   # ties to even: the even multiple has mantissa lsb 0
    v = np.where(finite, v, np.inf)
    v = np.minimum(v, E4M3_MAX)                # satfinite
    # encode v (a grid value or 0)
    sub = v < 2.0 ** -6
    m_sub = np.rint(v / 2.0 ** -9)
    _, kv = np.frexp(np.where(sub, 1.0, v))
    ev = kv - 1                                # v in [2^ev, 2^(ev+1))
    m_norm = np.rint(v / np.ldexp(1.0, ev) * 8.0 - 8.0)
    E = np.where(sub, 0, ev + 7)
    M = np.where(sub, m_sub, m_norm)
    code = (E.astype(np.int64) << 3) | M.astype(np.int64)
    code = code.astype(np.uint8) | sign
    code = np.where(np.isnan(x), np.uint8(E4M3_NAN), code)
    return code.astype(np.uint8)


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """E4M3 bit patterns -> float64 (exact)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = np.where((c >> 7) & 1 == 1, -1.0, 1.0)
    E = (c >> 3) & 0xF
    M = c & 0x7
    sub = M / 8.0 * 2.0 ** -6
    norm = (1.0 + M / 8.0) * np.ldexp(1.0, E - 7)
    v = np.where(E == 0, sub, norm)
    v = np.where((E == 15) & (M == 7), np.nan, v)
    return s * v


def encode(x: np.ndarray, dtype: str) -> np.ndarray:
    """fp32 values -> codes of the pool dtype."""
    x = np.asarray(x, dtype=np.float32)
    if dtype == "f32":
        return x.copy()
    if dtype == "bf16":
        return bf16_encode(x)
    if dtype == "e4m3":
        return e4m3_encode(x)
    raise ValueError(dtype)


def decode(codes: np.ndarray, dtype: str) -> np.ndarray:
    """Codes of the pool dtype -> float64 values."""
    if dtype == "f32":
        return np.asarray(codes, dtype=np.float32).astype(np.float64)
    if dtype == "bf16":
        return bf16_decode(codes)
    if dtype == "e4m3":
        return e4m3_decode(codes)
    raise ValueError(dtype)
