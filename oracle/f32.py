"""Binary32 / bf16 storage rules, written out exactly.

bf16 is storage only: a bf16 value widens to f32 by a 16-bit shift, and an f32
value reaches bf16 by one round to nearest, ties to even (presk "Native
execution", "bf16 is storage only"; NaN stays NaN, overflow goes to
infinity).  ``rn_f32`` rounds an exact rational to binary32 with gradual
underflow; the oracle uses it wherever a value is defined exactly (a
hyperparameter, a correctly rounded exp or erf) and must be stored in f32.
"""

from __future__ import annotations

from fractions import Fraction

import numpy as np

F32_MAX = float(np.finfo(np.float32).max)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float32 values (exact: a 16-bit shift)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """float32 -> uint16 bf16 bits, round to nearest even; NaN -> quiet NaN."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32)
    r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    nan = np.isnan(x)
    if nan.any():
        r = np.where(nan, (b >> np.uint32(16)) | np.uint32(0x0040), r)
    return r.astype(np.uint16)


def widen(arr: np.ndarray, dtype: str) -> np.ndarray:
    """Stored input -> f32 values ("f32" arrays pass through, "bf16" are bits)."""
    if dtype == "bf16":
        return bf16_to_f32(arr)
    if dtype == "f32":
        return np.asarray(arr, dtype=np.float32)
    raise ValueError(f"unknown storage dtype {dtype!r}")


def store(x32: np.ndarray, dtype: str) -> np.ndarray:
    """Round an f32 root to its storage type (f32: unchanged; bf16: bits)."""
    if dtype == "f32":
        return np.asarray(x32, dtype=np.float32)
    if dtype == "bf16":
        return f32_to_bf16(x32)
    raise ValueError(f"unknown storage dtype {dtype!r}")


def _floor_log2(q: Fraction) -> int:
    """floor(log2(q)) for a positive rational."""
    n, d = q.numerator, q.denominator
    e = n.bit_length() - d.bit_length()
    # 2^e <= q < 2^(e+1) after at most one correction step
    if (n << max(0, -e)) < (d << max(0, e)):
        e -= 1
    return e


def rn_f32(q) -> np.float32:
    """Round an exact rational (Fraction, int, or an exactly convertible value)
    to binary32: nearest, ties to even, gradual underflow, overflow to inf."""
    q = Fraction(q)
    if q == 0:
        return np.float32(0.0)
    neg = q < 0
    a = -q if neg else q
    e = _floor_log2(a)
    qe = max(e, -126) - 23            # exponent of one unit in the last place
    scaled = a / Fraction(2) ** qe
    m = scaled.numerator // scaled.denominator
    rem = scaled - m
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and (m & 1)):
        m += 1
    val = float(m) * 2.0 ** qe        # exact in binary64
    if val >= 2.0 ** 128:
        val = float("inf")
    out = np.float32(val)
    return -out if neg else out


def f32_ulp(x: float) -> float:
    """Spacing of binary32 numbers at |x| (towards +inf), as a binary64 value."""
    a = np.abs(np.float32(x))
    if np.isinf(a):
        return float("inf")
    nxt = np.nextafter(a, np.float32(np.inf))
    return float(nxt) - float(a)
