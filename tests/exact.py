"""Exact-arithmetic reference helpers for the oracle's pins (test-only).

Written independently of ``oracle``: binary32 rounding here searches the
neighbours of an approximation and keeps the one nearest to the exact rational
(ties to the even significand), where the oracle scales and rounds an integer.
"""

from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

_INF = float("inf")


def _neighbours(c: np.float32):
    lo = np.nextafter(c, np.float32(-np.inf))
    hi = np.nextafter(c, np.float32(np.inf))
    return [lo, c, hi]


def _even(c: np.float32) -> bool:
    return (int(np.asarray(c, dtype=np.float32).view(np.uint32)) & 1) == 0


def rn32(q: Fraction) -> np.float32:
    """Nearest binary32 to the rational q (ties to even), inf past the overflow
    boundary 2^128 - 2^103."""
    if q == 0:
        return np.float32(0.0)
    bound = Fraction(2) ** 128 - Fraction(2) ** 103
    if q >= bound:
        return np.float32(np.inf)
    if q <= -bound:
        return np.float32(-np.inf)
    try:
        approx = np.float32(float(q))
    except OverflowError:
        approx = np.float32(np.inf if q > 0 else -np.inf)
    if np.isinf(approx):
        approx = np.float32(np.finfo(np.float32).max) * np.float32(np.sign(float(q)))
    best, bestd = None, None
    for c in _neighbours(approx):
        if not np.isfinite(c):
            continue
        d = abs(Fraction(float(c)) - q)
        if bestd is None or d < bestd or (d == bestd and _even(c)):
            best, bestd = c, d
    return np.float32(best)


def sqrt32(q: Fraction) -> np.float32:
    """Correctly rounded binary32 sqrt of a non-negative rational."""
    if q == 0:
        return np.float32(0.0)
    c = np.float32(math.sqrt(float(q)))
    cands = [x for x in _neighbours(c) if np.isfinite(x) and x >= 0]
    cands = sorted(set(float(x) for x in cands))
    # pick the candidate whose rounding interval holds sqrt(q): compare squares
    best = None
    for a in cands:
        lo = a - (a - float(np.nextafter(np.float32(a), np.float32(-1.0)))) / 2 if a > 0 else 0.0
        hi = a + (float(np.nextafter(np.float32(a), np.float32(np.inf))) - a) / 2
        flo, fhi = Fraction(lo), Fraction(hi)
        inside_lo = q > flo * flo or (q == flo * flo and _even(np.float32(a)))
        inside_hi = q < fhi * fhi or (q == fhi * fhi and _even(np.float32(a)))
        if inside_lo and inside_hi:
            best = a
    assert best is not None, q
    return np.float32(best)


def f32_binop(name: str, a: np.float32, b: np.float32) -> np.float32:
    """IEEE binary32 add/sub/mul/div as exact rational then one rounding; specials
    (inf, nan, division by zero) follow IEEE 754."""
    a, b = np.float32(a), np.float32(b)
    if not (np.isfinite(a) and np.isfinite(b)) or (name == "DIV" and b == 0):
        # every such IEEE result is exact (an infinity, a NaN or a signed zero),
        # so binary64 computes it and the narrowing changes nothing
        with np.errstate(all="ignore"):
            fa, fb = np.float64(a), np.float64(b)
            r = {"ADD": fa + fb, "SUB": fa - fb, "MUL": fa * fb, "DIV": fa / fb}[name]
        return np.float32(r)
    A, B = Fraction(float(a)), Fraction(float(b))
    if name == "ADD":
        q = A + B
    elif name == "SUB":
        q = A - B
    elif name == "MUL":
        q = A * B
    elif name == "DIV":
        q = A / B
    else:
        raise ValueError(name)
    r = rn32(q)
    if r == 0:
        # sign of an exact zero result (IEEE 754 round to nearest)
        if q == 0:
            if name == "ADD":
                neg = np.signbit(a) and np.signbit(b)
            elif name == "SUB":
                neg = np.signbit(a) and not np.signbit(b)
            else:
                neg = np.signbit(a) != np.signbit(b)
        else:
            neg = q < 0
        r = np.float32(-0.0) if neg else np.float32(0.0)
    return r


def same_bits(x, y) -> bool:
    """Bitwise equality of binary32 values, any NaN equal to any NaN."""
    x = np.asarray(x, dtype=np.float32)
    y = np.asarray(y, dtype=np.float32)
    if x.shape != y.shape:
        return False
    both_nan = np.isnan(x) & np.isnan(y)
    eq = x.view(np.uint32) == y.view(np.uint32)
    return bool(np.all(eq | both_nan))


def mpf_fraction(v) -> Fraction:
    """An mpmath mpf as an exact Fraction."""
    sign, man, exp, _bc = v._mpf_
    q = Fraction(int(man)) * (Fraction(2) ** int(exp))
    return -q if sign else q
