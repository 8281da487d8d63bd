"""Correctly rounded binary32 exp and erf.

The pages fix that a fusion group computes every member in f32 and that gelu
is the exact x*Phi(x) through erf (presk "Native execution", realizations:
gelu is the exact x*Phi(x) through erf), and that every executor must compute
the same transcendental bits (presk "Native execution", The Cranelift
backend: one libm for all executors).  They do not fix which f32 function
that is.  The reading taken here: an exp or erf node returns the correctly
rounded value RN_f32(exp(x)) / RN_f32(erf(x)), nearest with ties to even,
gradual underflow, overflow to infinity.  That value has a plain definition,
so two independent implementations agree bit for bit without sharing code.

How it is evaluated (plainly, not fast): the function is computed in binary64
(error a few units of 2^-53) and rounded once to binary32.  That is the
correctly rounded result unless the binary64 value lies near a binary32
rounding boundary (a midpoint between two neighbours).  Those rare inputs --
within 2^-16 of a binary32 ulp of a midpoint, far wider than the binary64
error -- are recomputed exactly enough with Python's ``decimal`` module (exp:
``Decimal.exp`` at 60 digits, correctly rounded; erf: its Maclaurin series at
80 digits) and rounded from the exact rational.
"""

from __future__ import annotations

import math
from decimal import Decimal, localcontext
from fractions import Fraction

import numpy as np

from .f32 import rn_f32

try:  # vectorised binary64 erf; math.erf is the fallback
    from scipy.special import erf as _erf64
except Exception:  # pragma: no cover - scipy is present on both machines
    _erf64 = np.vectorize(math.erf, otypes=[np.float64])

_TWO_128 = 2.0 ** 128
_F32_MAX = float(np.finfo(np.float32).max)


def _ambiguous(yd: np.ndarray) -> np.ndarray:
    """True where the binary64 value yd (>= 0) lies within 2^-16 ulp of a binary32
    rounding boundary, so that rounding it once might not round the exact value."""
    with np.errstate(over="ignore", invalid="ignore"):
        y32 = yd.astype(np.float32)
        a = y32.astype(np.float64)
        up = np.nextafter(y32, np.float32(np.inf)).astype(np.float64)
        dn = np.nextafter(y32, np.float32(-np.inf)).astype(np.float64)
        # The boundary above FLT_MAX is FLT_MAX + ulp/2 = 2^128 - 2^103.
        up = np.where(y32 == np.float32(_F32_MAX), _TWO_128, up)
        isinf = np.isinf(a)
        dn = np.where(isinf, _F32_MAX, dn)
        a = np.where(isinf, _TWO_128, a)
        mid_hi = 0.5 * (a + up)
        mid_lo = 0.5 * (a + dn)
        gap = np.minimum(up - a, a - dn)
        tol = gap * 2.0 ** -16
        amb = (np.abs(yd - mid_hi) <= tol) | (np.abs(yd - mid_lo) <= tol)
    return amb & np.isfinite(yd)


def _check_decided(q: Fraction, digits: int) -> None:
    """Refuse a high-precision value that is itself too close to a rounding
    boundary to decide (never expected: the exact value is transcendental)."""
    r = rn_f32(q)
    a = Fraction(float(r)) if np.isfinite(r) else Fraction(2) ** 128
    up = np.nextafter(np.float32(abs(r)), np.float32(np.inf))
    dn = np.nextafter(np.float32(abs(r)), np.float32(-np.inf))
    aa = abs(a)
    up_f = Fraction(float(up)) if np.isfinite(up) else Fraction(2) ** 128
    for nb in (up_f, Fraction(float(dn))):
        mid = (aa + nb) / 2
        if abs(abs(q) - mid) <= abs(q) * Fraction(1, 10 ** (digits - 8)):
            raise ArithmeticError(f"rounding of {q} undecided at {digits} digits")


# -------------------------------------------------------------------- exp

def _exp_exact(x: np.float32) -> np.float32:
    with localcontext() as ctx:
        ctx.prec = 60
        v = Decimal(float(x)).exp()
    q = Fraction(v)
    _check_decided(q, 60)
    return rn_f32(q)


def exp_f32(x: np.ndarray) -> np.ndarray:
    """Correctly rounded binary32 exp, elementwise."""
    x = np.asarray(x, dtype=np.float32)
    with np.errstate(over="ignore", under="ignore", invalid="ignore"):
        yd = np.exp(x.astype(np.float64))
        y = yd.astype(np.float32)
    amb = _ambiguous(yd)
    if amb.any():
        flat_x = x.reshape(-1)
        flat_y = y.reshape(-1)
        for i in np.flatnonzero(amb.reshape(-1)):
            flat_y[i] = _exp_exact(flat_x[i])
        y = flat_y.reshape(x.shape)
    return y


# -------------------------------------------------------------------- erf

_PI_CACHE = {}


def _pi(prec: int) -> Decimal:
    """pi to prec digits by Machin's formula, pi = 16 atan(1/5) - 4 atan(1/239)."""
    if prec in _PI_CACHE:
        return _PI_CACHE[prec]
    with localcontext() as ctx:
        ctx.prec = prec + 10

        def atan_inv(n: int) -> Decimal:
            x = Decimal(1) / n
            x2 = x * x
            term, total, k = x, x, 1
            eps = Decimal(10) ** (-(prec + 8))
            while True:
                term = -term * x2
                k += 2
                t = term / k
                if abs(t) < eps:
                    break
                total += t
            return total

        p = 16 * atan_inv(5) - 4 * atan_inv(239)
    _PI_CACHE[prec] = +p
    return _PI_CACHE[prec]


def _erf_exact(x: np.float32) -> np.float32:
    """erf by its Maclaurin series, 2/sqrt(pi) * sum (-1)^n x^(2n+1) / (n! (2n+1)),
    at 80 digits; used only where |x| < 6 (beyond, erf rounds to +-1 by far)."""
    xf = float(x)
    if abs(xf) >= 6.0:
        return np.float32(math.copysign(1.0, xf))
    with localcontext() as ctx:
        ctx.prec = 80
        X = Decimal(xf)
        x2 = X * X
        term = X            # x^(2n+1) / n!
        total = X
        n = 0
        eps = Decimal(10) ** -85
        while True:
            n += 1
            term = -term * x2 / n
            t = term / (2 * n + 1)
            total += t
            if abs(t) < eps:
                break
        v = total * 2 / _pi(80).sqrt()
    q = Fraction(v)
    _check_decided(q, 60)
    return rn_f32(q)


def erf_f32(x: np.ndarray) -> np.ndarray:
    """Correctly rounded binary32 erf, elementwise (odd: erf(-x) = -erf(x))."""
    x = np.asarray(x, dtype=np.float32)
    ax = np.abs(x)
    with np.errstate(under="ignore", invalid="ignore"):
        yd = _erf64(ax.astype(np.float64))
        y = yd.astype(np.float32)
    amb = _ambiguous(yd)
    if amb.any():
        flat_x = ax.reshape(-1)
        flat_y = y.reshape(-1)
        for i in np.flatnonzero(amb.reshape(-1)):
            flat_y[i] = _erf_exact(flat_x[i])
        y = flat_y.reshape(x.shape)
    # odd symmetry: copy x's sign (keeps erf(-0) = -0 and NaN as NaN)
    return np.copysign(y, x).astype(np.float32)


# -------------------------------------------------------------------- log

def _log_exact(x: np.float32) -> np.float32:
    with localcontext() as ctx:
        ctx.prec = 60
        v = Decimal(float(x)).ln()
    q = Fraction(v)
    _check_decided(q, 60)
    return rn_f32(q)


def log_f32(x: np.ndarray) -> np.ndarray:
    """Correctly rounded binary32 natural logarithm, elementwise: log(+-0) =
    -inf, log(x < 0) = NaN, log(+inf) = +inf, log(1) = +0, NaN stays NaN."""
    x = np.asarray(x, dtype=np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        yd = np.log(x.astype(np.float64))
        y = yd.astype(np.float32)
    amb = _ambiguous(np.abs(yd))
    if amb.any():
        flat_x = x.reshape(-1)
        flat_y = y.reshape(-1)
        for i in np.flatnonzero(amb.reshape(-1)):
            flat_y[i] = _log_exact(flat_x[i])
        y = flat_y.reshape(x.shape)
    return y


# -------------------------------------------------------------------- tanh

def _tanh_exact(a: np.float32) -> np.float32:
    """tanh(a) = (e^(2a) - 1) / (e^(2a) + 1) at 120 digits, a >= 0 (the
    cancellation in the numerator costs at most 45 of them)."""
    with localcontext() as ctx:
        ctx.prec = 120
        e2 = (Decimal(float(a)) * 2).exp()
        v = (e2 - 1) / (e2 + 1)
    q = Fraction(v)
    _check_decided(q, 60)
    return rn_f32(q)


def tanh_f32(x: np.ndarray) -> np.ndarray:
    """Correctly rounded binary32 tanh, elementwise (odd: tanh(+-0) = +-0,
    tanh(+-inf) = +-1, NaN stays NaN)."""
    x = np.asarray(x, dtype=np.float32)
    ax = np.abs(x)
    with np.errstate(under="ignore", invalid="ignore"):
        yd = np.tanh(ax.astype(np.float64))
        y = yd.astype(np.float32)
    amb = _ambiguous(yd)
    if amb.any():
        flat_x = ax.reshape(-1)
        flat_y = y.reshape(-1)
        for i in np.flatnonzero(amb.reshape(-1)):
            flat_y[i] = _tanh_exact(flat_x[i])
        y = flat_y.reshape(x.shape)
    return np.copysign(y, x).astype(np.float32)
