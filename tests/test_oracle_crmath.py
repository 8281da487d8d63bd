"""Pins for the oracle's correctly rounded exp and erf.

An independent multiprecision library (mpmath, 200 bits) gives the exact value;
rounding it with the test's own neighbour search gives the correctly rounded
binary32 result the oracle must return, bit for bit.
"""

import math

import numpy as np
import pytest

from oracle import crmath
from tests.exact import mpf_fraction, rn32, same_bits

mpmath = pytest.importorskip("mpmath")
mpmath.mp.prec = 200


def _cr(fn, x):
    return np.array([rn32(mpf_fraction(fn(mpmath.mpf(float(v))))) for v in x], dtype=np.float32)


def _sample_binades(lo_exp, hi_exp, per, seed):
    rng = np.random.default_rng(seed)
    out = []
    for e in range(lo_exp, hi_exp + 1):
        m = rng.integers(0, 2 ** 23, per, dtype=np.uint64).astype(np.uint32)
        bits = (np.uint32(e + 127) << np.uint32(23)) | m
        v = bits.view(np.float32)
        out.append(v)
        out.append(-v)
    return np.concatenate(out)


def test_exp_correctly_rounded_across_binades():
    x = _sample_binades(-30, 6, 40, 1)
    x = x[(x > -104.0) & (x < 89.0)]
    assert same_bits(crmath.exp_f32(x), _cr(mpmath.exp, x))


def test_exp_subnormal_and_overflow_edges():
    x = np.array([-87.33654, -87.3366, -90.0, -100.0, -103.278, -103.97207, -103.972084, -104.0,
                  88.7228317, 88.72283935546875, 88.0, 89.0], dtype=np.float32)
    assert same_bits(crmath.exp_f32(x), _cr(mpmath.exp, x))


def test_exp_special_values():
    x = np.array([0.0, -0.0, np.inf, -np.inf, np.nan], dtype=np.float32)
    y = crmath.exp_f32(x)
    assert y[0] == 1.0 and y[1] == 1.0 and np.isposinf(y[2]) and y[3] == 0.0 and np.isnan(y[4])
    # below 2^-25 in magnitude the result rounds to 1 (or 1 - 2^-24 from below)
    assert crmath.exp_f32(np.float32(2 ** -26)) == 1.0
    assert crmath.exp_f32(np.float32(2 ** -24)) == np.float32(1.0 + 2 ** -23)


def test_exp_rare_boundary_cases_resolved_exactly():
    # inputs whose binary64 exp lands near a binary32 midpoint take the exact path
    x = np.linspace(-20, 20, 400_001, dtype=np.float32)
    yd = np.exp(x.astype(np.float64))
    amb = crmath._ambiguous(yd)
    assert amb.sum() >= 3
    xa = x[amb]
    assert same_bits(crmath.exp_f32(xa), _cr(mpmath.exp, xa))


def test_erf_correctly_rounded_across_binades():
    x = _sample_binades(-40, 2, 30, 2)
    assert same_bits(crmath.erf_f32(x), _cr(mpmath.erf, x))


def test_erf_rare_boundary_cases_and_saturation():
    import scipy.special as sp

    x = np.linspace(0, 4.5, 400_001, dtype=np.float32)
    amb = crmath._ambiguous(np.abs(sp.erf(x.astype(np.float64))))
    xa = np.concatenate([x[amb], np.array([3.9192, 3.9193, 3.92, 4.0, 5.0, 6.0, 10.0], dtype=np.float32)])
    assert amb.sum() >= 3
    assert same_bits(crmath.erf_f32(xa), _cr(mpmath.erf, xa))


def test_erf_symmetry_and_specials():
    rng = np.random.default_rng(5)
    x = rng.standard_normal(20000).astype(np.float32) * 2
    assert same_bits(crmath.erf_f32(-x), -crmath.erf_f32(x))
    sp = crmath.erf_f32(np.array([0.0, -0.0, np.inf, -np.inf, np.nan], dtype=np.float32))
    assert sp.view(np.uint32)[0] == 0 and sp.view(np.uint32)[1] == 0x80000000
    assert sp[2] == 1.0 and sp[3] == -1.0 and np.isnan(sp[4])
    # subnormal inputs: erf(x) ~ 2x/sqrt(pi), still correctly rounded
    tiny = np.array([1e-45, 3e-45, 1e-40, 1e-38], dtype=np.float32)
    assert same_bits(crmath.erf_f32(tiny), _cr(mpmath.erf, tiny))


def test_exp_error_bound_half_ulp_vs_binary64():
    # correct rounding implies at most half an ulp from the binary64 value
    rng = np.random.default_rng(9)
    x = rng.uniform(-80, 80, 100_000).astype(np.float32)
    y = crmath.exp_f32(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    ulp = np.spacing(np.abs(crmath.exp_f32(x))).astype(np.float64)
    assert np.all(np.abs(y - ref) <= 0.5 * ulp * (1 + 1e-6))
    assert math.isclose(float(crmath.exp_f32(np.float32(1.0))), math.e, rel_tol=1e-7)


# ---------------------------------------------------------------- log, tanh

def test_log_correctly_rounded_across_binades():
    x = np.abs(_sample_binades(-149 + 23, 127, 12, 21))
    x = np.concatenate([x, np.linspace(0.5, 2.0, 2001, dtype=np.float32)])
    assert same_bits(crmath.log_f32(x), _cr(mpmath.log, x))


def test_log_subnormals_specials_and_powers_of_two():
    tiny = np.array([1e-45, 3e-45, 1e-40, 1e-38, 1.1754942e-38], dtype=np.float32)
    assert same_bits(crmath.log_f32(tiny), _cr(mpmath.log, tiny))
    sp = crmath.log_f32(np.array([0.0, -0.0, -1.0, -np.inf, np.inf, np.nan, 1.0], dtype=np.float32))
    assert np.isneginf(sp[0]) and np.isneginf(sp[1]) and np.isnan(sp[2]) and np.isnan(sp[3])
    assert np.isposinf(sp[4]) and np.isnan(sp[5]) and sp.view(np.uint32)[6] == 0
    # log(2^k) is k ln2 rounded once
    k = np.arange(-149, 128)
    x = np.ldexp(np.float32(1.0), k).astype(np.float32)
    ln2 = mpf_fraction(mpmath.log(2))
    assert same_bits(crmath.log_f32(x), np.array([rn32(int(v) * ln2) for v in k], dtype=np.float32))


def test_log_rare_boundary_cases_resolved_exactly():
    x = np.linspace(0.25, 8.0, 400_001, dtype=np.float32)
    amb = crmath._ambiguous(np.abs(np.log(x.astype(np.float64))))
    assert amb.sum() >= 3
    xa = x[amb]
    assert same_bits(crmath.log_f32(xa), _cr(mpmath.log, xa))


def test_tanh_correctly_rounded_across_binades():
    x = _sample_binades(-40, 4, 30, 22)
    assert same_bits(crmath.tanh_f32(x), _cr(mpmath.tanh, x))


def test_tanh_small_arguments_saturation_and_specials():
    # below 2^-12 the cubic term is under half an ulp: tanh rounds to x
    rng = np.random.default_rng(23)
    tiny = np.concatenate([np.array([1e-45, 1e-40, 2.0 ** -13, 2.0 ** -12 * 0.999], dtype=np.float32),
                           rng.uniform(0, 2.0 ** -12, 200).astype(np.float32)])
    assert same_bits(crmath.tanh_f32(tiny), tiny)
    assert same_bits(crmath.tanh_f32(tiny), _cr(mpmath.tanh, tiny))
    big = np.array([9.0, 9.0109, 9.011, 9.5, 20.0, 1e30], dtype=np.float32)
    assert same_bits(crmath.tanh_f32(big), _cr(mpmath.tanh, big))
    assert crmath.tanh_f32(np.float32(9.5)) == 1.0
    sp = crmath.tanh_f32(np.array([0.0, -0.0, np.inf, -np.inf, np.nan], dtype=np.float32))
    assert sp.view(np.uint32)[0] == 0 and sp.view(np.uint32)[1] == 0x80000000
    assert sp[2] == 1.0 and sp[3] == -1.0 and np.isnan(sp[4])
    x = rng.standard_normal(20000).astype(np.float32) * 3
    assert same_bits(crmath.tanh_f32(-x), -crmath.tanh_f32(x))


def test_tanh_rare_boundary_cases_resolved_exactly():
    x = np.linspace(0, 9.5, 400_001, dtype=np.float32)
    amb = crmath._ambiguous(np.tanh(x.astype(np.float64)))
    assert amb.sum() >= 3
    xa = x[amb]
    assert same_bits(crmath.tanh_f32(xa), _cr(mpmath.tanh, xa))
