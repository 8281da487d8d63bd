"""The device exp/erf source, compiled for the host, against the oracle.

The library's kernels run the CUDA build of csrc/crmath.cuh; the same source
compiled as plain C++ (libpsk_hostmath.so) lets the CPU check every tier
element by element: tier 1's decision never keeps a wrong rounding, tiers 2
and 3 are correctly rounded on their own, and the composed functions equal the
oracle's correctly rounded exp and erf bit for bit.
"""

import ctypes
import os

import numpy as np
import pytest

from oracle.crmath import erf_f32, exp_f32
from tests.exact import same_bits

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def hm():
    from reduction_groups_gb300 import build as B

    B.build()
    L = ctypes.CDLL(os.path.join(ROOT, "reduction_groups_gb300", "_build", "libpsk_hostmath.so"))
    P = ctypes.c_void_p

    def unary(which, x):
        x = np.ascontiguousarray(x, dtype=np.float32)
        y = np.empty_like(x)
        L.psk_host_unary(ctypes.c_int(which), P(x.ctypes.data), P(y.ctypes.data), ctypes.c_long(x.size))
        return y

    def tier(which, t, x):
        x = np.ascontiguousarray(x, dtype=np.float32)
        y = np.empty_like(x)
        ok = np.empty(x.shape, dtype=np.uint8)
        L.psk_host_tier(ctypes.c_int(which), ctypes.c_int(t), P(x.ctypes.data), P(y.ctypes.data),
                        P(ok.ctypes.data), ctypes.c_long(x.size))
        return y, ok.astype(bool)

    return unary, tier


def _all_binades(lo, hi, per, seed):
    rng = np.random.default_rng(seed)
    out = []
    for e in range(lo, hi + 1):
        m = rng.integers(0, 2 ** 23, per, dtype=np.uint64).astype(np.uint32)
        v = ((np.uint32(e + 127) << np.uint32(23)) | m).view(np.float32)
        out += [v, -v]
    return np.concatenate(out)


def _specials():
    return np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 1e-45, -1e-45, 88.72283935546875, 88.7228317,
                     -87.33654, -103.97208, -103.97207, -104.0, 87.0, -87.0, 3.9192059, 3.9192057, 3.9375,
                     2 ** -60, 2 ** -61, 1.0, -1.0], dtype=np.float32)


def test_exp_composed_equals_oracle(hm):
    unary, _ = hm
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.uniform(-110, 95, 1_500_000).astype(np.float32), _all_binades(-149 + 23, 7, 2000, 2),
                        _specials()])
    assert same_bits(unary(0, x), exp_f32(x))


def test_erf_composed_equals_oracle(hm):
    unary, _ = hm
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.uniform(-4.5, 4.5, 1_500_000).astype(np.float32), _all_binades(-126, 2, 2000, 4),
                        _specials()])
    assert same_bits(unary(1, x), erf_f32(x))


def test_tier1_keeps_only_correct_roundings(hm):
    _, tier = hm
    rng = np.random.default_rng(5)
    x = rng.uniform(-87, 87, 2_000_000).astype(np.float32)
    y, ok = tier(0, 1, x)
    assert same_bits(y[ok], exp_f32(x[ok]))
    assert 1 - ok.mean() < 2.0 ** -12          # about one call in 2^14 falls through
    a = rng.uniform(2.0 ** -60, 3.919, 2_000_000).astype(np.float32)
    y, ok = tier(1, 1, a)
    assert same_bits(y[ok], erf_f32(a[ok]))
    assert 1 - ok.mean() < 2.0 ** -12


def test_erf_record_tables_give_the_same_bits(hm):
    """The group kernels read erf's Taylor coefficients as one record per
    interval (three 16-byte loads); tier 1 and the fast erf from the records
    equal tier 1 and the fast erf from the separate tables, bit for bit, over
    every interval (4·10^6 arguments and every binade below 1)."""
    unary, tier = hm
    rng = np.random.default_rng(13)
    a = np.concatenate([rng.uniform(2.0 ** -60, 3.919, 4_000_000).astype(np.float32),
                        np.abs(_all_binades(-60, 1, 2000, 4)),
                        (np.arange(126, dtype=np.float32) + np.float32(0.5)) / np.float32(32)])
    a = a[(a >= 2.0 ** -60) & (a < 3.919)]
    r_sep, _ = tier(1, 1, a)
    assert same_bits(unary(10, a), r_sep)
    x = np.concatenate([a, np.array([3.92, 4.0, 10.0, 0.0], dtype=np.float32)])
    assert same_bits(unary(11, x), unary(6, x))


@pytest.mark.parametrize("t", [2, 3])
def test_tiers_2_and_3_correctly_rounded_alone(hm, t):
    _, tier = hm
    rng = np.random.default_rng(7 + t)
    xe = np.concatenate([rng.uniform(-104, 89, 30000).astype(np.float32), _specials()[5:18]])
    y, _ = tier(0, t, xe)
    assert same_bits(y, exp_f32(xe))
    xr = np.concatenate([rng.uniform(0, 3.9375, 30000).astype(np.float32),
                         np.array([1e-30, 3e-20, 2 ** -61], dtype=np.float32)])
    y, _ = tier(1, t, xr)
    assert same_bits(y, erf_f32(xr))


def test_division_through_reciprocal_equals_ieee():
    """The softmax divides by the row sum through its reciprocal with
    Markstein's correction; on the operand ranges it accepts the result equals
    IEEE division (others fall back to it)."""
    from reduction_groups_gb300 import build as B

    B.build()
    L = ctypes.CDLL(os.path.join(ROOT, "reduction_groups_gb300", "_build", "libpsk_hostmath.so"))
    L.psk_host_div_check.restype = ctypes.c_long
    L.psk_host_div_check.argtypes = [ctypes.c_ulong, ctypes.c_long, ctypes.c_float, ctypes.c_float, ctypes.c_float]
    for seed, lo, hi, bmax in ((1, -100, 1, 4097.0), (2, -126, 1, 1e6), (3, -100, 100, 2.0 ** 20), (4, -30, 1, 3.0)):
        assert L.psk_host_div_check(seed, 5_000_000, lo, hi, bmax) == 0


def test_tier1_relative_error_below_the_decision_bound(hm):
    """Tier 1's decision assumes a relative error below 2^-41.  The value it
    returns, (R + d) 2^n, against binary64 exp and erf (errors below 2^-52) on
    every binade, uniform reals and the reduction's worst points (|r| at its
    ln2/2048 limit); measured over every float of their tier-1 ranges the
    bounds are 2^-43.3 (exp) and 2^-45.8 (erf)."""
    from scipy.special import erf as erf64

    L = ctypes.CDLL(os.path.join(ROOT, "reduction_groups_gb300", "_build", "libpsk_hostmath.so"))

    def value(which, x):
        x = np.ascontiguousarray(x, dtype=np.float32)
        y = np.empty(x.shape, dtype=np.float64)
        L.psk_host_tier1_value(ctypes.c_int(which), ctypes.c_void_p(x.ctypes.data), ctypes.c_void_p(y.ctypes.data),
                               ctypes.c_long(x.size))
        return y

    rng = np.random.default_rng(11)
    k = rng.integers(-128000, 128000, 400_000)
    edge = ((k + 0.5) * np.log(2) / 1024).astype(np.float32)           # |r| near ln2/2048
    xe = np.concatenate([_all_binades(-30, 6, 40_000, 12), rng.uniform(-87, 87, 1_000_000).astype(np.float32),
                         edge])
    xe = xe[np.abs(xe) <= 87]
    rel = np.abs(value(0, xe) / np.exp(xe.astype(np.float64)) - 1)
    assert rel.max() < 2.0 ** -42, np.log2(rel.max())
    xa = np.concatenate([_all_binades(-60, 1, 20_000, 13), rng.uniform(0, 3.919, 1_000_000).astype(np.float32)])
    xa = xa[(xa >= 2.0 ** -60) & (xa < 3.9192)]
    ref = erf64(xa.astype(np.float64))
    rel = np.abs(value(1, xa) / ref - 1)
    assert rel.max() < 2.0 ** -42, np.log2(rel.max())


# ---------------------------------------------------------------- log, tanh

def _positive_normals(n, seed):
    rng = np.random.default_rng(seed)
    return rng.integers(0x00800000, 0x7F800000, n, dtype=np.uint64).astype(np.uint32).view(np.float32)


def test_log_composed_equals_oracle(hm):
    from oracle.crmath import log_f32

    unary, _ = hm
    rng = np.random.default_rng(41)
    x = np.concatenate([_positive_normals(1_000_000, 42), (1 + rng.uniform(-2 ** -7, 2 ** -7, 300_000)).astype(np.float32),
                        rng.uniform(0, 2.0 ** -126, 20_000).astype(np.float32),
                        np.array([0.0, -0.0, -1.0, -1e-45, np.inf, -np.inf, np.nan, 1.0, 1e-45, 2.0, 0.5,
                                  np.sqrt(2), 3.4028235e38, 1.1754942e-38], dtype=np.float32)])
    assert same_bits(unary(3, x), log_f32(x))


def test_tanh_composed_equals_oracle(hm):
    from oracle.crmath import tanh_f32

    unary, _ = hm
    rng = np.random.default_rng(43)
    x = np.concatenate([rng.uniform(-10, 10, 1_000_000).astype(np.float32), _all_binades(-30, 3, 4000, 44),
                        rng.uniform(-2 ** -11, 2 ** -11, 20_000).astype(np.float32),
                        np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 1e-45, 2 ** -12, 9.010913, 9.0109135, 9.5,
                                  -9.5, 1e30], dtype=np.float32)])
    assert same_bits(unary(4, x), tanh_f32(x))


def test_log_tanh_tier1_keeps_only_correct_roundings_and_tiers_2_3_alone(hm):
    from oracle.crmath import log_f32, tanh_f32

    _, tier = hm
    x = _positive_normals(2_000_000, 45)
    y, ok = tier(2, 1, x)
    assert same_bits(y[ok], log_f32(x[ok]))
    assert 1 - ok.mean() < 2.0 ** -12
    bad = np.concatenate([x[~ok][:2000], x[:20000]])
    bad = bad[bad != 1]
    for t in (2, 3):
        y3, _ = tier(2, t, bad)
        assert same_bits(y3, log_f32(bad))
    rng = np.random.default_rng(46)
    a = rng.uniform(2.0 ** -12, 9.0109, 2_000_000).astype(np.float32)
    y, ok = tier(3, 1, a)
    assert same_bits(y[ok], tanh_f32(a[ok]))
    assert 1 - ok.mean() < 2.0 ** -12
    bad = np.concatenate([a[~ok][:2000], a[:20000]])
    for t in (2, 3):
        y3, _ = tier(3, t, bad)
        assert same_bits(y3, tanh_f32(bad))


def test_log_tanh_tier1_relative_error(hm):
    """Tier 1's decision assumes a relative error below 2^-41; over every float
    of their tier-1 ranges the bounds are 2^-42.1 (log, worst just above 1,
    where the cubic tail is largest against the result) and 2^-46.1 (tanh)."""
    L = ctypes.CDLL(os.path.join(ROOT, "reduction_groups_gb300", "_build", "libpsk_hostmath.so"))

    def value(which, x):
        x = np.ascontiguousarray(x, dtype=np.float32)
        y = np.empty(x.shape, dtype=np.float64)
        L.psk_host_tier1_value(ctypes.c_int(which), ctypes.c_void_p(x.ctypes.data), ctypes.c_void_p(y.ctypes.data),
                               ctypes.c_long(x.size))
        return y

    rng = np.random.default_rng(47)
    x = np.concatenate([_positive_normals(1_000_000, 48), (1 + rng.uniform(-2 ** -8, 2 ** -8, 1_000_000)).astype(np.float32),
                        (np.sqrt(2) * (1 + rng.uniform(-2 ** -8, 2 ** -8, 200_000))).astype(np.float32)])
    x = x[x != 1]
    rel = np.abs(value(2, x) / np.log(x.astype(np.float64)) - 1)
    assert rel.max() < 2.0 ** -41.5, np.log2(rel.max())
    a = np.concatenate([rng.uniform(2.0 ** -12, 9.0109, 1_000_000), np.exp2(rng.uniform(-12, 3, 500_000))]).astype(np.float32)
    a = a[(a >= 2.0 ** -12) & (a < 9.0109)]
    rel = np.abs(value(3, a) / np.tanh(a.astype(np.float64)) - 1)
    assert rel.max() < 2.0 ** -44, np.log2(rel.max())


# ------------------------------------------- the groups' fast math mode

def _ulps(a, b):
    def ordv(x):
        b_ = x.view(np.int32).astype(np.int64)
        return np.where(b_ < 0, -(b_ & 0x7FFFFFFF), b_)
    return np.abs(ordv(a) - ordv(b))


def test_fast_exp_and_erf_within_their_bounds(hm):
    """The fast mode's exp (one ulp) and erf (two ulp) against the correctly
    rounded oracle; measured over every float of their ranges the bounds are
    exactly 1 and 2."""
    unary, _ = hm
    rng = np.random.default_rng(61)
    sp = np.array([0.0, -0.0, np.inf, -np.inf, 88.72, 88.73, 89.0, -87.3, -103.97, -104.5, 1e-30, -1e-45],
                  dtype=np.float32)
    x = np.concatenate([rng.uniform(-110, 95, 1_000_000).astype(np.float32), _all_binades(-40, 6, 2000, 62), sp])
    y, ref = unary(5, x), exp_f32(x)
    assert np.array_equal(np.isnan(y), np.isnan(ref))
    assert _ulps(y, ref).max() <= 1
    a = np.concatenate([rng.uniform(-6, 6, 1_000_000).astype(np.float32), _all_binades(-149 + 23, 2, 2000, 63), sp])
    y, ref = unary(6, a), erf_f32(a)
    ok = ~np.isnan(ref)
    assert np.array_equal(np.isnan(y), np.isnan(ref))
    assert _ulps(y[ok], ref[ok]).max() <= 2


