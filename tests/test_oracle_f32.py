"""Pins for the oracle's storage rules (bf16 widening/rounding, exact f32 rounding)."""

from fractions import Fraction

import numpy as np
import pytest

from oracle import f32 as O
from tests.exact import rn32, same_bits


def _edge_f32():
    specials = np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, 3.4028235e38, -3.4028235e38,
                         1e-45, -1e-45, 1.1754944e-38, 1.1754942e-38, 65504.0, 3.3895314e38,
                         3.3961776e38, 1.0 + 2 ** -8, 1.0 + 2 ** -9, 1.0 + 3 * 2 ** -9], dtype=np.float32)
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2 ** 32, 200_000, dtype=np.uint64).astype(np.uint32)
    rand = bits.view(np.float32)
    rand = rand[np.isfinite(rand)]
    # exact ties at the bf16 rounding position, both parities
    tie_bits = (rng.integers(0, 2 ** 16, 2000, dtype=np.uint64).astype(np.uint32) << 16) | np.uint32(0x8000)
    ties = tie_bits.view(np.float32)
    ties = ties[np.isfinite(ties)]
    return np.concatenate([specials, rand, ties])


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    x = _edge_f32()
    ours = O.f32_to_bf16(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ours_f = O.bf16_to_f32(ours)
    ref_f = O.bf16_to_f32(ref)
    assert same_bits(ours_f, ref_f)


def test_bf16_widening_is_a_shift_and_round_trips():
    bits = np.arange(0, 2 ** 16, dtype=np.uint32).astype(np.uint16)
    f = O.bf16_to_f32(bits)
    # widening is exact: rounding back gives the same bits (NaN stays NaN)
    back = O.f32_to_bf16(f)
    nan = np.isnan(f)
    assert np.array_equal(back[~nan], bits[~nan])
    assert np.all(np.isnan(O.bf16_to_f32(back[nan])))
    assert f[0x3F80] == 1.0 and f[0xBF80] == -1.0 and np.isinf(f[0x7F80])


def test_bf16_nan_stays_quiet_nan():
    nan_bits = np.array([0x7F800001, 0xFF800001, 0x7FC00000, 0x7FFFFFFF], dtype=np.uint32)
    out = O.f32_to_bf16(nan_bits.view(np.float32))
    assert np.all(np.isnan(O.bf16_to_f32(out)))


def test_rn_f32_against_neighbour_search():
    rng = np.random.default_rng(11)
    qs = []
    for _ in range(3000):
        num = int(rng.integers(1, 2 ** 62)) * (1 if rng.random() < 0.5 else -1)
        den = int(rng.integers(1, 2 ** 62))
        sh = int(rng.integers(-200, 200))
        qs.append(Fraction(num, den) * Fraction(2) ** sh)
    # ties and the subnormal / overflow edges
    qs += [Fraction(1) + Fraction(1, 2 ** 24), Fraction(1) + Fraction(3, 2 ** 24),
           Fraction(1, 2 ** 150), Fraction(3, 2 ** 150), Fraction(1, 2 ** 151),
           Fraction(2) ** 128 - Fraction(2) ** 103, Fraction(2) ** 128 - Fraction(2) ** 103 - 1,
           Fraction(2) ** 127 * 3]
    for q in qs:
        a, b = O.rn_f32(q), rn32(q)
        assert same_bits(a, b), (q, a, b)


def test_rn_f32_matches_hardware_narrowing_of_doubles():
    # a binary64 value is a rational; the FPU's narrowing is correctly rounded
    rng = np.random.default_rng(3)
    d = rng.standard_normal(2000) * np.exp(rng.uniform(-100, 100, 2000))
    for v in d:
        assert same_bits(O.rn_f32(Fraction(float(v))), np.float32(v))
