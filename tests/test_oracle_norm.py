"""Pins of the normalization-region oracle (oracle/norm.py) against closed
forms, invariants and an independent library (PyTorch in float64)."""

import math

import numpy as np
import pytest

import oracle.norm as ON
from oracle.f32 import bf16_to_f32, f32_to_bf16

SEQ = ("sequential",)


def _f32(v):
    return np.float32(v)


def test_rms_of_a_constant_row_is_one():
    """sum of n ones is n exactly, its mean 1, sqrt 1: every output is 1 (eps = 0)."""
    for n in (1, 2, 3, 7, 64, 1000):
        x = np.ones((2, n), dtype=np.float32)
        for order in (SEQ, ("interleaved", 3)):
            y = ON.norm_region(x, "f32", "f32", "rms", 0.0, order=order)
            assert np.array_equal(y, np.ones_like(x))


def test_rms_closed_form_with_eps():
    """x = [3, 4], eps = 1/4: mean of squares 12.5, d = sqrt(12.75)."""
    x = np.array([[3.0, 4.0]], dtype=np.float32)
    y = ON.norm_region(x, "f32", "f32", "rms", 0.25)
    want = np.array([3.0, 4.0]) / math.sqrt(12.75)
    assert np.max(np.abs(y[0] / want - 1)) < 2.0 ** -22


def test_layer_norm_of_two_values_is_plus_minus_one():
    """n = 2, eps = 0: mu = (a + b)/2, c = +-(a - b)/2, var = c^2, y = +-1 exactly."""
    rng = np.random.default_rng(3)
    a = rng.integers(-1000, 1000, 50).astype(np.float32)
    b = a + 2 * rng.integers(1, 500, 50).astype(np.float32)
    x = np.stack([a, b], axis=1)
    y = ON.norm_region(x, "f32", "f32", "layer", 0.0)
    assert np.array_equal(y, np.tile(np.array([-1.0, 1.0], dtype=np.float32), (50, 1)))


def test_layer_norm_closed_form_four_values():
    x = np.array([[1.0, 2.0, 3.0, 4.0]], dtype=np.float32)
    y = ON.norm_region(x, "f32", "f32", "layer", 0.0)
    want = (np.array([1.0, 2.0, 3.0, 4.0]) - 2.5) / math.sqrt(1.25)
    assert np.max(np.abs(y[0] - want)) <= 2.0 ** -23


def test_layer_norm_constant_row_gives_the_bias():
    x = np.full((3, 16), 7.25, dtype=np.float32)
    beta = np.linspace(-2, 2, 16).astype(np.float32)
    gamma = np.full(16, 3.0, dtype=np.float32)
    y = ON.norm_region(x, "f32", "f32", "layer", 1e-5, gamma=gamma, beta=beta)
    assert np.array_equal(y, np.tile(beta, (3, 1)))


def test_scale_by_power_of_two_changes_no_bit():
    """eps = 0: every operation scales exactly, the outputs are identical."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((8, 100)).astype(np.float32)
    for kind in ("rms", "layer"):
        for order in (SEQ, ("interleaved", 4)):
            y0 = ON.norm_region(x, "f32", "f32", kind, 0.0, order=order)
            for k in (-20, -3, 5, 30):
                yk = ON.norm_region((x * np.float32(2.0 ** k)).astype(np.float32), "f32", "f32", kind, 0.0,
                                    order=order)
                assert np.array_equal(y0, yk)


def test_gamma_and_beta():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((5, 32)).astype(np.float32)
    y = ON.norm_region(x, "f32", "f32", "layer", 1e-5)
    y2 = ON.norm_region(x, "f32", "f32", "layer", 1e-5, gamma=np.full(32, 2.0, np.float32))
    assert np.array_equal(y2, y * 2)
    beta = rng.standard_normal(32).astype(np.float32)
    g = rng.standard_normal(32).astype(np.float32)
    y3 = ON.norm_region(x, "f32", "f32", "layer", 1e-5, gamma=g, beta=beta)
    assert np.array_equal(y3, ((y * g).astype(np.float32) + beta).astype(np.float32))
    gb = f32_to_bf16(g)
    y4 = ON.norm_region(x, "f32", "f32", "layer", 1e-5, gamma=gb, beta=f32_to_bf16(beta), param_dtype="bf16")
    assert np.array_equal(y4, ((y * bf16_to_f32(gb)).astype(np.float32) + bf16_to_f32(f32_to_bf16(beta)))
                          .astype(np.float32))


@pytest.mark.parametrize("kind", ["rms", "layer"])
def test_against_torch_float64(kind):
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F

    rng = np.random.default_rng(11)
    x = (rng.standard_normal((64, 768)) * 2 + 0.5).astype(np.float32)
    g = (1 + 0.1 * rng.standard_normal(768)).astype(np.float32)
    b = (0.1 * rng.standard_normal(768)).astype(np.float32)
    xt, gt, bt = (torch.from_numpy(v).double() for v in (x, g, b))
    if kind == "rms":
        y = ON.norm_region(x, "f32", "f32", "rms", 1e-6, gamma=g, order=("interleaved", 8))
        want = F.rms_norm(xt, (768,), gt, eps=float(np.float32(1e-6))).numpy()
    else:
        y = ON.norm_region(x, "f32", "f32", "layer", 1e-5, gamma=g, beta=b, order=("interleaved", 8))
        want = F.layer_norm(xt, (768,), gt, bt, eps=float(np.float32(1e-5))).numpy()
    # f32 rounding of O(1) values through a few operations; y + beta cancels
    # near zero, so the bound is absolute plus relative
    assert np.all(np.abs(y - want) <= 2e-6 + 2e-6 * np.abs(want))


def test_orders_follow_the_declared_trees():
    """Row sums in each order, seen through RMSNorm's divisor (eps = 0):
    sequential, interleaved(1) and blocked agree; on a row of squares
    1, 2^-24, 0, 2^-24, 0, ... the sequential chain rounds every 1 + 2^-24 back
    to 1, while interleaved(2) adds the 64 small squares in their own chain
    first (2^-18 exactly) and then 1 + 2^-18."""
    x = np.zeros((1, 129), dtype=np.float32)
    x[0, 0] = 1.0
    x[0, 1::2] = np.float32(2.0 ** -12)
    n = np.float32(129)
    stats = {}
    for name, order in (("seq", SEQ), ("i1", ("interleaved", 1)), ("blk", ("blocked", 4)), ("i2", ("interleaved", 2))):
        stats[name] = ON.norm_region(x, "f32", "f32", "rms", 0.0, order=order, return_stats=True)[2][0]
    assert stats["seq"] == stats["i1"] == stats["blk"]
    assert stats["seq"] == np.sqrt(np.float32(np.float32(1.0) / n))
    assert stats["i2"] == np.sqrt(np.float32(np.float32(1.0 + 2.0 ** -18) / n))
    assert stats["seq"] != stats["i2"]


def test_empty_and_nan_rows():
    y = ON.norm_region(np.zeros((3, 0), np.float32), "f32", "f32", "layer", 1e-5)
    assert y.shape == (3, 0)
    x = np.ones((2, 8), dtype=np.float32)
    x[1, 3] = np.nan
    y = ON.norm_region(x, "f32", "f32", "rms", 1e-6)
    assert not np.isnan(y[0]).any() and np.isnan(y[1]).all()
