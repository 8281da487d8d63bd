"""Reduction-rooted normalization regions: RMSNorm and LayerNorm over the last axis.

Test infrastructure: a plain CPU definition for the parity tests, the smoke
check and the bench's CPU baseline; nothing on the product path imports it.

Definitions followed: poot "Fusion and Planning", Reduction-rooted regions
(a last-axis, keepdim reduction followed by its pointwise epilogue; RMSNorm
as sum-of-squares -> sqrt -> div); presk PSK-Realize, "What it removes"
(layer normalization as (x - mu)^2 -> mean -> +eps -> sqrt -> divide, with
x - mu read by both the variance and the division); poot "Fusion and
Planning", Why this matters (a norm scale or bias stored in bf16 is widened
inside the region that reads it); presk "Native execution" for the numerics
(f32 arithmetic for bf16 storage, one rounding per operation, the root
rounded once to its storage type) and the summation ``order`` of the
region's reductions (the same trees as the softmax region's sum).

Readings taken here (the pages give the chains, not the f32 operation order):
* n is the row length, exact in f32; a mean is RN(sum / n) (IEEE division);
* eps is the binary64 argument rounded once to f32;
* RMSNorm:   ss = sum_j RN(x_j * x_j) in the declared order,
             d = sqrt(RN(RN(ss / n) + eps)),
             y_j = RN(x_j / d), then RN(y_j * gamma_j) when a scale is given;
* LayerNorm: S = sum_j x_j in the declared order, mu = RN(S / n),
             c_j = RN(x_j - mu), SS = sum_j RN(c_j * c_j) in the same order,
             d = sqrt(RN(RN(SS / n) + eps)),
             y_j = RN(c_j / d), then RN(y_j * gamma_j), then RN(y_j + beta_j),
             each step only when its parameter is given;
* the variance divides by n (a population variance, as "mean" says);
* sqrt and every division are IEEE (correctly rounded), never a reciprocal;
* gamma and beta are vectors of the row length, f32 or bf16 (widened exactly).
"""

from __future__ import annotations

import numpy as np

from .f32 import store, widen
from .softmax import row_sum

RMS, LAYER = "rms", "layer"


def _param(p, dtype, cols):
    if p is None:
        return None
    v = widen(np.asarray(p), dtype).reshape(-1)
    if v.size != cols:
        raise ValueError("a norm parameter must have one value per column")
    return v


def _mean(s: np.ndarray, n: np.float32) -> np.ndarray:
    """A row mean: RN(sum / n)."""
    return (s / n).astype(np.float32)


def _divisor(var: np.ndarray, e: np.float32) -> np.ndarray:
    """d = sqrt(RN(var + eps))."""
    return np.sqrt((var + e).astype(np.float32)).astype(np.float32)


def _affine(y: np.ndarray, g, b) -> np.ndarray:
    """RN(y * gamma), then RN(. + beta), each when given."""
    if g is not None:
        y = (y * g[None, :]).astype(np.float32)
    if b is not None:
        y = (y + b[None, :]).astype(np.float32)
    return y


def norm_region(x: np.ndarray, x_dtype: str, y_dtype: str, kind: str, eps: float, gamma=None, beta=None,
                param_dtype: str = "f32", order=("sequential",), return_stats: bool = False):
    """x: [rows, cols] stored (f32 values or bf16 bits); kind "rms" or "layer".
    Returns y in storage form, and optionally (mu, d): the row means (zeros for
    RMSNorm) and the row divisors, in f32."""
    x = np.asarray(x)
    rows, cols = x.shape
    if kind not in (RMS, LAYER):
        raise ValueError(f"unknown norm kind {kind!r}")
    if kind == RMS and beta is not None:
        raise ValueError("RMSNorm takes no bias")
    if rows == 0 or cols == 0:
        y = store(np.zeros((rows, cols), dtype=np.float32), y_dtype)
        z = np.zeros(rows, dtype=np.float32)
        return (y, z, z) if return_stats else y
    xf = widen(x, x_dtype).reshape(rows, cols)
    g = _param(gamma, param_dtype, cols)
    b = _param(beta, param_dtype, cols)
    n = np.float32(cols)
    e = np.float32(eps)
    with np.errstate(all="ignore"):
        if kind == RMS:
            mu = np.zeros(rows, dtype=np.float32)
            c = xf
        else:
            mu = _mean(row_sum(xf, order), n)
            c = (xf - mu[:, None]).astype(np.float32)
        sq = (c * c).astype(np.float32)
        var = _mean(row_sum(sq, order), n)
        d = _divisor(var, e)
        y = _affine((c / d[:, None]).astype(np.float32), g, b)
    out = store(y, y_dtype)
    return (out, mu, d) if return_stats else out
