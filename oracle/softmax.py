"""The reduction-rooted softmax region, Reduce(Max) -> Sub -> Exp -> Reduce(Sum) -> Div.

Definition followed: poot "Fusion and Planning", Reduction-rooted regions
(a last-axis, keepdim reduction followed by its pointwise epilogue) for the
region's shape; presk "Native execution", realizations, for the numerics
(softmax subtracts the row maximum; reductions accumulate in the arithmetic
type, f32 for bf16 storage; bf16 is widened exactly and the result is rounded
once) and for the summation ``order``: ``sequential`` and ``blocked(width)``
are bit-identical, ``interleaved(partials)`` reassociates.

Readings taken here (the pages fix the orders by name only):
* the max starts at element 0 and propagates NaN; it is exact, so its order
  does not matter, and the sign of a zero maximum changes no exp value;
* sequential: s = (((e0 + e1) + e2) + ...) + e_{n-1};
* blocked(width): register blocking keeps every addition in index order, so
  it is the sequential chain;
* interleaved(P): partial p sums e_j, j = p mod P, in increasing j starting
  from e_p; the partials are then combined left to right, ((p0 + p1) + p2) ...;
* y = RN(e / s) in f32 (IEEE division, no reciprocal), then rounded to the
  output's storage type;
* a row of zero columns is empty and produces nothing.

Masked softmax (presk "Native execution", numerics: a mask is an index buffer
of 0 and 1; the masked softmax takes its maximum from the allowed positions
and its sum over them, 0 where it refuses, a row it empties giving zeros, so
that its bits are those of the softmax of the scores with -inf at the refused
positions): the mask is one row [cols] shared by every row or a full
[rows, cols]; nonzero allows.  Refused positions contribute exp(-inf) = +0 to
the sum, which changes no bit of a chain, so the declared order is unchanged.

Softmax backward (presk "The language", automatic differentiation:
softmax's rule is y (ct - sum_axis(ct y))): per row s = sum_j RN(ct_j y_j) in
the declared order, dx_j = RN(y_j RN(ct_j - s)), y and ct widened from their
storage, dx rounded to its own.
"""

from __future__ import annotations

import numpy as np

from . import crmath
from .f32 import store, widen

SEQUENTIAL, BLOCKED, INTERLEAVED = "sequential", "blocked", "interleaved"


def _row_max(x: np.ndarray) -> np.ndarray:
    return np.max(x, axis=1).astype(np.float32)


def _sum_sequential(e: np.ndarray) -> np.ndarray:
    s = e[:, 0].copy()
    for j in range(1, e.shape[1]):
        s = (s + e[:, j]).astype(np.float32)
    return s


def _sum_interleaved(e: np.ndarray, partials: int) -> np.ndarray:
    n = e.shape[1]
    parts = []
    for p in range(min(partials, n)):
        acc = e[:, p].copy()
        for j in range(p + partials, n, partials):
            acc = (acc + e[:, j]).astype(np.float32)
        parts.append(acc)
    s = parts[0]
    for acc in parts[1:]:
        s = (s + acc).astype(np.float32)
    return s


def row_sum(e: np.ndarray, order) -> np.ndarray:
    kind = order[0]
    if kind in (SEQUENTIAL, BLOCKED):
        return _sum_sequential(e)
    if kind == INTERLEAVED:
        if int(order[1]) < 1:
            raise ValueError("interleaved needs at least one partial")
        return _sum_interleaved(e, int(order[1]))
    raise ValueError(f"unknown order {order!r}")


def _apply_mask(xf: np.ndarray, mask):
    """Scores with -inf at refused positions, and the rows the mask empties."""
    allow = np.broadcast_to(np.asarray(mask) != 0, xf.shape)
    return np.where(allow, xf, np.float32(-np.inf)).astype(np.float32), ~allow.any(axis=1)


def softmax_region(x: np.ndarray, x_dtype: str, y_dtype: str, order=(SEQUENTIAL,), return_stats: bool = False,
                   mask=None):
    """x: [rows, cols] stored (f32 values or bf16 bits); mask: None, or 0/1
    values of shape [cols] (every row) or [rows, cols].  Returns y in storage
    form, and optionally (m, s), the row maxima and row sums in f32."""
    x = np.asarray(x)
    rows, cols = x.shape
    if cols == 0 or rows == 0:
        y = store(np.zeros((rows, cols), dtype=np.float32), y_dtype)
        empty = np.zeros(rows, dtype=np.float32)
        return (y, empty, empty) if return_stats else y
    xf = widen(x, x_dtype).reshape(rows, cols)
    emptied = np.zeros(rows, dtype=bool)
    if mask is not None:
        xf, emptied = _apply_mask(xf, mask)
    with np.errstate(all="ignore"):
        m = _row_max(xf)
        m[emptied] = 0.0                       # every exp(-inf - 0) is 0: a zero sum
        d = (xf - m[:, None]).astype(np.float32)
        e = crmath.exp_f32(d)
        s = row_sum(e, order)
        y = (e / s[:, None]).astype(np.float32)
        y[emptied] = 0.0
    out = store(y, y_dtype)
    return (out, m, s) if return_stats else out


def softmax_backward(y: np.ndarray, ct: np.ndarray, y_dtype: str, ct_dtype: str, dx_dtype: str,
                     order=(SEQUENTIAL,)) -> np.ndarray:
    """dx = y (ct - sum(ct y)) per row; y, ct: [rows, cols] stored."""
    y = np.asarray(y)
    rows, cols = y.shape
    if rows == 0 or cols == 0:
        return store(np.zeros((rows, cols), dtype=np.float32), dx_dtype)
    yf = widen(y, y_dtype).reshape(rows, cols)
    cf = widen(np.asarray(ct), ct_dtype).reshape(rows, cols)
    with np.errstate(all="ignore"):
        p = (cf * yf).astype(np.float32)
        s = row_sum(p, order)
        dx = (yf * (cf - s[:, None]).astype(np.float32)).astype(np.float32)
    return store(dx, dx_dtype)
