"""The AdamW step as one parameter-tree group, every leaf, in f32.

Definition followed (presk "The language", The optimizer, adamw.step): AdamW
as PyTorch defines it, m' = b1 m + (1 - b1) g, v' = b2 v + (1 - b2) g^2,
m^ = m' / (1 - b1^t), v^ = v' / (1 - b2^t), theta' = theta - lr (m^ / (sqrt(v^)
+ eps) + wd theta), t counting steps from 1; hyperparameters are injected
exactly (presk: decimal literals injected exactly into the reals; a value
reaches f32 by one rounding at its injection).  A group of type ``params M``
is mapped over every leaf of the tree (PSK-Realize, Parameter trees).

Readings taken here:
* the scalars 1 - b1, 1 - b2, 1 - b1^t, 1 - b2^t are computed exactly from
  the binary64 values the caller passes, then rounded once to f32; lr, eps
  and wd are rounded once to f32;
* the per-parameter chain, each operation one f32 rounding, in this order:
    m1 = (b1*m) + (omb1*g)
    v1 = (b2*v) + (omb2*(g*g))
    mh = m1 / bc1 ;  vh = v1 / bc2
    q  = mh / (sqrt(vh) + eps)
    u  = q + (wd*theta)
    theta1 = theta - (lr*u)
* the schedule is constant and there is no gradient clipping; bf16 gradients
  widen exactly.
"""

from __future__ import annotations

from decimal import Decimal, localcontext
from fractions import Fraction

import numpy as np

from .f32 import rn_f32, widen


def _rn_decided(q: Fraction, rel_err: Fraction) -> np.float32:
    """RN_f32 of a value known to within rel_err, refusing an undecided one."""
    r = rn_f32(q)
    lo = rn_f32(q * (1 - rel_err))
    hi = rn_f32(q * (1 + rel_err))
    if lo != r or hi != r:
        raise ArithmeticError(f"f32 rounding of {float(q)} undecided")
    return r


def hyper_f32(lr: float, beta1: float, beta2: float, eps: float, weight_decay: float, t: int):
    """The f32 scalars the step reads: dict b1 b2 omb1 omb2 bc1 bc2 lr eps wd."""
    if t < 1:
        raise ValueError("t counts steps from 1")
    b1, b2 = Fraction(beta1), Fraction(beta2)
    with localcontext() as ctx:
        ctx.prec = 200
        p1 = Decimal(beta1) ** int(t)
        p2 = Decimal(beta2) ** int(t)
        bc1 = Fraction(1 - p1)
        bc2 = Fraction(1 - p2)
    tiny = Fraction(1, 10 ** 150)
    return {
        "b1": rn_f32(b1), "b2": rn_f32(b2),
        "omb1": rn_f32(1 - b1), "omb2": rn_f32(1 - b2),
        "bc1": _rn_decided(bc1, tiny), "bc2": _rn_decided(bc2, tiny),
        "lr": rn_f32(Fraction(lr)), "eps": rn_f32(Fraction(eps)), "wd": rn_f32(Fraction(weight_decay)),
    }


def step_leaf(theta: np.ndarray, m: np.ndarray, v: np.ndarray, grad: np.ndarray, grad_dtype: str, h: dict):
    """One AdamW step over one leaf; returns (theta', m', v') as new f32 arrays."""
    th = np.asarray(theta, dtype=np.float32)
    m = np.asarray(m, dtype=np.float32)
    v = np.asarray(v, dtype=np.float32)
    g = widen(grad, grad_dtype)
    with np.errstate(all="ignore"):
        m1 = (h["b1"] * m) + (h["omb1"] * g)
        v1 = (h["b2"] * v) + (h["omb2"] * (g * g))
        mh = m1 / h["bc1"]
        vh = v1 / h["bc2"]
        q = mh / (np.sqrt(vh) + h["eps"])
        u = q + (h["wd"] * th)
        th1 = th - (h["lr"] * u)
    f = np.float32
    return th1.astype(f), m1.astype(f), v1.astype(f)


def step_tree(leaves, grad_dtype: str, hp):
    """leaves: iterable of (theta, m, v, grad); hp has lr beta1 beta2 eps
    weight_decay t.  Returns a list of (theta', m', v') per leaf."""
    h = hyper_f32(hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, hp.t)
    return [step_leaf(th, m, v, g, grad_dtype, h) for th, m, v, g in leaves]
