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
* bf16 gradients widen exactly; a leaf stored in bf16 at rest (theta, m and v
  in bf16) widens exactly, runs the same f32 chain and rounds each of
  theta', m', v' once to bf16 (round to nearest even).

Schedules and clipping (the same passage: grad_clip = c scales the gradient
by min(1, c / (||g||_2 + 1e-6)), the global norm over the tree, as
clip_grad_norm_; schedules constant(), linear(warmup = w) -- lr t/w for
t <= w, then lr (total - t)/(total - w) -- and cosine(warmup = w) -- lr t/w,
then lr 1/2 (1 + cos(pi (t - w)/(total - w))) -- both reaching 0 at total).
Readings taken here:
* the scheduled lr is computed exactly (a rational, or cos at 300 bits, whose
  value is rational only where cos(pi r) is: r in {0, 1/3, 1/2, 2/3, 1}) and
  rounded once to f32; from t = total on it is 0 (the relu of the pages'
  piecewise form); warmup 0 has no warmup piece;
* ||g||^2 is summed in f32 over a declared tree: each leaf's RN(g_j^2) in
  blocks of 1024 consecutive elements (sequential within a block), the block
  sums in groups of 64 (sequential), the group sums of a leaf (sequential),
  then the leaves in tree order (sequential); the pages fix no order, and
  this one keeps every chain short on the GPU;
* scale = min(q, 1) with q = RN(c / RN(sqrt(||g||^2) + RN(1e-6))), min as the
  group's MIN (q < 1 ? q : 1, so a NaN q gives 1); every gradient is then
  RN(g * scale) in f32 before the step (scale 1 changes no bit).
"""

from __future__ import annotations

from decimal import Decimal, localcontext
from fractions import Fraction

import numpy as np

from .f32 import f32_to_bf16, rn_f32, widen


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


def step_leaf(theta: np.ndarray, m: np.ndarray, v: np.ndarray, grad: np.ndarray, grad_dtype: str, h: dict,
              param_dtype: str = "f32"):
    """One AdamW step over one leaf; returns (theta', m', v') as new arrays in
    the leaf's storage type (f32 values, or bf16 bits rounded once from the
    f32 results: a parameter at rest in bf16, presk "Native execution",
    params, keeps its moments in the same type, the tree type of adamw.init)."""
    if param_dtype == "bf16":
        t1, m1, v1 = step_leaf(widen(theta, "bf16"), widen(m, "bf16"), widen(v, "bf16"), grad, grad_dtype, h)
        return f32_to_bf16(t1), f32_to_bf16(m1), f32_to_bf16(v1)
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


# ------------------------------------------------------ schedules and clip
LR_CONSTANT, LR_LINEAR, LR_COSINE = "constant", "linear", "cosine"
SQ_BLOCK = 1024      # elements per block of the squared-norm tree
SQ_GROUP = 64        # blocks per group


def lr_factor(kind: str, warmup: int, total: int, t: int):
    """The schedule's factor at step t, exactly: a Fraction, or an mpmath value
    (cosine at an irrational point)."""
    if t < 1:
        raise ValueError("t counts steps from 1")
    if kind == LR_CONSTANT:
        return Fraction(1)
    if kind not in (LR_LINEAR, LR_COSINE):
        raise ValueError(f"unknown schedule {kind!r}")
    if not (0 <= warmup < total):
        raise ValueError("a schedule needs 0 <= warmup < total")
    if warmup > 0 and t <= warmup:
        return Fraction(t, warmup)
    if t >= total:
        return Fraction(0)
    num, den = t - warmup, total - warmup           # r = num / den in (0, 1)
    if kind == LR_LINEAR:
        return Fraction(den - num, den)
    exact = {Fraction(1, 3): Fraction(1, 2), Fraction(1, 2): Fraction(0), Fraction(2, 3): Fraction(-1, 2)}
    r = Fraction(num, den)
    if r in exact:
        return (1 + exact[r]) / 2
    import mpmath as mp

    with mp.workprec(300):
        return (1 + mp.cos(mp.pi * mp.mpf(num) / den)) / 2


def lr_scheduled(lr: float, kind: str, warmup: int, total: int, t: int) -> np.float32:
    """RN_f32(lr * factor(t)), the exact product rounded once."""
    f = lr_factor(kind, warmup, total, t)
    if isinstance(f, Fraction):
        return rn_f32(Fraction(lr) * f)
    import mpmath as mp

    with mp.workprec(300):
        v = mp.mpf(lr) * f
        man, exp = mp.frexp(v)
        q = Fraction(int(mp.floor(man * mp.mpf(2) ** 280)), 1) * Fraction(2) ** (int(exp) - 280)
    return _rn_decided(q, Fraction(1, 2 ** 250))


def _seq_sum_rows(a: np.ndarray) -> np.ndarray:
    """Sequential f32 sum along axis 1 of a 2-D array (rows in parallel)."""
    s = a[:, 0].copy()
    for j in range(1, a.shape[1]):
        s = (s + a[:, j]).astype(np.float32)
    return s


def leaf_group_sqsums(g, grad_dtype: str) -> np.ndarray:
    """The group sums of one leaf's ||g||^2 tree (see the module text): the
    RN(g^2) of each block of 1024 consecutive elements added in order, the
    block sums of each group of 64 added in order; f32, one per group."""
    gf = widen(np.asarray(g), grad_dtype).reshape(-1)
    if gf.size == 0:
        return np.zeros(0, dtype=np.float32)
    with np.errstate(all="ignore"):
        sq = (gf * gf).astype(np.float32)
        nb = -(-sq.size // SQ_BLOCK)
        blocks = _seq_sum_rows(np.pad(sq, (0, nb * SQ_BLOCK - sq.size)).reshape(nb, SQ_BLOCK))
        ng = -(-nb // SQ_GROUP)
        return _seq_sum_rows(np.pad(blocks, (0, ng * SQ_GROUP - nb)).reshape(ng, SQ_GROUP))


def sq_norm_from_groups(group_sums, groups_per_leaf) -> np.float32:
    """||g||^2 from the tree's group sums in leaf order: each leaf's groups
    added in order, then the non-empty leaves' sums in order."""
    group_sums = np.asarray(group_sums, dtype=np.float32).reshape(-1)
    total, at = None, 0
    with np.errstate(all="ignore"):
        for n in groups_per_leaf:
            if n == 0:
                continue
            leaf = group_sums[at]
            for v in group_sums[at + 1:at + n]:
                leaf = np.float32(leaf + v)
            at += n
            total = leaf if total is None else np.float32(total + leaf)
    return np.float32(0.0) if total is None else np.float32(total)


def grad_sq_norm(grads, grad_dtype: str) -> np.float32:
    """||g||^2 over the tree in the declared f32 tree (see the module text)."""
    groups = [leaf_group_sqsums(g, grad_dtype) for g in grads]
    return sq_norm_from_groups(np.concatenate(groups) if groups else np.zeros(0, np.float32),
                               [len(x) for x in groups])


def clip_scale(sq_norm: np.float32, grad_clip: float) -> np.float32:
    """min(RN(c / RN(sqrt(||g||^2) + RN(1e-6))), 1) in f32."""
    with np.errstate(all="ignore"):
        norm = np.sqrt(np.float32(sq_norm))
        den = np.float32(norm + np.float32(1e-6))
        q = np.float32(np.float32(grad_clip) / den)
    return q if q < np.float32(1.0) else np.float32(1.0)


def step_tree_scheduled(leaves, grad_dtype: str, hp, kind: str = LR_CONSTANT, warmup: int = 0, total: int = 1,
                        grad_clip: float = 0.0):
    """step_tree with the lr schedule and (grad_clip > 0) global-norm clipping.
    Returns (list of (theta', m', v'), scale or None)."""
    leaves = list(leaves)
    scale = None
    if grad_clip > 0:
        scale = clip_scale(grad_sq_norm([g for _, _, _, g in leaves], grad_dtype), grad_clip)
    return step_tree_scaled(leaves, grad_dtype, hp, scale, kind, warmup, total), scale


def step_tree_scaled(leaves, grad_dtype: str, hp, scale, kind: str = LR_CONSTANT, warmup: int = 0, total: int = 1):
    """The scheduled step with every gradient first scaled by `scale` (f32,
    RN(g * scale)) when scale is not None: a clipped step whose scale is
    known (for a tree split across ranks, from the gathered group sums)."""
    h = hyper_f32(hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, hp.t)
    h["lr"] = lr_scheduled(hp.lr, kind, warmup, total, hp.t)
    leaves = list(leaves)
    if scale is not None:
        with np.errstate(all="ignore"):
            leaves = [(th, m, v, (widen(np.asarray(g), grad_dtype) * np.float32(scale)).astype(np.float32))
                      for th, m, v, g in leaves]
        grad_dtype = "f32"
    return [step_leaf(th, m, v, g, grad_dtype, h) for th, m, v, g in leaves]
