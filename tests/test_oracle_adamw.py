"""Pins for the oracle's AdamW parameter-tree step.

* the injected f32 scalars equal the exact rationals rounded once (t small
  enough to compute beta^t exactly with fractions);
* at t = 1 with zero moments the step is theta - lr (sign(g) + wd theta) up
  to a few ulp (closed form);
* an independent implementation, torch.optim.AdamW in float64, agrees within
  the bound the f32 rounding of the chain allows;
* hand-picked scalars against exact rational arithmetic rounded per operation.
"""

import math
from fractions import Fraction

import numpy as np
import pytest

from oracle import adamw as OA
from synth import workloads as W
from tests.exact import f32_binop, rn32, same_bits, sqrt32


def test_hyper_injection_exact_rationals():
    for beta1, beta2 in ((0.9, 0.999), (0.8, 0.95), (0.5, 0.75)):
        for t in (1, 2, 3, 7, 10, 33, 100):
            h = OA.hyper_f32(3e-4, beta1, beta2, 1e-8, 0.01, t)
            b1, b2 = Fraction(beta1), Fraction(beta2)
            assert same_bits(h["bc1"], rn32(1 - b1 ** t))
            assert same_bits(h["bc2"], rn32(1 - b2 ** t))
            assert same_bits(h["omb1"], rn32(1 - b1)) and same_bits(h["omb2"], rn32(1 - b2))
            assert same_bits(h["b1"], np.float32(beta1)) and same_bits(h["lr"], np.float32(3e-4))
    with pytest.raises(ValueError):
        OA.hyper_f32(1e-3, 0.9, 0.999, 1e-8, 0.0, 0)


def test_first_step_closed_form():
    rng = np.random.default_rng(2)
    n = 10000
    th = (rng.standard_normal(n) * 0.02).astype(np.float32)
    g = (rng.standard_normal(n) * 1e-2).astype(np.float32)
    z = np.zeros(n, dtype=np.float32)
    h = OA.hyper_f32(3e-4, 0.9, 0.999, 1e-8, 0.01, 1)
    th1, m1, v1 = OA.step_leaf(th, z, z, g, "f32", h)
    # m^ = g, v^ = g^2 up to rounding, so q = g / (|g| + eps) ~ sign(g)
    want = th.astype(np.float64) - 3e-4 * (np.sign(g) * np.abs(g) / (np.abs(g) + 1e-8) + 0.01 * th)
    ulp = np.spacing(np.abs(th1)).astype(np.float64)
    assert np.all(np.abs(th1 - want) <= 2 * ulp + 3e-4 * 1e-6)
    assert np.allclose(m1, 0.1 * g.astype(np.float64), rtol=2 ** -22, atol=0)


def test_against_torch_adamw_float64():
    torch = pytest.importorskip("torch")
    tree = W.gpt_adamw_leaves()
    hp = tree.hp
    leaves = [tree.host_leaf(i) for i in range(6)]
    ours = OA.step_tree(leaves, "f32", hp)
    for (th, m, v, g), (th1, m1, v1) in zip(leaves, ours):
        p = torch.tensor(th, dtype=torch.float64, requires_grad=True)
        opt = torch.optim.AdamW([p], lr=hp.lr, betas=(hp.beta1, hp.beta2), eps=hp.eps,
                                weight_decay=hp.weight_decay, foreach=False)
        st = opt.state[p]
        st["step"] = torch.tensor(float(hp.t - 1), dtype=torch.float64)
        st["exp_avg"] = torch.tensor(m, dtype=torch.float64)
        st["exp_avg_sq"] = torch.tensor(v, dtype=torch.float64)
        p.grad = torch.tensor(g, dtype=torch.float64)
        opt.step()
        ref_th = p.detach().numpy()
        ref_m = st["exp_avg"].numpy()
        ref_v = st["exp_avg_sq"].numpy()
        # each moment is two products and a sum: a few units of 2^-24 relative
        assert np.all(np.abs(m1 - ref_m) <= 4 * 2.0 ** -24 * (np.abs(ref_m) + np.abs(0.1 * g)))
        assert np.all(np.abs(v1 - ref_v) <= 4 * 2.0 ** -24 * (np.abs(ref_v) + np.abs(0.001 * g * g)))
        # theta' = theta - lr u: the final rounding (1/2 ulp) plus lr |u| times the
        # chain's relative error (~10 roundings of 2^-24 in u)
        u = (th.astype(np.float64) - ref_th) / hp.lr
        bound = 0.5 * np.spacing(np.abs(th1)) + hp.lr * np.abs(u) * 12 * 2.0 ** -24 + 1e-12
        assert np.all(np.abs(th1 - ref_th) <= bound)


def test_hand_picked_scalars_exact_per_op():
    h = OA.hyper_f32(1e-3, 0.9, 0.999, 1e-8, 0.1, 5)
    cases = [(0.5, 0.25, 0.01, 0.125), (-1.0, 0.0, 0.0, 3.0), (0.0, -0.5, 1e-6, -2.0),
             (3.0, 1e-3, 2e-3, 1e-3)]
    for th, m, v, g in cases:
        th, m, v, g = (np.float32(a) for a in (th, m, v, g))
        r = OA.step_leaf(np.array([th]), np.array([m]), np.array([v]), np.array([g]), "f32", h)
        mul = lambda a, b: f32_binop("MUL", a, b)
        add = lambda a, b: f32_binop("ADD", a, b)
        div = lambda a, b: f32_binop("DIV", a, b)
        m1 = add(mul(h["b1"], m), mul(h["omb1"], g))
        v1 = add(mul(h["b2"], v), mul(h["omb2"], mul(g, g)))
        mh, vh = div(m1, h["bc1"]), div(v1, h["bc2"])
        q = div(mh, add(sqrt32(Fraction(float(vh))), h["eps"]))
        th1 = f32_binop("SUB", th, mul(h["lr"], add(q, mul(h["wd"], th))))
        assert same_bits(r[0][0], th1) and same_bits(r[1][0], m1) and same_bits(r[2][0], v1)


def test_bf16_grads_widen_exactly():
    rng = np.random.default_rng(6)
    g32 = (rng.standard_normal(512) * 1e-3).astype(np.float32)
    from oracle.f32 import bf16_to_f32, f32_to_bf16

    gb = f32_to_bf16(g32)
    th = np.full(512, 0.02, dtype=np.float32)
    z = np.zeros(512, dtype=np.float32)
    h = OA.hyper_f32(3e-4, 0.9, 0.999, 1e-8, 0.01, 1000)
    a = OA.step_leaf(th, z, z, gb, "bf16", h)
    b = OA.step_leaf(th, z, z, bf16_to_f32(gb), "f32", h)
    assert all(same_bits(x, y) for x, y in zip(a, b))


# ------------------------------------------------------ schedules and clip

def test_linear_schedule_closed_forms():
    lr, w, total = 3e-4, 100, 1000
    L = np.float32(lr)
    f = lambda t: OA.lr_scheduled(lr, "linear", w, total, t)  # noqa: E731
    assert f(w) == L and f(w // 2) == L / 2 and f(w // 4) == L / 4
    assert f(total) == 0 and f(total + 7) == 0
    assert f(w + (total - w) // 2) == L / 2                  # half way down: exactly half
    seq = [f(t) for t in range(1, total + 1)]
    assert all(a <= b for a, b in zip(seq[:w - 1], seq[1:w]))
    assert all(a >= b for a, b in zip(seq[w - 1:], seq[w:]))
    assert OA.lr_scheduled(lr, "linear", 0, 400, 100) == np.float32(3e-4 * 0.75) or \
        abs(float(OA.lr_scheduled(lr, "linear", 0, 400, 100)) - 2.25e-4) < 1e-11


def test_cosine_schedule_closed_forms_and_symmetry():
    lr, w, total = 1e-3, 50, 1050
    L = np.float32(lr)
    f = lambda t: OA.lr_scheduled(lr, "cosine", w, total, t)  # noqa: E731
    assert f(w) == L and f(total) == 0 and f(w // 2) == L / 2
    assert f(w + 500) == L / 2                                  # cos(pi/2) = 0
    assert f(w + 250) == np.float32(lr * 0.75 + 0) or abs(float(f(w + 250)) / (lr * (1 + np.cos(np.pi / 4)) / 2) - 1) < 2 ** -23
    for d in range(1, 500, 37):                                 # f(w+d) + f(total-d) = lr in exact reals
        s = float(f(w + d)) + float(f(total - d))
        assert abs(s - lr) <= float(np.spacing(L)) * 1.01
    for t in range(w + 1, total, 97):                           # the exact value, rounded once
        want = lr * 0.5 * (1 + math.cos(math.pi * (t - w) / (total - w)))
        assert abs(float(f(t)) - want) <= 0.5 * float(np.spacing(np.float32(want))) * 1.0001


def test_squared_norm_follows_the_declared_tree():
    """squares 1, then 2047 times 2^-24: a sequential chain keeps 1 (each
    1 + 2^-24 ties to 1); blocks of 1024 give 1 and 1024 * 2^-24 = 2^-14, so
    the leaf's sum is 1 + 2^-14 exactly."""
    g = np.full(2048, np.float32(2.0 ** -12), dtype=np.float32)
    g[0] = 1.0
    assert OA.grad_sq_norm([g], "f32") == np.float32(1 + 2.0 ** -14)
    # leaves combine in order, groups of 64 blocks inside a leaf
    big = np.full(64 * 1024 + 5, np.float32(0.5), dtype=np.float32)
    assert OA.grad_sq_norm([big, g], "f32") == np.float32(big.size * 0.25 + 1 + 2.0 ** -14)
    assert OA.grad_sq_norm([], "f32") == 0


def test_clip_scale_closed_form():
    """||g|| = 2^-10, c = 2^-12: q = c / (2^-10 + 1e-6), just below 1/4."""
    g = np.zeros(3000, dtype=np.float32)
    g[17] = np.float32(2.0 ** -10)
    sq = OA.grad_sq_norm([g], "f32")
    assert sq == np.float32(2.0 ** -20)
    q = OA.clip_scale(sq, 2.0 ** -12)
    want = Fraction(1, 4096) / (Fraction(1, 1024) + Fraction(float(np.float32(1e-6))))
    assert abs(Fraction(float(q)) - want) <= Fraction(float(np.spacing(np.float32(0.25)))) / 2
    assert q < 0.25
    assert OA.clip_scale(np.float32(4.0), 100.0) == 1.0          # below the threshold: no scaling


def test_clipped_scheduled_step_against_torch_float64():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(31)
    shapes = [(37, 19), (2500,), (3, 5, 7)]
    th = [(rng.standard_normal(s) * 0.02).astype(np.float32) for s in shapes]
    m = [(rng.standard_normal(s) * 1e-3).astype(np.float32) for s in shapes]
    v = [np.abs(rng.standard_normal(s) * 1e-4).astype(np.float32) for s in shapes]
    g = [(rng.standard_normal(s) * 0.5).astype(np.float32) for s in shapes]
    hp = W.AdamWHyper(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, t=7)
    out, scale = OA.step_tree_scheduled(zip(th, m, v, g), "f32", hp, "cosine", 3, 20, grad_clip=1.0)
    assert scale < 1
    params = [torch.nn.Parameter(torch.from_numpy(t.astype(np.float64))) for t in th]
    for p_, gg in zip(params, g):
        p_.grad = torch.from_numpy(gg.astype(np.float64))
    torch.nn.utils.clip_grad_norm_(params, 1.0)
    opt = torch.optim.AdamW(params, lr=float(OA.lr_scheduled(1e-3, "cosine", 3, 20, 7)), betas=(0.9, 0.999),
                            eps=1e-8, weight_decay=0.01)
    for p_, mm, vv in zip(params, m, v):
        st = opt.state[p_]
        st["step"] = torch.tensor(6.0, dtype=torch.float64)
        st["exp_avg"] = torch.from_numpy(mm.astype(np.float64))
        st["exp_avg_sq"] = torch.from_numpy(vv.astype(np.float64))
    opt.step()
    for (t1, m1, v1), p_, mm in zip(out, params, m):
        assert np.allclose(t1, p_.detach().numpy(), rtol=0, atol=3e-7)
        assert np.allclose(m1, opt.state[p_]["exp_avg"].numpy(), rtol=3e-6, atol=1e-9)


def test_bf16_leaf_at_rest_is_the_f32_chain_rounded_once():
    """A bf16 leaf: widen theta, m, v exactly, the f32 step, one RNE per output
    (checked against PyTorch's own bf16 rounding of the f32 results)."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(51)
    n = 4000
    th32 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m32 = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    v32 = np.abs(rng.standard_normal(n) * 1e-4).astype(np.float32)
    g = (rng.standard_normal(n) * 1e-2).astype(np.float32)
    to_b = lambda a: torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    thb, mb, vb = to_b(th32), to_b(m32), to_b(v32)
    h = OA.hyper_f32(1e-3, 0.9, 0.999, 1e-8, 0.01, 4)
    got = OA.step_leaf(thb, mb, vb, g, "f32", h, param_dtype="bf16")
    wide = lambda b: (b.astype(np.uint32) << 16).view(np.float32)  # noqa: E731
    want32 = OA.step_leaf(wide(thb), wide(mb), wide(vb), g, "f32", h)
    for a, w in zip(got, want32):
        assert a.dtype == np.uint16 and np.array_equal(a, to_b(w))
