"""Pins for the oracle's AdamW parameter-tree step.

* the injected f32 scalars equal the exact rationals rounded once (t small
  enough to compute beta^t exactly with fractions);
* at t = 1 with zero moments the step is theta - lr (sign(g) + wd theta) up
  to a few ulp (closed form);
* an independent implementation, torch.optim.AdamW in float64, agrees within
  the bound the f32 rounding of the chain allows;
* hand-picked scalars against exact rational arithmetic rounded per operation.
"""

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
