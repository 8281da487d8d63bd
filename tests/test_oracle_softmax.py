"""Pins for the oracle's reduction-rooted softmax region.

* tiny rows against exact arithmetic: mpmath exp rounded to f32, the declared
  bracketing tree in exact rationals rounded per addition, IEEE division;
* rows sum to one within the f32 error bound; the interleaved and sequential
  sums lie within the recursive-summation bound of the exact sum;
* a shift of every logit by an exactly representable constant changes no bit;
* sequential = blocked(w) = interleaved(1), bit for bit;
* NaN propagates; an empty row is empty.
"""

from fractions import Fraction
import math

import numpy as np
import pytest

from oracle import softmax as OS
from oracle.f32 import bf16_to_f32
from synth import workloads as W
from tests.exact import f32_binop, mpf_fraction, rn32, same_bits

SEQ = ("sequential",)


def _exact_softmax(row: np.ndarray, order):
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.prec = 200
    m = max(row.tolist())
    d = [f32_binop("SUB", np.float32(v), np.float32(m)) for v in row]
    e = [rn32(mpf_fraction(mpmath.exp(mpmath.mpf(float(v))))) for v in d]
    n = len(e)
    if order[0] == "interleaved":
        P = order[1]
        parts = []
        for p in range(min(P, n)):
            acc = e[p]
            for j in range(p + P, n, P):
                acc = f32_binop("ADD", acc, e[j])
            parts.append(acc)
        s = parts[0]
        for acc in parts[1:]:
            s = f32_binop("ADD", s, acc)
    else:
        s = e[0]
        for v in e[1:]:
            s = f32_binop("ADD", s, v)
    return np.array([f32_binop("DIV", v, s) for v in e], dtype=np.float32), s


@pytest.mark.parametrize("order", [SEQ, ("interleaved", 3), ("interleaved", 8)])
def test_tiny_rows_exact(order):
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((6, 21)) * 3).astype(np.float32)
    y, m, s = OS.softmax_region(x, "f32", "f32", order, return_stats=True)
    for r in range(x.shape[0]):
        want, ws = _exact_softmax(x[r], order)
        assert same_bits(y[r], want)
        assert same_bits(s[r], ws)


def test_rows_sum_to_one():
    wl = W.softmax_rows(64, 1000)
    x = wl.host_x()
    for order in (SEQ, ("interleaved", 8)):
        y = OS.softmax_region(x, "bf16", "f32", order)
        tot = np.array([math.fsum(r) for r in y.astype(np.float64)])
        # e/s rounded per element (<= 2^-24 relative each) and s's own rounding
        # (<= (n-1) 2^-24 relative): |sum - 1| <= n 2^-24 + O(2^-48)
        assert np.all(np.abs(tot - 1.0) <= 1001 * 2.0 ** -24)


@pytest.mark.parametrize("order", [SEQ, ("interleaved", 8)])
def test_sum_within_recursive_summation_bound(order):
    wl = W.softmax_rows(16, 4096)
    x = wl.host_x()
    _, m, s = OS.softmax_region(x, "bf16", "f32", order, return_stats=True)
    from oracle.crmath import exp_f32

    xf = bf16_to_f32(x)
    e = exp_f32((xf - m[:, None]).astype(np.float32)).astype(np.float64)
    n = x.shape[1]
    chain = n - 1 if order[0] == "sequential" else (n // order[1] - 1) + (order[1] - 1)
    gamma = chain * 2.0 ** -24 / (1 - chain * 2.0 ** -24)
    for r in range(x.shape[0]):
        exact = math.fsum(e[r])
        assert abs(float(s[r]) - exact) <= gamma * exact


def test_shift_invariance_bitwise():
    rng = np.random.default_rng(8)
    # logits on a 2^-12 grid within (-8, 8): adding an integer is exact in f32
    x = (np.round(rng.uniform(-8, 8, (12, 333)) * 4096) / 4096).astype(np.float32)
    for order in (SEQ, ("interleaved", 8)):
        y0 = OS.softmax_region(x, "f32", "f32", order)
        for c in (1.0, -5.0, 100.0):
            y1 = OS.softmax_region((x + np.float32(c)).astype(np.float32), "f32", "f32", order)
            assert same_bits(y0, y1)


def test_sequential_blocked_interleaved1_identical():
    x = W.softmax_rows(8, 777).host_x()
    a = OS.softmax_region(x, "bf16", "bf16", SEQ)
    b = OS.softmax_region(x, "bf16", "bf16", ("blocked", 16))
    c = OS.softmax_region(x, "bf16", "bf16", ("interleaved", 1))
    assert np.array_equal(a, b) and np.array_equal(a, c)
    d = OS.softmax_region(x, "bf16", "bf16", ("interleaved", 8))
    assert not np.array_equal(OS.softmax_region(x, "bf16", "f32", SEQ),
                              OS.softmax_region(x, "bf16", "f32", ("interleaved", 8))) or np.array_equal(a, d)


def test_nan_and_empty_rows():
    x = np.zeros((3, 5), dtype=np.float32)
    x[1, 2] = np.nan
    y = OS.softmax_region(x, "f32", "f32", SEQ)
    assert np.all(np.isnan(y[1])) and np.allclose(y[0], 0.2) and np.allclose(y[2], 0.2)
    e = OS.softmax_region(np.zeros((4, 0), dtype=np.float32), "f32", "f32", SEQ)
    assert e.shape == (4, 0)
    one = OS.softmax_region(np.array([[3.5]], dtype=np.float32), "f32", "f32", SEQ)
    assert one[0, 0] == 1.0


# ------------------------------------------------------------ masked softmax

@pytest.mark.parametrize("order", [SEQ, ("interleaved", 3)])
def test_masked_equals_scores_with_minus_infinity(order):
    """The pages' definition: the bits of the softmax of the scores with -inf
    at every refused position (rows the mask does not empty)."""
    rng = np.random.default_rng(41)
    x = (rng.standard_normal((30, 77)) * 3).astype(np.float32)
    mask = (rng.random((30, 77)) < 0.6).astype(np.uint8)
    mask[:, 5] = 1
    got = OS.softmax_region(x, "f32", "f32", order, mask=mask)
    want = OS.softmax_region(np.where(mask != 0, x, -np.inf).astype(np.float32), "f32", "f32", order)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    assert np.all(got[mask == 0] == 0)
    row = (rng.random(77) < 0.5).astype(np.uint8)
    row[0] = 1
    assert np.array_equal(OS.softmax_region(x, "f32", "f32", order, mask=row),
                          OS.softmax_region(x, "f32", "f32", order, mask=np.tile(row, (30, 1))))


def test_mask_emptied_rows_give_zeros_and_full_mask_changes_nothing():
    rng = np.random.default_rng(42)
    x = (rng.standard_normal((6, 40)) * 3).astype(np.float32)
    mask = np.ones((6, 40), dtype=np.uint8)
    mask[2] = 0
    y = OS.softmax_region(x, "f32", "f32", SEQ, mask=mask)
    assert np.all(y[2] == 0) and not np.signbit(y[2]).any()
    assert np.array_equal(np.delete(y, 2, axis=0), np.delete(OS.softmax_region(x, "f32", "f32", SEQ), 2, axis=0))
    x2 = x.copy()
    x2[4, :] = -np.inf                          # allowed but -inf everywhere: NaN, as without a mask
    y2 = OS.softmax_region(x2, "f32", "f32", SEQ, mask=np.ones(40, np.uint8))
    assert np.isnan(y2[4]).all()


# ----------------------------------------------------------- softmax backward

def test_backward_one_hot_cotangent_closed_form():
    """ct = e_k: s = y_k exactly, dx_j = RN(y_j * -y_k) (j != k),
    dx_k = RN(y_k * RN(1 - y_k))."""
    rng = np.random.default_rng(43)
    y = OS.softmax_region((rng.standard_normal((4, 33)) * 2).astype(np.float32), "f32", "f32", SEQ)
    for k in (0, 7, 32):
        ct = np.zeros_like(y)
        ct[:, k] = 1.0
        dx = OS.softmax_backward(y, ct, "f32", "f32", "f32")
        want = (y * -y[:, k:k + 1]).astype(np.float32)
        want[:, k] = (y[:, k] * (np.float32(1) - y[:, k]).astype(np.float32)).astype(np.float32)
        assert np.array_equal(dx.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("order", [SEQ, ("interleaved", 8)])
def test_backward_against_torch_autograd_float64(order):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(44)
    x = (rng.standard_normal((16, 300)) * 2).astype(np.float32)
    ct = rng.standard_normal((16, 300)).astype(np.float32)
    xt = torch.from_numpy(x.astype(np.float64)).requires_grad_(True)
    torch.softmax(xt, dim=1).backward(torch.from_numpy(ct.astype(np.float64)))
    y = OS.softmax_region(x, "f32", "f32", order)
    dx = OS.softmax_backward(y, ct, "f32", "f32", "f32", order)
    want = xt.grad.numpy()
    assert np.all(np.abs(dx - want) <= 1e-6 * np.abs(want) + 1e-8)
    assert np.all(np.abs(dx.astype(np.float64).sum(axis=1)) < 1e-6)   # sum_j y_j (ct_j - s) = 0 in exact reals
