"""Pins for the oracle's node-by-node group evaluation.

* every program of up to two op nodes over two inputs, and random deeper
  programs with re-read (REF) nodes, against an element-by-element evaluator in
  exact rational arithmetic with one binary32 rounding per node;
* the small 6-node workload against mpmath's erf and exact arithmetic;
* the exp-clamp node, clamped by the builtins' rule and exponentiated by
  mpmath, inside, at and beyond the bounds, at the infinities and at NaN;
* broadcasting equals evaluating over the materialised expansion, bit for bit;
* bf16 storage: interior values stay in f32 (rounding each node to bf16
  changes results);
* every malformed program is refused.
"""

import itertools
from fractions import Fraction

import numpy as np
import pytest

from oracle import group as OG
from oracle.f32 import bf16_to_f32, f32_to_bf16
from synth import workloads as W
from tests.exact import f32_binop, mpf_fraction, rn32, same_bits, sqrt32

BIN = ["ADD", "SUB", "MUL", "DIV", "MAX", "MIN"]
UN = ["NEG", "ABS", "SQRT", "SQRTA", "RECIP"]


def _exact_node(name, a, b=None):
    """One node on scalars, IEEE binary32, computed without the oracle."""
    a = np.float32(a)
    if name in ("ADD", "SUB", "MUL", "DIV"):
        return f32_binop(name, a, np.float32(b))
    if name == "MAX":
        return np.float32(a) if a > b else np.float32(b)
    if name == "MIN":
        return np.float32(a) if a < b else np.float32(b)
    if name == "NEG":
        return np.float32(-a)
    if name == "ABS":
        return np.float32(abs(a))
    if name == "RECIP":
        return f32_binop("DIV", np.float32(1.0), a)
    if name in ("SQRT", "SQRTA"):
        v = abs(a) if name == "SQRTA" else a
        if np.isnan(v) or v < 0:
            return np.float32(np.nan)
        if np.isinf(v):
            return np.float32(np.inf)
        if v == 0:
            return np.float32(v)  # sqrt(-0) = -0
        return sqrt32(Fraction(float(v)))
    raise ValueError(name)


def _exact_eval(seq, vals):
    """seq: [(name, arg)]; vals: per input a 1-D f32 array.  Element by element."""
    n = len(vals[0])
    out = np.empty(n, dtype=np.float32)
    for i in range(n):
        stack, nodes = [], []
        for name, arg in seq:
            if name == "IN":
                stack.append(vals[arg][i])
            elif name == "REF":
                stack.append(nodes[arg])
            elif name in BIN:
                b = stack.pop()
                a = stack.pop()
                r = _exact_node(name, a, b)
                nodes.append(r)
                stack.append(r)
            else:
                r = _exact_node(name, stack.pop())
                nodes.append(r)
                stack.append(r)
        out[i] = stack.pop()
    return out


def _test_inputs():
    a = np.array([1.5, -2.25, 3.0, 0.1, -0.0, 0.0, 1e-40, -7.0, 2.0, 1e30, -3.0, 0.75, 5e-39, 6.5e4, np.inf, -1.0],
                 dtype=np.float32)
    b = np.array([1.5, 0.5, -3.0, 0.3, 0.0, -0.0, 3e-41, 2.0, -1e-20, 1e20, -3.0, 7.0, -2e-38, 6.5e4, 1.0, np.nan],
                 dtype=np.float32)
    return [a, b]


def _trees(depth):
    """All expression trees with exactly `depth` op nodes over inputs 0, 1 (postfix)."""
    if depth == 0:
        return [[("IN", 0)], [("IN", 1)]]
    out = []
    for u in UN:
        for t in _trees(depth - 1):
            out.append(t + [(u, 0)])
    for bop in BIN:
        for i in range(depth):
            for l, r in itertools.product(_trees(i), _trees(depth - 1 - i)):
                out.append(l + r + [(bop, 0)])
    return out


def _run_oracle(seq, vals):
    toks = W.encode([(n, a) if n in ("IN", "IMM", "REF") else (n,) for n, a in seq])
    inputs = [(v, "f32", (1,)) for v in vals]
    return OG.evaluate(toks, [], inputs, (len(vals[0]),), "f32")


def test_all_programs_up_to_two_nodes_bitwise():
    vals = _test_inputs()
    progs = _trees(1) + _trees(2)
    assert len(progs) > 500
    for seq in progs:
        assert same_bits(_run_oracle(seq, vals), _exact_eval(seq, vals)), seq


def test_random_deep_programs_with_reads_bitwise():
    rng = np.random.default_rng(21)
    vals = _test_inputs()
    for _ in range(150):
        n_ops = int(rng.integers(3, 12))
        seq = [("IN", int(rng.integers(0, 2)))]
        for i in range(n_ops):
            op = (BIN + UN)[int(rng.integers(0, len(BIN) + len(UN)))]
            if op in BIN:
                c = int(rng.integers(0, 2 + i))
                seq.append(("IN", c) if c < 2 else ("REF", c - 2))
            seq.append((op, 0))
        assert same_bits(_run_oracle(seq, vals), _exact_eval(seq, vals)), seq


def test_max_min_tie_gives_second_operand():
    a = np.array([0.0, -0.0, 1.0, np.nan, 2.0], dtype=np.float32)
    b = np.array([-0.0, 0.0, 1.0, 3.0, np.nan], dtype=np.float32)
    mx = _run_oracle([("IN", 0), ("IN", 1), ("MAX", 0)], [a, b])
    mn = _run_oracle([("IN", 0), ("IN", 1), ("MIN", 0)], [a, b])
    assert same_bits(mx, b) and same_bits(mn, b)


def test_small_group_against_mpmath_per_node():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.prec = 200
    wl = W.small_group(8, 16)
    ins = wl.host_inputs()
    y = OG.evaluate(wl.tokens, wl.imm, [(a, dt, s.strides) for (a, dt), s in zip(ins, wl.inputs)],
                    wl.out_shape, wl.out_dtype)
    x, b, s, r = (a for a, _ in ins)
    k = rn32(Fraction(1) / mpf_fraction(mpmath.sqrt(2)))
    for i in range(8):
        for j in range(16):
            t = f32_binop("MUL", x[i, j], np.float32(1.7))
            t = f32_binop("ADD", t, b[j])
            u = f32_binop("MUL", t, k)
            e = rn32(mpf_fraction(mpmath.erf(mpmath.mpf(float(u)))))
            g = f32_binop("MUL", t, f32_binop("MUL", np.float32(0.5), f32_binop("ADD", np.float32(1.0), e)))
            want = f32_binop("ADD", f32_binop("MUL", g, s), r[i, j])
            assert same_bits(y[i, j], want), (i, j)


def _expc_reference(a):
    """exp(clamp(a, -4, 4)) without the oracle: clamp(x, lo, hi) =
    min(max(x, lo), hi) with the builtins' tie rule (max(a, b) = a if a > b
    else b, min likewise), so a NaN gives the second operand at each step and
    leaves the clamp as -4; then the exponential at 200 bits, rounded once."""
    import mpmath

    mpmath.mp.prec = 200
    a = float(a)
    c = a if a > -4.0 else -4.0
    c = c if c < 4.0 else 4.0
    return rn32(mpf_fraction(mpmath.exp(mpmath.mpf(c))))


def test_expc_clamp_bounds_against_mpmath():
    pytest.importorskip("mpmath")
    f = np.float32
    special = [0.0, -0.0, 1.0, -1.0, 3.999999, -3.999999, 4.0, -4.0,
               float(np.nextafter(f(4), f(np.inf))), float(np.nextafter(f(-4), f(-np.inf))),
               4.0000005, -4.0000005, 5.0, -5.0, 7.99, -7.99, 8.0, -8.0, 10.0, -10.0, 1e30, -1e30,
               1e-40, -1e-40, np.inf, -np.inf, np.nan]
    rng = np.random.default_rng(34)
    x = np.concatenate([np.array(special, dtype=np.float32),
                        (rng.random(400) * 24 - 12).astype(np.float32)])
    y = OG.evaluate(W.encode([("IN", 0), ("EXPC",)]), [], [(x, "f32", (1,))], x.shape, "f32")
    want = np.array([_expc_reference(v) for v in x], dtype=np.float32)
    assert same_bits(y, want)
    # the bounds are the only values it takes outside (-4, 4); NaN reads as -4
    assert y[np.isnan(x)][0] == want[special.index(-4.0)]
    assert y[x == np.float32(1e30)][0] == want[special.index(4.0)]


def test_broadcast_equals_materialised_expansion():
    wl = W.cap_group(24, 40, n_ops=20)
    ins = wl.host_inputs()
    bcast = [(a, dt, s.strides) for (a, dt), s in zip(ins, wl.inputs)]
    y1 = OG.evaluate(wl.tokens, wl.imm, bcast, wl.out_shape, wl.out_dtype)
    R, C = wl.out_shape
    full = []
    for (a, dt), spec in zip(ins, wl.inputs):
        f = bf16_to_f32(a) if dt == "bf16" else a
        full.append((np.broadcast_to(f.reshape(spec.shape) if spec.shape else f, (R, C)).copy()
                     if spec.shape != (R, 1) else np.repeat(f.reshape(R, 1), C, axis=1), "f32", (C, 1)))
    y2 = OG.evaluate(wl.tokens, wl.imm, full, wl.out_shape, wl.out_dtype)
    assert np.array_equal(y1, y2)


def test_interior_values_stay_f32_under_bf16():
    # Rounding every node to bf16 (the unfused bf16 chain) changes the root on
    # this workload: the oracle keeps the interior in f32.
    wl = W.cap_group(16, 64, n_ops=64)
    ins = wl.host_inputs()
    inputs = [(a, dt, s.strides) for (a, dt), s in zip(ins, wl.inputs)]
    y, nodes = OG.evaluate(wl.tokens, wl.imm, inputs, wl.out_shape, "bf16", return_nodes=True)
    assert np.array_equal(y, f32_to_bf16(nodes[-1]))
    prog = OG.decode(wl.tokens, 4, 0)
    vals = [OG.broadcast_input(a, dt, st, wl.out_shape) for a, dt, st in inputs]
    stack, rnodes = [], []
    for name, arg in prog:
        if name == "IN":
            stack.append(vals[arg])
        elif name == "REF":
            stack.append(rnodes[arg])
        else:
            args = [stack.pop()] if name in OG.UNARY else [stack.pop(), stack.pop()][::-1]
            r = bf16_to_f32(f32_to_bf16(OG.apply_op(name, *args)))
            rnodes.append(r)
            stack.append(r)
    assert not np.array_equal(f32_to_bf16(rnodes[-1]), y)


def test_gelu_special_values():
    x = np.array([0.0, -0.0, 10.0, -10.0, np.inf, -np.inf, np.nan], dtype=np.float32)
    g = OG.gelu(x)
    assert g[0] == 0.0 and g[2] == 10.0 and g[3] == 0.0 and np.isposinf(g[4])
    assert np.isnan(g[5]) and np.isnan(g[6])   # -inf * 0 is NaN in this op order


@pytest.mark.parametrize("seq,n_in,n_imm", [
    ([], 1, 0),
    ([("IN", 0)], 1, 0),                                   # no op node
    ([("IN", 0), ("ADD",)], 1, 0),                         # underflow
    ([("IN", 0), ("IN", 0)], 1, 0),                        # no op, depth 2
    ([("IN", 0), ("IN", 0), ("ADD",), ("IN", 0)], 1, 0),   # two values left
    ([("IN", 1), ("NEG",)], 1, 0),                         # input out of range
    ([("IMM", 0), ("NEG",)], 1, 0),                        # immediate out of range
    ([("IN", 0), ("REF", 0), ("ADD",)], 1, 0),             # REF before it exists
])
def test_malformed_programs_are_refused(seq, n_in, n_imm):
    toks = W.encode(seq) if seq else np.zeros(0, dtype=np.uint32)
    with pytest.raises(OG.ProgramError):
        OG.decode(toks, n_in, n_imm)


def test_cap_of_64_nodes():
    ok = W.encode([("IN", 0)] + [("NEG",)] * 64)
    assert len(OG.decode(ok, 1, 0)) == 65
    with pytest.raises(OG.ProgramError):
        OG.decode(W.encode([("IN", 0)] + [("NEG",)] * 65), 1, 0)
    with pytest.raises(OG.ProgramError):
        OG.decode(np.array([0x7F000000], dtype=np.uint32), 1, 0)


# ------------------------------------------------- SELECT, LOG, TANH, sigmoid

def _select_program():
    # c a b SELECT with a = x * 2 and b = log(y): each branch a node of its own
    return W.encode([("IN", 0), ("IN", 1), ("IMM", 0), ("MUL",), ("IN", 2), ("LOG",), ("SELECT",)])


def test_select_moves_the_picked_bits_and_never_the_other_branch():
    c = np.array([1, 0, 7, 0, -1, 0, 1, 0], dtype=np.int32)
    x = np.array([1.5, np.nan, np.inf, 2.0, -0.0, 1e38, 3.0, np.float32(-np.inf)], dtype=np.float32)
    y = np.array([-1.0, 4.0, np.nan, 0.0, 5.0, -2.0, -np.inf, 1.0], dtype=np.float32)
    inputs = [(c, "i32", (1,)), (x, "f32", (1,)), (y, "f32", (1,))]
    out = OG.evaluate(_select_program(), [2.0], inputs, (8,), "f32")
    want = []
    for ci, xi, yi in zip(c, x, y):
        if ci != 0:
            want.append(f32_binop("MUL", xi, np.float32(2.0)))
        else:
            want.append(rn32(mpf_fraction(__import__("mpmath").log(float(yi)))) if 0 < yi < np.inf
                        else {0.0: -np.inf, np.inf: np.inf}.get(float(yi), np.nan) if yi >= 0 else np.nan)
    assert same_bits(out, np.array(want, dtype=np.float32))
    # an unpicked NaN or infinity never reaches the result (x[1] NaN, y[6] = -inf);
    # a picked one does (x[2] = inf doubled, log(0) = -inf)
    assert np.isfinite(out[1]) and np.isfinite(out[6])
    assert np.isposinf(out[2]) and np.isneginf(out[3])


def test_select_of_bf16_branches_equals_the_stored_branch():
    rng = np.random.default_rng(31)
    a = f32_to_bf16(rng.standard_normal(64).astype(np.float32))
    b = f32_to_bf16(rng.standard_normal(64).astype(np.float32))
    c = rng.integers(0, 2, 64).astype(np.int32)
    toks = W.encode([("IN", 0), ("IN", 1), ("IN", 2), ("SELECT",)])
    out = OG.evaluate(toks, [], [(c, "i32", (1,)), (a, "bf16", (1,)), (b, "bf16", (1,))], (64,), "bf16")
    assert np.array_equal(out, np.where(c != 0, a, b))


def test_select_condition_broadcast_row_mask():
    rng = np.random.default_rng(32)
    m = rng.integers(0, 2, 5).astype(np.int32)
    x = rng.standard_normal((3, 5)).astype(np.float32)
    toks = W.encode([("IN", 0), ("IN", 1), ("IMM", 0), ("SELECT",)])
    out = OG.evaluate(toks, [-7.0], [(m, "i32", (0, 1)), (x, "f32", (5, 1))], (3, 5), "f32")
    assert same_bits(out, np.where(m[None, :] != 0, x, np.float32(-7.0)))


@pytest.mark.parametrize("seq,dtypes", [
    ([("IN", 0), ("IN", 1), ("IN", 1), ("SELECT",)], ["f32", "f32"]),          # condition not i32
    ([("IMM", 0), ("IN", 1), ("IN", 1), ("SELECT",)], ["i32", "f32"]),         # condition not an input token
    ([("IN", 1), ("NEG",), ("IN", 1), ("IN", 1), ("SELECT",)], ["i32", "f32"]),  # condition a node
    ([("IN", 0), ("NEG",)], ["i32"]),                                          # i32 read as a value
    ([("IN", 0), ("IN", 0), ("IN", 1), ("SELECT",)], ["i32", "f32"]),          # i32 as a branch
    ([("IN", 0), ("IN", 1), ("SELECT",)], ["i32", "f32"]),                     # two operands
])
def test_select_typing_is_refused(seq, dtypes):
    with pytest.raises(OG.ProgramError):
        OG.decode(W.encode(seq), len(dtypes), 1, dtypes)


def test_log_tanh_and_sigmoid_chain_against_mpmath():
    import mpmath

    mpmath.mp.prec = 200
    rng = np.random.default_rng(33)
    x = np.concatenate([rng.standard_normal(300).astype(np.float32) * 4,
                        np.array([0.0, -0.0, 1e-30, 20.0, -20.0, -90.0, 90.0], dtype=np.float32)])
    # sigmoid(x) = 1 / (1 + exp(-x)), four nodes; then log(sigmoid) and tanh(x)
    sig = W.encode([("IN", 0), ("NEG",), ("EXP",), ("IMM", 0), ("ADD",), ("RECIP",)])
    s, nodes = OG.evaluate(sig, [1.0], [(x, "f32", (1,))], x.shape, "f32", return_nodes=True)
    for xi, e, d, si in zip(x, nodes[1], nodes[2], s):
        assert e == rn32(mpf_fraction(mpmath.exp(-mpmath.mpf(float(xi))))) or (np.isinf(e) and float(xi) < -88)
        assert d == f32_binop("ADD", np.float32(1.0), e)
        assert same_bits(np.float32(si), f32_binop("DIV", np.float32(1.0), d))
    ls = OG.evaluate(W.encode([("IN", 0), ("LOG",)]), [], [(s, "f32", (1,))], x.shape, "f32")
    want = [rn32(mpf_fraction(mpmath.log(float(v)))) if v > 0 else np.float32(-np.inf) for v in s]
    assert same_bits(ls, np.array(want, dtype=np.float32))
    th = OG.evaluate(W.encode([("IN", 0), ("TANH",)]), [], [(x, "f32", (1,))], x.shape, "f32")
    want = [rn32(mpf_fraction(mpmath.tanh(float(v)))) if v != 0 else v for v in x]
    assert same_bits(th, np.array(want, dtype=np.float32))
