"""The group interpreter (psk_group_run_interp: one precompiled kernel that
walks the program's node list per element) through the C ABI, against the
oracle and against the kernel specialised for the program (psk_group_run):
the same bits in both math modes, for every op, every input layout, both
vector widths, and the same refusals."""

import ctypes

import numpy as np
import pytest

import oracle.group as OG
from oracle.f32 import bf16_to_f32
from synth import workloads as W
from tests.guard import guarded

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import reduction_groups_gb300 as R

    return R


def _to_dev(a, dtype):
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    if dtype == "i32":
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def _to_host(t):
    if t.dtype == torch.bfloat16:
        return t.cpu().view(torch.int16).numpy().view(np.uint16)
    return t.cpu().numpy()


def _same(a, b, dtype):
    x = bf16_to_f32(a) if dtype == "bf16" else np.asarray(a, dtype=np.float32)
    y = bf16_to_f32(b) if dtype == "bf16" else np.asarray(b, dtype=np.float32)
    return (x.view(np.uint32) == y.view(np.uint32)) | (np.isnan(x) & np.isnan(y))


def _both(dev, toks, imm, dins, shape, odt, math):
    """The specialised kernel's output and the interpreter's, each into a
    poisoned, guarded output."""
    outs = []
    for fn in (dev.psk_group_run, dev.psk_group_run_interp):
        g = guarded(shape, torch.bfloat16 if odt == "bf16" else torch.float32)
        fn(toks, imm, dins, g.tensor, math=math)
        torch.cuda.synchronize()
        assert g.intact(), "a store landed outside the output"
        outs.append(_to_host(g.tensor))
    return outs


@pytest.mark.parametrize("shape", [(96, 200), (37, 53), (130, 1024), (1, 4)])
@pytest.mark.parametrize("math", ["exact", "fast"])
def test_cap_group_interpreter_same_bits(dev, shape, math):
    """The 64-node program (EXPC, GELU, SQRTA and binary nodes over row,
    column and scalar broadcasts); 53 columns take the one-element path."""
    wl = W.cap_group(*shape)
    ins = wl.host_inputs()
    dins = [(_to_dev(a, dt), spec.strides) for (a, dt), spec in zip(ins, wl.inputs)]
    jit, interp = _both(dev, wl.tokens, wl.imm, dins, wl.out_shape, wl.out_dtype, math)
    ok = _same(interp, jit, "bf16")
    assert ok.all(), f"{(~ok).sum()} differ from the specialised kernel"
    if math == "exact":
        want = OG.evaluate(wl.tokens, wl.imm, [(a, dt, spec.strides) for (a, dt), spec in zip(ins, wl.inputs)],
                           wl.out_shape, wl.out_dtype)
        assert _same(interp, want, "bf16").all()


def _random_program(rng, n_in_f32):
    """A random program over every op: operands from the f32 inputs, two
    immediates and earlier nodes; SELECTs on the int32 input n_in_f32."""
    ops_b = ["ADD", "SUB", "MUL", "DIV", "MAX", "MIN"]
    ops_u = ["NEG", "ABS", "EXP", "EXPC", "GELU", "SQRT", "SQRTA", "ERF", "RECIP", "LOG", "TANH"]
    seq = [("IN", 0)]
    nodes = 0
    for i in range(int(rng.integers(8, 60))):
        if nodes >= 60:
            break
        r = rng.random()
        if r < 0.4:
            c = int(rng.integers(0, n_in_f32 + 1 + i))
            if c < n_in_f32:
                seq.append(("IN", c))
            elif c == n_in_f32 or c - n_in_f32 - 1 >= nodes:
                seq.append(("IMM", int(rng.integers(0, 2))))
            else:
                seq.append(("REF", c - n_in_f32 - 1))
            seq.append((str(rng.choice(ops_b)),))
            nodes += 1
        elif r < 0.5:
            # select(condition, acc, input): the condition pushed under the accumulator
            seq = [("IN", n_in_f32)] + seq + [("IN", int(rng.integers(0, n_in_f32))), ("SELECT",)]
            nodes += 1
        else:
            seq.append((str(rng.choice(ops_u)),))
            nodes += 1
    return W.encode(seq)


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("odt", ["f32", "bf16"])
def test_random_programs_interpreter_same_bits(dev, seed, odt):
    rng = np.random.default_rng(300 + seed)
    R_, C_ = 41, 64
    x = (rng.standard_normal((R_, C_)) * 3).astype(np.float32)
    x.flat[:12] = [0.0, -0.0, np.inf, -np.inf, np.nan, 1e-45, -1e-40, 3e38, 88.8, -104.0, 4.0, 1.0]
    rowv = (rng.standard_normal(C_) * 2).astype(np.float32)
    col = (rng.standard_normal(R_) * 2).astype(np.float32)
    cond = rng.integers(0, 2, (R_, C_)).astype(np.int32)
    toks = _random_program(rng, 3)
    imm = np.array([0.5, -1.25], dtype=np.float32)
    inputs = [(x, "f32", (C_, 1)), (rowv, "f32", (0, 1)), (col, "f32", (1, 0)), (cond, "i32", (C_, 1))]
    dins = [(_to_dev(a, dt), st) for a, dt, st in inputs]
    want = OG.evaluate(toks, imm, inputs, (R_, C_), odt)
    for math in ("exact", "fast"):
        jit, interp = _both(dev, toks, imm, dins, (R_, C_), odt, math)
        assert _same(interp, jit, odt).all()
        if math == "exact":
            ok = _same(interp, want, odt)
            assert ok.all(), f"{(~ok).sum()} differ from the oracle"


def test_interpreter_gathered_input_and_rank3(dev):
    """An input read with a stride of 2 along the last axis (the gather path)
    into a rank-3 output, with a broadcast middle axis."""
    rng = np.random.default_rng(77)
    A, B, C = 3, 5, 24
    a = rng.standard_normal((A, B, 2 * C)).astype(np.float32)
    b = rng.standard_normal((A, 1, C)).astype(np.float32)
    toks = W.encode([("IN", 0), ("IN", 1), ("MUL",), ("EXP",), ("IN", 0), ("ADD",)])
    inputs = [(a, "f32", (B * 2 * C, 2 * C, 2)), (b, "f32", (C, 0, 1))]
    dins = [(_to_dev(a_, dt), st) for a_, dt, st in inputs]
    want = OG.evaluate(toks, [], inputs, (A, B, C), "f32")
    jit, interp = _both(dev, toks, [], dins, (A, B, C), "f32", "exact")
    assert _same(interp, want, "f32").all()
    assert _same(interp, jit, "f32").all()


def test_interpreter_refusals_and_empty_output(dev):
    x = torch.zeros((4, 8), device="cuda")
    y = torch.empty((4, 8), device="cuda")
    too_many = W.encode([("IN", 0)] + [("NEG",)] * 65)
    with pytest.raises(dev.PskError) as e:
        dev.psk_group_run_interp(too_many, [], [(x, (8, 1))], y)
    assert e.value.name == "PSK_E_TOO_MANY_NODES"
    with pytest.raises(dev.PskError) as e:
        dev.psk_group_run_interp(W.encode([("IN", 1), ("NEG",)]), [], [(x, (8, 1))], y)
    assert e.value.name == "PSK_E_PROGRAM"
    with pytest.raises(KeyError):          # the binding knows two math modes
        dev.psk_group_run_interp(W.encode([("IN", 0), ("NEG",)]), [], [(x, (8, 1))], y, math="other")
    # the C ABI refuses any other mode value before launching
    from reduction_groups_gb300 import _native as N
    from reduction_groups_gb300 import ops

    p, keep = ops._program(W.encode([("IN", 0), ("NEG",)]), [])
    arr, n, o = ops._group_args([(x, (8, 1))], y)
    assert N.lib().psk_group_run_interp(ctypes.byref(p), arr, n, ctypes.byref(o), 7, None) == -9   # PSK_E_ARG
    empty = torch.empty((0, 8), device="cuda")
    dev.psk_group_run_interp(W.encode([("IN", 0), ("NEG",)]), [], [(torch.zeros((0, 8), device="cuda"), (8, 1))],
                             empty)
    torch.cuda.synchronize()
