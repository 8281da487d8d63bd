"""Parity of the extended group op set (RECIP, LOG, TANH, SELECT with int32
conditions) on the GPU, through the C ABI, with the CPU oracle: bit for bit.

LOG and TANH are correctly rounded on both sides; RECIP is the IEEE quotient;
SELECT moves the picked operand's bits, so NaN and infinities planted in the
branch it does not pick must never show in the result.
"""

import numpy as np
import pytest

import oracle.group as OG
from oracle.f32 import bf16_to_f32, f32_to_bf16
from synth import workloads as W

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


def _run(R, toks, imm, inputs, out_shape, out_dtype):
    """inputs: [(host array, dtype, strides)]; returns (device result, oracle)."""
    want = OG.evaluate(toks, imm, inputs, out_shape, out_dtype)
    out = torch.empty(out_shape, dtype=torch.bfloat16 if out_dtype == "bf16" else torch.float32, device="cuda")
    out.fill_(float("nan"))      # poisoned: every element must be written
    R.psk_group_run(toks, imm, [(_to_dev(a, dt), st) for a, dt, st in inputs], out)
    torch.cuda.synchronize()
    return _to_host(out), want


@pytest.mark.parametrize("op", ["LOG", "TANH", "RECIP"])
def test_unary_node_over_many_inputs(dev, op):
    rng = np.random.default_rng(70)
    n = (1 << 22) + 3        # a ragged tail: the scalar path
    if op == "LOG":
        x = np.concatenate([rng.uniform(0, 4, n // 2), (1 + rng.uniform(-2 ** -7, 2 ** -7, n - n // 2))])
    elif op == "TANH":
        x = rng.uniform(-10, 10, n)
    else:
        x = rng.standard_normal(n) * 1e3
    x = x.astype(np.float32)
    x[: n // 4] = rng.integers(0, 2 ** 32, n // 4, dtype=np.uint64).astype(np.uint32).view(np.float32)
    x[:20] = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 1e-45, -1e-45, 1.0, -1.0, 2 ** -12, 9.0109135, 9.010913,
                       1.1754942e-38, 3.4028235e38, 2.0, 0.5, np.sqrt(2), 1e-40, -3.0, 8.5e37], dtype=np.float32)
    toks = W.encode([("IN", 0), (op,)])
    got, want = _run(dev, toks, [], [(x, "f32", (1,))], (n,), "f32")
    ok = _same(got, want, "f32")
    assert ok.all(), f"{(~ok).sum()} differ, e.g. x={x[~ok][:5]}"


def test_sigmoid_chain_and_log_sigmoid_bitwise(dev):
    rng = np.random.default_rng(71)
    x = (rng.standard_normal((257, 129)) * 6).astype(np.float32)
    x.flat[:8] = [0.0, -0.0, 90.0, -90.0, np.inf, -np.inf, np.nan, 1e-30]
    # log(1 / (1 + exp(-x))) with the sigmoid as its four-node chain
    toks = W.encode([("IN", 0), ("NEG",), ("EXP",), ("IMM", 0), ("ADD",), ("RECIP",), ("LOG",)])
    for odt in ("f32", "bf16"):
        got, want = _run(dev, toks, [1.0], [(x, "f32", (129, 1))], x.shape, odt)
        assert _same(got, want, odt).all()


def _conditions(shape, rng):
    c = rng.integers(0, 2, shape).astype(np.int32)
    flat = c.reshape(-1)
    flat[: min(6, flat.size)] = np.array([0, 1, -1, 2 ** 31 - 1, -2 ** 31, 7], dtype=np.int32)[: min(6, flat.size)]
    return c


@pytest.mark.parametrize("layout", ["full", "row_mask", "col_mask", "scalar", "gathered"])
@pytest.mark.parametrize("odt", ["f32", "bf16"])
def test_select_never_passes_the_unpicked_branch(dev, layout, odt):
    rng = np.random.default_rng(72)
    R_, C_ = 67, 96
    if layout == "full":
        c, cst = _conditions((R_, C_), rng), (C_, 1)
    elif layout == "row_mask":
        c, cst = _conditions((C_,), rng), (0, 1)
    elif layout == "col_mask":
        c, cst = _conditions((R_,), rng), (1, 0)
    elif layout == "scalar":
        c, cst = np.array([3], dtype=np.int32), (0, 0)
    else:
        c, cst = _conditions((R_, 2 * C_), rng), (2 * C_, 2)
    a = rng.standard_normal((R_, C_)).astype(np.float32)
    b = rng.standard_normal((R_, C_)).astype(np.float32)
    # poison both branches: whichever side is not picked carries NaN and infinities
    a[::3, ::5] = np.nan
    b[1::4, ::3] = np.inf
    b[2::5, 1::7] = np.nan
    # select(c, log(a), tanh(b)) then * 2: the branches are nodes, the select a node
    toks = W.encode([("IN", 0), ("IN", 1), ("LOG",), ("IN", 2), ("TANH",), ("SELECT",), ("IMM", 0), ("MUL",)])
    inputs = [(c, "i32", cst), (a, "f32", (C_, 1)), (b, "f32", (C_, 1))]
    got, want = _run(dev, toks, [2.0], inputs, (R_, C_), odt)
    ok = _same(got, want, odt)
    assert ok.all(), f"{(~ok).sum()} differ"


def test_select_of_stored_bf16_moves_the_stored_bits(dev):
    rng = np.random.default_rng(73)
    n = 4099
    a = f32_to_bf16(rng.standard_normal(n).astype(np.float32))
    b = f32_to_bf16(rng.standard_normal(n).astype(np.float32) * 1e30)
    a[:4] = [0x7F80, 0xFF80, 0x8000, 0x0001]     # inf, -inf, -0, the least subnormal
    c = rng.integers(0, 2, n).astype(np.int32)
    toks = W.encode([("IN", 0), ("IN", 1), ("IN", 2), ("SELECT",)])
    got, want = _run(dev, toks, [], [(c, "i32", (1,)), (a, "bf16", (1,)), (b, "bf16", (1,))], (n,), "bf16")
    assert np.array_equal(got, want)
    assert np.array_equal(got, np.where(c != 0, a, b))


def test_unaligned_condition_takes_the_scalar_path(dev):
    rng = np.random.default_rng(74)
    c = torch.from_numpy(rng.integers(0, 2, 4 * 64 + 1).astype(np.int32)).cuda()[1:]   # 4-byte, not 16-byte aligned
    x = torch.from_numpy(rng.standard_normal(4 * 64).astype(np.float32)).cuda()
    out = torch.empty(4, 64, device="cuda")
    toks = W.encode([("IN", 0), ("IN", 1), ("IMM", 0), ("SELECT",)])
    dev.psk_group_run(toks, [-5.0], [(c, (64, 1)), (x, (64, 1))], out)
    torch.cuda.synchronize()
    want = np.where(c.cpu().numpy().reshape(4, 64) != 0, x.cpu().numpy().reshape(4, 64), np.float32(-5.0))
    assert np.array_equal(out.cpu().numpy().view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("seed", range(6))
def test_random_programs_extended_op_set_bitwise(dev, seed):
    rng = np.random.default_rng(200 + seed)
    ops_b = ["ADD", "SUB", "MUL", "DIV", "MAX", "MIN"]
    ops_u = ["NEG", "ABS", "EXP", "EXPC", "GELU", "SQRT", "SQRTA", "ERF", "RECIP", "LOG", "TANH"]
    R_, C_ = 41, 72 + seed        # ragged widths on odd seeds
    seq, nodes = [("IN", 0)], 0
    while nodes < int(rng.integers(8, 60)):
        r = rng.random()
        if r < 0.35:
            c = int(rng.integers(0, 4 + nodes))
            seq.append(("IN", c) if c < 3 else (("IMM", int(rng.integers(0, 2))) if c == 3 else ("REF", c - 4)))
            seq.append((str(rng.choice(ops_b)),))
            nodes += 1
        elif r < 0.5 and nodes > 0:
            # acc, then select(cond, acc, other) combined back into acc
            other = ("IN", int(rng.integers(0, 3))) if rng.random() < 0.6 else ("IMM", int(rng.integers(0, 2)))
            branches = [("REF", nodes - 1), other] if rng.random() < 0.5 else [other, ("REF", nodes - 1)]
            seq += [("IN", 3)] + branches + [("SELECT",), (str(rng.choice(ops_b)),)]
            nodes += 2
        else:
            seq.append((str(rng.choice(ops_u)),))
            nodes += 1
    toks = W.encode(seq)
    imm = np.array([0.5, -1.25], dtype=np.float32)
    x = (rng.standard_normal((R_, C_)) * 3).astype(np.float32)
    x.flat[:12] = [0.0, -0.0, np.inf, -np.inf, np.nan, 1e-45, -1e-40, 3e38, 1.0, -1.0, 2 ** -13, 9.5]
    rowv = (rng.standard_normal(C_) * 2).astype(np.float32)
    col = (rng.standard_normal(R_) * 2).astype(np.float32)
    cond = rng.integers(-1, 2, (R_, C_)).astype(np.int32)
    inputs = [(x, "f32", (C_, 1)), (rowv, "f32", (0, 1)), (col, "f32", (1, 0)), (cond, "i32", (C_, 1))]
    odt = "bf16" if seed % 2 else "f32"
    got, want = _run(dev, toks, imm, inputs, (R_, C_), odt)
    ok = _same(got, want, odt)
    assert ok.all(), f"{(~ok).sum()} differ"


def test_extended_ops_are_refused_with_wrong_types(dev):
    x = torch.zeros(8, 8, device="cuda")
    c = torch.zeros(8, 8, dtype=torch.int32, device="cuda")
    sel = W.encode([("IN", 0), ("IN", 1), ("IN", 1), ("SELECT",)])
    with pytest.raises(dev.PskError) as e:
        dev.psk_group_run(sel, [], [(x, (8, 1)), (x, (8, 1))], torch.empty(8, 8, device="cuda"))
    assert e.value.name == "PSK_E_DTYPE"
    with pytest.raises(dev.PskError) as e:
        dev.psk_group_run(W.encode([("IN", 0), ("LOG",)]), [], [(c, (8, 1))], torch.empty(8, 8, device="cuda"))
    assert e.value.name == "PSK_E_DTYPE"


def test_select_group_full_size_sampled_rows(dev):
    """The select/log/tanh group at its full size [8192, 8192] (int32 row mask,
    bf16 in and out), launched as the benchmark launches it; sampled rows
    against the oracle."""
    wl = W.select_group()
    dins = wl.device_inputs()
    out = torch.empty(wl.out_shape, dtype=torch.bfloat16, device="cuda")
    dev.psk_group_run(wl.tokens, wl.imm, [(t, s.strides) for t, s in zip(dins, wl.inputs)], out)
    torch.cuda.synchronize()
    rows = np.array([0, 1, 4095, 8191] + list(np.random.default_rng(2).integers(0, 8192, 8)))
    idx = torch.from_numpy(rows).cuda()
    x = _to_host(dins[0][idx])
    mask = dins[1].cpu().numpy()
    assert mask.dtype == np.int32 and 0.6 < mask.mean() < 0.8
    ins = [(x, "bf16", (8192, 1)), (mask, "i32", (0, 1))]
    want = OG.evaluate(wl.tokens, wl.imm, ins, (len(rows), 8192), "bf16")
    ok = _same(_to_host(out[idx]), want, "bf16")
    assert ok.all(), f"{(~ok).sum()} differ"
