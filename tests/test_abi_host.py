"""Host-side checks of the C-ABI library (no GPU needed): it loads, exports
every entry point include/psk.h declares, validates programs exactly as the
oracle's definition does, and injects the AdamW scalars the oracle computes."""

import ctypes
import os
import re

import numpy as np
import pytest

import oracle.adamw as OA
import oracle.group as OG
from synth import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def native():
    from reduction_groups_gb300 import build as B

    B.build()
    from reduction_groups_gb300 import _native as N

    return N


def test_library_exports_every_declared_symbol(native):
    header = open(os.path.join(ROOT, "include", "psk.h")).read()
    declared = set(re.findall(r"^\s*(?:int|const char\*)\s+(psk_\w+)\s*\(", header, re.M))
    assert declared == set(native.EXPORTS)
    L = native.lib()
    for name in declared:
        assert hasattr(L, name), name


def test_opcodes_agree_across_header_oracle_and_inputs():
    header = open(os.path.join(ROOT, "include", "psk.h")).read()
    hdr = {k: int(v, 16) for k, v in re.findall(r"#define PSK_OP_(\w+) (0x[0-9a-fA-F]+)", header)}
    assert hdr == OG.OP
    assert hdr == W.OPCODES


def _rand_program(rng, n_in, n_imm, valid=True):
    ops_b = ["ADD", "SUB", "MUL", "DIV", "MAX", "MIN"]
    ops_u = ["NEG", "ABS", "EXP", "EXPC", "GELU", "SQRT", "SQRTA", "ERF", "RECIP", "LOG", "TANH"]
    seq, depth, nodes = [], 0, 0
    n_ops = int(rng.integers(1, 70))
    while nodes < n_ops:
        r = rng.random()
        if depth < 2 or r < 0.35:
            kind = rng.choice(["IN", "IMM", "REF"] if nodes else ["IN", "IMM"])
            if kind == "IN":
                seq.append(("IN", int(rng.integers(0, n_in))))
            elif kind == "IMM" and n_imm:
                seq.append(("IMM", int(rng.integers(0, n_imm))))
            elif kind == "REF":
                seq.append(("REF", int(rng.integers(0, nodes))))
            else:
                continue
            depth += 1
        elif r < 0.6:
            seq.append((str(rng.choice(ops_u)),))
            nodes += 1
        elif r < 0.68 and depth >= 3:
            seq.append(("SELECT",))     # valid only where the condition slot holds an IN token
            depth -= 2
            nodes += 1
        else:
            seq.append((str(rng.choice(ops_b)),))
            depth -= 1
            nodes += 1
    while depth > 1:
        seq.append(("ADD",))
        depth -= 1
        nodes += 1
    if not valid:
        k = int(rng.integers(0, 5))
        if k == 0:
            seq.append(("ADD",))                      # underflow
        elif k == 1:
            seq.insert(0, ("IN", n_in))               # input out of range
        elif k == 2:
            seq.append(("IN", 0))                     # two values left
        elif k == 3:
            seq.insert(1, ("REF", 99))                # REF ahead
        else:
            seq += [("NEG",)] * 70                    # past the cap
    return W.encode(seq)


def test_program_check_matches_oracle_definition(native):
    from reduction_groups_gb300 import ops

    rng = np.random.default_rng(12)
    for trial in range(600):
        valid = trial % 3 != 0
        toks = _rand_program(rng, 3, 2, valid)
        imm = np.array([1.5, -2.0], dtype=np.float32)
        try:
            prog = OG.decode(toks, 3, 2)
            want = ("ok", sum(1 for n, _ in prog if n not in ("IN", "IMM", "REF")))
        except OG.ProgramError:
            want = ("refused", None)
        try:
            nn, ns = ops.psk_group_check(toks, 3, imm)
            got = ("ok", nn)
            assert 1 <= ns <= nn + 3
        except native.PskError as e:
            assert e.name in ("PSK_E_PROGRAM", "PSK_E_TOO_MANY_NODES")
            got = ("refused", None)
        assert got == want, (toks, got, want)


def test_refusals_name_the_fault(native):
    from reduction_groups_gb300 import ops

    with pytest.raises(native.PskError) as e:
        ops.psk_group_check(W.encode([("IN", 0)] + [("NEG",)] * 65), 1)
    assert e.value.name == "PSK_E_TOO_MANY_NODES" and "cap" in str(e.value)
    with pytest.raises(native.PskError) as e:
        ops.psk_group_check(np.array([0x7F000000], dtype=np.uint32), 1)
    assert e.value.name == "PSK_E_PROGRAM" and "opcode" in str(e.value)
    with pytest.raises(native.PskError):
        ops.psk_group_check(W.encode([("IN", 0), ("NEG",)]), 17)


def test_interpreter_refuses_before_any_device_work(native):
    """psk_group_run_interp validates exactly as psk_group_run does and
    refuses before touching a device (host tensors stand in for the
    pointers, which a refusal never dereferences)."""
    import torch

    from reduction_groups_gb300 import ops

    x = torch.zeros((4, 8))
    y = torch.empty((4, 8))
    L = native.lib()

    def call(tokens, inputs, out, math=0):
        p, keep = ops._program(tokens, [])
        arr, n, o = ops._group_args(inputs, out)
        rc = L.psk_group_run_interp(ctypes.byref(p), arr, n, ctypes.byref(o), math, None)
        return rc, L.psk_last_error().decode()

    rc, msg = call(W.encode([("IN", 0)] + [("NEG",)] * 65), [(x, (8, 1))], y)
    assert rc == -2 and "cap" in msg                                 # PSK_E_TOO_MANY_NODES
    rc, _ = call(W.encode([("IN", 1), ("NEG",)]), [(x, (8, 1))], y)
    assert rc == -1                                                   # PSK_E_PROGRAM
    rc, _ = call(W.encode([("IN", 0), ("NEG",)]), [(x, (8, 1))], y, math=3)
    assert rc == -9                                                   # PSK_E_ARG
    # an input overlapping the output with another layout
    buf = torch.zeros(64)
    rc, msg = call(W.encode([("IN", 0), ("NEG",)]), [(buf[1:33].view(4, 8), (8, 1))], buf[:32].view(4, 8))
    assert rc == -8                                                   # PSK_E_ALIAS


def test_adamw_scalars_equal_oracle_injection(native):
    from reduction_groups_gb300 import ops

    rng = np.random.default_rng(3)
    ts = list(range(1, 3001)) + [int(t) for t in rng.integers(3001, 1_000_001, 400)] + [1_000_000]
    for beta1, beta2 in ((0.9, 0.999), (0.8, 0.95), (0.99, 0.9999), (0.3, 0.7)):
        for t in ts if beta1 == 0.9 else ts[::10]:
            hp = W.AdamWHyper(lr=3e-4, beta1=beta1, beta2=beta2, eps=1e-8, weight_decay=0.01, t=t)
            got = ops.psk_adamw_scalars(hp)
            h = OA.hyper_f32(hp.lr, beta1, beta2, hp.eps, hp.weight_decay, t)
            want = np.array([h[k] for k in ("b1", "b2", "omb1", "omb2", "bc1", "bc2", "lr", "eps", "wd")],
                            dtype=np.float32)
            assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), (beta1, beta2, t, got, want)


def test_adamw_scalars_refuse_bad_hyperparameters(native):
    from reduction_groups_gb300 import ops

    for bad in (dict(t=0), dict(beta1=1.0), dict(beta2=0.0), dict(lr=float("nan"))):
        hp = W.AdamWHyper(**bad)
        with pytest.raises(native.PskError):
            ops.psk_adamw_scalars(hp)


def test_group_prepare_compiles_every_op_and_layout(native):
    """The kernel generator and the run-time compiler on the host (no device):
    one program with every op, in each storage type, access mode and vector
    width; tensors are inspected, never read."""
    torch = pytest.importorskip("torch")
    from reduction_groups_gb300 import ops

    seq = [("IN", 0), ("IN", 1), ("ADD",), ("IN", 2), ("SUB",), ("IMM", 0), ("MUL",), ("IN", 0), ("DIV",),
           ("REF", 0), ("MAX",), ("IN", 1), ("MIN",), ("NEG",), ("ABS",), ("EXP",), ("EXPC",), ("GELU",),
           ("SQRT",), ("SQRTA",), ("ERF",), ("IMM", 1), ("REF", 2), ("SUB",), ("ADD",)]
    toks = W.encode(seq)
    imm = np.array([0.5, -3.0], dtype=np.float32)
    for din in (torch.float32, torch.bfloat16):
        for dout in (torch.float32, torch.bfloat16):
            for cols, step in ((16, 1), (15, 1), (16, 2)):     # contiguous, V = 1, gathered
                x = torch.zeros(8, cols * step, dtype=din)
                row = torch.zeros(cols, dtype=din)
                col = torch.zeros(8, 1, dtype=din)
                out = torch.zeros(8, cols, dtype=dout)
                ops.psk_group_prepare(toks, imm, [(x, (cols * step, step)), (row, (0, 1)), (col, (1, 0))], out)


def test_group_prepare_compiles_the_extended_op_set(native):
    """RECIP, LOG, TANH and SELECT with an int32 condition in every access
    mode, and the sigmoid chain."""
    torch = pytest.importorskip("torch")
    from reduction_groups_gb300 import ops

    seq = [("IN", 0), ("IN", 1), ("RECIP",), ("IN", 1), ("LOG",), ("SELECT",), ("TANH",),
           ("IN", 1), ("NEG",), ("EXP",), ("IMM", 0), ("ADD",), ("RECIP",), ("ADD",)]
    toks = W.encode(seq)
    for din in (torch.float32, torch.bfloat16):
        for cols, cstride in ((16, (16, 1)), (16, (0, 1)), (15, (15, 1)), (16, (1, 0))):
            c = torch.zeros(8, cols, dtype=torch.int32)
            x = torch.zeros(8, cols, dtype=din)
            out = torch.zeros(8, cols, dtype=torch.float32)
            ops.psk_group_prepare(toks, np.array([1.0], np.float32), [(c, cstride), (x, (cols, 1))], out)


def test_select_typing_refusals(native):
    torch = pytest.importorskip("torch")
    from reduction_groups_gb300 import ops

    c = torch.zeros(4, 4, dtype=torch.int32)
    x = torch.zeros(4, 4)
    out = torch.zeros(4, 4)
    sel = W.encode([("IN", 0), ("IN", 1), ("IN", 1), ("SELECT",)])
    ops.psk_group_prepare(sel, None, [(c, (4, 1)), (x, (4, 1))], out)
    with pytest.raises(native.PskError) as e:                      # condition is f32
        ops.psk_group_prepare(sel, None, [(x, (4, 1)), (x, (4, 1))], out)
    assert e.value.name == "PSK_E_DTYPE" and "condition" in str(e.value)
    with pytest.raises(native.PskError) as e:                      # i32 read as a value
        ops.psk_group_prepare(W.encode([("IN", 0), ("NEG",)]), None, [(c, (4, 1))], out)
    assert e.value.name == "PSK_E_DTYPE"
    with pytest.raises(native.PskError) as e:                      # condition is a node
        ops.psk_group_check(W.encode([("IN", 1), ("NEG",), ("IN", 1), ("IN", 1), ("SELECT",)]), 2)
    assert e.value.name == "PSK_E_PROGRAM" and "condition" in str(e.value)
    with pytest.raises(native.PskError) as e:                      # an i32 output
        ops.psk_group_prepare(sel, None, [(c, (4, 1)), (x, (4, 1))], torch.zeros(4, 4, dtype=torch.int32))
    assert e.value.name == "PSK_E_DTYPE"


def test_group_prepare_compiles_the_fast_math_mode(native):
    torch = pytest.importorskip("torch")
    from reduction_groups_gb300 import ops

    toks = W.encode([("IN", 0), ("EXP",), ("EXPC",), ("ERF",), ("GELU",), ("LOG",), ("TANH",)])
    x = torch.zeros(8, 16)
    ops.psk_group_prepare(toks, None, [(x, (16, 1))], torch.zeros(8, 16), math="fast")
    ops.psk_group_prepare(toks, None, [(x, (16, 1))], torch.zeros(8, 16, dtype=torch.bfloat16), math="fast")
    from reduction_groups_gb300 import _native as N

    p, keep = ops._program(toks, None)
    arr, n, o = ops._group_args([(x, (16, 1))], torch.zeros(8, 16))
    assert N.lib().psk_group_prepare_ex(ctypes.byref(p), arr, n, ctypes.byref(o), 7) == -9   # PSK_E_ARG


def test_test_hook_refuses_bad_rows(native):
    from reduction_groups_gb300 import ops

    with pytest.raises(native.PskError) as e:
        ops.psk_test_drop_row(-2)
    assert e.value.name == "PSK_E_ARG"


def test_group_prepare_refuses_as_check(native):
    torch = pytest.importorskip("torch")
    from reduction_groups_gb300 import ops

    x = torch.zeros(4, 4)
    bad = W.encode([("IN", 0)] + [("NEG",)] * 65)
    with pytest.raises(native.PskError) as e:
        ops.psk_group_prepare(bad, None, [(x, (4, 1))], torch.zeros(4, 4))
    assert e.value.name == "PSK_E_TOO_MANY_NODES"
    ops.psk_group_prepare(W.encode([("IN", 0), ("NEG",)]), None, [(x, (4, 1))], x)      # in place: allowed
    with pytest.raises(native.PskError) as e:                                             # transposed: races
        ops.psk_group_prepare(W.encode([("IN", 0), ("NEG",)]), None, [(x, (1, 4))], x)
    assert e.value.name == "PSK_E_ALIAS"


def test_scheduled_lr_equals_oracle(native):
    """The host's exact schedule (binary64 pairs, double-double cos) against the
    oracle's (rationals, mpmath): the same f32 for every step, including lrs
    and lengths whose quotients fall on or next to f32 rounding midpoints."""
    from reduction_groups_gb300 import ops

    rng = np.random.default_rng(17)
    cases = [(3e-4, "linear", 100, 1000), (1e-3, "cosine", 50, 1050), (2.0 ** -10, "linear", 2 ** 12, 2 ** 20),
             (2.0 ** -7 * 3, "cosine", 0, 3 * 2 ** 10), (6e-4, "cosine", 2000, 100000), (1.0, "linear", 0, 7),
             (0.1, "constant", 0, 1)]
    for lr, kind, w, total in cases:
        ts = sorted(set([1, 2, w, w + 1, total - 1, total, total + 3, max(1, w // 2), w + (total - w) // 3,
                         w + (total - w) // 2, w + 2 * (total - w) // 3] +
                        [int(t) for t in rng.integers(1, total + 5, 300)]))
        for t in ts:
            if t < 1:
                continue
            hp = W.AdamWHyper(lr=lr, t=int(t))
            got = ops.psk_adamw_lr(hp, kind, w, total)
            want = OA.lr_scheduled(lr, kind, w, total, int(t))
            assert got.view(np.uint32) == np.float32(want).view(np.uint32), (lr, kind, w, total, t, got, want)


def test_adamw_workspace_and_schedule_refusals(native):
    torch = pytest.importorskip("torch")
    from reduction_groups_gb300 import ops

    leaves = [tuple(torch.zeros(n) for _ in range(4)) for n in (5, 0, 3000, 70000)]
    assert ops.psk_adamw_workspace(leaves) == 0
    nb = 1 + 3 + 69                                   # blocks of 1024
    ng = 1 + 1 + 2                                    # groups of 64 blocks
    want = 16 + ((4 * nb + 15) // 16) * 16 + ((4 * ng + 15) // 16) * 16 + ((4 * 3 + 15) // 16) * 16
    assert ops.psk_adamw_workspace(leaves, grad_clip=1.0) == want
    hp = W.AdamWHyper(t=3)
    with pytest.raises(native.PskError) as e:
        ops.psk_adamw_lr(hp, "linear", 10, 10)
    assert e.value.name == "PSK_E_ARG"
    with pytest.raises(native.PskError):
        ops.psk_adamw_workspace(leaves, grad_clip=float("nan"))


def test_static_scratch_refuses_trees_beyond_its_buffer(native):
    """The fixed buffer's size check happens on the host, before any device
    work: a tree needing more clipping scratch is refused (no device here, so a
    check that let it through would fail with PSK_E_CUDA instead)."""
    torch = pytest.importorskip("torch")
    from reduction_groups_gb300 import _native as N

    t = torch.zeros(4)
    arr = (N.psk_leaf * 1)()
    arr[0].theta = arr[0].m = arr[0].v = arr[0].grad = t.data_ptr()
    arr[0].grad_dtype = N.PSK_F32
    arr[0].numel = 3 * 10 ** 9                     # never dereferenced: refused first
    h = N.psk_adamw_hparams(3e-4, 0.9, 0.999, 1e-8, 0.01, 1)
    sc = N.psk_adamw_schedule(N.PSK_LR_CONSTANT, 0, 1, 1.0)
    rc = N.lib().psk_adamw_tree_static(arr, 1, ctypes.byref(h), ctypes.byref(sc), None)
    assert N.ERRORS.get(rc) == "PSK_E_ARG" and "fixed buffer" in N.lib().psk_last_error().decode()
