"""A fusion group evaluated node by node (the unfused chain), in f32.

Definition followed (PSK-Realize, "What a group is" and "What it buys"): a
group is a connected chain of elementwise primitives over one loop nest whose
inputs may be smaller and broadcast; every member is computed in the root's
arithmetic type (f32, also for bf16 storage) and only the root is rounded to
its storage type; fusion reassociates nothing, so the fused result is the
unfused chain's.  The oracle is that unfused chain: one full f32 array per
node, in program order.

Program format (postfix, one 32-bit token per item, opcode in the top byte,
argument in the low 24 bits):

  operand tokens  IN k (input k), IMM k (immediate k), REF k (op node k's value)
  binary ops      ADD SUB MUL DIV MAX MIN    (a b OP -> OP(a, b))
  unary ops       NEG ABS EXP EXPC GELU SQRT SQRTA ERF RECIP LOG TANH
  ternary op      SELECT                     (c a b SELECT -> a where c != 0, else b)

Readings of the pages taken here:
* the 64-node cap ("past sixty-four nodes the group stops growing") counts op
  nodes; operand tokens are not nodes.  A REF re-reads a node's value, which
  is the value a re-emitted expression would compute again;
* max(a, b) = a if a > b else b and min(a, b) = a if a < b else b, so a tie
  (and +0 against -0) gives the second operand (presk "The language",
  builtins max/min); clamp(x, lo, hi) = min(max(x, lo), hi);
* EXPC(a) = exp(clamp(a, -4, 4)) and SQRTA(a) = sqrt(|a|), one node each;
* gelu(a) = a * (0.5 * (1 + erf(a * RN(1/sqrt 2)))), exp and erf correctly
  rounded (``oracle.crmath``);
* broadcasting: each input gives an element stride per output axis, 0 where
  it is broadcast (trailing-axis alignment, presk "The language",
  Broadcasting; a length-1 column [R, 1] is read with stride (1, 0));
* the op set beyond the configurations' follows poot "Fusion and Planning",
  Pointwise chains (the unaries Neg, Exp, Log, Sqrt, Recip, Tanh and Erf, and
  Select): RECIP is the IEEE quotient 1/a, LOG and TANH are correctly rounded
  like EXP and ERF; SELECT's condition is an I32 region input (the operand
  just before the two branches must be an IN token of an "i32" input), c != 0
  picks a, and the select moves the picked value's bits without arithmetic,
  so a NaN or an infinity in the other branch never reaches the result.  An
  I32 input is read by SELECT conditions only; any other use is refused.
  Sigmoid is not an op of its own: it is written as the chain
  1 / (1 + exp(-a)).
"""

from __future__ import annotations

import numpy as np

from . import crmath
from .f32 import store, widen

OP = {
    "IN": 0x01, "IMM": 0x02, "REF": 0x03,
    "ADD": 0x10, "SUB": 0x11, "MUL": 0x12, "DIV": 0x13, "MAX": 0x14, "MIN": 0x15,
    "NEG": 0x20, "ABS": 0x21, "EXP": 0x22, "EXPC": 0x23, "GELU": 0x24,
    "SQRT": 0x25, "SQRTA": 0x26, "ERF": 0x27, "RECIP": 0x28, "LOG": 0x29, "TANH": 0x2A,
    "SELECT": 0x30,
}
NAME = {v: k for k, v in OP.items()}
BINARY = {"ADD", "SUB", "MUL", "DIV", "MAX", "MIN"}
UNARY = {"NEG", "ABS", "EXP", "EXPC", "GELU", "SQRT", "SQRTA", "ERF", "RECIP", "LOG", "TANH"}
TERNARY = {"SELECT"}
MAX_NODES = 64
MAX_TOKENS = 1024

INV_SQRT2 = np.float32(0.7071067811865476)   # RN_f32(1/sqrt(2))


class ProgramError(ValueError):
    """A program that is not a group: refused, never run."""


def decode(tokens, n_inputs: int, n_imm: int, input_dtypes=None):
    """Validate a token program and return [(name, arg)].  Refuses: an empty
    program or no op node; more than 64 op nodes; an unknown opcode; an operand
    index out of range; a REF to a node not yet computed; a stack underflow; a
    final stack that is not exactly the root; a SELECT whose condition is not an
    input token.  With ``input_dtypes`` also refuses a condition input that is
    not "i32" and an "i32" input read as anything but a condition."""
    toks = [int(t) for t in np.asarray(tokens, dtype=np.uint32).reshape(-1)]
    if not toks or len(toks) > MAX_TOKENS:
        raise ProgramError("program length out of range")
    prog, depth, nodes = [], 0, 0
    kinds = []   # per stack slot: ("IN", k) for an input token, None otherwise
    for pos, t in enumerate(toks):
        code, arg = t >> 24, t & 0xFFFFFF
        name = NAME.get(code)
        if name is None:
            raise ProgramError(f"token {pos}: unknown opcode {code:#x}")
        if name == "IN":
            if arg >= n_inputs:
                raise ProgramError(f"token {pos}: input {arg} of {n_inputs}")
            depth += 1
            kinds.append(("IN", arg))
        elif name == "IMM":
            if arg >= n_imm:
                raise ProgramError(f"token {pos}: immediate {arg} of {n_imm}")
            depth += 1
            kinds.append(None)
        elif name == "REF":
            if arg >= nodes:
                raise ProgramError(f"token {pos}: REF {arg} before it exists")
            depth += 1
            kinds.append(None)
        else:
            need = 3 if name in TERNARY else (2 if name in BINARY else 1)
            if depth < need:
                raise ProgramError(f"token {pos}: {name} needs {need} operands")
            ops = kinds[len(kinds) - need:]
            del kinds[len(kinds) - need:]
            if name in TERNARY and ops[0] is None:
                raise ProgramError(f"token {pos}: a SELECT condition must be an input token")
            if input_dtypes is not None:
                for j, o in enumerate(ops):
                    is_cond = name in TERNARY and j == 0
                    if o is not None and (input_dtypes[o[1]] == "i32") != is_cond:
                        raise ProgramError(f"token {pos}: input {o[1]} is "
                                           + ("not i32" if is_cond else "i32 and only a SELECT condition reads it"))
            depth -= need - 1
            kinds.append(None)
            nodes += 1
            if nodes > MAX_NODES:
                raise ProgramError("more than 64 op nodes")
        prog.append((name, arg))
    if nodes == 0:
        raise ProgramError("no op node")
    if depth != 1:
        raise ProgramError(f"{depth} values left on the stack")
    return prog


def _max(a, b):
    return np.where(a > b, a, b).astype(np.float32)


def _min(a, b):
    return np.where(a < b, a, b).astype(np.float32)


def gelu(a: np.ndarray) -> np.ndarray:
    with np.errstate(all="ignore"):
        t = a * INV_SQRT2
        e = crmath.erf_f32(t)
        u = np.float32(1.0) + e
        h = np.float32(0.5) * u
        return (a * h).astype(np.float32)


def apply_op(name: str, a: np.ndarray, b: np.ndarray | None = None) -> np.ndarray:
    """One node in f32 (every operation rounded once, no contraction)."""
    with np.errstate(all="ignore"):
        if name == "ADD":
            r = a + b
        elif name == "SUB":
            r = a - b
        elif name == "MUL":
            r = a * b
        elif name == "DIV":
            r = a / b
        elif name == "MAX":
            r = _max(a, b)
        elif name == "MIN":
            r = _min(a, b)
        elif name == "NEG":
            r = -a
        elif name == "ABS":
            r = np.abs(a)
        elif name == "EXP":
            r = crmath.exp_f32(a)
        elif name == "EXPC":
            r = crmath.exp_f32(_min(_max(a, np.float32(-4.0)), np.float32(4.0)))
        elif name == "GELU":
            r = gelu(a)
        elif name == "SQRT":
            r = np.sqrt(a)
        elif name == "SQRTA":
            r = np.sqrt(np.abs(a))
        elif name == "ERF":
            r = crmath.erf_f32(a)
        elif name == "RECIP":
            r = np.float32(1.0) / a
        elif name == "LOG":
            r = crmath.log_f32(a)
        elif name == "TANH":
            r = crmath.tanh_f32(a)
        else:
            raise ProgramError(f"not an op: {name}")
    return np.asarray(r, dtype=np.float32)


def select(c: np.ndarray, a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """SELECT: a where the i32 condition is nonzero, else b; the picked value's
    bits are moved, never computed on."""
    return np.where(np.asarray(c) != 0, a, b).astype(np.float32)


def broadcast_input(arr: np.ndarray, dtype: str, strides, out_shape) -> np.ndarray:
    """The value each output element reads from a stored input: element
    (i0, i1, ...) reads arr.flat[sum_k i_k * strides[k]] (f32 for "f32" and
    "bf16" storage, int32 for an "i32" condition input)."""
    out_shape = tuple(int(s) for s in out_shape)
    if dtype == "i32":
        vals = np.asarray(arr).reshape(-1).astype(np.int32)
    else:
        vals = widen(np.asarray(arr).reshape(-1), dtype)
    if len(out_shape) == 0:
        return vals[:1].reshape(())
    off = np.zeros(out_shape, dtype=np.int64)
    for k, n in enumerate(out_shape):
        shp = [1] * len(out_shape)
        shp[k] = n
        off = off + np.arange(n, dtype=np.int64).reshape(shp) * int(strides[k])
    return vals[off]


def evaluate(tokens, imm, inputs, out_shape, out_dtype: str, return_nodes: bool = False):
    """Run a group program node by node.

    inputs: list of (stored array, dtype "f32"|"bf16"|"i32", strides per
    output axis).  Returns the root in storage form (f32 array, or bf16 bit
    patterns)."""
    imm = np.asarray(imm, dtype=np.float32).reshape(-1)
    prog = decode(tokens, len(inputs), len(imm), [dt for _, dt, _ in inputs])
    out_shape = tuple(int(s) for s in out_shape)
    vals = [broadcast_input(a, dt, st, out_shape) for a, dt, st in inputs]
    stack, nodes = [], []
    for name, arg in prog:
        if name == "IN":
            stack.append(vals[arg])
        elif name == "IMM":
            stack.append(np.full(out_shape, imm[arg], dtype=np.float32))
        elif name == "REF":
            stack.append(nodes[arg])
        elif name in BINARY:
            b = stack.pop()
            a = stack.pop()
            r = apply_op(name, a, b)
            nodes.append(r)
            stack.append(r)
        elif name in TERNARY:
            b = stack.pop()
            a = stack.pop()
            c = stack.pop()
            r = select(c, a, b)
            nodes.append(r)
            stack.append(r)
        else:
            r = apply_op(name, stack.pop())
            nodes.append(r)
            stack.append(r)
    root = np.broadcast_to(stack.pop(), out_shape).astype(np.float32)
    out = store(root, out_dtype)
    return (out, nodes) if return_nodes else out
