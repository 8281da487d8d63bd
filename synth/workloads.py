"""The five synthetic workloads of the fusion-group hot path, by what they are.

* ``small_group``      6-node elementwise group y = gelu(x*1.7 + b)*s + r, f32 [64, 64]
* ``gpt_adamw_leaves`` AdamW parameter tree of a 2-layer GPT (V=92, D=64, H=2, T=32)
* ``softmax_rows``     reduction-rooted softmax region over bf16 logits [32768, 4096]
* ``cap_group``        64-node (the cap) elementwise group over bf16 [8192, 8192]
* ``llama_adamw_leaves`` AdamW parameter tree of a Llama-style 1.1B model

Each workload is described by shapes, dtypes and value distributions; the
arrays are drawn on demand with the generators of this package, seed 1000 + k
for the k-th workload in the order above.  Node programs are written in the
group program format (postfix 32-bit tokens, opcode in the top byte, argument
in the low 24 bits), spelled out here from the format's definition.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import generators as G

# ----------------------------------------------------------- program format
# Operand tokens push a value; op tokens pop their operands and push a node.
OPCODES = {
    "IN": 0x01, "IMM": 0x02, "REF": 0x03,
    "ADD": 0x10, "SUB": 0x11, "MUL": 0x12, "DIV": 0x13, "MAX": 0x14, "MIN": 0x15,
    "NEG": 0x20, "ABS": 0x21, "EXP": 0x22, "EXPC": 0x23, "GELU": 0x24,
    "SQRT": 0x25, "SQRTA": 0x26, "ERF": 0x27, "RECIP": 0x28, "LOG": 0x29, "TANH": 0x2A,
    "SELECT": 0x30,
}
BINARY_OPS = ("ADD", "SUB", "MUL", "DIV", "MAX", "MIN")
UNARY_OPS = ("NEG", "ABS", "EXP", "EXPC", "GELU", "SQRT", "SQRTA", "ERF", "RECIP", "LOG", "TANH")


def tok(name: str, arg: int = 0) -> int:
    return (OPCODES[name] << 24) | (int(arg) & 0xFFFFFF)


def encode(seq) -> np.ndarray:
    """[("IN", 0), ("IMM", 0), ("MUL",), ...] -> uint32 tokens."""
    return np.array([tok(*t) for t in seq], dtype=np.uint32)


SEED_BASE = 1000


@dataclass
class InputSpec:
    name: str
    shape: tuple          # stored shape (contiguous, row-major)
    strides: tuple        # element stride per OUTPUT axis (0 = broadcast)
    dtype: str            # "f32" | "bf16" | "i32"
    dist: tuple           # ("normal", std) | ("uniform", lo, hi) | ("const", value) | ("bernoulli", p)


@dataclass
class GroupWorkload:
    name: str
    seed: int
    tokens: np.ndarray
    imm: np.ndarray
    inputs: list
    out_shape: tuple
    out_dtype: str
    n_ops: int = field(default=0)

    def host_inputs(self):
        """Draw every input on the host: list of (array, dtype) with f32 arrays or
        uint16 bf16 bit patterns, each contiguous in its stored shape."""
        out = []
        for i, spec in enumerate(self.inputs):
            out.append((_host_draw(spec, self.seed, i), spec.dtype))
        return out

    def device_inputs(self, device="cuda"):
        import torch

        out = []
        for i, spec in enumerate(self.inputs):
            dt = torch.bfloat16 if spec.dtype == "bf16" else torch.float32
            kind = spec.dist[0]
            if kind == "bernoulli":
                u = G.device_uniform(spec.shape, 0.0, 1.0, self.seed, i, device, torch.float32)
                out.append((u < spec.dist[1]).to(torch.int32))
                continue
            if kind == "normal":
                t = G.device_normal(spec.shape, spec.dist[1], self.seed, i, device, dt)
            elif kind == "uniform":
                t = G.device_uniform(spec.shape, spec.dist[1], spec.dist[2], self.seed, i, device, dt)
            else:
                t = torch.full(spec.shape, float(spec.dist[1]), dtype=dt, device=device)
            out.append(t)
        return out

    def algorithmic_bytes(self) -> int:
        """Bytes a fused launch must move: every stored input once, the output once."""
        b = 0
        for spec in self.inputs:
            b += int(np.prod(spec.shape, dtype=np.int64)) * (2 if spec.dtype == "bf16" else 4)   # i32: 4
        b += int(np.prod(self.out_shape, dtype=np.int64)) * (2 if self.out_dtype == "bf16" else 4)
        return b


def _host_draw(spec: InputSpec, seed: int, tensor_id: int) -> np.ndarray:
    kind = spec.dist[0]
    if kind == "bernoulli":
        return (G.host_uniform(spec.shape, 0.0, 1.0, seed, tensor_id) < spec.dist[1]).astype(np.int32)
    if kind == "normal":
        v = G.host_normal(spec.shape, spec.dist[1], seed, tensor_id)
    elif kind == "uniform":
        v = G.host_uniform(spec.shape, spec.dist[1], spec.dist[2], seed, tensor_id)
    else:
        v = np.full(spec.shape, spec.dist[1], dtype=np.float32)
    return G.host_bf16_bits(v) if spec.dtype == "bf16" else v


# --------------------------------------------------------------- workloads

def small_group(rows: int = 64, cols: int = 64) -> GroupWorkload:
    """y = gelu(x*1.7 + b)*s + r: x, r ~N(0,1) [rows, cols], b ~N(0,0.1) [cols]
    broadcast along rows, s = 0.5 a scalar input; f32 in and out."""
    prog = [("IN", 0), ("IMM", 0), ("MUL",), ("IN", 1), ("ADD",), ("GELU",),
            ("IN", 2), ("MUL",), ("IN", 3), ("ADD",)]
    inputs = [
        InputSpec("x", (rows, cols), (cols, 1), "f32", ("normal", 1.0)),
        InputSpec("b", (cols,), (0, 1), "f32", ("normal", 0.1)),
        InputSpec("s", (), (0, 0), "f32", ("const", 0.5)),
        InputSpec("r", (rows, cols), (cols, 1), "f32", ("normal", 1.0)),
    ]
    return GroupWorkload("small_group", SEED_BASE + 0, encode(prog),
                         np.array([1.7], dtype=np.float32), inputs, (rows, cols), "f32", 5)


def select_group(rows: int = 8192, cols: int = 8192, seed: int = SEED_BASE + 7) -> GroupWorkload:
    """The extended op set on one group: y = select(mask, log(sigmoid(x)),
    tanh(x)) with sigmoid as 1 / (1 + exp(-x)); x bf16 [rows, cols] ~N(0, 3),
    mask an int32 row vector [cols] (70 % ones) broadcast down the rows; bf16
    out.  Seven nodes: NEG EXP ADD RECIP LOG TANH SELECT."""
    prog = [("IN", 1), ("IN", 0), ("NEG",), ("EXP",), ("IMM", 0), ("ADD",), ("RECIP",), ("LOG",),
            ("IN", 0), ("TANH",), ("SELECT",)]
    inputs = [
        InputSpec("x", (rows, cols), (cols, 1), "bf16", ("normal", 3.0)),
        InputSpec("mask", (cols,), (0, 1), "i32", ("bernoulli", 0.7)),
    ]
    return GroupWorkload("select_group", seed, encode(prog), np.array([1.0], dtype=np.float32), inputs,
                         (rows, cols), "bf16", 7)


CAP_OPS = ("ADD", "MUL", "SUB", "MAX", "EXPC", "GELU", "SQRTA")


def cap_program(seed: int, n_ops: int = 64) -> np.ndarray:
    """A connected chain of n_ops nodes drawn by seed: node i's first operand is
    node i-1 (node 0 reads x); a binary node's second operand is drawn uniformly
    from the four inputs (x, row, col, scalar) and the nodes before it."""
    raw = G._stream(seed, 99).random_raw(2 * n_ops)
    seq = [("IN", 0)]
    for i in range(n_ops):
        op = CAP_OPS[int(raw[2 * i] % np.uint64(len(CAP_OPS)))]
        if op in BINARY_OPS:
            c = int(raw[2 * i + 1] % np.uint64(4 + i))
            seq.append(("IN", c) if c < 4 else ("REF", c - 4))
        seq.append((op,))
    return encode(seq)


def cap_group(rows: int = 8192, cols: int = 8192, n_ops: int = 64, seed: int = SEED_BASE + 3) -> GroupWorkload:
    """64-node group over bf16 x [rows, cols] ~U(-2,2) with a row vector [cols], a
    column vector [rows, 1] and a scalar broadcast in, all bf16 ~U(-2,2); bf16 out."""
    inputs = [
        InputSpec("x", (rows, cols), (cols, 1), "bf16", ("uniform", -2.0, 2.0)),
        InputSpec("row", (cols,), (0, 1), "bf16", ("uniform", -2.0, 2.0)),
        InputSpec("col", (rows, 1), (1, 0), "bf16", ("uniform", -2.0, 2.0)),
        InputSpec("scalar", (), (0, 0), "bf16", ("uniform", -2.0, 2.0)),
    ]
    return GroupWorkload("cap_group", seed, cap_program(seed, n_ops),
                         np.zeros(0, dtype=np.float32), inputs, (rows, cols), "bf16", n_ops)


@dataclass
class SoftmaxWorkload:
    name: str
    seed: int
    rows: int
    cols: int
    x_dtype: str
    y_dtype: str
    std: float

    def host_x(self) -> np.ndarray:
        v = G.host_normal((self.rows, self.cols), self.std, self.seed, 0)
        return G.host_bf16_bits(v) if self.x_dtype == "bf16" else v

    def device_x(self, device="cuda"):
        import torch

        dt = torch.bfloat16 if self.x_dtype == "bf16" else torch.float32
        return G.device_normal((self.rows, self.cols), self.std, self.seed, 0, device, dt)

    def algorithmic_bytes(self) -> int:
        n = self.rows * self.cols
        return n * (2 if self.x_dtype == "bf16" else 4) + n * (2 if self.y_dtype == "bf16" else 4)


def softmax_rows(rows: int = 32768, cols: int = 4096) -> SoftmaxWorkload:
    """Rows of bf16 logits ~N(0, 3^2), f32 arithmetic, bf16 output."""
    return SoftmaxWorkload("softmax_rows", SEED_BASE + 2, rows, cols, "bf16", "bf16", 3.0)


@dataclass
class NormWorkload:
    """Rows of activations x ~N(mean, std^2) for a normalization region, a scale
    gamma ~1 + N(0, 0.1^2) and (LayerNorm) a bias beta ~N(0, 0.1^2), stored in
    x_dtype / param_dtype."""
    name: str
    seed: int
    rows: int
    cols: int
    kind: str            # "rms" or "layer"
    eps: float
    x_dtype: str = "bf16"
    y_dtype: str = "bf16"
    param_dtype: str = "bf16"
    std: float = 1.0
    mean: float = 0.25

    def _store(self, v, dtype):
        return G.host_bf16_bits(v) if dtype == "bf16" else v

    def host_x(self) -> np.ndarray:
        v = (G.host_normal((self.rows, self.cols), self.std, self.seed, 0) + np.float32(self.mean)).astype(np.float32)
        return self._store(v, self.x_dtype)

    def host_gamma(self) -> np.ndarray:
        v = (G.host_normal((self.cols,), 0.1, self.seed, 1) + np.float32(1.0)).astype(np.float32)
        return self._store(v, self.param_dtype)

    def host_beta(self):
        if self.kind != "layer":
            return None
        return self._store(G.host_normal((self.cols,), 0.1, self.seed, 2), self.param_dtype)

    def device_x(self, device="cuda"):
        import torch

        dt = torch.bfloat16 if self.x_dtype == "bf16" else torch.float32
        v = G.device_normal((self.rows, self.cols), self.std, self.seed, 0, device, torch.float32) + self.mean
        return v.to(dt)

    def device_params(self, device="cuda"):
        """(gamma, beta or None) on the device, drawn on the host (they are small)."""
        import torch

        def dev(a):
            if a is None:
                return None
            if self.param_dtype == "bf16":
                return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
            return torch.from_numpy(a).to(device)

        return dev(self.host_gamma()), dev(self.host_beta())

    def algorithmic_bytes(self) -> int:
        n = self.rows * self.cols
        return n * (2 if self.x_dtype == "bf16" else 4) + n * (2 if self.y_dtype == "bf16" else 4)


def norm_rows(kind: str, rows: int = 32768, cols: int = 4096) -> NormWorkload:
    """RMSNorm (eps 1e-6) or LayerNorm (eps 1e-5) over bf16 rows, bf16 scale and
    bias, f32 arithmetic, bf16 output: the softmax region's shape."""
    if kind == "rms":
        return NormWorkload("rms_rows", SEED_BASE + 5, rows, cols, "rms", 1e-6)
    return NormWorkload("layer_rows", SEED_BASE + 6, rows, cols, "layer", 1e-5)


# ----------------------------------------------------------- parameter trees

@dataclass
class AdamWHyper:
    lr: float = 3e-4
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01
    t: int = 10


@dataclass
class LeafTree:
    name: str
    seed: int
    leaves: list          # [(path, shape)]
    grad_dtype: str
    hp: AdamWHyper
    grad_std: float = 1e-2

    @property
    def numels(self):
        return [int(np.prod(s, dtype=np.int64)) for _, s in self.leaves]

    @property
    def n_params(self) -> int:
        return int(sum(self.numels))

    def bytes_per_param(self) -> int:
        # theta, m, v read and written (f32), grad read once.
        return 3 * 8 + (2 if self.grad_dtype == "bf16" else 4)

    def host_leaf(self, i: int):
        """(theta, m, v, grad) of leaf i drawn on the host; grad as f32 or bf16 bits."""
        shape = self.leaves[i][1]
        th = G.host_normal(shape, 0.02, self.seed, 4 * i)
        g = G.host_normal(shape, self.grad_std, self.seed, 4 * i + 1)
        m = G.host_normal(shape, 1e-3, self.seed, 4 * i + 2)
        v = np.abs(G.host_normal(shape, 1e-4, self.seed, 4 * i + 3))
        if self.grad_dtype == "bf16":
            g = G.host_bf16_bits(g)
        return th.reshape(-1), m.reshape(-1), v.reshape(-1), g.reshape(-1)

    def device_leaf(self, i: int, device="cuda"):
        import torch

        n = self.numels[i]
        th = G.device_normal((n,), 0.02, self.seed, 4 * i, device)
        gdt = torch.bfloat16 if self.grad_dtype == "bf16" else torch.float32
        g = G.device_normal((n,), self.grad_std, self.seed, 4 * i + 1, device, gdt)
        m = G.device_normal((n,), 1e-3, self.seed, 4 * i + 2, device)
        v = G.device_abs_normal((n,), 1e-4, self.seed, 4 * i + 3, device)
        return th, m, v, g


def gpt_adamw_leaves() -> LeafTree:
    """Leaves of a 2-layer GPT, V=92, D=64, H=2, T=32, f32 grads ~N(0, 1e-2^2), t=10."""
    V, D, T, L = 92, 64, 32, 2
    leaves = [("tok_emb", (V, D)), ("pos_emb", (T, D))]
    for l in range(L):
        p = f"blocks.{l}."
        leaves += [
            (p + "ln1.w", (D,)), (p + "ln1.b", (D,)),
            (p + "qkv.w", (D, 3 * D)), (p + "qkv.b", (3 * D,)),
            (p + "proj.w", (D, D)), (p + "proj.b", (D,)),
            (p + "ln2.w", (D,)), (p + "ln2.b", (D,)),
            (p + "fc1.w", (D, 4 * D)), (p + "fc1.b", (4 * D,)),
            (p + "fc2.w", (4 * D, D)), (p + "fc2.b", (D,)),
        ]
    leaves += [("lnf.w", (D,)), ("lnf.b", (D,))]
    return LeafTree("gpt_adamw_leaves", SEED_BASE + 1, leaves, "f32", AdamWHyper(t=10), 1e-2)


def llama_adamw_leaves(layers: int = 22, D: int = 2048, F: int = 5632, KV: int = 256, V: int = 32000) -> LeafTree:
    """Leaves of a Llama-style 1.1B model: embed and lm_head [V, D]; per layer
    q, o [D, D], k, v [D, KV], gate, up [D, F], down [F, D], two RMSNorm w [D].
    f32 params/m/v, bf16 grads ~N(0, 1e-3^2), t=1000."""
    leaves = [("embed", (V, D))]
    for l in range(layers):
        p = f"layers.{l}."
        leaves += [
            (p + "attn_norm.w", (D,)),
            (p + "q", (D, D)), (p + "k", (D, KV)), (p + "v", (D, KV)), (p + "o", (D, D)),
            (p + "mlp_norm.w", (D,)),
            (p + "gate", (D, F)), (p + "up", (D, F)), (p + "down", (F, D)),
        ]
    leaves += [("lm_head", (V, D))]
    return LeafTree("llama_adamw_leaves", SEED_BASE + 4, leaves, "bf16", AdamWHyper(t=1000), 1e-3)
