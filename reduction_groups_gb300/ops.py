"""Python binding of the C ABI with the same names: psk_group_run,
psk_softmax_region, psk_norm_region, psk_adamw_tree (plus the host-only psk_group_check and
psk_adamw_scalars).  Each function marshals torch tensors (device memory and
the current stream) or plain host arrays into the C structs and calls the
library; every step of the hot path runs in the library's kernels.
"""

from __future__ import annotations

import ctypes

import numpy as np

from . import _native as N


def _dtype_code(t) -> int:
    """The psk_dtype of a tensor; which entry point takes which type is the
    library's to check (int32 is a group's SELECT condition type only)."""
    import torch

    if t.dtype == torch.float32:
        return N.PSK_F32
    if t.dtype == torch.bfloat16:
        return N.PSK_BF16
    if t.dtype == torch.int32:
        return N.PSK_I32
    raise TypeError(f"storage type {t.dtype} is not f32, bf16 or int32")


def _stream_handle(stream) -> int:
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _program(tokens, imm):
    toks = np.ascontiguousarray(np.asarray(tokens, dtype=np.uint32).reshape(-1))
    ims = np.ascontiguousarray(np.asarray(imm if imm is not None else [], dtype=np.float32).reshape(-1))
    p = N.psk_program()
    p.tokens = toks.ctypes.data_as(ctypes.POINTER(ctypes.c_uint32))
    p.n_tokens = int(toks.size)
    p.imm = ims.ctypes.data_as(ctypes.POINTER(ctypes.c_float)) if ims.size else None
    p.n_imm = int(ims.size)
    return p, (toks, ims)


def psk_group_check(tokens, n_inputs: int, imm=None):
    """Validate a program on the host; returns (n_nodes, n_values)."""
    p, keep = _program(tokens, imm)
    nn, ns = ctypes.c_int32(0), ctypes.c_int32(0)
    N.check(N.lib().psk_group_check(ctypes.byref(p), int(n_inputs), ctypes.byref(nn), ctypes.byref(ns)))
    return nn.value, ns.value


def _group_args(inputs, out):
    n = len(inputs)
    arr = (N.psk_input * max(n, 1))()
    for i, (t, strides) in enumerate(inputs):
        arr[i].ptr = t.data_ptr()
        arr[i].dtype = _dtype_code(t)
        st = list(strides) + [0] * (N.PSK_MAX_RANK - len(strides))
        for k in range(N.PSK_MAX_RANK):
            arr[i].stride[k] = int(st[k])
    if not out.is_contiguous():
        raise ValueError("the output must be contiguous (row-major)")
    o = N.psk_output()
    o.ptr = out.data_ptr()
    o.dtype = _dtype_code(out)
    o.rank = out.dim()
    for k, s in enumerate(out.shape):
        o.shape[k] = int(s)
    return arr, n, o


_MATH = {"exact": 0, "fast": 1}


def psk_group_prepare(tokens, imm, inputs, out, math: str = "exact") -> None:
    """Validate and compile (cached) the kernel psk_group_run would launch for
    these arguments; needs no device (tensors are inspected, not read)."""
    p, keep = _program(tokens, imm)
    arr, n, o = _group_args(inputs, out)
    N.check(N.lib().psk_group_prepare_ex(ctypes.byref(p), arr, n, ctypes.byref(o), _MATH[math]))


def psk_group_run(tokens, imm, inputs, out, stream=None, math: str = "exact") -> None:
    """inputs: list of (tensor, strides) with one element stride per output axis
    (0 = broadcast), f32 or bf16 values or int32 SELECT conditions; out: a
    contiguous row-major tensor (f32 or bf16).  math "exact" (every node
    correctly rounded) or "fast" (EXP within one f32 ulp, EXPC and ERF within
    two; GELU, LOG and TANH stay correctly rounded)."""
    p, keep = _program(tokens, imm)
    arr, n, o = _group_args(inputs, out)
    N.check(N.lib().psk_group_run_ex(ctypes.byref(p), arr, n, ctypes.byref(o), _MATH[math], _stream_handle(stream)))


def psk_group_run_interp(tokens, imm, inputs, out, stream=None, math: str = "exact") -> None:
    """psk_group_run through the library's precompiled interpreter kernel (no
    run-time compilation): the same arguments and the same result bits,
    slower."""
    p, keep = _program(tokens, imm)
    arr, n, o = _group_args(inputs, out)
    N.check(N.lib().psk_group_run_interp(ctypes.byref(p), arr, n, ctypes.byref(o), _MATH[math],
                                         _stream_handle(stream)))


_ORDER = {"sequential": N.PSK_ORDER_SEQUENTIAL, "blocked": N.PSK_ORDER_BLOCKED,
          "interleaved": N.PSK_ORDER_INTERLEAVED}


def psk_softmax_region(x, y, order=("sequential",), exp_mode: str = "exact", stream=None) -> None:
    """Row softmax of the 2-D tensor x into y (same shape; row strides may
    exceed the row length).  order: ("sequential",), ("blocked", w) or
    ("interleaved", P); exp_mode: "exact" (correctly rounded) or "fast"."""
    if x.dim() != 2 or y.dim() != 2 or tuple(x.shape) != tuple(y.shape):
        raise ValueError("x and y must be 2-D tensors of one shape")
    if x.stride(1) != 1 or y.stride(1) != 1:
        raise ValueError("rows must be contiguous")
    o = N.psk_order(_ORDER[order[0]], int(order[1]) if len(order) > 1 else 0)
    em = {"exact": N.PSK_EXP_EXACT, "fast": N.PSK_EXP_FAST}[exp_mode]
    rows, cols = x.shape
    N.check(N.lib().psk_softmax_region(x.data_ptr(), _dtype_code(x), y.data_ptr(), _dtype_code(y), rows, cols,
                                       max(x.stride(0), cols), max(y.stride(0), cols), o, em, _stream_handle(stream)))


def _rows2d(*ts):
    for t in ts:
        if t.dim() != 2 or t.stride(1) != 1:
            raise ValueError("row regions take 2-D tensors with contiguous rows")
    if len({tuple(t.shape) for t in ts}) != 1:
        raise ValueError("the row tensors must share one shape")


def psk_softmax_masked(x, y, mask, order=("sequential",), exp_mode: str = "exact", stream=None) -> None:
    """Masked softmax of the rows of x into y; mask: a uint8/bool device tensor
    of shape [cols] (every row) or [rows, cols] (contiguous rows), nonzero
    allows."""
    import torch

    _rows2d(x, y)
    rows, cols = x.shape
    if mask.dtype not in (torch.uint8, torch.bool):
        raise TypeError("the mask must be uint8 or bool")
    if mask.dim() == 1:
        if mask.numel() != cols or (cols > 1 and mask.stride(0) != 1):
            raise ValueError("a mask row must hold cols contiguous values")
        ldm = 0
    else:
        if tuple(mask.shape) != (rows, cols) or mask.stride(1) != 1:
            raise ValueError("a full mask must be [rows, cols] with contiguous rows")
        ldm = max(mask.stride(0), cols)
    o = N.psk_order(_ORDER[order[0]], int(order[1]) if len(order) > 1 else 0)
    em = {"exact": N.PSK_EXP_EXACT, "fast": N.PSK_EXP_FAST}[exp_mode]
    N.check(N.lib().psk_softmax_masked(x.data_ptr(), _dtype_code(x), y.data_ptr(), _dtype_code(y), rows, cols,
                                       max(x.stride(0), cols), max(y.stride(0), cols), mask.data_ptr(), ldm, o, em,
                                       _stream_handle(stream)))


def psk_softmax_backward(y, ct, dx, order=("sequential",), stream=None) -> None:
    """dx = y (ct - sum(ct y)) per row (the softmax region's backward)."""
    _rows2d(y, ct, dx)
    rows, cols = y.shape
    o = N.psk_order(_ORDER[order[0]], int(order[1]) if len(order) > 1 else 0)
    N.check(N.lib().psk_softmax_backward(y.data_ptr(), _dtype_code(y), ct.data_ptr(), _dtype_code(ct),
                                         dx.data_ptr(), _dtype_code(dx), rows, cols, max(y.stride(0), cols),
                                         max(ct.stride(0), cols), max(dx.stride(0), cols), o,
                                         _stream_handle(stream)))


def psk_norm_region(x, y, kind: str, eps: float, gamma=None, beta=None, order=("sequential",),
                    stream=None) -> None:
    """RMSNorm (kind "rms") or LayerNorm ("layer") of the rows of the 2-D
    tensor x into y; gamma / beta: optional 1-D tensors of x's row length, both
    of one storage type."""
    if x.dim() != 2 or y.dim() != 2 or tuple(x.shape) != tuple(y.shape):
        raise ValueError("x and y must be 2-D tensors of one shape")
    if x.stride(1) != 1 or y.stride(1) != 1:
        raise ValueError("rows must be contiguous")
    params = [t for t in (gamma, beta) if t is not None]
    for t in params:
        if t.dim() != 1 or t.numel() != x.shape[1] or (t.numel() > 1 and t.stride(0) != 1):
            raise ValueError("gamma and beta must be contiguous vectors of the row length")
    if len(params) == 2 and gamma.dtype != beta.dtype:
        raise TypeError("gamma and beta must share one storage type")
    pdt = _dtype_code(params[0]) if params else N.PSK_F32
    o = N.psk_order(_ORDER[order[0]], int(order[1]) if len(order) > 1 else 0)
    k = {"rms": N.PSK_NORM_RMS, "layer": N.PSK_NORM_LAYER}[kind]
    rows, cols = x.shape
    N.check(N.lib().psk_norm_region(x.data_ptr(), _dtype_code(x), y.data_ptr(), _dtype_code(y), rows, cols,
                                    max(x.stride(0), cols), max(y.stride(0), cols), k, float(eps),
                                    gamma.data_ptr() if gamma is not None else None,
                                    beta.data_ptr() if beta is not None else None, pdt, o, _stream_handle(stream)))


def psk_device_status(reset: bool = False) -> int:
    """The pipelined kernels' status word (0: no bounded wait ever timed out)."""
    v = ctypes.c_uint32(0)
    N.check(N.lib().psk_device_status(ctypes.byref(v), 1 if reset else 0))
    return v.value


def psk_test_drop_row(row: int) -> None:
    """Test hook: the pipelined row-region kernels stop producing at local row
    `row` of every CTA (their bounded waits then run out); -1 turns it off."""
    N.check(N.lib().psk_test_drop_row(int(row)))


def psk_test_fast_exp(x, y, stream=None) -> None:
    """Test hook: y = the softmax region's fast exp of x elementwise (f32
    device tensors of equal size, x <= 0)."""
    import torch

    if x.dtype != torch.float32 or y.dtype != torch.float32 or x.numel() != y.numel():
        raise TypeError("x and y must be f32 tensors of equal size")
    if not (x.is_contiguous() and y.is_contiguous()):
        raise ValueError("x and y must be contiguous")
    N.check(N.lib().psk_test_fast_exp(x.data_ptr(), y.data_ptr(), x.numel(), _stream_handle(stream)))


def _hparams(hp) -> N.psk_adamw_hparams:
    h = N.psk_adamw_hparams()
    h.lr, h.beta1, h.beta2 = float(hp.lr), float(hp.beta1), float(hp.beta2)
    h.eps, h.weight_decay, h.t = float(hp.eps), float(hp.weight_decay), int(hp.t)
    return h


def psk_adamw_scalars(hp):
    """The nine f32 scalars the step reads (b1, b2, 1-b1, 1-b2, 1-b1^t, 1-b2^t, lr, eps, wd)."""
    h = _hparams(hp)
    out = (ctypes.c_float * 9)()
    N.check(N.lib().psk_adamw_scalars(ctypes.byref(h), out))
    return np.array(list(out), dtype=np.float32)


def _leaf_table(leaves):
    n = len(leaves)
    arr = (N.psk_leaf * max(n, 1))()
    for i, (th, m, v, g) in enumerate(leaves):
        arr[i].theta, arr[i].m, arr[i].v, arr[i].grad = th.data_ptr(), m.data_ptr(), v.data_ptr(), g.data_ptr()
        arr[i].grad_dtype = _dtype_code(g)
        arr[i].param_dtype = _dtype_code(th)
        if _dtype_code(m) != arr[i].param_dtype or _dtype_code(v) != arr[i].param_dtype:
            raise TypeError("theta, m and v of a leaf must share one storage type")
        arr[i].numel = int(th.numel())
    return arr, n


_LR = {"constant": N.PSK_LR_CONSTANT, "linear": N.PSK_LR_LINEAR, "cosine": N.PSK_LR_COSINE}


def _schedule(kind="constant", warmup=0, total=1, grad_clip=0.0) -> N.psk_adamw_schedule:
    return N.psk_adamw_schedule(_LR[kind], int(warmup), int(total), float(grad_clip))


def psk_adamw_tree(leaves, hp, stream=None) -> None:
    """leaves: list of (theta, m, v, grad) tensors, updated in place."""
    arr, n = _leaf_table(leaves)
    h = _hparams(hp)
    N.check(N.lib().psk_adamw_tree(arr, n, ctypes.byref(h), _stream_handle(stream)))


def psk_adamw_lr(hp, kind="constant", warmup=0, total=1) -> np.float32:
    """The scheduled f32 lr of step hp.t (host only)."""
    h, sc, out = _hparams(hp), _schedule(kind, warmup, total), ctypes.c_float(0)
    N.check(N.lib().psk_adamw_lr(ctypes.byref(h), ctypes.byref(sc), ctypes.byref(out)))
    return np.float32(out.value)


def psk_adamw_workspace(leaves, kind="constant", warmup=0, total=1, grad_clip=0.0) -> int:
    """Device workspace bytes psk_adamw_tree_ex needs (0 without clipping)."""
    arr, n = _leaf_table(leaves)
    sc, out = _schedule(kind, warmup, total, grad_clip), ctypes.c_uint64(0)
    N.check(N.lib().psk_adamw_workspace(arr, n, ctypes.byref(sc), ctypes.byref(out)))
    return int(out.value)


def psk_adamw_tree_ex(leaves, hp, kind="constant", warmup=0, total=1, grad_clip=0.0, workspace=None,
                      stream=None) -> None:
    """psk_adamw_tree with a schedule and global-norm clipping; workspace: a
    device tensor of at least psk_adamw_workspace bytes (needed when clipping)."""
    arr, n = _leaf_table(leaves)
    h, sc = _hparams(hp), _schedule(kind, warmup, total, grad_clip)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    N.check(N.lib().psk_adamw_tree_ex(arr, n, ctypes.byref(h), ctypes.byref(sc), ws_ptr, ws_bytes,
                                      _stream_handle(stream)))


def psk_adamw_group_sqsums(leaves, group_sums, workspace, stream=None) -> None:
    """The squared-norm tree's group sums of `leaves` (pieces of a tree's
    leaves, each starting on a 65,536-element boundary of its leaf), leaf
    after leaf, into the f32 device tensor group_sums; workspace as for
    psk_adamw_tree_ex with clipping."""
    arr, n = _leaf_table(leaves)
    N.check(N.lib().psk_adamw_group_sqsums(arr, n, group_sums.data_ptr(), workspace.data_ptr(),
                                           workspace.numel() * workspace.element_size(), _stream_handle(stream)))


def psk_adamw_clip_scale(group_sums, groups_per_leaf, grad_clip, scale, stream=None) -> None:
    """The clip scale from a whole tree's group sums (f32 device tensor, leaf
    order) and its leaves' group counts (ints), into the one-element f32
    device tensor scale."""
    counts = (ctypes.c_int64 * max(1, len(groups_per_leaf)))(*[int(c) for c in groups_per_leaf])
    N.check(N.lib().psk_adamw_clip_scale(group_sums.data_ptr() if group_sums.numel() else None, counts,
                                         len(groups_per_leaf), float(grad_clip), scale.data_ptr(),
                                         _stream_handle(stream)))


def psk_adamw_tree_scaled(leaves, hp, scale, kind="constant", warmup=0, total=1, stream=None) -> None:
    """psk_adamw_tree_ex with every gradient scaled by the device scalar
    `scale` (a sharded step's clip scale) and the schedule's lr."""
    arr, n = _leaf_table(leaves)
    h, sc = _hparams(hp), _schedule(kind, warmup, total, 0.0)
    N.check(N.lib().psk_adamw_tree_scaled(arr, n, ctypes.byref(h), ctypes.byref(sc), scale.data_ptr(),
                                          _stream_handle(stream)))


def psk_adamw_tree_static(leaves, hp, kind="constant", warmup=0, total=1, grad_clip=0.0, stream=None) -> None:
    """psk_adamw_tree_ex whose clipping scratch is the library's fixed device
    buffer (no workspace argument; overlapping calls on one device race)."""
    arr, n = _leaf_table(leaves)
    h, sc = _hparams(hp), _schedule(kind, warmup, total, grad_clip)
    N.check(N.lib().psk_adamw_tree_static(arr, n, ctypes.byref(h), ctypes.byref(sc), _stream_handle(stream)))
