"""ctypes view of the C ABI in include/psk.h (argument marshalling only).

Loads ``_build/libpsk.so`` from this package's directory.  There is no
fallback: if the library is missing, importing the binding raises.
"""

from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libpsk.so")

PSK_F32, PSK_BF16, PSK_I32 = 0, 1, 2
PSK_ORDER_SEQUENTIAL, PSK_ORDER_BLOCKED, PSK_ORDER_INTERLEAVED = 0, 1, 2
PSK_EXP_EXACT, PSK_EXP_FAST = 0, 1
PSK_NORM_RMS, PSK_NORM_LAYER = 0, 1
PSK_LR_CONSTANT, PSK_LR_LINEAR, PSK_LR_COSINE = 0, 1, 2
PSK_MAX_RANK = 4
PSK_ADAMW_MAX_LEAVES = 512

ERRORS = {
    -1: "PSK_E_PROGRAM", -2: "PSK_E_TOO_MANY_NODES", -3: "PSK_E_SHAPE", -4: "PSK_E_DTYPE",
    -5: "PSK_E_NULL", -6: "PSK_E_ORDER", -7: "PSK_E_CUDA", -8: "PSK_E_ALIAS", -9: "PSK_E_ARG",
}

EXPORTS = ("psk_group_run", "psk_group_run_ex", "psk_group_run_interp", "psk_group_check", "psk_group_prepare", "psk_group_prepare_ex", "psk_softmax_region", "psk_softmax_masked",
           "psk_softmax_backward", "psk_norm_region",
           "psk_adamw_tree", "psk_adamw_tree_ex", "psk_adamw_tree_static", "psk_adamw_lr", "psk_adamw_workspace",
           "psk_adamw_scalars", "psk_adamw_group_sqsums", "psk_adamw_clip_scale", "psk_adamw_tree_scaled",
           "psk_device_status", "psk_test_drop_row", "psk_test_fast_exp", "psk_last_error")


class psk_program(ctypes.Structure):
    _fields_ = [("tokens", ctypes.POINTER(ctypes.c_uint32)), ("n_tokens", ctypes.c_int32),
                ("imm", ctypes.POINTER(ctypes.c_float)), ("n_imm", ctypes.c_int32)]


class psk_input(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("stride", ctypes.c_int64 * PSK_MAX_RANK)]


class psk_output(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("rank", ctypes.c_int32),
                ("shape", ctypes.c_int64 * PSK_MAX_RANK)]


class psk_order(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("param", ctypes.c_int32)]


class psk_leaf(ctypes.Structure):
    _fields_ = [("theta", ctypes.c_void_p), ("m", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("grad", ctypes.c_void_p), ("grad_dtype", ctypes.c_int32), ("param_dtype", ctypes.c_int32),
                ("numel", ctypes.c_int64)]


class psk_adamw_hparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double), ("beta2", ctypes.c_double),
                ("eps", ctypes.c_double), ("weight_decay", ctypes.c_double), ("t", ctypes.c_int64)]


class psk_adamw_schedule(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("warmup", ctypes.c_int64), ("total", ctypes.c_int64),
                ("grad_clip", ctypes.c_double)]


class PskError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code
        self.name = ERRORS.get(code, str(code))


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.POINTER
        L.psk_group_run.argtypes = [P(psk_program), P(psk_input), ctypes.c_int32, P(psk_output), ctypes.c_void_p]
        L.psk_group_check.argtypes = [P(psk_program), ctypes.c_int32, P(ctypes.c_int32), P(ctypes.c_int32)]
        L.psk_group_prepare.argtypes = [P(psk_program), P(psk_input), ctypes.c_int32, P(psk_output)]
        L.psk_group_run_ex.argtypes = [P(psk_program), P(psk_input), ctypes.c_int32, P(psk_output), ctypes.c_int32,
                                       ctypes.c_void_p]
        L.psk_group_prepare_ex.argtypes = [P(psk_program), P(psk_input), ctypes.c_int32, P(psk_output), ctypes.c_int32]
        L.psk_group_run_interp.argtypes = [P(psk_program), P(psk_input), ctypes.c_int32, P(psk_output),
                                           ctypes.c_int32, ctypes.c_void_p]
        L.psk_softmax_region.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32,
                                         ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                         psk_order, ctypes.c_int32, ctypes.c_void_p]
        L.psk_softmax_masked.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32,
                                         ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.c_void_p, ctypes.c_int64, psk_order, ctypes.c_int32, ctypes.c_void_p]
        L.psk_softmax_backward.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32,
                                           ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64,
                                           ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, psk_order, ctypes.c_void_p]
        L.psk_norm_region.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32,
                                      ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                      ctypes.c_int32, ctypes.c_double, ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_int32, psk_order, ctypes.c_void_p]
        L.psk_adamw_tree.argtypes = [P(psk_leaf), ctypes.c_int32, P(psk_adamw_hparams), ctypes.c_void_p]
        L.psk_adamw_scalars.argtypes = [P(psk_adamw_hparams), P(ctypes.c_float)]
        L.psk_adamw_lr.argtypes = [P(psk_adamw_hparams), P(psk_adamw_schedule), P(ctypes.c_float)]
        L.psk_adamw_workspace.argtypes = [P(psk_leaf), ctypes.c_int32, P(psk_adamw_schedule), P(ctypes.c_uint64)]
        L.psk_adamw_tree_ex.argtypes = [P(psk_leaf), ctypes.c_int32, P(psk_adamw_hparams), P(psk_adamw_schedule),
                                        ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p]
        L.psk_adamw_tree_static.argtypes = [P(psk_leaf), ctypes.c_int32, P(psk_adamw_hparams),
                                            P(psk_adamw_schedule), ctypes.c_void_p]
        L.psk_device_status.argtypes = [P(ctypes.c_uint32), ctypes.c_int32]
        L.psk_test_drop_row.argtypes = [ctypes.c_int64]
        L.psk_test_fast_exp.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
        L.psk_adamw_group_sqsums.argtypes = [P(psk_leaf), ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_uint64, ctypes.c_void_p]
        L.psk_adamw_clip_scale.argtypes = [ctypes.c_void_p, P(ctypes.c_int64), ctypes.c_int32, ctypes.c_double,
                                           ctypes.c_void_p, ctypes.c_void_p]
        L.psk_adamw_tree_scaled.argtypes = [P(psk_leaf), ctypes.c_int32, P(psk_adamw_hparams),
                                            P(psk_adamw_schedule), ctypes.c_void_p, ctypes.c_void_p]
        L.psk_last_error.restype = ctypes.c_char_p
        for f in ("psk_group_run", "psk_group_run_ex", "psk_group_run_interp", "psk_group_check", "psk_group_prepare", "psk_group_prepare_ex",
                  "psk_softmax_region", "psk_norm_region",
                  "psk_softmax_masked", "psk_softmax_backward",
                  "psk_adamw_tree",
                  "psk_adamw_scalars", "psk_adamw_lr", "psk_adamw_workspace", "psk_adamw_tree_ex",
                  "psk_adamw_tree_static",
                  "psk_adamw_group_sqsums", "psk_adamw_clip_scale", "psk_adamw_tree_scaled",
                  "psk_device_status", "psk_test_drop_row", "psk_test_fast_exp"):
            getattr(L, f).restype = ctypes.c_int
        _lib = L
    return _lib


def check(rc: int) -> None:
    if rc != 0:
        raise PskError(rc, lib().psk_last_error().decode())
