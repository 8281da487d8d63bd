"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in the oracle (on the CPU, through monkeypatch)
and checks that the pin written for that part of the oracle now fails.
"""

import numpy as np
import pytest

import oracle.adamw as OA
import oracle.crmath as OC
import oracle.f32 as OF
import oracle.group as OG
import oracle.norm as ON
import oracle.softmax as OS
from tests import test_oracle_adamw as TA
from tests import test_oracle_crmath as TC
from tests import test_oracle_f32 as TF
from tests import test_oracle_group as TG
from tests import test_oracle_norm as TN
from tests import test_oracle_softmax as TS


def _sub_reversed(monkeypatch):
    real = OG.apply_op

    def wrong(name, a, b=None):
        return real("SUB", b, a) if name == "SUB" else real(name, a, b)

    monkeypatch.setattr(OG, "apply_op", wrong)


def _max_tie_first(monkeypatch):
    monkeypatch.setattr(OG, "_max", lambda a, b: np.where(a >= b, a, b).astype(np.float32))


def _gelu_half_off(monkeypatch):
    monkeypatch.setattr(OG, "INV_SQRT2", np.float32(0.7071068))


def _expc_clamp_at_eight(monkeypatch):
    real = OG.apply_op

    def wrong(name, a, b=None):
        if name == "EXPC":
            return real("EXP", OG._min(OG._max(a, np.float32(-8.0)), np.float32(8.0)))
        return real(name, a, b)

    monkeypatch.setattr(OG, "apply_op", wrong)


def _expc_min_max_swapped(monkeypatch):
    real = OG.apply_op

    def wrong(name, a, b=None):
        if name == "EXPC":
            return real("EXP", OG._max(OG._min(a, np.float32(4.0)), np.float32(-4.0)))
        return real(name, a, b)

    monkeypatch.setattr(OG, "apply_op", wrong)


def _bf16_truncates(monkeypatch):
    monkeypatch.setattr(OF, "f32_to_bf16",
                        lambda x: (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16))


def _exp_in_binary32(monkeypatch):
    monkeypatch.setattr(OC, "exp_f32", lambda x: np.exp(np.asarray(x, dtype=np.float32)))


def _interleaved_combined_backwards(monkeypatch):
    real = OS._sum_interleaved

    def wrong(e, partials):
        return real(e[:, ::-1].copy(), partials)

    monkeypatch.setattr(OS, "_sum_interleaved", wrong)


def _adamw_no_bias_correction(monkeypatch):
    real = OA.hyper_f32

    def wrong(*a, **k):
        h = dict(real(*a, **k))
        h["bc2"] = np.float32(1.0)
        return h

    monkeypatch.setattr(OA, "hyper_f32", wrong)


def _adamw_eps_inside_sqrt(monkeypatch):
    def wrong(theta, m, v, grad, grad_dtype, h):
        th = np.asarray(theta, dtype=np.float32)
        g = OF.widen(grad, grad_dtype)
        m1 = (h["b1"] * m) + (h["omb1"] * g)
        v1 = (h["b2"] * v) + (h["omb2"] * (g * g))
        q = (m1 / h["bc1"]) / np.sqrt((v1 / h["bc2"]) + h["eps"])
        return (th - h["lr"] * (q + h["wd"] * th)).astype(np.float32), m1, v1

    monkeypatch.setattr(OA, "step_leaf", wrong)


def _norm_variance_over_n_minus_1(monkeypatch):
    calls = {"k": 0}

    def wrong(s, n):
        calls["k"] += 1
        return (s / (n - np.float32(1))).astype(np.float32) if calls["k"] % 2 == 0 else (s / n).astype(np.float32)

    monkeypatch.setattr(ON, "_mean", wrong)


def _norm_eps_after_sqrt(monkeypatch):
    monkeypatch.setattr(ON, "_divisor", lambda var, e: (np.sqrt(var).astype(np.float32) + e).astype(np.float32))


def _norm_no_mean_in_rms(monkeypatch):
    real = ON._mean
    monkeypatch.setattr(ON, "_mean", lambda s, n: real(s, np.float32(1)))


def _norm_bias_before_scale(monkeypatch):
    def wrong(y, g, b):
        if b is not None:
            y = (y + b[None, :]).astype(np.float32)
        if g is not None:
            y = (y * g[None, :]).astype(np.float32)
        return y

    monkeypatch.setattr(ON, "_affine", wrong)


def _cosine_without_half(monkeypatch):
    real = OA.lr_factor

    def wrong(kind, warmup, total, t):
        f = real(kind, warmup, total, t)
        return f * 2 if kind == "cosine" and warmup < t < total else f

    monkeypatch.setattr(OA, "lr_factor", wrong)


def _linear_decay_from_zero(monkeypatch):
    real = OA.lr_factor

    def wrong(kind, warmup, total, t):
        from fractions import Fraction
        if kind == "linear" and warmup < t < total:
            return Fraction(total - t, total)
        return real(kind, warmup, total, t)

    monkeypatch.setattr(OA, "lr_factor", wrong)


def _sq_norm_one_chain(monkeypatch):
    def wrong(grads, grad_dtype):
        total = np.float32(0)
        for g in grads:
            for v in OF.widen(np.asarray(g), grad_dtype).reshape(-1):
                total = np.float32(total + np.float32(v * v))
        return total

    monkeypatch.setattr(OA, "grad_sq_norm", wrong)


def _clip_without_epsilon(monkeypatch):
    def wrong(sq_norm, grad_clip):
        q = np.float32(np.float32(grad_clip) / np.sqrt(np.float32(sq_norm)))
        return q if q < 1 else np.float32(1)

    monkeypatch.setattr(OA, "clip_scale", wrong)


def _mask_keeps_emptied_rows(monkeypatch):
    real = OS._apply_mask

    def wrong(xf, mask):
        xm, emptied = real(xf, mask)
        return xm, np.zeros_like(emptied)

    monkeypatch.setattr(OS, "_apply_mask", wrong)


def _backward_sign_flipped(monkeypatch):
    def wrong(y, ct, y_dtype, ct_dtype, dx_dtype, order=("sequential",)):
        yf, cf = OF.widen(np.asarray(y), y_dtype), OF.widen(np.asarray(ct), ct_dtype)
        s = OS.row_sum((cf * yf).astype(np.float32), order)
        return OF.store((yf * (s[:, None] - cf).astype(np.float32)).astype(np.float32), dx_dtype)

    monkeypatch.setattr(OS, "softmax_backward", wrong)


def _log_in_binary32(monkeypatch):
    def wrong(x):
        with np.errstate(all="ignore"):
            return np.log(np.asarray(x, dtype=np.float32))

    monkeypatch.setattr(OC, "log_f32", wrong)


def _tanh_through_exp_in_binary32(monkeypatch):
    def wrong(x):
        x = np.asarray(x, dtype=np.float32)
        with np.errstate(all="ignore"):
            e = np.exp(np.float32(2) * x)
            return ((e - np.float32(1)) / (e + np.float32(1))).astype(np.float32)

    monkeypatch.setattr(OC, "tanh_f32", wrong)


def _select_by_arithmetic(monkeypatch):
    def wrong(c, a, b):
        k = (np.asarray(c) != 0).astype(np.float32)
        with np.errstate(all="ignore"):
            return (k * a + (np.float32(1) - k) * b).astype(np.float32)

    monkeypatch.setattr(OG, "select", wrong)


def _select_picks_on_zero(monkeypatch):
    monkeypatch.setattr(OG, "select", lambda c, a, b: np.where(np.asarray(c) == 0, a, b).astype(np.float32))


CASES = [
    (_sub_reversed, TG.test_all_programs_up_to_two_nodes_bitwise),
    (_max_tie_first, TG.test_max_min_tie_gives_second_operand),
    (_gelu_half_off, TG.test_small_group_against_mpmath_per_node),
    (_expc_clamp_at_eight, TG.test_expc_clamp_bounds_against_mpmath),
    (_expc_min_max_swapped, TG.test_expc_clamp_bounds_against_mpmath),
    (_bf16_truncates, TF.test_bf16_rounding_matches_torch),
    (_exp_in_binary32, TC.test_exp_correctly_rounded_across_binades),
    (_interleaved_combined_backwards, lambda: TS.test_tiny_rows_exact(("interleaved", 3))),
    (_adamw_no_bias_correction, TA.test_against_torch_adamw_float64),
    (_adamw_eps_inside_sqrt, TA.test_first_step_closed_form),
    (_norm_variance_over_n_minus_1, TN.test_layer_norm_of_two_values_is_plus_minus_one),
    (_norm_eps_after_sqrt, TN.test_rms_closed_form_with_eps),
    (_norm_no_mean_in_rms, TN.test_rms_of_a_constant_row_is_one),
    (_norm_bias_before_scale, TN.test_gamma_and_beta),
    (_cosine_without_half, TA.test_cosine_schedule_closed_forms_and_symmetry),
    (_linear_decay_from_zero, TA.test_linear_schedule_closed_forms),
    (_sq_norm_one_chain, TA.test_squared_norm_follows_the_declared_tree),
    (_clip_without_epsilon, TA.test_clip_scale_closed_form),
    (_mask_keeps_emptied_rows, TS.test_mask_emptied_rows_give_zeros_and_full_mask_changes_nothing),
    (_backward_sign_flipped, TS.test_backward_one_hot_cotangent_closed_form),
    (_log_in_binary32, TC.test_log_correctly_rounded_across_binades),
    (_tanh_through_exp_in_binary32, TC.test_tanh_correctly_rounded_across_binades),
    (_select_by_arithmetic, TG.test_select_moves_the_picked_bits_and_never_the_other_branch),
    (_select_picks_on_zero, TG.test_select_condition_broadcast_row_mask),
]


@pytest.mark.parametrize("plant,pin", CASES, ids=[c[0].__name__ for c in CASES])
def test_planted_mistake_is_caught(monkeypatch, plant, pin):
    plant(monkeypatch)
    with pytest.raises(AssertionError):
        pin()
