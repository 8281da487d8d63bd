// Pairs of binary32 values for the sm_100-class packed f32x2 instructions
// (fma / add / mul .rn.f32x2: one issue slot, two IEEE operations, each
// rounded to nearest even with gradual underflow, exactly as two scalar
// operations), the softmax region's fast exp (on pairs and alone) and the
// groups' fast exp-clamp (device code only: the exps take the multifunction
// unit's ex2.approx, so their bounds are measured on the GPU).

#pragma once

#include "crmath.cuh"

namespace psk {

typedef float2 f2;
// A pair product must never feed a pair sum whose rounding matters: the
// assembler has been seen to fuse such a product and sum into one fma (both
// through these intrinsics and through PTX that states the rounding), where
// scalar products (mul.rn) are never fused.  Here no pair product feeds a
// sum except exact ones (the exps' power-of-two scalings).
PSK_HD f2 f2_fma(f2 a, f2 b, f2 c) { return __ffma2_rn(a, b, c); }
PSK_HD f2 f2_add(f2 a, f2 b) { return __fadd2_rn(a, b); }
PSK_HD f2 f2_mul(f2 a, f2 b) { return __fmul2_rn(a, b); }
// max with NaN propagation (either operand NaN gives NaN)
PSK_HD float fmax_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}
PSK_HD f2 f2_splat(float v) { return f2{v, v}; }

constexpr float PAIR_EXP_MAGIC = 12582912.0f;   // 1.5 * 2^23

// 2^f for |f| <= 1/2 by the multifunction unit's ex2.approx (device only).
__device__ __forceinline__ float ex2_unit(float f) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(f));
  return r;
}

// The softmax region's fast exp, of t <= 0 (NaN and -inf allowed: the
// region's x - max), within two f32 ulp of exp(t), subnormal results
// included (device only):
//   t is held at -104.5 (exp below it rounds to +0; -inf, whose reduction
//   would be NaN, becomes that; NaN stays NaN);
//   k = nearest integer to t log2(e) by one fma with 1.5 * 2^23 (the sum lands
//   in the binade whose ulp is 1, so its low bits hold k);
//   f = t log2(e) - k in two fmas, log2(e) split as L + L' (L = RN(log2 e)):
//   t L - k is rounded once, to 2^-26 (|f| <= 1/2 + 2^-20), and t L' adds a
//   term below 2^-24.6 rounded to 2^-50 (Cody and Waite's reduction, in the
//   base-2 exponent);
//   2^f by the multifunction unit's ex2.approx;
//   2^k applied as 2^(k+64), an exact scaling, then 2^-64, the one rounding
//   where the result is subnormal.  The exponent field of 2^(k+64) is the
//   sum's bit pattern shifted left by 23 (its high bits fall out) plus 191.
// The bound is measured over every float of [-104.5, 0] on the GPU against
// the correctly rounded exp (91 % exact, 9 % one ulp, 0.03 % two ulp).  Pair
// and scalar forms do the same operations on each element: the same bits.
constexpr float PAIR_LOG2E_LO = 1.9259629911783687e-08f;   // RN(log2 e - RN(log2 e))
__device__ __forceinline__ f2 exp2_unit_nonpos(f2 t) {
  const f2 tc{fmax_nan(t.x, -104.5f), fmax_nan(t.y, -104.5f)};
  const f2 z = f2_fma(tc, f2_splat(PSK_FEXP_INV_LN2), f2_splat(PAIR_EXP_MAGIC));
  const f2 nk = f2_fma(z, f2_splat(-1.0f), f2_splat(PAIR_EXP_MAGIC));   // -k (exact)
  f2 f = f2_fma(tc, f2_splat(PSK_FEXP_INV_LN2), nk);
  f = f2_fma(tc, f2_splat(PAIR_LOG2E_LO), f);
  const f2 p{ex2_unit(f.x), ex2_unit(f.y)};
  const f2 s{u2f(f2u(z.x) * (1u << 23) + (191u << 23)), u2f(f2u(z.y) * (1u << 23) + (191u << 23))};
  return f2_mul(f2_mul(p, s), f2_splat(0x1p-64f));
}

__device__ __forceinline__ float exp_unit_nonpos(float t) {
  const float tc = fmax_nan(t, -104.5f);
  const float z = fmaf(tc, PSK_FEXP_INV_LN2, PAIR_EXP_MAGIC);
  const float kf = __fadd_rn(z, -PAIR_EXP_MAGIC);
  float f = fmaf(tc, PSK_FEXP_INV_LN2, -kf);
  f = fmaf(tc, PAIR_LOG2E_LO, f);
  const float p = ex2_unit(f);
  const float s = u2f(f2u(z) * (1u << 23) + (191u << 23));
  return __fmul_rn(__fmul_rn(p, s), 0x1p-64f);
}

// The groups' fast EXP-clamp node: exp of t in [-4, 4] (the clamped
// argument) by the same split and ex2.approx as above; k is in [-6, 6] and
// every result normal, so 2^k goes on in one step (exponent field: the sum's
// bit pattern shifted left by 23, plus 127) and the product is the one
// rounding after ex2.approx.  Within two f32 ulp over [-4, 4] (measured on
// the GPU against the correctly rounded exp).  Pair and scalar forms: the
// same bits.
__device__ __forceinline__ f2 exp2_unit_mid(f2 t) {
  const f2 z = f2_fma(t, f2_splat(PSK_FEXP_INV_LN2), f2_splat(PAIR_EXP_MAGIC));
  const f2 nk = f2_fma(z, f2_splat(-1.0f), f2_splat(PAIR_EXP_MAGIC));   // -k (exact)
  f2 f = f2_fma(t, f2_splat(PSK_FEXP_INV_LN2), nk);
  f = f2_fma(t, f2_splat(PAIR_LOG2E_LO), f);
  const f2 p{ex2_unit(f.x), ex2_unit(f.y)};
  const f2 s{u2f(f2u(z.x) * (1u << 23) + (127u << 23)), u2f(f2u(z.y) * (1u << 23) + (127u << 23))};
  return f2_mul(p, s);
}

__device__ __forceinline__ float exp_unit_mid(float t) {
  const float z = fmaf(t, PSK_FEXP_INV_LN2, PAIR_EXP_MAGIC);
  const float kf = __fadd_rn(z, -PAIR_EXP_MAGIC);
  float f = fmaf(t, PSK_FEXP_INV_LN2, -kf);
  f = fmaf(t, PAIR_LOG2E_LO, f);
  return __fmul_rn(ex2_unit(f), u2f(f2u(z) * (1u << 23) + (127u << 23)));
}

}  // namespace psk
