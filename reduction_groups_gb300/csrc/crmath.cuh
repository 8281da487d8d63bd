// Correctly rounded binary32 exp and erf for the group and softmax kernels.
//
// An exp or erf node of a fusion group returns RN_f32(exp(x)) / RN_f32(erf(x))
// (nearest, ties to even, gradual underflow, overflow to infinity).  The pages
// ask that every executor compute the same transcendental bits ("Native
// execution", The Cranelift backend: one libm for all executors); a correctly
// rounded function has one value, so any correct implementation gives it.
//
// Each function has three tiers (Ziv's strategy: evaluate with an error bound,
// keep the result when the bound decides the rounding, else retry more
// accurately):
//   1. binary32 float-float arithmetic, relative error below 2^-41; the result
//      is kept when it lies more than the error bound away from every rounding
//      boundary (one call in about 2^14 fails the test);
//   2. binary64, relative error below 2^-50, kept unless within 2^-48 of a
//      boundary (one call in about 2^25 of the calls reaching it);
//   3. double-double Taylor series, error below 2^-95.
// Tier 1 is all that runs in practice; tiers 2 and 3 are separate functions.
//
// The same source compiles as CUDA device code (the library) and as plain C++
// for the host (a test build that checks the tiers element by element).

#pragma once

#if !defined(__CUDACC_RTC__)   // the run-time compiler has its own built-ins
#include <stdint.h>
#include <math.h>
#include <string.h>
#endif

// PSK_TAB: tables read with a uniform index (constant memory on the device);
// PSK_GTAB: tables read with a per-lane index (global memory, cached in L1,
// or staged by a kernel into shared memory).
#if defined(PSK_HOST_BUILD)
#define PSK_HD static inline
#define PSK_NOINLINE static
#define PSK_TAB static const
#define PSK_GTAB alignas(16) static const
#else
#define PSK_HD __device__ __forceinline__
#define PSK_NOINLINE static __device__ __noinline__
#define PSK_TAB static __constant__ const
#define PSK_GTAB static __device__ const __attribute__((aligned(16)))
#endif

#include "crmath_tables.inc"

namespace psk {

// ------------------------------------------------------------ bit helpers
PSK_HD uint32_t f2u(float f) {
#if defined(PSK_HOST_BUILD)
  uint32_t u; memcpy(&u, &f, 4); return u;
#else
  return __float_as_uint(f);
#endif
}
PSK_HD float u2f(uint32_t u) {
#if defined(PSK_HOST_BUILD)
  float f; memcpy(&f, &u, 4); return f;
#else
  return __uint_as_float(u);
#endif
}
PSK_HD float d2f_rn(double d) {
#if defined(PSK_HOST_BUILD)
  return (float)d;
#else
  return __double2float_rn(d);
#endif
}

// ------------------------------------------------- error-free transforms
// (Knuth's TwoSum, Dekker's Fast2Sum, and the product error by fma.)
PSK_HD void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}
PSK_HD void fast_two_sum(float a, float b, float& s, float& e) {  // |a| >= |b| or a == 0
  s = a + b;
  e = b - (s - a);
}
PSK_HD void two_prod(float a, float b, float& p, float& e) {
  p = a * b;
  e = fmaf(a, b, -p);
}
PSK_HD void two_sum_d(double a, double b, double& s, double& e) {
  s = a + b;
  double bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}
PSK_HD void fast_two_sum_d(double a, double b, double& s, double& e) {
  s = a + b;
  e = b - (s - a);
}

// double-double value hi + lo, |lo| <= ulp(hi)/2
struct dd { double hi, lo; };

PSK_HD dd dd_add(dd a, dd b) {
  double s, e, t, f;
  two_sum_d(a.hi, b.hi, s, e);
  two_sum_d(a.lo, b.lo, t, f);
  e += t;
  fast_two_sum_d(s, e, s, e);
  e += f;
  fast_two_sum_d(s, e, s, e);
  return dd{s, e};
}
PSK_HD dd dd_mul(dd a, dd b) {
  double p = a.hi * b.hi;
  double e = fma(a.hi, b.hi, -p);
  e = fma(a.hi, b.lo, e);
  e = fma(a.lo, b.hi, e);
  double s;
  fast_two_sum_d(p, e, s, e);
  return dd{s, e};
}
PSK_HD dd dd_div_d(dd a, double b) {  // a / b, b a small exact value
  double q1 = a.hi / b;
  double p = q1 * b;
  double pe = fma(q1, b, -p);
  double r = ((a.hi - p) - pe) + a.lo;
  double q2 = r / b;
  double s, e;
  fast_two_sum_d(q1, q2, s, e);
  return dd{s, e};
}

PSK_HD dd dd_neg(dd a) { return dd{-a.hi, -a.lo}; }

// a / b in double-double: three quotient digits, each from the residual
// a - q b evaluated in double-double (relative error below 2^-100).
PSK_HD dd dd_div(dd a, dd b) {
  double q1 = a.hi / b.hi;
  dd r = dd_add(a, dd_neg(dd_mul(b, dd{q1, 0.0})));
  double q2 = r.hi / b.hi;
  r = dd_add(r, dd_neg(dd_mul(b, dd{q2, 0.0})));
  double q3 = r.hi / b.hi;
  double s, e;
  fast_two_sum_d(q1, q2, s, e);
  return dd_add(dd{s, e}, dd{q3, 0.0});
}

// ------------------------------------------------------------ rounding
// RN_f32 of a binary64 value y known to within rel*|y|; ok = false when the
// interval of possible exact values reaches a binary32 rounding boundary.
PSK_HD float round_checked(double y, double rel, bool& ok) {
  float r = d2f_rn(y);
  double ay = fabs(y);
  float ar = fabsf(r);
  double a = (double)ar, up, dn;
  if (isinf(ar)) {
    a = 0x1p128;
    dn = 0x1.fffffep127;
    up = 0x1p129;
  } else {
    up = (ar == 0x1.fffffep127f) ? 0x1p128 : (double)nextafterf(ar, INFINITY);
    dn = (ar == 0.0f) ? -0x1p-149 : (double)nextafterf(ar, 0.0f);
  }
  double tol = rel * ay;
  ok = (fabs(ay - 0.5 * (a + up)) > tol) && (fabs(ay - 0.5 * (a + dn)) > tol);
  return r;
}

// RN_f32 of the double-double value hi + lo (|lo| <= ulp(hi)/2).  Rounding hi
// alone is right unless hi is exactly halfway between two binary32 values;
// then the sign of lo says on which side the exact value lies.
PSK_HD float dd_to_f32(dd v) {
  double A = fabs(v.hi);
  double L = (v.hi < 0) ? -v.lo : v.lo;     // exact magnitude is A + L
  float r = d2f_rn(A);
  if ((double)r == A) return copysignf(r, (float)v.hi);
  double below, above;                       // binary32 neighbours around A
  if (isinf(r)) {
    below = 0x1.fffffep127; above = 0x1p128;
  } else if ((double)r > A) {
    above = (double)r; below = (r == 0.0f) ? 0.0 : (double)nextafterf(r, 0.0f);
  } else {
    below = (double)r;
    above = (r == 0x1.fffffep127f) ? 0x1p128 : (double)nextafterf(r, INFINITY);
  }
  double mid = 0.5 * (below + above);
  float out = r;
  if (A == mid && L != 0.0) out = (L > 0) ? (above >= 0x1p128 ? INFINITY : (float)above) : (float)below;
  return copysignf(out, (float)v.hi);
}

// ====================================================================== exp

// exp(x) = 2^k exp(r), r = x - k ln2, with exp(r) by its Taylor series in
// double-double (to 2^-106); returns exp(r) and k.
PSK_HD dd exp_dd_reduced(double x, int& k) {
  const dd LN2 = {PSK_DD_LN2_HI, PSK_DD_LN2_LO};
  double kd = rint(x * PSK_DD_INV_LN2);
  dd kl = dd_mul(LN2, dd{kd, 0.0});
  dd r = dd_add(dd{x, 0.0}, dd{-kl.hi, -kl.lo});
  dd term = {1.0, 0.0}, sum = {1.0, 0.0};
  for (int n = 1; n < 40; ++n) {
    term = dd_div_d(dd_mul(term, r), (double)n);
    sum = dd_add(sum, term);
    if (fabs(term.hi) < 0x1p-110 * fabs(sum.hi)) break;
  }
  k = (int)kd;
  return sum;
}

// Tier 3: double-double.
PSK_NOINLINE float exp_tier3(float xf) {
  int ki;
  dd sum = exp_dd_reduced((double)xf, ki);
  return dd_to_f32(dd{ldexp(sum.hi, ki), ldexp(sum.lo, ki)});
}

// Tier 2: binary64, table 2^(j/32) and a degree-6 polynomial on |r| <= ln2/64.
PSK_NOINLINE float exp_tier2(float xf) {
  if (isnan(xf)) return xf + xf;
  if (xf > 89.0f) return INFINITY;
  if (xf < -104.0f) return 0.0f;
  double x = (double)xf;
  double kd = rint(x * PSK_EXP_INV_LD);
  int k = (int)kd;
  double r = fma(-kd, PSK_EXP_L1D, x);  // exact
  r = fma(-kd, PSK_EXP_L2D, r);
  double p = 1.0 / 720.0;
  p = fma(p, r, 1.0 / 120.0);
  p = fma(p, r, 1.0 / 24.0);
  p = fma(p, r, 1.0 / 6.0);
  p = fma(p, r, 0.5);
  p = fma(p, r * r, r);                 // e^r - 1
  int j = k & 31, n = k >> 5;
  double T = psk_exp_tab_d[j];
  double y = ldexp(fma(T, p, T), n);
  bool ok;
  float res = round_checked(y, 0x1p-48, ok);
  return ok ? res : exp_tier3(xf);
}

// Entry j of a table of float pairs (hi, lo) stored interleaved; one 8-byte
// load on the device (the table is 8-byte aligned).
PSK_HD void load_pair(const float* tab2, int j, float& hi, float& lo) {
#if defined(PSK_HOST_BUILD)
  hi = tab2[2 * j];
  lo = tab2[2 * j + 1];
#else
  const float2 t = *reinterpret_cast<const float2*>(tab2 + 2 * j);
  hi = t.x;
  lo = t.y;
#endif
}

// Tier 1 core, |x| <= 87 (normal results).  tab2: 2^(j/1024), j = 0..1023,
// as float pairs (hi, lo) interleaved.  Returns R (the nearest float to the
// approximation) and d, with exp(x) = (R + d) 2^n (1 + delta), |delta| < 2^-42.
//
// x = k ln2/1024 + r, |r| <= ln2/2048 (< 2^-11.4), k = 1024 n + j; and
// r = r1 + c with r1 = x - k L1 exact (L1 = RN(ln2/1024): r1 is a multiple
// of 2^-35 below 2^-11, so 24 bits hold it) and c = -k (L2 + L3),
// |c| < 2^-21.99.  Then e^r - 1 = r1 + ql with
//   ql = c (1 + r1) + r1^2 (1/2 + r1/6)
// (dropped: r^4/24, c^2/2 and c r1^2/2, each below 2^-45), and
//   exp(x) 2^-n = Th + Th r1 + [Th ql + Tl (1 + r1)]
// (dropped: Tl ql < 2^-45), where Th r1 is split exactly (two_prod) and the
// bracket (< 2^-20.5) takes one rounding of its own; R = RN(Th + RN(m1 +
// low)) and the residual d = ((Th - R) + m1) + low, whose first two steps
// are exact (Th - R by Sterbenz; the sum below ulp(R) on the grid of m1).
PSK_HD void exp_tier1_core(float x, const float* tab2, float& R, float& d, int& n) {
  const float kf = rintf(x * PSK_EXP_INV_L);
  const int k = (int)kf;
  n = k >> 10;
  const int j = k & 1023;
  const float r1 = fmaf(-kf, PSK_EXP_L1, x);
  const float c = fmaf(-kf, PSK_EXP_L2, -kf * PSK_EXP_L3);
  float Th, Tl;
  load_pair(tab2, j, Th, Tl);
  const float s = r1 * r1;
  const float p = fmaf(r1, 1.0f / 6.0f, 0.5f);
  const float u = fmaf(c, r1, c);
  const float ql = fmaf(s, p, u);
  float m1, e1;
  two_prod(Th, r1, m1, e1);
  const float t = fmaf(Tl, r1, Tl + e1);
  const float low = fmaf(Th, ql, t);
  R = Th + (m1 + low);
  d = ((Th - R) + m1) + low;   // Th - R exact (Sterbenz), + m1 exact but for < 2^-47
}

// Keep R when R + d (1 + 2^-14) still rounds to R (R finite): fma rounds the
// exact sum once, so this tests |d| against the half-gap to R's neighbour on
// d's side -- the smaller gap below a power of two included -- with a margin
// of 2^-14 of it, in two instructions.  An approximation R + d of relative
// error below 2^-41 lies within 2^-16 of a half-gap above (2^-15 of the one
// below a power of two) of the exact value, so a kept R is its correct
// rounding.
PSK_HD bool tier1_decided(float R, float d) {
  return fmaf(d, 0x1.0004p+0f, R) == R;
}

PSK_HD bool exp_tier1(float x, const float* tab2, float& out) {
  float R, d;
  int n;
  exp_tier1_core(x, tab2, R, d, n);
  out = u2f((uint32_t)((int32_t)f2u(R) + n * (1 << 23)));
  return tier1_decided(R, d);
}

// Correctly rounded exp; tab2 points at the 2^(j/1024) float-pair table
// (psk_exp_tab2, or a copy of it in shared memory).
PSK_HD float exp_cr(float x, const float* tab2) {
  float r;
  if (fabsf(x) <= 87.0f && exp_tier1(x, tab2, r)) return r;
  return exp_tier2(x);
}

// ====================================================================== erf

// Tier 3: Maclaurin series in double-double (|a| < 4), error below 2^-95.
PSK_NOINLINE float erf_tier3(float af) {
  double a = (double)af;
  dd a2 = dd_mul(dd{a, 0.0}, dd{a, 0.0});
  dd term = {a, 0.0};      // a^(2n+1) / n!
  dd sum = {a, 0.0};
  for (int n = 1; n < 200; ++n) {
    term = dd_div_d(dd_mul(term, a2), (double)n);
    dd t = dd_div_d(term, (double)(2 * n + 1));
    if (n & 1) t = dd{-t.hi, -t.lo};
    sum = dd_add(sum, t);
    if (fabs(t.hi) < 0x1p-112 * fabs(sum.hi)) break;
  }
  return dd_to_f32(dd_mul(sum, dd{PSK_DD_TWO_OVER_SQRTPI_HI, PSK_DD_TWO_OVER_SQRTPI_LO}));
}

// Tier 2: binary64 Taylor polynomials of degree 12 about i/8.  a = |x|.
PSK_NOINLINE float erf_tier2(float af) {
  double a = (double)af, y;
  if (af < 0x1p-60f) {
    y = PSK_TWO_OVER_SQRTPI_D * a;
  } else {
    int i = (int)rint(a * 8.0);
    double t = a - 0.125 * i;
    y = psk_erf_c64[PSK_ERF_D64][i];
    for (int k = PSK_ERF_D64 - 1; k >= 0; --k) y = fma(y, t, psk_erf_c64[k][i]);
  }
  bool ok;
  float res = round_checked(y, 0x1p-48, ok);
  return ok ? res : erf_tier3(af);
}

// Tier 1 core of a function tabulated as Taylor polynomials about i/32
// (interval width 1/32), N intervals, degree D, coefficients 0..NPAIR-1 as
// float pairs [k][interval][hi, lo] in p2 and NPAIR..D as floats
// [k - NPAIR][interval] in h.  Returns R + d = f(a)(1 + delta).
//
// t = a - i/32 (exact, |t| <= 1/64).  Coefficients NPAIR..D by Horner in
// binary32 (their terms stay below 2^-18 of f(a)); then V_k = c_k + t V_{k+1}
// for k = NPAIR-1..0 in float-float, each product split exactly (two_prod)
// and each sum renormalised: by Fast2Sum where |c_k| >= |t V_{k+1}| or
// c_k = 0 holds on every interval (checked when the tables are generated),
// by TwoSum at the steps set in TWOSUM (bit k: step k).
template <int N, int D, int NPAIR, int TWOSUM>
PSK_HD void taylor32_tier1_core(float a, const float* p2, const float* h, float& R, float& d) {
  const float fi = rintf(a * 32.0f);
  const int i = (int)fi;
  const float t = fmaf(fi, -0.03125f, a);   // exact
  float H = h[(D - NPAIR) * N + i];
#pragma unroll
  for (int k = D - 1; k >= NPAIR; --k) H = fmaf(H, t, h[(k - NPAIR) * N + i]);
  float p, pe, vh, vl, ch, cl;
  two_prod(t, H, p, pe);
  load_pair(p2 + (NPAIR - 1) * 2 * N, i, ch, cl);
  if (TWOSUM & (1 << (NPAIR - 1))) two_sum(ch, p, vh, vl);
  else fast_two_sum(ch, p, vh, vl);
  vl = vl + (pe + cl);
#pragma unroll
  for (int k = NPAIR - 2; k >= 0; --k) {
    two_prod(t, vh, p, pe);
    pe = fmaf(t, vl, pe);
    load_pair(p2 + k * 2 * N, i, ch, cl);
    if (TWOSUM & (1 << k)) two_sum(ch, p, vh, vl);
    else fast_two_sum(ch, p, vh, vl);
    vl = vl + (pe + cl);
  }
  R = vh + vl;
  d = vl - (R - vh);
}

// The same tables as one record of 12 floats per interval (three 16-byte
// groups: coefficients 7, 6, 5, 4; then 3 and 2 as (hi, lo) pairs; then 1
// and 0), so that a lookup is three 16-byte loads instead of eight: record i
// is rec[12 i .. 12 i + 11].
PSK_HD void erf_record(const float* p2, const float* h, int i, float* rec) {
  for (int k = 0; k < 4; ++k) rec[k] = h[(3 - k) * PSK_ERF_N32 + i];
  for (int k = 0; k < 4; ++k) {
    rec[4 + 2 * k] = p2[(3 - k) * 2 * PSK_ERF_N32 + 2 * i];
    rec[5 + 2 * k] = p2[(3 - k) * 2 * PSK_ERF_N32 + 2 * i + 1];
  }
}

PSK_HD void load_record12(const float* rec, int i, float* v) {
#if defined(PSK_HOST_BUILD)
  for (int k = 0; k < 12; ++k) v[k] = rec[12 * i + k];
#else
  const float4* r = reinterpret_cast<const float4*>(rec) + 3 * i;
  const float4 a = r[0], b = r[1], c = r[2];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  v[8] = c.x; v[9] = c.y; v[10] = c.z; v[11] = c.w;
#endif
}

// erf tier 1 from the record tables: the same operations on the same
// coefficients as erf_tier1_core (degree 7, four float-float steps), so the
// same R and d.
PSK_HD void erf_tier1_core_rec(float a, const float* rec, float& R, float& d) {
  static_assert(PSK_ERF_D32 == 7 && PSK_ERF_NPAIR == 4, "erf record layout");
  const float fi = rintf(a * 32.0f);
  const int i = (int)fi;
  const float t = fmaf(fi, -0.03125f, a);   // exact
  float c[12];
  load_record12(rec, i, c);
  float H = c[0];
  H = fmaf(H, t, c[1]);
  H = fmaf(H, t, c[2]);
  H = fmaf(H, t, c[3]);
  float p, pe, vh, vl;
  two_prod(t, H, p, pe);
  fast_two_sum(c[4], p, vh, vl);
  vl = vl + (pe + c[5]);
#pragma unroll
  for (int k = 1; k < 4; ++k) {
    two_prod(t, vh, p, pe);
    pe = fmaf(t, vl, pe);
    float sh, sl;
    fast_two_sum(c[4 + 2 * k], p, sh, sl);
    vh = sh;
    vl = sl + (pe + c[5 + 2 * k]);
  }
  R = vh + vl;
  d = vl - (R - vh);
}

// erf tier 1, 2^-60 <= a < PSK_ERF_ONE_FROM (< 3.9375): p2 / h are
// psk_erf_p2 / psk_erf_h or copies in shared memory.  Relative error below
// 2^-42 (the coefficients' terms from 4 on stay below 2^-18 of erf(a)).
PSK_HD void erf_tier1_core(float a, const float* p2, const float* h, float& R, float& d) {
  taylor32_tier1_core<PSK_ERF_N32, PSK_ERF_D32, PSK_ERF_NPAIR, 0>(a, p2, h, R, d);
}

PSK_HD bool erf_tier1(float a, const float* p2, const float* h, float& out) {
  float d;
  erf_tier1_core(a, p2, h, out, d);
  return tier1_decided(out, d);
}

// erf of |x| outside tier 1's reach or undecided by it: NaN, 0, tiny
// arguments and undecided ones by tier 2, saturation at 1.
PSK_NOINLINE float erf_abs_rest(float a) {
  if (!(a == a)) return a + a;
  if (a >= PSK_ERF_ONE_FROM) return 1.0f;   // erfc(a) < 2^-25 from here on: rounds to 1
  if (a == 0.0f) return 0.0f;
  return erf_tier2(a);
}

// Correctly rounded erf (odd; erf(+-0) = +-0, erf(+-inf) = +-1, NaN stays NaN).
PSK_HD float erf_cr(float x, const float* p2, const float* h) {
  const float a = fabsf(x);
  const bool inr = a < PSK_ERF_ONE_FROM && a >= 0x1p-60f;
  float r;
  if (!(inr && erf_tier1(a, p2, h, r))) r = erf_abs_rest(a);
  return copysignf(r, x);
}

// ===================================================================== tanh
// tanh(a) rounds to a below 2^-12 (a^3/3 is under half an ulp there) and to 1
// from PSK_TANH_ONE_FROM (1 - tanh(a) <= 2^-25); between, tier 1 is the
// Taylor table (psk_tanh_p2 / psk_tanh_h, erf's layout), tier 2 the math
// library's binary64 tanh and tier 3 the double-double (1 - e^-2a) /
// (1 + e^-2a) (cancellation costs at most 11 of its 106 bits).

// Tier 3: 2^-12 <= a < PSK_TANH_ONE_FROM.
PSK_NOINLINE float tanh_tier3(float af) {
  int k;
  dd E = exp_dd_reduced(-2.0 * (double)af, k);
  E = dd{ldexp(E.hi, k), ldexp(E.lo, k)};        // e^-2a >= 2^-27: no underflow
  dd num = dd_add(dd{1.0, 0.0}, dd_neg(E));
  dd den = dd_add(dd{1.0, 0.0}, E);
  return dd_to_f32(dd_div(num, den));
}

PSK_HD void tanh_tier1_core(float a, const float* p2, const float* h, float& R, float& d) {
  taylor32_tier1_core<PSK_TANH_N32, PSK_TANH_D32, PSK_ERF_NPAIR, PSK_TANH_TWOSUM_MASK>(a, p2, h, R, d);
}

PSK_HD bool tanh_tier1(float a, const float* p2, const float* h, float& out) {
  float d;
  tanh_tier1_core(a, p2, h, out, d);
  return tier1_decided(out, d);
}

// Tier 2: the math library's binary64 tanh (within a few ulp of binary64,
// relative error below 2^-50), kept unless within 2^-48 of a rounding
// boundary; else tier 3.  2^-12 <= a < PSK_TANH_ONE_FROM.
PSK_NOINLINE float tanh_tier2(float af) {
  bool ok;
  const float r = round_checked(tanh((double)af), 0x1p-48, ok);
  return ok ? r : tanh_tier3(af);
}

// tanh of a = |x| where tier 1 does not reach or decide: NaN, small
// arguments, saturation, the undecided rest by tiers 2 and 3.
PSK_NOINLINE float tanh_abs_rest(float a) {
  if (!(a == a)) return a + a;
  if (a < 0x1p-12f) return a;
  if (a >= PSK_TANH_ONE_FROM) return 1.0f;
  return tanh_tier2(a);
}

// Correctly rounded tanh (odd; tanh(+-0) = +-0, tanh(+-inf) = +-1).
PSK_HD float tanh_cr(float x, const float* p2, const float* h) {
  const float a = fabsf(x);
  const bool inr = a >= 0x1p-12f && a < PSK_TANH_ONE_FROM;
  float r;
  if (!(inr && tanh_tier1(a, p2, h, r))) r = tanh_abs_rest(a);
  return copysignf(r, x);
}

// ====================================================================== log
// x = 2^e m, m in [1, 2); on the intervals above sqrt 2 (table flag s = 1) m
// is read as m/2 and e as e + 1, so that log(x) = e' ln2 + log(m') with
// m' in [0.707, 1.414).  The table entry of m's top nine bits gives c (a
// multiple of 2^-10 near 1/m, so r = m c - 1 is exact and |r| < 2^-9) and
// T = -log(c 2^s), so log(x) = e' ln2 + T + log1p(r).  Entries 0 and 511 (m
// next to 1 and 2) have c = 1 and 1/2, T = 0: near x = 1 the result is
// log1p(r) with no cancellation.

// Tier 3: log(m') = 2 atanh(u), u = (m' - 1)/(m' + 1) (|u| < 0.172), by its
// series in double-double; x positive, finite, normal.
PSK_NOINLINE float log_tier3(float xf, int ebias) {
  int e = (int)((f2u(xf) >> 23) & 0xffu) - 127 + ebias;
  double m = (double)u2f((f2u(xf) & 0x007fffffu) | 0x3f800000u);
  if (m > 0x1.6a09e667f3bcdp+0) { m *= 0.5; e += 1; }
  dd u = dd_div_d(dd{m - 1.0, 0.0}, m + 1.0);    // m - 1 and m + 1 exact
  dd u2 = dd_mul(u, u);
  dd term = u, sum = u;
  for (int n = 1; n < 40; ++n) {
    term = dd_mul(term, u2);
    dd t = dd_div_d(term, (double)(2 * n + 1));
    sum = dd_add(sum, t);
    if (fabs(t.hi) < 0x1p-110 * fabs(sum.hi)) break;
  }
  const dd LN2 = {PSK_DD_LN2_HI, PSK_DD_LN2_LO};
  dd r = dd_add(dd_mul(LN2, dd{(double)e, 0.0}), dd{2.0 * sum.hi, 2.0 * sum.lo});
  return dd_to_f32(r);
}

// Entry i of the log table: (c, T hi, T lo, s), one 16-byte load on the
// device (the table is 16-byte aligned).
PSK_HD void load_quad(const float* tab4, int i, float& c, float& th, float& tl, float& s) {
#if defined(PSK_HOST_BUILD)
  c = tab4[4 * i]; th = tab4[4 * i + 1]; tl = tab4[4 * i + 2]; s = tab4[4 * i + 3];
#else
  const float4 q = *reinterpret_cast<const float4*>(tab4 + 4 * i);
  c = q.x; th = q.y; tl = q.z; s = q.w;
#endif
}

// Tier 1 core: x positive, finite and normal (a subnormal is passed scaled
// by 2^24 with ebias = -24).  log(x) = R + d to a relative error below
// 2^-41 (at most 2^-42.1 over every positive normal float):
//   log1p(r) = r - r^2/2 + r^3 (1/3 - r/4 + r^2/5)   (dropped: r^6/6 < 2^-56),
// r^2 split exactly (two_prod).  T hi, r, -r^2/2, e' L1 and e' L2 (exact: L1
// and L2 carry 16 bits, |e'| < 2^8) are added exactly, each by Fast2Sum (the
// table holds T = 0 or |T hi| >= |r|; |r^2/2| < |T hi + r|; e' L1 is 0 or
// above 0.69 > |log m'|; |e' L2| < 2^-11 |e' L1 + log m'|); the rest -- the
// Fast2Sum errors, T lo, e' L3, the product error of r^2 and the cubic tail,
// each below 2^-19 of the result -- is summed in binary32.
PSK_HD void log_tier1_core(float x, int ebias, const float* tab4, float& R, float& d) {
  const uint32_t u = f2u(x);
  const int i = (int)((u >> 14) & 511u);
  const float m = u2f((u & 0x007fffffu) | 0x3f800000u);
  float c, th, tl, sf;
  load_quad(tab4, i, c, th, tl, sf);
  const float ef = (float)((int)(u >> 23) - 127 + ebias) + sf;
  const float r = fmaf(m, c, -1.0f);               // exact
  float s2, se;
  two_prod(r, r, s2, se);
  const float hs = -0.5f * s2;                     // exact
  float a1, b1, a2, b2, a3, b3, H, b4;
  fast_two_sum(th, r, a1, b1);
  fast_two_sum(a1, hs, a2, b2);
  fast_two_sum(ef * PSK_LOG_L1, a2, a3, b3);
  fast_two_sum(a3, ef * PSK_LOG_L2, H, b4);
  const float p = fmaf(fmaf(r, 0.2f, -0.25f), r, 0x1.555556p-2f);
  const float tail = fmaf(-0.5f, se, (s2 * r) * p);
  const float low = ((b1 + b2) + (b3 + b4)) + (fmaf(ef, PSK_LOG_L3, tl) + tail);
  fast_two_sum(H, low, R, d);
}

// Tier 2: the math library's binary64 log (within a few ulp of binary64,
// relative error below 2^-50), kept unless within 2^-48 of a rounding
// boundary; else tier 3.  x positive, finite, not 1.
PSK_NOINLINE float log_tier2(float x) {
  bool ok;
  const float r = round_checked(log((double)x), 0x1p-48, ok);
  if (ok) return r;
  return x < 0x1p-126f ? log_tier3(x * 0x1p24f, -24) : log_tier3(x, 0);
}

// log of x outside tier 1's reach or undecided by it: NaN, zero, negative,
// infinite, 1 (exactly 0) and the undecided rest by tiers 2 and 3.
PSK_NOINLINE float log_rest(float x) {
  if (!(x == x)) return x + x;
  if (x == 0.0f) return -INFINITY;
  if (x < 0.0f) return u2f(0x7fc00000u);
  if (isinf(x)) return x;
  if (x == 1.0f) return 0.0f;
  return log_tier2(x);
}

// Correctly rounded natural logarithm.
PSK_HD float log_cr(float x, const float* tab4) {
  const bool inr = x > 0.0f && x < INFINITY && x != 1.0f;
  float r = 0.0f;
  bool ok = false;
  if (inr) {
    const bool sub = x < 0x1p-126f;
    float d;
    log_tier1_core(sub ? x * 0x1p24f : x, sub ? -24 : 0, tab4, r, d);
    ok = tier1_decided(r, d);
  }
  return ok ? r : log_rest(x);
}

// ================================================ division by a fixed b
// a / b correctly rounded from rb = RN(1/b), for |a| >= 2^-100, 1 <= b < 2^20
// (Markstein's correction: q = RN(a rb) is within an ulp of a/b, the residual
// r = a - b q is exact by fma, and RN(q + r rb) is the correctly rounded
// quotient).  Other operands go to IEEE division.
PSK_HD float div_by_recip(float a, float b, float rb) {
  if (!(fabsf(a) >= 0x1p-100f) || !(b >= 1.0f && b < 0x1p20f) || isinf(a)) return a / b;
  float q = a * rb;
  float r = fmaf(-q, b, a);
  return fmaf(r, rb, q);
}

// ====================================== faithful exp and erf for groups
// A group's declared fast realization of its EXP and ERF nodes (math mode
// FAST): within one and two f32 ulp of the correctly rounded value (measured
// over their ranges by the host tests), not correctly rounded and not
// bit-identical to the oracle.  (The EXP-clamp node's fast exp is in
// pair.cuh; GELU keeps the correctly rounded erf.)

// exp over every f32: x clamped to [-104.5, 89] (beyond, the result is 0 or
// infinity either way), 2^k applied in two exact halves and one rounding at
// the end (subnormal and overflowing results included), NaN passed through.
PSK_HD float exp_fast(float x) {
  const float xc = fminf(fmaxf(x, -104.5f), 89.0f);
  const float kf = rintf(xc * PSK_FEXP_INV_LN2);
  float r = fmaf(-kf, PSK_FEXP_LN2_HI, xc);
  r = fmaf(-kf, PSK_FEXP_LN2_LO, r);
  float p = 1.0f / 5040.0f;
  p = fmaf(p, r, 1.0f / 720.0f);
  p = fmaf(p, r, 1.0f / 120.0f);
  p = fmaf(p, r, 1.0f / 24.0f);
  p = fmaf(p, r, 1.0f / 6.0f);
  p = fmaf(p, r, 0.5f);
  p = fmaf(p, r, 1.0f);
  p = fmaf(p, r, 1.0f);
  const int k = (int)kf;                           // -151 .. 128
  const int k1 = k >> 1, k2 = k - k1;              // each in [-76, 64]: 2^k1, 2^k2 normal
  const float y = (p * u2f((uint32_t)(k1 + 127) << 23)) * u2f((uint32_t)(k2 + 127) << 23);
  return x == x ? y : x;
}

// erf of a = |x| from the correctly rounded erf's Taylor tables (their
// binary32 coefficients, the pairs' high parts) by plain binary32 Horner of
// degree DF (4 is enough for two ulp: the higher terms stay below 2^-30 of
// erf on an interval of width 1/32; measured over every float of [0, 5]); a
// past PSK_ERF_ONE_FROM gives 1.  p2 / h as for erf_tier1_core.
constexpr int ERF_FAST_DEGREE = 4;
template <int DF = ERF_FAST_DEGREE>
PSK_HD float erf_fast_abs(float a, const float* p2, const float* h) {
  const float ac = fminf(a, 3.9f);
  const float fi = rintf(ac * 32.0f);
  const int i = (int)fi;
  const float t = fmaf(fi, -0.03125f, ac);         // exact
  float H = h[(DF - PSK_ERF_NPAIR) * PSK_ERF_N32 + i];
#pragma unroll
  for (int k = DF - 1; k >= PSK_ERF_NPAIR; --k) H = fmaf(H, t, h[(k - PSK_ERF_NPAIR) * PSK_ERF_N32 + i]);
#pragma unroll
  for (int k = PSK_ERF_NPAIR - 1; k >= 0; --k) H = fmaf(H, t, p2[k * 2 * PSK_ERF_N32 + 2 * i]);
  return a >= PSK_ERF_ONE_FROM ? 1.0f : H;
}

// erf_fast_abs from the record tables (the same operations on the same
// coefficients: the same result): coefficient 4 and the high parts of 3..0.
PSK_HD float erf_fast_abs_rec(float a, const float* rec) {
  static_assert(ERF_FAST_DEGREE == 4, "erf record layout");
  const float ac = fminf(a, 3.9f);
  const float fi = rintf(ac * 32.0f);
  const int i = (int)fi;
  const float t = fmaf(fi, -0.03125f, ac);         // exact
  float c[12];
  load_record12(rec, i, c);
  float H = c[3];
  H = fmaf(H, t, c[4]);
  H = fmaf(H, t, c[6]);
  H = fmaf(H, t, c[8]);
  H = fmaf(H, t, c[10]);
  return a >= PSK_ERF_ONE_FROM ? 1.0f : H;
}


}  // namespace psk
