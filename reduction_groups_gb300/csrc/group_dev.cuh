// Device side of a fusion group (PSK-Realize, "What a group is"): the kernel
// parameter block and the pieces every specialised group kernel is built
// from -- coordinates of a vector of V output elements, input loads, the node
// operations, the root's store.  The host generates, per program, a kernel
// that calls these pieces in the program's node order and compiles it at run
// time; this header is part of that kernel's source (no host headers).
#pragma once

#include "../../include/psk.h"
#include "devcommon.cuh"
#include "crmath.cuh"
#include "pair.cuh"

namespace psk {

constexpr int GROUP_THREADS = 128;

// How an input walks the last (collapsed) output axis.
enum : int32_t { IN_CONTIG = 0, IN_BCAST = 1, IN_GATHER = 2 };

struct GroupInput {
  const void* ptr;
  int64_t stride[4];   // elements per step of each collapsed output axis
  int32_t dtype;
  int32_t mode;
};

// The launch parameter (a __grid_constant__ block in the constant bank).
struct GroupParams {
  GroupInput in[PSK_MAX_INPUTS];
  float imm[PSK_MAX_IMM];
  void* out;
  uint32_t rank;            // collapsed rank, 1..4 (axes padded at the front)
  uint32_t dim[4];          // collapsed dims (dim[3] = last axis)
  FastDiv div_cv;           // vectors per row: dim[3] / V
  FastDiv div2, div1;       // dim[2], dim[1]
  uint64_t v_begin;         // first vector of this launch
  uint32_t n_vec;           // vectors in this launch
};

// exp and erf tables staged once per CTA in shared memory.
struct MathTables {
  float2 exp_tab[PSK_EXP_TAB_N];   // 2^(j/1024) as (hi, lo)
  float4 erf_rec[3 * PSK_ERF_N32];  // erf's Taylor coefficients, one 48-byte record per interval (erf_record)
};

__device__ __forceinline__ void load_tables(MathTables& t) {
  const float2* src = reinterpret_cast<const float2*>(psk_exp_tab2);
  for (int i = threadIdx.x; i < PSK_EXP_TAB_N; i += blockDim.x) t.exp_tab[i] = src[i];
  for (int i = threadIdx.x; i < PSK_ERF_N32; i += blockDim.x)
    erf_record(&psk_erf_p2[0][0], &psk_erf_h[0][0], i, reinterpret_cast<float*>(&t.erf_rec[3 * i]));
}

// log and tanh tables, staged per CTA only by kernels with such nodes.
struct LogTables {
  float4 tab[512];                                             // (c, T hi, T lo, s) per interval
};
struct TanhTables {
  float2 p2[PSK_ERF_NPAIR * PSK_TANH_N32];                     // coefficients 0..3 as (hi, lo)
  float h[(PSK_TANH_D32 + 1 - PSK_ERF_NPAIR) * PSK_TANH_N32];  // coefficients 4..D
};

__device__ __forceinline__ void load_log_tables(LogTables& t) {
  const float4* src = reinterpret_cast<const float4*>(psk_log_tab);
  for (int i = threadIdx.x; i < 512; i += blockDim.x) t.tab[i] = src[i];
}

__device__ __forceinline__ void load_tanh_tables(TanhTables& t) {
  const float2* p2 = reinterpret_cast<const float2*>(&psk_tanh_p2[0][0]);
  for (int i = threadIdx.x; i < PSK_ERF_NPAIR * PSK_TANH_N32; i += blockDim.x) t.p2[i] = p2[i];
  for (int i = threadIdx.x; i < (PSK_TANH_D32 + 1 - PSK_ERF_NPAIR) * PSK_TANH_N32; i += blockDim.x)
    t.h[i] = (&psk_tanh_h[0][0])[i];
}

template <int V> struct Vec { float v[V]; };

// The EXP-clamp node's min(max(a, -4), 4) with the group's selects
// (max(a, b) = a > b ? a : b): fmaxf / fminf give the same value for every a
// (a NaN gives -4 either way; the bounds are not zeros), in one min / max
// instruction each.
__device__ __forceinline__ float clamp_pm4(float a) { return fminf(fmaxf(a, -4.0f), 4.0f); }

template <int V>
__device__ __forceinline__ Vec<V> splat(float q) {
  Vec<V> r;
#pragma unroll
  for (int j = 0; j < V; ++j) r.v[j] = q;
  return r;
}

// Output vector v -> coordinates (i0, i1, i2, i3) of its first element in the
// collapsed output (i3 along the last axis).
template <int V>
__device__ __forceinline__ void vec_coords(const GroupParams& P, uint64_t v, uint32_t& i0, uint32_t& i1, uint32_t& i2,
                                           uint32_t& i3) {
  const uint32_t vlo = (uint32_t)v;   // a call never indexes past 2^32 vectors
  const uint32_t row = P.div_cv.div(vlo);
  i3 = (vlo - row * (P.dim[3] / V)) * V;
  i2 = row;
  i1 = 0;
  i0 = 0;
  if (P.rank > 2) {
    const uint32_t q2 = P.div2.div(row);
    i2 = row - q2 * P.dim[2];
    if (P.rank > 3) {
      const uint32_t q1 = P.div1.div(q2);
      i1 = q2 - q1 * P.dim[1];
      i0 = q1;
    } else {
      i1 = q2;
    }
  }
}

// Input k at the vector's coordinates: contiguous inputs load 16 B (f32,
// i32) or 8 B (bf16) at once, broadcast ones one element, the rest gather.
// An i32 input (a SELECT condition) keeps its bits in the value's register.
template <int V, int DT, int MODE>
__device__ __forceinline__ Vec<V> load_in(const GroupInput& in, uint32_t i0, uint32_t i1, uint32_t i2, uint32_t i3) {
  const int64_t off = (int64_t)i0 * in.stride[0] + (int64_t)i1 * in.stride[1] + (int64_t)i2 * in.stride[2] +
                      (int64_t)i3 * in.stride[3];
  Vec<V> r;
  if (DT == PSK_I32) {
    const uint32_t* p = (const uint32_t*)in.ptr + off;
    if (V == 4 && MODE == IN_CONTIG) {
      const uint4 q = __ldg((const uint4*)p);
      r.v[0] = __uint_as_float(q.x); r.v[1 % V] = __uint_as_float(q.y);
      r.v[2 % V] = __uint_as_float(q.z); r.v[3 % V] = __uint_as_float(q.w);
    } else if (MODE == IN_BCAST) {
      r = splat<V>(__uint_as_float(__ldg(p)));
    } else {
#pragma unroll
      for (int j = 0; j < V; ++j) r.v[j] = __uint_as_float(__ldg(p + j * in.stride[3]));
    }
  } else if (DT == PSK_F32) {
    const float* p = (const float*)in.ptr + off;
    if (V == 4 && MODE == IN_CONTIG) {
      const float4 q = __ldg((const float4*)p);
      r.v[0] = q.x; r.v[1 % V] = q.y; r.v[2 % V] = q.z; r.v[3 % V] = q.w;
    } else if (MODE == IN_BCAST) {
      r = splat<V>(__ldg(p));
    } else {
#pragma unroll
      for (int j = 0; j < V; ++j) r.v[j] = __ldg(p + j * in.stride[3]);
    }
  } else {
    const uint16_t* p = (const uint16_t*)in.ptr + off;
    if (V == 4 && MODE == IN_CONTIG) {
      const uint2 q = __ldg((const uint2*)p);
      r.v[0] = __uint_as_float(q.x << 16);
      r.v[1 % V] = __uint_as_float(q.x & 0xFFFF0000u);
      r.v[2 % V] = __uint_as_float(q.y << 16);
      r.v[3 % V] = __uint_as_float(q.y & 0xFFFF0000u);
    } else if (MODE == IN_BCAST) {
      r = splat<V>(bf16_bits_to_f32(__ldg(p)));
    } else {
#pragma unroll
      for (int j = 0; j < V; ++j) r.v[j] = bf16_bits_to_f32(__ldg(p + j * in.stride[3]));
    }
  }
  return r;
}

// ------------------------------------------------------------- node ops
// Binary nodes: IEEE binary32, one rounding; max(a, b) = a > b ? a : b and
// min(a, b) = a < b ? a : b (a tie, and NaN, give the second operand).
#define PSK_NODE2(NAME, EXPR)                                                        \
  template <int V>                                                                   \
  __device__ __forceinline__ Vec<V> NAME(const Vec<V>& A, const Vec<V>& B) {         \
    Vec<V> r;                                                                        \
    _Pragma("unroll") for (int j = 0; j < V; ++j) {                                  \
      const float a = A.v[j], b = B.v[j];                                            \
      r.v[j] = (EXPR);                                                               \
    }                                                                                \
    return r;                                                                        \
  }
PSK_NODE2(node_add, __fadd_rn(a, b))
PSK_NODE2(node_sub, __fsub_rn(a, b))
PSK_NODE2(node_mul, __fmul_rn(a, b))
PSK_NODE2(node_div, __fdiv_rn(a, b))
PSK_NODE2(node_max, a > b ? a : b)
PSK_NODE2(node_min, a < b ? a : b)
#undef PSK_NODE2

#define PSK_NODE1(NAME, EXPR)                                                        \
  template <int V>                                                                   \
  __device__ __forceinline__ Vec<V> NAME(const Vec<V>& A) {                          \
    Vec<V> r;                                                                        \
    _Pragma("unroll") for (int j = 0; j < V; ++j) {                                  \
      const float a = A.v[j];                                                        \
      r.v[j] = (EXPR);                                                               \
    }                                                                                \
    return r;                                                                        \
  }
PSK_NODE1(node_neg, -a)
PSK_NODE1(node_abs, fabsf(a))
PSK_NODE1(node_sqrt, __fsqrt_rn(a))
PSK_NODE1(node_sqrta, __fsqrt_rn(fabsf(a)))
PSK_NODE1(node_recip, __frcp_rn(a))
#undef PSK_NODE1

// SELECT: C holds the condition's i32 bits; the picked operand is moved as is.
template <int V>
__device__ __forceinline__ Vec<V> node_select(const Vec<V>& C, const Vec<V>& A, const Vec<V>& B) {
  Vec<V> r;
#pragma unroll
  for (int j = 0; j < V; ++j) r.v[j] = __float_as_uint(C.v[j]) != 0u ? A.v[j] : B.v[j];
  return r;
}

// exp, exp(clamp(a, -4, 4)), erf and gelu: one out-of-line copy each, called
// by every such node (the kernel's code stays small enough for the
// instruction cache).  The tier-1 cores of the V elements run side by side
// (independent chains for the scheduler); one branch per call sends the
// undecided elements on to the slower tiers.
// The exp-clamp node at a clamp bound takes the correctly rounded constant
// (RN(e^4) = 0x1.b4c902p+5, RN(e^-4) = 0x1.2c155cp-6), and a warp whose
// every argument sits at a bound skips tier 1.
constexpr float PSK_EXP_P4 = 0x1.b4c902p+5f;
constexpr float PSK_EXP_M4 = 0x1.2c155cp-6f;
template <int V, bool CLAMP>
__device__ __noinline__ Vec<V> node_exp_any(Vec<V> A, const MathTables& tab) {
  float a[V], R[V], d[V];
  int n[V];
  bool ok[V], bnd[V];
  bool any = !CLAMP;
#pragma unroll
  for (int j = 0; j < V; ++j) {
    a[j] = A.v[j];
    if (CLAMP) {
      a[j] = clamp_pm4(a[j]);                         // NaN clamps to -4
    }
    bnd[j] = CLAMP && fabsf(a[j]) == 4.0f;
    any = any || !bnd[j];
    R[j] = 1.0f;
    d[j] = 0.0f;
    n[j] = 0;
  }
  bool all = true;
  if (!CLAMP || __any_sync(__activemask(), any)) {
#pragma unroll
    for (int j = 0; j < V; ++j) {
      const bool inr = CLAMP || fabsf(a[j]) <= 87.0f;   // a clamped argument is in range
      exp_tier1_core(inr ? a[j] : 0.0f, reinterpret_cast<const float*>(tab.exp_tab), R[j], d[j], n[j]);
      ok[j] = (inr && tier1_decided(R[j], d[j])) || bnd[j];
      all = all && ok[j];
    }
  }
  Vec<V> r;
#pragma unroll
  for (int j = 0; j < V; ++j) {
    r.v[j] = u2f((uint32_t)((int32_t)f2u(R[j]) + n[j] * (1 << 23)));
    if (bnd[j]) r.v[j] = a[j] > 0.0f ? PSK_EXP_P4 : PSK_EXP_M4;
  }
  if (!all) {   // one branch per call; the elements tier 1 left undecided
#pragma unroll
    for (int j = 0; j < V; ++j)
      if (!ok[j]) r.v[j] = exp_tier2(a[j]);
  }
  return r;
}

// gelu(a) = a * (0.5 * (1 + erf(a * RN(1/sqrt 2)))), every step rounded.
// Where |t| >= PSK_ERF_ONE_FROM (infinities included) erf(|t|) rounds to 1:
// taken here, without the slow tiers; a warp none of whose elements is in
// tier 1's range skips tier 1 altogether.
template <int V, bool GELU>
__device__ __noinline__ Vec<V> node_erf_any(Vec<V> A, const MathTables& tab) {
  float tt[V], aa[V], R[V], d[V];
  bool ok[V], inr[V];
  bool any = false;
#pragma unroll
  for (int j = 0; j < V; ++j) {
    tt[j] = GELU ? __fmul_rn(A.v[j], PSK_INV_SQRT2) : A.v[j];
    aa[j] = fabsf(tt[j]);
    inr[j] = aa[j] < PSK_ERF_ONE_FROM && aa[j] >= 0x1p-60f;
    any = any || inr[j];
    R[j] = 1.0f;
    d[j] = 0.0f;
  }
  if (__any_sync(__activemask(), any)) {
#pragma unroll
    for (int j = 0; j < V; ++j)
      erf_tier1_core_rec(inr[j] ? aa[j] : 0.5f, reinterpret_cast<const float*>(tab.erf_rec), R[j], d[j]);
  }
  bool all = true;
#pragma unroll
  for (int j = 0; j < V; ++j) {
    const bool sat = aa[j] >= PSK_ERF_ONE_FROM;               // false for NaN
    ok[j] = (inr[j] && tier1_decided(R[j], d[j])) || sat;
    if (sat) R[j] = 1.0f;
    all = all && ok[j];
  }
  if (!all) {
#pragma unroll
    for (int j = 0; j < V; ++j)
      if (!ok[j]) R[j] = erf_abs_rest(fabsf(tt[j]));
  }
  Vec<V> r;
#pragma unroll
  for (int j = 0; j < V; ++j) {
    const float e = copysignf(R[j], tt[j]);
    r.v[j] = GELU ? __fmul_rn(A.v[j], __fmul_rn(0.5f, __fadd_rn(1.0f, e))) : e;
  }
  return r;
}

// log: tier 1 for positive finite x other than 1 (subnormals scaled by
// 2^24), the rest and undecided elements out of line.
template <int V>
__device__ __noinline__ Vec<V> node_log(Vec<V> A, const LogTables& tab) {
  float R[V], d[V];
  bool ok[V];
  bool all = true;
#pragma unroll
  for (int j = 0; j < V; ++j) {
    const float a = A.v[j];
    const bool inr = a > 0.0f && a < INFINITY && a != 1.0f;
    const bool sub = a < 0x1p-126f;
    log_tier1_core(inr ? (sub ? a * 0x1p24f : a) : 2.0f, (inr && sub) ? -24 : 0,
                   reinterpret_cast<const float*>(tab.tab), R[j], d[j]);
    ok[j] = inr && tier1_decided(R[j], d[j]);
    all = all && ok[j];
  }
  Vec<V> r;
#pragma unroll
  for (int j = 0; j < V; ++j) r.v[j] = R[j];
  if (!all) {
#pragma unroll
    for (int j = 0; j < V; ++j)
      if (!ok[j]) r.v[j] = log_rest(A.v[j]);
  }
  return r;
}

// tanh: tier 1 on 2^-12 <= |a| < PSK_TANH_ONE_FROM, the rest out of line.
template <int V>
__device__ __noinline__ Vec<V> node_tanh(Vec<V> A, const TanhTables& tab) {
  float R[V], d[V];
  bool ok[V];
  bool all = true;
#pragma unroll
  for (int j = 0; j < V; ++j) {
    const float aa = fabsf(A.v[j]);
    const bool inr = aa >= 0x1p-12f && aa < PSK_TANH_ONE_FROM;
    tanh_tier1_core(inr ? aa : 0.5f, reinterpret_cast<const float*>(tab.p2), tab.h, R[j], d[j]);
    ok[j] = inr && tier1_decided(R[j], d[j]);
    all = all && ok[j];
  }
  if (!all) {
#pragma unroll
    for (int j = 0; j < V; ++j)
      if (!ok[j]) R[j] = tanh_abs_rest(fabsf(A.v[j]));
  }
  Vec<V> r;
#pragma unroll
  for (int j = 0; j < V; ++j) r.v[j] = copysignf(R[j], A.v[j]);
  return r;
}

// The fast realization (math mode FAST) of the exp, exp-clamp and erf nodes:
// a faithful exp (at most one ulp) for EXP, the multifunction unit's 2^f
// after an exact split for EXP-clamp (at most two ulp; the clamped argument
// needs no special cases) and a faithful erf (at most two ulp).
// Short enough to inline at every node (1.22 -> 1.11 ms on the 64-node group
// against one out-of-line copy each).
template <int V, bool CLAMP>
__device__ __forceinline__ Vec<V> node_exp_fast_any(Vec<V> A) {
  Vec<V> r;
  if constexpr (CLAMP && V % 2 == 0) {   // two at a time (packed f32x2 arithmetic)
#pragma unroll
    for (int j = 0; j < V; j += 2) {
      float a = A.v[j], b = A.v[j + 1];
      a = clamp_pm4(a);
      b = clamp_pm4(b);
      const f2 e = exp2_unit_mid(f2{a, b});
      r.v[j] = e.x;
      r.v[j + 1] = e.y;
    }
    return r;
  }
#pragma unroll
  for (int j = 0; j < V; ++j) {
    float a = A.v[j];
    if (CLAMP) {
      a = clamp_pm4(a);
      r.v[j] = exp_unit_mid(a);
    } else {
      r.v[j] = exp_fast(a);
    }
  }
  return r;
}

template <int V, bool GELU>
__device__ __forceinline__ Vec<V> node_erf_fast_any(Vec<V> A, const MathTables& tab) {
  Vec<V> r;
#pragma unroll
  for (int j = 0; j < V; ++j) {
    const float t = GELU ? __fmul_rn(A.v[j], PSK_INV_SQRT2) : A.v[j];
    const float aa = fabsf(t);
    float e = erf_fast_abs_rec(aa, reinterpret_cast<const float*>(tab.erf_rec));
    e = t == t ? copysignf(e, t) : t;
    r.v[j] = GELU ? __fmul_rn(A.v[j], __fmul_rn(0.5f, __fadd_rn(1.0f, e))) : e;
  }
  return r;
}

template <int V> __device__ __forceinline__ Vec<V> node_exp_fast(const Vec<V>& a, const MathTables&) { return node_exp_fast_any<V, false>(a); }
template <int V> __device__ __forceinline__ Vec<V> node_expc_fast(const Vec<V>& a, const MathTables&) { return node_exp_fast_any<V, true>(a); }
template <int V> __device__ __forceinline__ Vec<V> node_erf_fast(const Vec<V>& a, const MathTables& t) { return node_erf_fast_any<V, false>(a, t); }
// gelu keeps the correctly rounded erf in the fast mode too: where erf(t) <
// -1/2, 1 + erf(t) is exact and cancels, so one ulp of erf becomes 2^k ulp of
// a result 2^-k below 1, and no approximate erf stays within two ulp of the
// correctly rounded gelu there.
template <int V> __device__ __forceinline__ Vec<V> node_gelu_fast(const Vec<V>& a, const MathTables& t) { return node_erf_any<V, true>(a, t); }

template <int V> __device__ __forceinline__ Vec<V> node_exp(const Vec<V>& a, const MathTables& t) { return node_exp_any<V, false>(a, t); }
template <int V> __device__ __forceinline__ Vec<V> node_expc(const Vec<V>& a, const MathTables& t) { return node_exp_any<V, true>(a, t); }
template <int V> __device__ __forceinline__ Vec<V> node_erf(const Vec<V>& a, const MathTables& t) { return node_erf_any<V, false>(a, t); }
template <int V> __device__ __forceinline__ Vec<V> node_gelu(const Vec<V>& a, const MathTables& t) { return node_erf_any<V, true>(a, t); }

// The root, rounded once to its storage type, row-major.
template <int V, int OUT>
__device__ __forceinline__ void store_root(const GroupParams& P, uint64_t v, const Vec<V>& r) {
  const uint64_t e0 = v * V;
  if (OUT == PSK_F32) {
    float* o = (float*)P.out + e0;
    if (V == 4) *(float4*)o = make_float4(r.v[0], r.v[1 % V], r.v[2 % V], r.v[3 % V]);
    else o[0] = r.v[0];
  } else {
    uint16_t* o = (uint16_t*)P.out + e0;
    if (V == 4) {
      uint2 q;
      q.x = f32x2_to_bf16x2(r.v[0], r.v[1 % V]);
      q.y = f32x2_to_bf16x2(r.v[2 % V], r.v[3 % V]);
      *(uint2*)o = q;
    } else {
      o[0] = f32_to_bf16_bits(r.v[0]);
    }
  }
}

}  // namespace psk
