// Row-region arithmetic shared by the row kernels (regions.cu) and the
// lane-per-row softmax kernel (lanes.cu): the launch parameters, the exact
// NaN-propagating max, the region's exp (correctly rounded or fast) and
// the row division e / s, so that every kernel computing a softmax row does
// the same operations on the same values and gives the same bits.
#pragma once

#include "common.cuh"
#include "crmath.cuh"
#include "pair.cuh"

namespace psk {

constexpr int SM_THREADS = 256;
constexpr int SM_EPT = 16;                      // row elements per thread when resident
constexpr int SM_CAP = SM_THREADS * SM_EPT;     // 4096
constexpr int SM_MAX_PARTIALS = 64;

// Region kinds of the row kernels.
enum : int { REGION_SOFTMAX = 0, REGION_RMS = 1, REGION_LAYER = 2, REGION_SOFTMAX_BWD = 3 };

struct RegionParams {
  const void* x;
  void* y;
  int64_t rows, cols, ldx, ldy;
  int32_t partials;     // 1 for sequential / blocked
  int32_t nb;           // rows per batch (resident kernel) / per chain group (pipelined)
  int32_t estride;      // floats between row buffers in shared memory
  int32_t sx, se;       // pipelined kernel: x and value ring slots
  // normalization regions
  const void* gamma;    // scale per column, NULL if none
  const void* beta;     // bias per column (LayerNorm), NULL if none
  int32_t param_dtype;  // storage type of gamma and beta
  float eps;            // RN_f32 of the eps argument
  // masked softmax
  const uint8_t* mask;  // 0 refuses, nonzero allows; NULL if none
  int64_t ldm;          // mask row stride (0: one mask row for every row)
  // softmax backward (x is y)
  const void* ct;       // cotangent rows
  int64_t ldc;
  int32_t ct_dtype;
};

// NaN-propagating max (exact; the order of a max reduction changes no bit
// except the sign of a zero maximum, which no exp(x - m) can see).
__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// The same on a pair of bf16 values (exact: the max of widened bf16 values
// is a bf16 value).
__device__ __forceinline__ uint32_t bf16x2_max_nan(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

template <int EXPM>
__device__ __forceinline__ float region_exp(float d) {
  if (EXPM == PSK_EXP_FAST) return exp_unit_nonpos(d);
  return exp_cr(d, psk_exp_tab2);
}

// exp of eight values: the correctly rounded tier-1 cores run side by side
// (independent chains for the scheduler), the rare undecided lanes after.
// tab2: the 2^(j/1024) pair table (psk_exp_tab2 or its copy in shared
// memory: the lookups' indices differ per lane, and a shared-memory load of
// 32 random pairs takes a few bank wavefronts where the global table's takes
// one L1 wavefront per distinct 128-byte line, about 25).
template <int EXPM>
__device__ __forceinline__ void region_exp8(float* v, const float* tab2 = psk_exp_tab2) {
  if constexpr (EXPM == PSK_EXP_FAST) {
#pragma unroll
    for (int q = 0; q < 8; ++q) v[q] = exp_unit_nonpos(v[q]);
  } else {
    float R[8], d[8];
    int n[8];
    bool ok[8];
    bool all = true;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const bool inr = fabsf(v[q]) <= 87.0f;
      exp_tier1_core(inr ? v[q] : 0.0f, tab2, R[q], d[q], n[q]);
      ok[q] = inr && tier1_decided(R[q], d[q]);
      all = all && ok[q];
    }
    float out[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) out[q] = u2f((uint32_t)((int32_t)f2u(R[q]) + n[q] * (1 << 23)));
    if (!all) {   // one branch for the eight; the undecided elements
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (!ok[q]) out[q] = exp_tier2(v[q]);
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) v[q] = out[q];
  }
}

// e / s for one row: Markstein's correction through rs = RN(1/s) when the row
// sum allows it (1 <= s < 2^20, true of every finite row), IEEE division for
// the rare tiny e and for rows with a NaN or infinite sum.
__device__ __forceinline__ float row_div(float e, float s, float rs, bool fast_ok) {
  float q = e * rs;
  float r = fmaf(-q, s, e);
  float y = fmaf(r, rs, q);
  if (!(fast_ok && e >= 0x1p-100f)) y = __fdiv_rn(e, s);
  return y;
}

// N quotients e_q / s at once: Markstein's correction for all, one test for
// the whole group, and the per-element path (IEEE division where the
// correction's operand range is left) only for a group that needs it.  The
// dividends are exp values (>= +0): +0, a masked position's, gives +0 through
// the correction as well.
template <int N>
__device__ __forceinline__ void row_div_n(float* o, float s, float rs, bool fast_ok) {
  float y[N];
  bool bad = !fast_ok;
#pragma unroll
  for (int q = 0; q < N; ++q) {
    const float e = o[q];
    const float qq = e * rs;
    const float r = fmaf(-qq, s, e);
    y[q] = fmaf(r, rs, qq);
    bad = bad || !(e >= 0x1p-100f || e == 0.0f);
  }
  if (bad) {
#pragma unroll
    for (int q = 0; q < N; ++q) y[q] = row_div(o[q], s, rs, fast_ok);
  }
#pragma unroll
  for (int q = 0; q < N; ++q) o[q] = y[q];
}

// Division by a row's divisor d > 0 of any magnitude (the norms' sqrt):
// d = dd 2^-k with dd in [1, 2); a / d = (a 2^k) / dd exactly, and for
// 2^-100 <= |a 2^k| <= 2^100 Markstein's correction through RN(1/dd) gives the
// IEEE quotient; a zero dividend gives itself (+-0 / d = +-0 for d > 0; the
// correction would turn -0 into +0); other operands, and rows whose d is not
// a normal number below 2^127, take IEEE division.
struct RowDivisor {
  float d, dd, rdd, scale;
  bool ok;
};

__device__ __forceinline__ RowDivisor make_divisor(float d) {
  RowDivisor r;
  r.d = d;
  const uint32_t b = __float_as_uint(d);
  const int e = (int)((b >> 23) & 0xFFu) - 127;
  r.ok = d > 0.0f && e >= -126 && e <= 126;
  r.dd = __uint_as_float((b & 0x007FFFFFu) | 0x3F800000u);
  r.scale = __uint_as_float((uint32_t)(r.ok ? 127 - e : 127) << 23);
  r.rdd = __frcp_rn(r.dd);
  return r;
}

template <int N>
__device__ __forceinline__ void divide_n(float* o, const RowDivisor& D) {
  float y[N];
  bool bad = !D.ok;
#pragma unroll
  for (int q = 0; q < N; ++q) {
    const float a = __fmul_rn(o[q], D.scale);
    const float qq = a * D.rdd;
    const float r = fmaf(-qq, D.dd, a);
    y[q] = fmaf(r, D.rdd, qq);
    const float aa = fabsf(a);
    if (aa == 0.0f) y[q] = a;
    bad = bad || !((aa >= 0x1p-100f && aa <= 0x1p100f) || aa == 0.0f);
  }
  if (bad) {
#pragma unroll
    for (int q = 0; q < N; ++q) y[q] = __fdiv_rn(o[q], D.d);
  }
#pragma unroll
  for (int q = 0; q < N; ++q) o[q] = y[q];
}

// Launch the lane-per-row kernel (lanes.cu) for rows it takes: bf16 x and y,
// 16-byte aligned rows of 64 to 4096 columns (a multiple of 8), enough rows
// to fill the GPU, the one-chain orders (sequential, blocked); for the softmax
// its fast realization; for the norms kind REGION_RMS or REGION_LAYER; the
// softmax backward with bf16 y, ct and dx.
// *taken is false, and nothing is launched, for other rows.
int softmax_lanes(const RegionParams& P, int exp_mode, cudaStream_t stream, bool* taken);
int norm_lanes(const RegionParams& P, int kind, cudaStream_t stream, bool* taken);
int softmax_bwd_lanes(const RegionParams& P, cudaStream_t stream, bool* taken);
// The lane kernel's status word (read, then zeroed if `reset`) and its copy
// of the lost-copy test hook (lanes.cu keeps its own, like every unit).
int lanes_status(unsigned int* v, bool reset);
int lanes_set_drop_row(long long row);

}  // namespace psk
