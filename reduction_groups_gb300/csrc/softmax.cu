// psk_softmax_region: the reduction-rooted row region Reduce(Max) -> Sub ->
// Exp -> Reduce(Sum) -> Div over the last axis, in one kernel: the row is
// reduced on chip, then the pointwise epilogue runs in the same kernel (poot
// "Fusion and Planning", Reduction-rooted regions).  Arithmetic is f32 for
// bf16 storage, the sum follows the declared order's bracketing tree (presk
// "Native execution", the realization's order; metrale "The LKB in
// Mathematics", section 2: bit parity is the same bracketing tree):
//   sequential / blocked(w): one chain ((e0 + e1) + e2) + ... in index order;
//   interleaved(P): P chains, chain p over j = p mod P in increasing j, then
//   the P partials added left to right.
//
// One CTA works on one row at a time (grid-stride over rows).  A row of up to
// 4096 columns stays in registers (16 per thread, read with 16-byte vector
// loads); exp(x - m) is computed once, kept in registers for the division and
// staged in shared memory, where the chain threads add it in the declared
// order.  Longer rows stream through in chunks of 4096: a max pass, a sum
// pass (the chain threads carry their sums from chunk to chunk) and an
// output pass that recomputes exp (deterministic, so the same bits).

#include "common.cuh"
#include "crmath.cuh"

namespace psk {

constexpr int SM_THREADS = 256;
constexpr int SM_EPT = 16;                      // row elements per thread when resident
constexpr int SM_CAP = SM_THREADS * SM_EPT;     // 4096
constexpr int SM_MAX_PARTIALS = 64;

struct SoftmaxParams {
  const void* x;
  void* y;
  int64_t rows, cols, ldx, ldy;
  int32_t order_kind, partials;   // partials: 1 for sequential / blocked
};

// NaN-propagating max (exact; the order of a max reduction changes no bit
// except the sign of a zero maximum, which no exp(x - m) can see).
__device__ __forceinline__ float max_nan(float a, float b) { return (a > b || a != a) ? a : b; }

template <int XT>
__device__ __forceinline__ float load_x1(const void* base, int64_t off) {
  if (XT == PSK_F32) return __ldg((const float*)base + off);
  return bf16_bits_to_f32(__ldg((const uint16_t*)base + off));
}

template <int XT>
__device__ __forceinline__ void load_x8(const void* base, int64_t off, float* v) {
  if (XT == PSK_F32) {
    const float4* p = (const float4*)((const float*)base + off);
    float4 a = __ldg(p), b = __ldg(p + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else {
    uint4 q = __ldg((const uint4*)((const uint16_t*)base + off));
    uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
}

template <int YT>
__device__ __forceinline__ void store_y1(void* base, int64_t off, float v) {
  if (YT == PSK_F32) ((float*)base)[off] = v;
  else ((uint16_t*)base)[off] = f32_to_bf16_bits(v);
}

template <int YT>
__device__ __forceinline__ void store_y8(void* base, int64_t off, const float* v) {
  if (YT == PSK_F32) {
    float4* p = (float4*)((float*)base + off);
    p[0] = make_float4(v[0], v[1], v[2], v[3]);
    p[1] = make_float4(v[4], v[5], v[6], v[7]);
  } else {
    uint4 q;
    q.x = f32x2_to_bf16x2(v[0], v[1]);
    q.y = f32x2_to_bf16x2(v[2], v[3]);
    q.z = f32x2_to_bf16x2(v[4], v[5]);
    q.w = f32x2_to_bf16x2(v[6], v[7]);
    *(uint4*)((uint16_t*)base + off) = q;
  }
}

template <int EXPM>
__device__ __forceinline__ float region_exp(float d, const float* thi, const float* tlo) {
  if (EXPM == PSK_EXP_FAST) return exp_faithful(d);
  return exp_cr(d, thi, tlo);
}

struct SoftmaxShared {
  float E[SM_CAP];                 // exp(x - m) of the row (or chunk), index order
  float exp_hi[32], exp_lo[32];
  float red[SM_THREADS / 32];
  float part[SM_MAX_PARTIALS];
  float bcast;
};

__device__ __forceinline__ float block_max(float v, SoftmaxShared& sh) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max_nan(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) sh.red[w] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = sh.red[0];
    for (int i = 1; i < SM_THREADS / 32; ++i) m = max_nan(m, sh.red[i]);
    sh.bcast = m;
  }
  __syncthreads();
  float m = sh.bcast;
  __syncthreads();
  return m;
}

// Chain threads add E[0..n) into their running sums in the declared order.
// Global index of E[i] is base + i; chain p owns indices j = p (mod P).
__device__ __forceinline__ void chain_add(const SoftmaxShared& sh, int n, int64_t base, int P, float& acc, bool& started) {
  const int p = threadIdx.x;
  if (p >= P) return;
  int i0 = (int)(((int64_t)p - base) % P);
  if (i0 < 0) i0 += P;
  int i = i0;
  if (!started && i < n) { acc = sh.E[i]; started = true; i += P; }
  if (P == 1) {
    // one chain: read four at a time (16-byte aligned), add in order
    for (; (i & 3) != 0 && i < n; ++i) acc = __fadd_rn(acc, sh.E[i]);
    for (; i + 3 < n; i += 4) {
      float4 q = *reinterpret_cast<const float4*>(&sh.E[i]);
      acc = __fadd_rn(acc, q.x); acc = __fadd_rn(acc, q.y); acc = __fadd_rn(acc, q.z); acc = __fadd_rn(acc, q.w);
    }
  }
  for (; i < n; i += P) acc = __fadd_rn(acc, sh.E[i]);
}

__device__ __forceinline__ float combine_partials(SoftmaxShared& sh, int P, float acc) {
  if ((int)threadIdx.x < P) sh.part[threadIdx.x] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = sh.part[0];
    for (int p = 1; p < P; ++p) s = __fadd_rn(s, sh.part[p]);
    sh.bcast = s;
  }
  __syncthreads();
  float s = sh.bcast;
  __syncthreads();
  return s;
}

template <int XT, int YT, int EXPM, bool VEC>
__global__ void __launch_bounds__(SM_THREADS) softmax_kernel(const __grid_constant__ SoftmaxParams P) {
  __shared__ __align__(16) SoftmaxShared sh;
  const int t = threadIdx.x;
  if (EXPM == PSK_EXP_EXACT) {
    if (t < 32) { sh.exp_hi[t] = psk_exp_tab_hi[t]; sh.exp_lo[t] = psk_exp_tab_lo[t]; }
    __syncthreads();
  }
  const int64_t cols = P.cols;
  const int parts = P.partials;
  const int nP = (int)(cols < parts ? cols : parts);   // chains that have elements

  for (int64_t row = blockIdx.x; row < P.rows; row += gridDim.x) {
    const void* xr = (const void*)((const char*)P.x + row * P.ldx * (XT == PSK_F32 ? 4 : 2));
    void* yr = (void*)((char*)P.y + row * P.ldy * (YT == PSK_F32 ? 4 : 2));
    if (cols <= SM_CAP) {
      // ---------------- resident row: x and e in registers
      float v[SM_EPT];
      float m = -INFINITY;
      if (VEC) {
#pragma unroll
        for (int k = 0; k < SM_EPT / 8; ++k) {
          int64_t j = ((int64_t)k * SM_THREADS + t) * 8;
          if (j < cols) load_x8<XT>(xr, j, v + 8 * k);
          else {
#pragma unroll
            for (int q = 0; q < 8; ++q) v[8 * k + q] = -INFINITY;
          }
        }
      } else {
#pragma unroll
        for (int k = 0; k < SM_EPT; ++k) {
          int64_t j = (int64_t)k * SM_THREADS + t;
          v[k] = j < cols ? load_x1<XT>(xr, j) : -INFINITY;
        }
      }
#pragma unroll
      for (int k = 0; k < SM_EPT; ++k) m = max_nan(m, v[k]);
      m = block_max(m, sh);
#pragma unroll
      for (int k = 0; k < SM_EPT; ++k) {
        int64_t j = VEC ? ((int64_t)(k / 8) * SM_THREADS + t) * 8 + (k % 8) : (int64_t)k * SM_THREADS + t;
        if (j < cols) {
          v[k] = region_exp<EXPM>(__fsub_rn(v[k], m), sh.exp_hi, sh.exp_lo);
          sh.E[j] = v[k];
        }
      }
      __syncthreads();
      float acc = 0.0f;
      bool started = false;
      chain_add(sh, (int)cols, 0, nP, acc, started);
      float s = combine_partials(sh, nP, acc);
      if (VEC) {
#pragma unroll
        for (int k = 0; k < SM_EPT / 8; ++k) {
          int64_t j = ((int64_t)k * SM_THREADS + t) * 8;
          if (j < cols) {
            float o[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) o[q] = __fdiv_rn(v[8 * k + q], s);
            store_y8<YT>(yr, j, o);
          }
        }
      } else {
#pragma unroll
        for (int k = 0; k < SM_EPT; ++k) {
          int64_t j = (int64_t)k * SM_THREADS + t;
          if (j < cols) store_y1<YT>(yr, j, __fdiv_rn(v[k], s));
        }
      }
    } else {
      // ---------------- streaming row: chunks of SM_CAP columns
      float m = -INFINITY;
      for (int64_t j = t; j < cols; j += SM_THREADS) m = max_nan(m, load_x1<XT>(xr, j));
      m = block_max(m, sh);
      float acc = 0.0f;
      bool started = false;
      for (int64_t base = 0; base < cols; base += SM_CAP) {
        int n = (int)((cols - base) < SM_CAP ? (cols - base) : SM_CAP);
        for (int i = t; i < n; i += SM_THREADS)
          sh.E[i] = region_exp<EXPM>(__fsub_rn(load_x1<XT>(xr, base + i), m), sh.exp_hi, sh.exp_lo);
        __syncthreads();
        chain_add(sh, n, base, nP, acc, started);
        __syncthreads();
      }
      float s = combine_partials(sh, nP, acc);
      for (int64_t j = t; j < cols; j += SM_THREADS) {
        float e = region_exp<EXPM>(__fsub_rn(load_x1<XT>(xr, j), m), sh.exp_hi, sh.exp_lo);
        store_y1<YT>(yr, j, __fdiv_rn(e, s));
      }
    }
    __syncthreads();
  }
}

template <int XT, int YT, int EXPM, bool VEC>
static int launch_softmax(const SoftmaxParams& P, cudaStream_t stream) {
  int dev = 0, sms = 1, per_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, softmax_kernel<XT, YT, EXPM, VEC>, SM_THREADS, 0);
  if (per_sm < 1) per_sm = 1;
  int64_t cap = (int64_t)sms * per_sm;
  unsigned grid = (unsigned)(P.rows < cap ? P.rows : cap);
  softmax_kernel<XT, YT, EXPM, VEC><<<grid, SM_THREADS, 0, stream>>>(P);
  return check_launch("softmax region kernel");
}

template <int XT, int YT>
static int dispatch_softmax(const SoftmaxParams& P, int exp_mode, bool vec, cudaStream_t s) {
  if (exp_mode == PSK_EXP_EXACT)
    return vec ? launch_softmax<XT, YT, PSK_EXP_EXACT, true>(P, s) : launch_softmax<XT, YT, PSK_EXP_EXACT, false>(P, s);
  return vec ? launch_softmax<XT, YT, PSK_EXP_FAST, true>(P, s) : launch_softmax<XT, YT, PSK_EXP_FAST, false>(P, s);
}

}  // namespace psk

using namespace psk;

extern "C" int psk_softmax_region(const void* x, int32_t xt, void* y, int32_t yt, int64_t rows, int64_t cols,
                                  int64_t ldx, int64_t ldy, psk_order order, int32_t exp_mode, void* stream) {
  clear_error();
  if (!dtype_ok(xt)) return fail(PSK_E_DTYPE, "x dtype %d", xt);
  if (!dtype_ok(yt)) return fail(PSK_E_DTYPE, "y dtype %d", yt);
  if (rows < 0 || cols < 0) return fail(PSK_E_SHAPE, "rows %lld, cols %lld", (long long)rows, (long long)cols);
  if (exp_mode != PSK_EXP_EXACT && exp_mode != PSK_EXP_FAST) return fail(PSK_E_ARG, "exp_mode %d", exp_mode);
  int partials = 1;
  switch (order.kind) {
    case PSK_ORDER_SEQUENTIAL: break;
    case PSK_ORDER_BLOCKED:
      if (order.param < 1) return fail(PSK_E_ORDER, "blocked width %d < 1", order.param);
      break;
    case PSK_ORDER_INTERLEAVED:
      if (order.param < 1 || order.param > SM_MAX_PARTIALS)
        return fail(PSK_E_ORDER, "interleaved partials %d (1..%d)", order.param, SM_MAX_PARTIALS);
      partials = order.param;
      break;
    default:
      return fail(PSK_E_ORDER, "order kind %d", order.kind);
  }
  if (rows == 0 || cols == 0) return PSK_OK;
  if (!x || !y) return fail(PSK_E_NULL, "x or y is NULL");
  if (ldx < cols || ldy < cols) return fail(PSK_E_SHAPE, "leading dimension below cols");
  // overlap: only the exact in-place form is allowed
  const char* xlo = (const char*)x;
  const char* xhi = xlo + ((rows - 1) * ldx + cols) * dtype_size(xt);
  const char* ylo = (const char*)y;
  const char* yhi = ylo + ((rows - 1) * ldy + cols) * dtype_size(yt);
  if (xlo < yhi && ylo < xhi && !(x == y && xt == yt && ldx == ldy))
    return fail(PSK_E_ALIAS, "y overlaps x and is not the same buffer");
  SoftmaxParams P{x, y, rows, cols, ldx, ldy, order.kind, partials};
  bool vec = (cols % 8 == 0) && (ldx % 8 == 0) && (ldy % 8 == 0) && ((uintptr_t)x % 16 == 0) &&
             ((uintptr_t)y % 16 == 0) && cols <= SM_CAP;
  cudaStream_t s = (cudaStream_t)stream;
  if (xt == PSK_BF16 && yt == PSK_BF16) return dispatch_softmax<PSK_BF16, PSK_BF16>(P, exp_mode, vec, s);
  if (xt == PSK_BF16 && yt == PSK_F32) return dispatch_softmax<PSK_BF16, PSK_F32>(P, exp_mode, vec, s);
  if (xt == PSK_F32 && yt == PSK_BF16) return dispatch_softmax<PSK_F32, PSK_BF16>(P, exp_mode, vec, s);
  return dispatch_softmax<PSK_F32, PSK_F32>(P, exp_mode, vec, s);
}
