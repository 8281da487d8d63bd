// psk_softmax_region: the reduction-rooted row region Reduce(Max) -> Sub ->
// Exp -> Reduce(Sum) -> Div over the last axis, in one kernel: the row is
// reduced on chip, then the pointwise epilogue runs in the same kernel (poot
// "Fusion and Planning", Reduction-rooted regions).  Arithmetic is f32 for
// bf16 storage, and the sum follows the declared order's bracketing tree
// (presk "Native execution", the realization's order; metrale "The LKB in
// Mathematics", section 2: bit parity is the same bracketing tree):
//   sequential / blocked(w): one chain ((e0 + e1) + e2) + ... in index order;
//   interleaved(P): P chains, chain p over j = p mod P in increasing j, then
//   the P partials added left to right.
//
// Rows of up to 4096 columns (the resident kernel): a CTA of 256 threads takes
// NB rows at a time (4 for bf16 input, 2 for f32).  Each thread loads 16
// elements of every row with 16-byte loads and keeps them packed in
// registers; the NB row maxima are reduced together (warp shuffles, one
// barrier); e = exp(x - m) goes to a shared-memory buffer per row; then one
// warp runs every chain of the batch at once -- lane (b, p) adds chain p of
// row b, eight loads issued ahead of each eight dependent adds -- and combines
// each row's partials left to right; finally every thread divides its
// elements by the row sum (Markstein's reciprocal correction, bit-identical to
// IEEE division) and stores.  While one CTA's chain warp works, the other
// CTAs on the SM compute, so the chain latency (512 dependent adds per chain
// under interleaved(8), 4096 under sequential) overlaps the streaming work.
// Longer rows stream through a second kernel in chunks of 4096.

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
  int32_t partials;     // 1 for sequential / blocked
  int32_t nb;           // rows per batch (resident kernel)
  int32_t estride;      // floats between row buffers in shared memory
};

// NaN-propagating max (exact; the order of a max reduction changes no bit
// except the sign of a zero maximum, which no exp(x - m) can see).
__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

template <int EXPM>
__device__ __forceinline__ float region_exp(float d, const float* thi, const float* tlo) {
  if (EXPM == PSK_EXP_FAST) return exp_faithful_nonpos(d);
  return exp_cr(d, thi, tlo);
}

// exp of eight values: the correctly rounded tier-1 cores run side by side
// (independent chains for the scheduler), the rare undecided lanes after.
template <int EXPM>
__device__ __forceinline__ void region_exp8(float* v, const float* thi, const float* tlo) {
  if (EXPM == PSK_EXP_FAST) {
#pragma unroll
    for (int q = 0; q < 8; ++q) v[q] = exp_faithful_nonpos(v[q]);
    return;
  }
  float R[8], d[8];
  int n[8];
  bool inr[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    inr[q] = fabsf(v[q]) <= 87.0f;
    exp_tier1_core(inr[q] ? v[q] : 0.0f, thi, tlo, R[q], d[q], n[q]);
  }
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    float out = u2f((uint32_t)((int32_t)f2u(R[q]) + n[q] * (1 << 23)));
    if (!(inr[q] && tier1_decided(R[q], d[q]))) out = exp_tier2(v[q]);
    v[q] = out;
  }
}

template <int XT>
__device__ __forceinline__ float load_x1(const void* base, int64_t off) {
  if (XT == PSK_F32) return __ldg((const float*)base + off);
  return bf16_bits_to_f32(__ldg((const uint16_t*)base + off));
}

template <int YT>
__device__ __forceinline__ void store_y1(void* base, int64_t off, float v) {
  if (YT == PSK_F32) ((float*)base)[off] = v;
  else ((uint16_t*)base)[off] = f32_to_bf16_bits(v);
}

// Raw storage of 8 consecutive elements: bf16 as 4 words, f32 as 8 floats.
template <int XT> struct Raw8;
template <> struct Raw8<PSK_BF16> { uint4 w; };
template <> struct Raw8<PSK_F32> { float4 a, b; };

template <int XT>
__device__ __forceinline__ void raw_load(Raw8<XT>& r, const void* base, int64_t off);
template <>
__device__ __forceinline__ void raw_load<PSK_BF16>(Raw8<PSK_BF16>& r, const void* base, int64_t off) {
  r.w = __ldcs((const uint4*)((const uint16_t*)base + off));
}
template <>
__device__ __forceinline__ void raw_load<PSK_F32>(Raw8<PSK_F32>& r, const void* base, int64_t off) {
  const float4* p = (const float4*)((const float*)base + off);
  r.a = __ldcs(p);
  r.b = __ldcs(p + 1);
}
__device__ __forceinline__ void raw_unpack(const Raw8<PSK_BF16>& r, float* v) {
  const uint32_t w[4] = {r.w.x, r.w.y, r.w.z, r.w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ void raw_unpack(const Raw8<PSK_F32>& r, float* v) {
  v[0] = r.a.x; v[1] = r.a.y; v[2] = r.a.z; v[3] = r.a.w;
  v[4] = r.b.x; v[5] = r.b.y; v[6] = r.b.z; v[7] = r.b.w;
}
__device__ __forceinline__ void raw_fill(Raw8<PSK_BF16>& r) { r.w = make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u); }
__device__ __forceinline__ void raw_fill(Raw8<PSK_F32>& r) {
  r.a = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
  r.b = r.a;
}

template <int YT>
__device__ __forceinline__ void store_y8(void* base, int64_t off, const float* v) {
  if (YT == PSK_F32) {
    float4* p = (float4*)((float*)base + off);
    __stcs(p, make_float4(v[0], v[1], v[2], v[3]));
    __stcs(p + 1, make_float4(v[4], v[5], v[6], v[7]));
  } else {
    uint4 q;
    q.x = f32x2_to_bf16x2(v[0], v[1]);
    q.y = f32x2_to_bf16x2(v[2], v[3]);
    q.z = f32x2_to_bf16x2(v[4], v[5]);
    q.w = f32x2_to_bf16x2(v[6], v[7]);
    __stcs((uint4*)((uint16_t*)base + off), q);
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

// One chain: acc over E[p], E[p+P], ... (n elements in the row), in index order.
__device__ __forceinline__ float run_chain(const float* E, int n, int p, int P) {
  float acc = E[p];
  int j = p + P;
  if (P == 1) {
    for (; (j & 3) != 0 && j < n; ++j) acc = __fadd_rn(acc, E[j]);
    for (; j + 15 < n; j += 16) {
      float4 a = *(const float4*)&E[j], b = *(const float4*)&E[j + 4];
      float4 c = *(const float4*)&E[j + 8], d = *(const float4*)&E[j + 12];
      acc = __fadd_rn(acc, a.x); acc = __fadd_rn(acc, a.y); acc = __fadd_rn(acc, a.z); acc = __fadd_rn(acc, a.w);
      acc = __fadd_rn(acc, b.x); acc = __fadd_rn(acc, b.y); acc = __fadd_rn(acc, b.z); acc = __fadd_rn(acc, b.w);
      acc = __fadd_rn(acc, c.x); acc = __fadd_rn(acc, c.y); acc = __fadd_rn(acc, c.z); acc = __fadd_rn(acc, c.w);
      acc = __fadd_rn(acc, d.x); acc = __fadd_rn(acc, d.y); acc = __fadd_rn(acc, d.z); acc = __fadd_rn(acc, d.w);
    }
  } else {
    for (; j + 7 * P < n; j += 8 * P) {
      float v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = E[j + i * P];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc = __fadd_rn(acc, v[i]);
    }
  }
  for (; j < n; j += P) acc = __fadd_rn(acc, E[j]);
  return acc;
}

// --------------------------------------------------- resident rows (<= 4096)
template <int XT, int YT, int EXPM, bool VEC>
__global__ void __launch_bounds__(SM_THREADS, 3) softmax_batch_kernel(const __grid_constant__ SoftmaxParams P) {
  constexpr int NBMAX = (XT == PSK_BF16) ? 4 : 2;
  extern __shared__ __align__(16) float smem[];
  __shared__ float exp_hi[32], exp_lo[32];
  __shared__ float red[SM_THREADS / 32][NBMAX];
  __shared__ float rowsum[NBMAX], rowrcp[NBMAX];
  const int t = threadIdx.x, w = t >> 5, l = t & 31;
  if (EXPM == PSK_EXP_EXACT && t < 32) { exp_hi[t] = psk_exp_tab_hi[t]; exp_lo[t] = psk_exp_tab_lo[t]; }
  const int cols = (int)P.cols;
  const int nb = P.nb;
  const int parts = P.partials < cols ? P.partials : cols;
  const int64_t nbatch = (P.rows + nb - 1) / nb;
  const size_t xsz = XT == PSK_F32 ? 4 : 2, ysz = YT == PSK_F32 ? 4 : 2;

  Raw8<XT> raw[NBMAX][2];
  float xs[NBMAX][SM_EPT];                         // scalar path only
  // loads of one batch into registers (issued a batch ahead, so their latency
  // overlaps the previous batch's chain and output phases)
  auto load_batch = [&](int64_t bt) {
    const int64_t r0 = bt * nb;
    const int nrr = bt < nbatch ? (int)((P.rows - r0) < nb ? (P.rows - r0) : nb) : 0;
#pragma unroll
    for (int b = 0; b < NBMAX; ++b) {
      const void* xr = (const char*)P.x + (r0 + b) * P.ldx * xsz;
      if (VEC) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int j = (k * SM_THREADS + t) * 8;
          if (b < nrr && j < cols) raw_load<XT>(raw[b][k], xr, j); else raw_fill(raw[b][k]);
        }
      } else {
#pragma unroll
        for (int k = 0; k < SM_EPT; ++k) {
          const int j = k * SM_THREADS + t;
          xs[b][k] = (b < nrr && j < cols) ? load_x1<XT>(xr, j) : -INFINITY;
        }
      }
    }
  };
  load_batch(blockIdx.x);
  for (int64_t bt = blockIdx.x; bt < nbatch; bt += gridDim.x) {
    const int64_t row0 = bt * nb;
    const int nr = (int)((P.rows - row0) < nb ? (P.rows - row0) : nb);
    // 1. local maxima of the batch held in registers
    float mloc[NBMAX];
#pragma unroll
    for (int b = 0; b < NBMAX; ++b) {
      mloc[b] = -INFINITY;
      if (VEC) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          float v[8];
          raw_unpack(raw[b][k], v);
#pragma unroll
          for (int q = 0; q < 8; ++q) mloc[b] = max_nan(mloc[b], v[q]);
        }
      } else {
#pragma unroll
        for (int k = 0; k < SM_EPT; ++k) mloc[b] = max_nan(mloc[b], xs[b][k]);
      }
    }
    // 2. the NB row maxima, one barrier
#pragma unroll
    for (int b = 0; b < NBMAX; ++b) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mloc[b] = max_nan(mloc[b], __shfl_xor_sync(0xffffffffu, mloc[b], o));
      if (l == 0) red[w][b] = mloc[b];
    }
    __syncthreads();
    float m[NBMAX];
#pragma unroll
    for (int b = 0; b < NBMAX; ++b) {
      m[b] = red[0][b];
#pragma unroll
      for (int i = 1; i < SM_THREADS / 32; ++i) m[b] = max_nan(m[b], red[i][b]);
    }
    // 3. e = exp(x - m) into the row buffers
#pragma unroll
    for (int b = 0; b < NBMAX; ++b) {
      if (b >= nr) continue;
      float* E = smem + b * P.estride;
      if (VEC) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int j = (k * SM_THREADS + t) * 8;
          if (j < cols) {
            float v[8];
            raw_unpack(raw[b][k], v);
#pragma unroll
            for (int q = 0; q < 8; ++q) v[q] = __fsub_rn(v[q], m[b]);
            region_exp8<EXPM>(v, exp_hi, exp_lo);
            *(float4*)&E[j] = make_float4(v[0], v[1], v[2], v[3]);
            *(float4*)&E[j + 4] = make_float4(v[4], v[5], v[6], v[7]);
          }
        }
      } else {
#pragma unroll
        for (int k = 0; k < SM_EPT; ++k) {
          const int j = k * SM_THREADS + t;
          if (j < cols) E[j] = region_exp<EXPM>(__fsub_rn(xs[b][k], m[b]), exp_hi, exp_lo);
        }
      }
    }
    __syncthreads();
    load_batch(bt + gridDim.x);
    // 4. every chain of the batch in warp 0: lane (b, p) sums chain p of row b
    if (w == 0) {
      const int nlanes = nr * parts;
      for (int base = 0; base < nlanes; base += 32) {
        const int lane_id = base + l;
        float acc = 0.0f;
        int b = 0, p = 0;
        if (lane_id < nlanes) {
          b = lane_id / parts;
          p = lane_id - b * parts;
          acc = run_chain(smem + b * P.estride, cols, p, parts);
        }
        // partials of row b sit in lanes b*parts .. b*parts+parts-1 of this
        // pass when parts divides 32; otherwise they are combined through smem
        if (parts <= 32 && (32 % parts) == 0) {
          float s = acc;
          for (int q = 1; q < parts; ++q) {
            float o = __shfl_sync(0xffffffffu, acc, (l - p + q) & 31);
            if (lane_id < nlanes) s = __fadd_rn(s, o);
          }
          if (lane_id < nlanes && p == 0) { rowsum[b] = s; rowrcp[b] = __frcp_rn(s); }
        } else {
          float* part = smem + nb * P.estride;     // scratch after the row buffers
          if (lane_id < nlanes) part[lane_id] = acc;
          __syncwarp();
          if (base + 32 >= nlanes) {
            for (int bb = l; bb < nr; bb += 32) {
              float s = part[bb * parts];
              for (int q = 1; q < parts; ++q) s = __fadd_rn(s, part[bb * parts + q]);
              rowsum[bb] = s;
              rowrcp[bb] = __frcp_rn(s);
            }
          }
          __syncwarp();
        }
      }
    }
    __syncthreads();
    // 5. y = e / s, stored
#pragma unroll
    for (int b = 0; b < NBMAX; ++b) {
      if (b >= nr) continue;
      const float* E = smem + b * P.estride;
      const float s = rowsum[b], rs = rowrcp[b];
      const bool fast_ok = s >= 1.0f && s < 0x1p20f;
      void* yr = (char*)P.y + (row0 + b) * P.ldy * ysz;
      if (VEC) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int j = (k * SM_THREADS + t) * 8;
          if (j < cols) {
            float4 a = *(const float4*)&E[j], c = *(const float4*)&E[j + 4];
            float o[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
            for (int q = 0; q < 8; ++q) o[q] = row_div(o[q], s, rs, fast_ok);
            store_y8<YT>(yr, j, o);
          }
        }
      } else {
#pragma unroll
        for (int k = 0; k < SM_EPT; ++k) {
          const int j = k * SM_THREADS + t;
          if (j < cols) store_y1<YT>(yr, j, row_div(E[j], s, rs, fast_ok));
        }
      }
    }
    __syncthreads();
  }
}

// ------------------------------------------------- streaming rows (> 4096)
struct StreamShared {
  float E[SM_CAP];
  float exp_hi[32], exp_lo[32];
  float red[SM_THREADS / 32];
  float part[SM_MAX_PARTIALS];
  float bcast;
};

__device__ __forceinline__ float block_max(float v, StreamShared& sh) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max_nan(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) sh.red[threadIdx.x >> 5] = v;
  __syncthreads();
  float m = sh.red[0];
  for (int i = 1; i < SM_THREADS / 32; ++i) m = max_nan(m, sh.red[i]);
  __syncthreads();
  return m;
}

template <int XT, int YT, int EXPM>
__global__ void __launch_bounds__(SM_THREADS) softmax_stream_kernel(const __grid_constant__ SoftmaxParams P) {
  __shared__ __align__(16) StreamShared sh;
  const int t = threadIdx.x;
  if (EXPM == PSK_EXP_EXACT && t < 32) { sh.exp_hi[t] = psk_exp_tab_hi[t]; sh.exp_lo[t] = psk_exp_tab_lo[t]; }
  __syncthreads();
  const int64_t cols = P.cols;
  const int nP = (int)(cols < P.partials ? cols : P.partials);
  for (int64_t row = blockIdx.x; row < P.rows; row += gridDim.x) {
    const void* xr = (const char*)P.x + row * P.ldx * (XT == PSK_F32 ? 4 : 2);
    void* yr = (char*)P.y + row * P.ldy * (YT == PSK_F32 ? 4 : 2);
    float m = -INFINITY;
    for (int64_t j = t; j < cols; j += SM_THREADS) m = max_nan(m, load_x1<XT>(xr, j));
    m = block_max(m, sh);
    float acc = 0.0f;
    for (int64_t base = 0; base < cols; base += SM_CAP) {
      const int n = (int)((cols - base) < SM_CAP ? (cols - base) : SM_CAP);
      for (int i = t; i < n; i += SM_THREADS)
        sh.E[i] = region_exp<EXPM>(__fsub_rn(load_x1<XT>(xr, base + i), m), sh.exp_hi, sh.exp_lo);
      __syncthreads();
      if (t < nP) {
        // chain t continues over the indices j = t (mod nP) of this chunk
        int i = (int)(((int64_t)t - base) % nP);
        if (i < 0) i += nP;
        if (base == 0) { acc = sh.E[i]; i += nP; }
        for (; i < n; i += nP) acc = __fadd_rn(acc, sh.E[i]);
      }
      __syncthreads();
    }
    if (t < nP) sh.part[t] = acc;
    __syncthreads();
    if (t == 0) {
      float s = sh.part[0];
      for (int q = 1; q < nP; ++q) s = __fadd_rn(s, sh.part[q]);
      sh.bcast = s;
    }
    __syncthreads();
    const float s = sh.bcast, rs = __frcp_rn(s);
    for (int64_t j = t; j < cols; j += SM_THREADS) {
      float e = region_exp<EXPM>(__fsub_rn(load_x1<XT>(xr, j), m), sh.exp_hi, sh.exp_lo);
      store_y1<YT>(yr, j, div_by_recip(e, s, rs));
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ host
static int sm_count_softmax() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
  }
  return n;
}

template <int XT, int YT, int EXPM, bool VEC>
static int launch_batch(SoftmaxParams P, cudaStream_t stream) {
  constexpr int NBMAX = (XT == PSK_BF16) ? 4 : 2;
  // row buffers padded so that lanes of different rows start in different
  // banks: buffer b begins at b * estride, estride = cols rounded to 32 plus
  // the partial count rounded up to 4
  const int pad = ((P.partials + 3) / 4) * 4;
  P.nb = NBMAX;
  P.estride = (int)(((P.cols + 31) / 32) * 32 + (pad % 32));
  const size_t smem = (size_t)(P.nb * P.estride + P.nb * P.partials + 64) * sizeof(float);
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(softmax_batch_kernel<XT, YT, EXPM, VEC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         100 * 1024);
    attr = true;
  }
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, softmax_batch_kernel<XT, YT, EXPM, VEC>, SM_THREADS, smem);
  if (per_sm < 1) per_sm = 1;
  const int64_t nbatch = (P.rows + P.nb - 1) / P.nb;
  const int64_t cap = (int64_t)sm_count_softmax() * per_sm;
  const unsigned grid = (unsigned)(nbatch < cap ? nbatch : cap);
  softmax_batch_kernel<XT, YT, EXPM, VEC><<<grid, SM_THREADS, smem, stream>>>(P);
  return check_launch("softmax region kernel");
}

template <int XT, int YT, int EXPM>
static int launch_stream(const SoftmaxParams& P, cudaStream_t stream) {
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, softmax_stream_kernel<XT, YT, EXPM>, SM_THREADS, 0);
  if (per_sm < 1) per_sm = 1;
  const int64_t cap = (int64_t)sm_count_softmax() * per_sm;
  const unsigned grid = (unsigned)(P.rows < cap ? P.rows : cap);
  softmax_stream_kernel<XT, YT, EXPM><<<grid, SM_THREADS, 0, stream>>>(P);
  return check_launch("softmax region kernel (streaming rows)");
}

template <int XT, int YT, int EXPM>
static int dispatch_exp(const SoftmaxParams& P, bool vec, cudaStream_t s) {
  if (P.cols > SM_CAP) return launch_stream<XT, YT, EXPM>(P, s);
  return vec ? launch_batch<XT, YT, EXPM, true>(P, s) : launch_batch<XT, YT, EXPM, false>(P, s);
}

template <int XT, int YT>
static int dispatch_softmax(const SoftmaxParams& P, int exp_mode, bool vec, cudaStream_t s) {
  return exp_mode == PSK_EXP_EXACT ? dispatch_exp<XT, YT, PSK_EXP_EXACT>(P, vec, s)
                                   : dispatch_exp<XT, YT, PSK_EXP_FAST>(P, vec, s);
}

}  // namespace psk

using namespace psk;

extern "C" int psk_softmax_region(const void* x, int32_t xt, void* y, int32_t yt, int64_t rows, int64_t cols,
                                  int64_t ldx, int64_t ldy, psk_order order, int32_t exp_mode, void* stream) {
  clear_error();
  if (!dtype_ok(xt)) return fail(PSK_E_DTYPE, "x dtype %d", xt);
  if (!dtype_ok(yt)) return fail(PSK_E_DTYPE, "y dtype %d", yt);
  if (rows < 0 || cols < 0) return fail(PSK_E_SHAPE, "rows %lld, cols %lld", (long long)rows, (long long)cols);
  if (cols > 0x7FFFFFFF) return fail(PSK_E_SHAPE, "cols %lld above 2^31-1", (long long)cols);
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
  SoftmaxParams P{x, y, rows, cols, ldx, ldy, partials, 1, 0};
  const bool vec = (cols % 8 == 0) && (ldx % 8 == 0) && (ldy % 8 == 0) && ((uintptr_t)x % 16 == 0) &&
                   ((uintptr_t)y % 16 == 0);
  cudaStream_t s = (cudaStream_t)stream;
  if (xt == PSK_BF16 && yt == PSK_BF16) return dispatch_softmax<PSK_BF16, PSK_BF16>(P, exp_mode, vec, s);
  if (xt == PSK_BF16 && yt == PSK_F32) return dispatch_softmax<PSK_BF16, PSK_F32>(P, exp_mode, vec, s);
  if (xt == PSK_F32 && yt == PSK_BF16) return dispatch_softmax<PSK_F32, PSK_BF16>(P, exp_mode, vec, s);
  return dispatch_softmax<PSK_F32, PSK_F32>(P, exp_mode, vec, s);
}
