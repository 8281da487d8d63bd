// Reduction-rooted row regions: a last-axis, keepdim reduction followed by
// its pointwise epilogue, in one kernel -- the row is reduced on chip and the
// epilogue runs in the same kernel (poot "Fusion and Planning",
// Reduction-rooted regions).  Arithmetic is f32 for bf16 storage, one rounding
// per operation, and every sum follows the declared order's bracketing tree
// (presk "Native execution", the realization's order; metrale "The LKB in
// Mathematics", section 2: bit parity is the same bracketing tree):
//   sequential / blocked(w): one chain ((v0 + v1) + v2) + ... in index order;
//   interleaved(P): P chains, chain p over j = p mod P in increasing j, then
//   the P partials added left to right.
//
// Regions:
//   psk_softmax_region  Reduce(Max) -> Sub -> Exp -> Reduce(Sum) -> Div;
//   psk_norm_region     RMSNorm: Reduce(Sum of x^2) -> mean -> +eps -> sqrt ->
//                       Div (-> * gamma); LayerNorm: Reduce(Sum) -> mean ->
//                       x - mu -> Reduce(Sum of squares) -> mean -> +eps ->
//                       sqrt -> Div (-> * gamma -> + beta) (PSK-Realize,
//                       "What it removes").
//
// Kernels:
//   region_pipe_kernel   rows of <= 4096 columns, 16-byte aligned, <= 32
//                        partials (both regions): a warp-specialised pipeline,
//                        described where it is defined;
//   softmax_batch_kernel other softmax rows of <= 4096 columns: NB rows per
//                        CTA, warp 0 runs the chains;
//   softmax_stream_kernel softmax rows longer than 4096, in chunks (exp
//                        recomputed in the output pass, bit-identical);
//   region_row_kernel    other norm rows, masked softmax rows and backward
//                        rows: one row at a time per CTA, held in shared
//                        memory as f32.

#include "common.cuh"
#include "crmath.cuh"
#include "pipe.cuh"
#include "pair.cuh"
#include "rowmath.cuh"

namespace psk {

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

// Value transforms a chain applies to each stored element before adding it.
struct ChainIdentity {
  __device__ __forceinline__ float operator()(float v) const { return v; }
};
struct ChainSquare {            // RN(v * v)
  __device__ __forceinline__ float operator()(float v) const { return __fmul_rn(v, v); }
};
struct ChainCenteredSquare {    // RN(RN(v - mu)^2)
  float mu;
  __device__ __forceinline__ float operator()(float v) const {
    const float c = __fsub_rn(v, mu);
    return __fmul_rn(c, c);
  }
};

// A chain continued over f(E[j]), f(E[j+P]), ... for j < end, in index
// order (j is left past the last element added).  Loads run ahead of the
// dependent adds in a register ring of D16 blocks of 16 (P = 1) or D8 blocks
// of 8 (P > 1), D - 1 blocks ahead (no moves: each block's registers are
// refilled right after it is added), so the chain runs at the add latency
// while the shared-memory latency stays below that of the blocks ahead.
template <int D16, int D8, class F>
__device__ __forceinline__ float chain_range(float acc, const float* E, int& j, int end, int P, F f) {
#define PSK_ADD4(q) acc = __fadd_rn(acc, f(q.x)); acc = __fadd_rn(acc, f(q.y)); \
                    acc = __fadd_rn(acc, f(q.z)); acc = __fadd_rn(acc, f(q.w));
  if (P == 1) {
    constexpr int D = D16;
    for (; (j & 3) != 0 && j < end; ++j) acc = __fadd_rn(acc, f(E[j]));
    if (j + D * 16 <= end) {
      float4 r[D][4];
#pragma unroll
      for (int d = 0; d < D; ++d)
#pragma unroll
        for (int q = 0; q < 4; ++q) r[d][q] = *(const float4*)&E[j + 16 * d + 4 * q];
      for (; j + 2 * D * 16 <= end; j += D * 16) {
#pragma unroll
        for (int d = 0; d < D; ++d) {
#pragma unroll
          for (int q = 0; q < 4; ++q) { PSK_ADD4(r[d][q]) }
#pragma unroll
          for (int q = 0; q < 4; ++q) r[d][q] = *(const float4*)&E[j + 16 * (d + D) + 4 * q];
        }
      }
#pragma unroll
      for (int d = 0; d < D; ++d)
#pragma unroll
        for (int q = 0; q < 4; ++q) { PSK_ADD4(r[d][q]) }
      j += D * 16;
    }
  } else {
    constexpr int D = D8;
    if (j + (8 * D - 1) * P < end) {
      float r[D][8];
#pragma unroll
      for (int d = 0; d < D; ++d)
#pragma unroll
        for (int i = 0; i < 8; ++i) r[d][i] = E[j + (8 * d + i) * P];
      for (; j + (16 * D - 1) * P < end; j += 8 * D * P) {
#pragma unroll
        for (int d = 0; d < D; ++d) {
#pragma unroll
          for (int i = 0; i < 8; ++i) acc = __fadd_rn(acc, f(r[d][i]));
#pragma unroll
          for (int i = 0; i < 8; ++i) r[d][i] = E[j + (8 * (d + D) + i) * P];
        }
      }
#pragma unroll
      for (int d = 0; d < D; ++d)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc = __fadd_rn(acc, f(r[d][i]));
      j += 8 * D * P;
    }
  }
#undef PSK_ADD4
  for (; j < end; j += P) acc = __fadd_rn(acc, f(E[j]));
  return acc;
}

// The same through chain_range's register ring (the pipelined kernel's chain
// warps, whose shared-memory loads compete with the teams' traffic).
template <int D16, int D8, class F>
__device__ __forceinline__ float run_chain_deep(const float* E, int n, int p, int P, F f) {
  float acc = f(E[p]);
  int j = p + P;
  return chain_range<D16, D8>(acc, E, j, n, P, f);
}

// One chain: acc over f(E[p]), f(E[p+P]), ... (n elements in the row), in
// index order.  The loads of the next block are issued before the dependent
// adds of the current one (registers double-buffered), so the chain runs at
// the add latency instead of add + shared-memory latency per block.
template <class F>
__device__ __forceinline__ float run_chain(const float* E, int n, int p, int P, F f) {
  float acc = f(E[p]);
  int j = p + P;
#define PSK_ADD4(q) acc = __fadd_rn(acc, f(q.x)); acc = __fadd_rn(acc, f(q.y)); \
                    acc = __fadd_rn(acc, f(q.z)); acc = __fadd_rn(acc, f(q.w));
  if (P == 1) {
    for (; (j & 3) != 0 && j < n; ++j) acc = __fadd_rn(acc, f(E[j]));
    if (j + 15 < n) {
      float4 a = *(const float4*)&E[j], b = *(const float4*)&E[j + 4];
      float4 c = *(const float4*)&E[j + 8], d = *(const float4*)&E[j + 12];
      for (; j + 31 < n; j += 16) {
        const float4 na = *(const float4*)&E[j + 16], nb = *(const float4*)&E[j + 20];
        const float4 nc = *(const float4*)&E[j + 24], nd = *(const float4*)&E[j + 28];
        PSK_ADD4(a) PSK_ADD4(b) PSK_ADD4(c) PSK_ADD4(d)
        a = na; b = nb; c = nc; d = nd;
      }
      PSK_ADD4(a) PSK_ADD4(b) PSK_ADD4(c) PSK_ADD4(d)
      j += 16;
    }
  } else if (j + 7 * P < n) {
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = E[j + i * P];
    for (; j + 15 * P < n; j += 8 * P) {
      float nv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) nv[i] = E[j + (8 + i) * P];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc = __fadd_rn(acc, f(v[i]));
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = nv[i];
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) acc = __fadd_rn(acc, f(v[i]));
    j += 8 * P;
  }
#undef PSK_ADD4
  for (; j < n; j += P) acc = __fadd_rn(acc, f(E[j]));
  return acc;
}

__device__ __forceinline__ float run_chain(const float* E, int n, int p, int P) {
  return run_chain(E, n, p, P, ChainIdentity());
}

// --------------------------------------------------- resident rows (<= 4096)
template <int XT, int YT, int EXPM, bool VEC>
__global__ void __launch_bounds__(SM_THREADS, 3) softmax_batch_kernel(const __grid_constant__ RegionParams P) {
  constexpr int NBMAX = (XT == PSK_BF16) ? 4 : 2;
  extern __shared__ __align__(16) float smem[];
  __shared__ float red[SM_THREADS / 32][NBMAX];
  __shared__ float rowsum[NBMAX], rowrcp[NBMAX];
  const int t = threadIdx.x, w = t >> 5, l = t & 31;
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
            region_exp8<EXPM>(v);
            *(float4*)&E[j] = make_float4(v[0], v[1], v[2], v[3]);
            *(float4*)&E[j + 4] = make_float4(v[4], v[5], v[6], v[7]);
          }
        }
      } else {
#pragma unroll
        for (int k = 0; k < SM_EPT; ++k) {
          const int j = k * SM_THREADS + t;
          if (j < cols) E[j] = region_exp<EXPM>(__fsub_rn(xs[b][k], m[b]));
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
            row_div_n<8>(o, s, rs, fast_ok);
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


// ------------------------------------- pipelined rows (<= 4096 columns)
// One persistent CTA per SM with three roles:
//   a producer warp streams this CTA's rows (bf16 or f32) into a shared ring
//   of SX slots with 1-D bulk copies (TMA) that complete on the slot's
//   mbarrier;
//   4 teams of 4 compute warps each take every 4th row of the CTA (so four
//   rows are in the compute stage at once, each team synchronising only
//   within itself) and write the row's values into a shared ring of SE f32
//   rows -- softmax: e = exp(x - max) (the max by warp shuffles and a team
//   barrier); norms: x widened -- then, LAG = SE/4 - 1 team rows later, once
//   the chain warps have published the row's reductions, the epilogue
//   (softmax: e / s; RMSNorm: x / d, * gamma; LayerNorm: (x - mu) / d,
//   * gamma, + beta), stored with streaming stores;
//   3 chain warps own the value ring's slot groups (G <= 4 consecutive rows):
//   lane (row, p) adds chain p of its row in index order, the partials are
//   combined left to right by shuffles and the row's scalars published on
//   the row's mbarrier (LayerNorm runs two chains per row, the sum and then
//   the sum of squares about the mean).
// A row's chain is a serial run of cols/P dependent adds, so about 4 LAG
// rows chain at once; long chains (sequential order) get a deeper value ring
// and a shallower x ring.  Every wait is bounded (pipe.cuh).
constexpr int PIPE_TEAMS = 4;
constexpr int PIPE_TW = 4;                                   // warps per team
constexpr int PIPE_CW = PIPE_TEAMS * PIPE_TW;                // compute warps (16)
constexpr int PIPE_TT = PIPE_TW * 32;                        // threads per team (128)
constexpr int PIPE_EPT = SM_CAP / PIPE_TT;                   // row elements per team thread (32)
constexpr int PIPE_KW = 3;                                   // chain warps
constexpr int PIPE_THREADS = (PIPE_CW + PIPE_KW + 1) * 32;   // + producer warp
constexpr int PIPE_SX_MAX = 16;                              // x ring slots (barrier arrays)
constexpr int PIPE_SX_DEEP = 8;                              // the deep x ring of the default depths
constexpr int PIPE_SE_MAX = 16;                              // value ring slots (a multiple of the teams)
constexpr size_t PIPE_SMEM_BUDGET = 225 * 1024;              // dynamic shared memory of one CTA
constexpr int PIPE_EXP_TAB_BYTES = 2048 * 4;                 // the exact softmax's copy of psk_exp_tab2

// Four consecutive stored elements at j, widened.
template <int T>
__device__ __forceinline__ void load4(const void* base, int j, float* v) {
  if (T == PSK_F32) {
    const float4 q = *reinterpret_cast<const float4*>((const float*)base + j);
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
  } else {
    const uint2 q = *reinterpret_cast<const uint2*>((const uint16_t*)base + j);
    v[0] = __uint_as_float(q.x << 16);
    v[1] = __uint_as_float(q.x & 0xFFFF0000u);
    v[2] = __uint_as_float(q.y << 16);
    v[3] = __uint_as_float(q.y & 0xFFFF0000u);
  }
}

// The same from global memory through the read-only path (norm parameters).
__device__ __forceinline__ void load4_param(const void* base, int dtype, int j, float* v) {
  if (dtype == PSK_F32) {
    const float4 q = __ldg(reinterpret_cast<const float4*>((const float*)base + j));
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
  } else {
    const uint2 q = __ldg(reinterpret_cast<const uint2*>((const uint16_t*)base + j));
    v[0] = __uint_as_float(q.x << 16);
    v[1] = __uint_as_float(q.x & 0xFFFF0000u);
    v[2] = __uint_as_float(q.y << 16);
    v[3] = __uint_as_float(q.y & 0xFFFF0000u);
  }
}

// Storage of four consecutive norm parameters (one 16- or 8-byte load).
template <int PT> struct Param4;
template <> struct Param4<PSK_F32> {
  float4 q;
  __device__ __forceinline__ void load(const void* base, int j) { q = __ldg(reinterpret_cast<const float4*>(base) + (j >> 2)); }
  __device__ __forceinline__ void widen(float* v) const { v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w; }
};
template <> struct Param4<PSK_BF16> {
  uint2 q;
  __device__ __forceinline__ void load(const void* base, int j) { q = __ldg(reinterpret_cast<const uint2*>(base) + (j >> 2)); }
  __device__ __forceinline__ void widen(float* v) const {
    v[0] = __uint_as_float(q.x << 16);
    v[1] = __uint_as_float(q.x & 0xFFFF0000u);
    v[2] = __uint_as_float(q.y << 16);
    v[3] = __uint_as_float(q.y & 0xFFFF0000u);
  }
};

// A norm row's epilogue for one team thread (its 8 chunks of 4 columns): bf16
// scale and bias chunks are loaded first (16 registers each), so they arrive
// while the thread waits for the row's mean and divisor; f32 ones are loaded
// chunk by chunk.  Then (x - mu) / d, * gamma, + beta, rounded to the output
// and stored.  False if the wait gave up.
// One chunk of a norm row's epilogue: (x - mu) / d, * gamma, + beta, rounded
// to the output and stored.
template <int KIND, int YT, int PT>
__device__ __forceinline__ void norm_chunk(const float* Er, char* yr, int j, const RowDivisor& D, float mu,
                                           const Param4<PT>* g, const Param4<PT>* b) {
  const float4 e = *reinterpret_cast<const float4*>(Er + j);
  float o4[4] = {e.x, e.y, e.z, e.w};
  if (KIND == REGION_LAYER) {
#pragma unroll
    for (int q = 0; q < 4; ++q) o4[q] = __fsub_rn(o4[q], mu);
  }
  divide_n<4>(o4, D);
  if (g) {
    float g4[4];
    g->widen(g4);
#pragma unroll
    for (int q = 0; q < 4; ++q) o4[q] = __fmul_rn(o4[q], g4[q]);
  }
  if (b) {
    float b4[4];
    b->widen(b4);
#pragma unroll
    for (int q = 0; q < 4; ++q) o4[q] = __fadd_rn(o4[q], b4[q]);
  }
  if (YT == PSK_F32) {
    __stcs(reinterpret_cast<float4*>(yr) + (j >> 2), make_float4(o4[0], o4[1], o4[2], o4[3]));
  } else {
    uint2 q;
    q.x = f32x2_to_bf16x2(o4[0], o4[1]);
    q.y = f32x2_to_bf16x2(o4[2], o4[3]);
    __stcs(reinterpret_cast<uint2*>(yr) + (j >> 2), q);
  }
}

// A norm row's epilogue for one team thread (its 8 chunks of 4 columns).  bf16
// scale and bias chunks are loaded first (16 registers each), so they arrive
// while the thread waits for the row's mean and divisor; f32 ones are loaded
// chunk by chunk.  False if the wait gave up.
template <int KIND, int YT, int PT>
__device__ __forceinline__ bool norm_epilogue(const RegionParams& P, const float* Er, char* yr, int tt, int cols,
                                              uint64_t* ready, uint32_t parity, const float* d_slot,
                                              const float* mu_slot) {
  constexpr int NC = PIPE_EPT / 4;
  const bool hg = P.gamma != nullptr;
  const bool hb = KIND == REGION_LAYER && P.beta != nullptr;
  if constexpr (PT == PSK_BF16) {
    Param4<PT> g[NC], b[NC];
#pragma unroll
    for (int c4 = 0; c4 < NC; ++c4) {
      const int j = c4 * (PIPE_TT * 4) + 4 * tt;
      if (j < cols) {
        if (hg) g[c4].load(P.gamma, j);
        if (hb) b[c4].load(P.beta, j);
      }
    }
    if (!mbar_wait(ready, parity)) return false;
    const RowDivisor D = make_divisor(*d_slot);
    const float mu = *mu_slot;
#pragma unroll
    for (int c4 = 0; c4 < NC; ++c4) {
      const int j = c4 * (PIPE_TT * 4) + 4 * tt;
      if (j < cols) norm_chunk<KIND, YT, PT>(Er, yr, j, D, mu, hg ? &g[c4] : nullptr, hb ? &b[c4] : nullptr);
    }
  } else {
    if (!mbar_wait(ready, parity)) return false;
    const RowDivisor D = make_divisor(*d_slot);
    const float mu = *mu_slot;
#pragma unroll 2
    for (int c4 = 0; c4 < NC; ++c4) {
      const int j = c4 * (PIPE_TT * 4) + 4 * tt;
      if (j < cols) {
        Param4<PT> g, b;
        if (hg) g.load(P.gamma, j);
        if (hb) b.load(P.beta, j);
        norm_chunk<KIND, YT, PT>(Er, yr, j, D, mu, hg ? &g : nullptr, hb ? &b : nullptr);
      }
    }
  }
  return true;
}

// A backward row's epilogue for one team thread: y and ct (back from L2: the
// producer read them moments ago) loaded before the wait for the row's sum
// when they are bf16, chunk by chunk when f32; dx = RN(y RN(ct - s)).
template <int XT, int YT>
__device__ __forceinline__ bool bwd_epilogue(const RegionParams& P, char* yr, int64_t row, int tt, int cols,
                                             uint64_t* ready, uint32_t parity, const float* s_slot) {
  constexpr int NC = PIPE_EPT / 4;
  const void* ybase = (const char*)P.x + row * P.ldx * (XT == PSK_F32 ? 4 : 2);
  const void* cbase = (const char*)P.ct + row * P.ldc * (XT == PSK_F32 ? 4 : 2);
  auto finish = [&](int j, const float* y4, const float* c4v, float s) {
    float o4[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) o4[q] = __fmul_rn(y4[q], __fsub_rn(c4v[q], s));
    if (YT == PSK_F32) {
      __stcs(reinterpret_cast<float4*>(yr) + (j >> 2), make_float4(o4[0], o4[1], o4[2], o4[3]));
    } else {
      uint2 q;
      q.x = f32x2_to_bf16x2(o4[0], o4[1]);
      q.y = f32x2_to_bf16x2(o4[2], o4[3]);
      __stcs(reinterpret_cast<uint2*>(yr) + (j >> 2), q);
    }
  };
  if constexpr (XT == PSK_BF16) {
    Param4<PSK_BF16> yv[NC], cv[NC];
#pragma unroll
    for (int c4 = 0; c4 < NC; ++c4) {
      const int j = c4 * (PIPE_TT * 4) + 4 * tt;
      if (j < cols) { yv[c4].load(ybase, j); cv[c4].load(cbase, j); }
    }
    if (!mbar_wait(ready, parity)) return false;
    const float s = *s_slot;
#pragma unroll
    for (int c4 = 0; c4 < NC; ++c4) {
      const int j = c4 * (PIPE_TT * 4) + 4 * tt;
      if (j < cols) {
        float y4[4], c4v[4];
        yv[c4].widen(y4);
        cv[c4].widen(c4v);
        finish(j, y4, c4v, s);
      }
    }
  } else {
    if (!mbar_wait(ready, parity)) return false;
    const float s = *s_slot;
#pragma unroll 2
    for (int c4 = 0; c4 < NC; ++c4) {
      const int j = c4 * (PIPE_TT * 4) + 4 * tt;
      if (j < cols) {
        Param4<PSK_F32> yv, cv;
        yv.load(ybase, j);
        cv.load(cbase, j);
        float y4[4], c4v[4];
        yv.widen(y4);
        cv.widen(c4v);
        finish(j, y4, c4v, s);
      }
    }
  }
  return true;
}

// TAB: the correctly rounded exp's table copied into shared memory (the
// launch's choice: short chains), read from there with shared loads.
template <int KIND, int XT, int YT, int EXPM, bool MASK, bool TAB = false>
__global__ void __launch_bounds__(PIPE_THREADS, 1) region_pipe_kernel(const __grid_constant__ RegionParams P) {
  extern __shared__ __align__(128) unsigned char pipe_smem[];
  __shared__ __align__(8) uint64_t xfull[PIPE_SX_MAX], xempty[PIPE_SX_MAX], efull[PIPE_SE_MAX], sready[PIPE_SE_MAX];
  __shared__ float rowsum[PIPE_SE_MAX], rowrcp[PIPE_SE_MAX];   // softmax: s, RN(1/s); norms: d, mu
  __shared__ float red[PIPE_TEAMS][2][PIPE_TW];
  __shared__ int red_any[PIPE_TEAMS][2][PIPE_TW];            // masked softmax: does the row allow a position
  __shared__ volatile int abort_flag;

  constexpr uint32_t XSZ = XT == PSK_F32 ? 4u : 2u;
  constexpr bool BWD = KIND == REGION_SOFTMAX_BWD;
  // fast softmax over bf16 rows: the max on the stored pairs, exp and the
  // division on f32 pairs
  constexpr bool FASTSM = KIND == REGION_SOFTMAX && EXPM == PSK_EXP_FAST && XT == PSK_BF16;
  // the softmax with the correctly rounded exp: one copy of the eight-wide
  // exp in a rolled loop over x re-read from its slot (four unrolled copies
  // overflowed the instruction cache), the slot freed by each warp after it
  constexpr bool REXP = KIND == REGION_SOFTMAX && EXPM == PSK_EXP_EXACT && !MASK;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int cols = (int)P.cols;
  const uint32_t rbytes = (uint32_t)cols * XSZ;               // one stored row
  const uint32_t xbytes = BWD ? 2u * rbytes : rbytes;         // backward: the row of y, then the row of ct
  const uint32_t xslot = ((xbytes + 127u) / 128u) * 128u;     // ring slot stride in bytes
  const int SX = P.sx, SE = P.se, LAG = P.se / PIPE_TEAMS - 1;
  unsigned char* X = pipe_smem;
  float* E = reinterpret_cast<float*>(pipe_smem + (size_t)SX * xslot);
  const int estride = P.estride;
  // the correctly rounded exp's pair table, copied after the value ring
  constexpr bool STAGE_TAB = TAB && KIND == REGION_SOFTMAX && EXPM == PSK_EXP_EXACT;
  static_assert(sizeof(psk_exp_tab2) == PIPE_EXP_TAB_BYTES, "exp table size");
  float* tab_smem = E + (size_t)SE * estride;
  if (STAGE_TAB) {
    for (int q = tid; q < PIPE_EXP_TAB_BYTES / 16; q += PIPE_THREADS)
      reinterpret_cast<float4*>(tab_smem)[q] = reinterpret_cast<const float4*>(psk_exp_tab2)[q];
  }
  const float* tab = STAGE_TAB ? tab_smem : psk_exp_tab2;
  const int parts = P.partials < cols ? P.partials : cols;  // a partial beyond the row is empty
  const int G = P.nb;                                        // rows per chain group
  const int n_local = blockIdx.x < P.rows ? (int)((P.rows - 1 - blockIdx.x) / gridDim.x + 1) : 0;

  if (tid == 0) {
    for (int i = 0; i < SX; ++i) { mbar_init(&xfull[i], 1); mbar_init(&xempty[i], REXP ? PIPE_TW : 1); }
    for (int i = 0; i < SE; ++i) { mbar_init(&efull[i], PIPE_TT); mbar_init(&sready[i], 1); }
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (w == PIPE_CW + PIPE_KW) {
    // ---------------- producer
    if (lane == 0) {
      int issued = 0;
      const unsigned char* src = (const unsigned char*)P.x + (int64_t)blockIdx.x * P.ldx * XSZ;
      const int64_t step = (int64_t)gridDim.x * P.ldx * XSZ;
      const unsigned char* csrc = BWD ? (const unsigned char*)P.ct + (int64_t)blockIdx.x * P.ldc * XSZ : nullptr;
      const int64_t cstep = (int64_t)gridDim.x * P.ldc * XSZ;
      const long long drop = g_pipe_drop_row;
      for (int i = 0; i < n_local; ++i) {
        const int s = i % SX;
        if (i == drop) break;                               // test hook: the copies from here on are "lost"
        if (i >= SX && !mbar_wait(&xempty[s], (uint32_t)((i / SX) - 1) & 1u)) { abort_flag = 1; break; }
        if (abort_flag) break;
        mbar_arrive_expect_tx(&xfull[s], xbytes);
        bulk_copy_g2s(X + (size_t)s * xslot, src, rbytes, &xfull[s]);
        if (BWD) {
          bulk_copy_g2s(X + (size_t)s * xslot + rbytes, csrc, rbytes, &xfull[s]);
          csrc += cstep;
        }
        src += step;
        issued = i + 1;
      }
      if (abort_flag)   // copies still in flight land before the CTA retires
        for (int i = issued > SX ? issued - SX : 0; i < issued; ++i) mbar_wait(&xfull[i % SX], (uint32_t)(i / SX) & 1u);
    }
    return;
  }

  if (w >= PIPE_CW) {
    // ---------------- chain warps
    // A parity wait must never run two phases ahead of its barrier (it would
    // pass at once), so every slot group of the value ring (G consecutive
    // slots) belongs to one chain warp, which visits its phases in order.
    const int c = w - PIPE_CW;
    const int b = lane / parts, p = lane - (lane / parts) * parts;
    const int n_groups = SE / G;
    const float n_f = (float)cols;                           // exact: cols <= 4096
    for (int g = 0; g * G < n_local; ++g) {
      if ((g % n_groups) % PIPE_KW != c) continue;
      if (abort_flag) break;
      const int j = g * G + b;
      const bool act = b < G && j < n_local;
      const int se = j % SE;
      bool ok = true;
      if (act) ok = mbar_wait(&efull[se], (uint32_t)(j / SE) & 1u);
      if (__any_sync(0xffffffffu, !ok)) { abort_flag = 1; break; }
      const float* Er = E + (size_t)se * estride;
      // partials of the row are combined left to right in lane p = 0
      auto combine = [&](float acc) {
        float sum = acc;
        for (int q = 1; q < parts; ++q) {
          const float o = __shfl_sync(0xffffffffu, acc, (lane - p + q) & 31);
          if (act) sum = __fadd_rn(sum, o);
        }
        return sum;
      };
      if (KIND == REGION_SOFTMAX || BWD) {
        const float sum = combine(act ? run_chain_deep<3, 4>(Er, cols, p, parts, ChainIdentity()) : 0.0f);
        if (act && p == 0) {
          rowsum[se] = sum;
          rowrcp[se] = __frcp_rn(sum);
        }
      } else {
        float mu = 0.0f;
        float ss;
        if (KIND == REGION_LAYER) {
          const float s1 = combine(act ? run_chain_deep<3, 4>(Er, cols, p, parts, ChainIdentity()) : 0.0f);
          mu = __fdiv_rn(s1, n_f);
          mu = __shfl_sync(0xffffffffu, mu, (lane - p) & 31);   // the row's mean, to every lane of the row
          ss = combine(act ? run_chain_deep<3, 4>(Er, cols, p, parts, ChainCenteredSquare{mu}) : 0.0f);
        } else {
          ss = combine(act ? run_chain_deep<3, 4>(Er, cols, p, parts, ChainSquare()) : 0.0f);
        }
        if (act && p == 0) {
          const float var = __fdiv_rn(ss, n_f);
          rowsum[se] = __fsqrt_rn(__fadd_rn(var, P.eps));
          rowrcp[se] = mu;
        }
      }
      if (act && p == 0) mbar_arrive(&sready[se]);
    }
    return;
  }

  // ---------------- compute teams: team t takes rows t, t + 4, ...; team
  // thread tt owns elements 4 tt + 512 k (+0..3), k = 0..7.  After a timeout
  // (`dead`) a team skips every wait and all work but keeps meeting its
  // barrier, so every thread leaves in bounded time.
  const int team = w / PIPE_TW, tw = w % PIPE_TW, tt = tid % PIPE_TT;
  bool dead = false;
  const size_t ysz = YT == PSK_F32 ? 4 : 2;
  // ring positions of the rows i and o below, kept without a division per
  // row: i advances by the team count, which divides SX and SE; o starts at
  // team - PIPE_TEAMS * LAG >= -SE (SE = PIPE_TEAMS * (LAG + 1)), its
  // position and phase taken with floor division
  int xs = team, xpar = 0;                                    // i % SX, (i / SX) & 1
  int ei = team;                                              // i % SE
  const int o0 = team - PIPE_TEAMS * LAG;
  int eo = o0 >= 0 ? o0 % SE : o0 + SE;                       // o % SE
  int opar = o0 >= 0 ? (o0 / SE) & 1 : 1;                     // floor(o / SE) & 1
  auto advance = [&]() {
    xs += PIPE_TEAMS;
    if (xs >= SX) { xs -= SX; xpar ^= 1; }
    ei += PIPE_TEAMS;
    if (ei >= SE) ei -= SE;
    eo += PIPE_TEAMS;
    if (eo >= SE) { eo -= SE; opar ^= 1; }
  };
  for (int k = 0;; ++k, advance()) {
    const int i = team + PIPE_TEAMS * k;                     // row produced in this team iteration
    const int o = i - PIPE_TEAMS * LAG;                      // row output in this team iteration
    if (o >= n_local) break;
    dead = dead || abort_flag;
    if (i < n_local) {
      const int s = xs;
      // masked softmax: the row's mask words, loaded before the wait for x
      constexpr bool masked = KIND == REGION_SOFTMAX && MASK;
      uint32_t mk[PIPE_EPT / 4];
      if (masked) {
        const uint8_t* mrow = P.mask + ((int64_t)blockIdx.x + (int64_t)i * gridDim.x) * P.ldm;
#pragma unroll
        for (int c4 = 0; c4 < PIPE_EPT / 4; ++c4) {
          const int j = c4 * (PIPE_TT * 4) + 4 * tt;
          mk[c4] = j < cols ? __ldg(reinterpret_cast<const uint32_t*>(mrow + j)) : 0u;
        }
      }
      if (!dead && !mbar_wait(&xfull[s], (uint32_t)xpar)) { abort_flag = 1; dead = true; }
      const unsigned char* xs = X + (size_t)s * xslot;
      float v[FASTSM ? 1 : PIPE_EPT];
      uint2 xw[FASTSM ? PIPE_EPT / 4 : 1];                   // fast softmax: the row's bf16 pairs as stored
      float m = -INFINITY;
      int any = 0;
      if constexpr (FASTSM) {
        uint32_t mb = 0xFF80FF80u;                           // (-inf, -inf)
#pragma unroll
        for (int c4 = 0; c4 < PIPE_EPT / 4; ++c4) {
          const int j = c4 * (PIPE_TT * 4) + 4 * tt;
          xw[c4] = (j < cols && !dead) ? *reinterpret_cast<const uint2*>(xs + 2 * j) : make_uint2(0xFF80FF80u, 0xFF80FF80u);
          if (masked) {
            // a refused position (mask byte 0; byte q is element j + q) reads
            // as bf16 -inf, as the f32 path's -INFINITY
            const uint32_t w = mk[c4];
            const uint32_t ka = ((w & 0xFFu) ? 0x0000FFFFu : 0u) | ((w & 0xFF00u) ? 0xFFFF0000u : 0u);
            const uint32_t kb = ((w & 0xFF0000u) ? 0x0000FFFFu : 0u) | ((w & 0xFF000000u) ? 0xFFFF0000u : 0u);
            xw[c4].x = (xw[c4].x & ka) | (0xFF80FF80u & ~ka);
            xw[c4].y = (xw[c4].y & kb) | (0xFF80FF80u & ~kb);
            any |= (w != 0u);
          }
          mb = bf16x2_max_nan(mb, bf16x2_max_nan(xw[c4].x, xw[c4].y));
        }
        m = max_nan(__uint_as_float(mb << 16), __uint_as_float(mb & 0xFFFF0000u));
      } else {
#pragma unroll
      for (int c4 = 0; c4 < PIPE_EPT / 4; ++c4) {
        const int j = c4 * (PIPE_TT * 4) + 4 * tt;
        if (j < cols && !dead) {
          load4<XT>(xs, j, &v[4 * c4]);
          if (BWD) {                                           // p = RN(ct y)
            float c[4];
            load4<XT>(xs + rbytes, j, c);
#pragma unroll
            for (int q = 0; q < 4; ++q) v[4 * c4 + q] = __fmul_rn(c[q], v[4 * c4 + q]);
          }
          if (masked) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const bool allow = ((mk[c4] >> (8 * q)) & 0xFFu) != 0u;
              any |= allow;
              if (!allow) v[4 * c4 + q] = -INFINITY;
            }
          }
        } else {
          v[4 * c4 + 0] = v[4 * c4 + 1] = v[4 * c4 + 2] = v[4 * c4 + 3] = -INFINITY;
        }
        if (KIND == REGION_SOFTMAX) {
#pragma unroll
          for (int q = 0; q < 4; ++q) m = max_nan(m, v[4 * c4 + q]);
        }
      }
      }
      if (KIND == REGION_SOFTMAX) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = max_nan(m, __shfl_xor_sync(0xffffffffu, m, off));
        if (lane == 0) red[team][k & 1][tw] = m;
        if (masked) {
          any = __any_sync(0xffffffffu, any);
          if (lane == 0) red_any[team][k & 1][tw] = any;
        }
      }
      named_barrier(1 + team, PIPE_TT);                      // every team thread has read x
      if (KIND == REGION_SOFTMAX) {
        m = red[team][k & 1][0];
#pragma unroll
        for (int q = 1; q < PIPE_TW; ++q) m = max_nan(m, red[team][k & 1][q]);
        if (masked) {
          int team_any = 0;
#pragma unroll
          for (int q = 0; q < PIPE_TW; ++q) team_any |= red_any[team][k & 1][q];
          if (!team_any) m = 0.0f;                           // a row the mask empties: every exp is 0
        }
      }
      if (!REXP && tt == 0) mbar_arrive(&xempty[s]);
      const int se = ei;
      float* Er = E + (size_t)se * estride;
      if (FASTSM && !dead) {
        // e = exp(x - m) two at a time: x - m as x + (-m) (the same rounding)
        const f2 nm = f2_splat(-m);
#pragma unroll
        for (int c4 = 0; c4 < PIPE_EPT / 4; ++c4) {
          const int j = c4 * (PIPE_TT * 4) + 4 * tt;
          if (j < cols) {
            const f2 a = exp2_unit_nonpos(f2_add(
                f2{__uint_as_float(xw[c4].x << 16), __uint_as_float(xw[c4].x & 0xFFFF0000u)}, nm));
            const f2 b = exp2_unit_nonpos(f2_add(
                f2{__uint_as_float(xw[c4].y << 16), __uint_as_float(xw[c4].y & 0xFFFF0000u)}, nm));
            *reinterpret_cast<float4*>(Er + j) = make_float4(a.x, a.y, b.x, b.y);
          }
        }
      } else if (REXP && !dead) {
#pragma unroll 1
        for (int h = 0; h < PIPE_EPT / 8; ++h) {
          float u[8];
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const int j = (2 * h + kk) * (PIPE_TT * 4) + 4 * tt;
            if (j < cols) {
              load4<XT>(xs, j, u + 4 * kk);
            } else {
              u[4 * kk] = u[4 * kk + 1] = u[4 * kk + 2] = u[4 * kk + 3] = -INFINITY;
            }
          }
#pragma unroll
          for (int q = 0; q < 8; ++q) u[q] = __fsub_rn(u[q], m);
          region_exp8<EXPM>(u, tab);
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const int j = (2 * h + kk) * (PIPE_TT * 4) + 4 * tt;
            if (j < cols)
              *reinterpret_cast<float4*>(Er + j) = make_float4(u[4 * kk], u[4 * kk + 1], u[4 * kk + 2], u[4 * kk + 3]);
          }
        }
      } else if (!dead) {
#pragma unroll
        for (int h = 0; h < PIPE_EPT / 8; ++h) {
          float u[8];
          if (KIND == REGION_SOFTMAX) {
#pragma unroll
            for (int q = 0; q < 8; ++q) u[q] = __fsub_rn(v[8 * h + q], m);
            region_exp8<EXPM>(u, tab);
          } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) u[q] = v[8 * h + q];
          }
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const int j = (2 * h + kk) * (PIPE_TT * 4) + 4 * tt;
            if (j < cols)
              *reinterpret_cast<float4*>(Er + j) = make_float4(u[4 * kk], u[4 * kk + 1], u[4 * kk + 2], u[4 * kk + 3]);
          }
        }
      }
      if (REXP) {                                            // this warp has read its x
        __syncwarp();
        if (lane == 0) mbar_arrive(&xempty[s]);
      }
      mbar_arrive(&efull[se]);
    }
    if (o >= 0 && !dead) {
      const int se = eo;
      const uint32_t par = (uint32_t)opar;
      const float* Er = E + (size_t)se * estride;
      char* yr = (char*)P.y + ((int64_t)blockIdx.x + (int64_t)o * gridDim.x) * P.ldy * ysz;
      if (BWD) {
        if (!bwd_epilogue<XT, YT>(P, yr, blockIdx.x + (int64_t)o * gridDim.x, tt, cols, &sready[se], par, &rowsum[se])) {
          abort_flag = 1;
          dead = true;
        }
        continue;
      }
      if (KIND != REGION_SOFTMAX) {
        const bool ok = P.param_dtype == PSK_BF16
                            ? norm_epilogue<KIND, YT, PSK_BF16>(P, Er, yr, tt, cols, &sready[se], par, &rowsum[se], &rowrcp[se])
                            : norm_epilogue<KIND, YT, PSK_F32>(P, Er, yr, tt, cols, &sready[se], par, &rowsum[se], &rowrcp[se]);
        if (!ok) { abort_flag = 1; dead = true; }
        continue;
      }
      if (!mbar_wait(&sready[se], par)) { abort_flag = 1; dead = true; continue; }
      const float sm = rowsum[se], rs = rowrcp[se];
      const bool fast_ok = sm >= 1.0f && sm < 0x1p20f;
      if (FASTSM && fast_ok) {
        // Markstein's correction two at a time; exp values below 2^-100 are
        // not sent to IEEE division here (their quotient may be an ulp off,
        // within the fast realization's tolerance)
        const f2 rs2 = f2_splat(rs), ns2 = f2_splat(-sm);
#pragma unroll
        for (int c4 = 0; c4 < PIPE_EPT / 4; ++c4) {
          const int j = c4 * (PIPE_TT * 4) + 4 * tt;
          if (j < cols) {
            const float4 e = *reinterpret_cast<const float4*>(Er + j);
            const f2 ea{e.x, e.y}, eb{e.z, e.w};
            const f2 qa = f2_mul(ea, rs2), qb = f2_mul(eb, rs2);
            const f2 ya = f2_fma(f2_fma(qa, ns2, ea), rs2, qa);
            const f2 yb = f2_fma(f2_fma(qb, ns2, eb), rs2, qb);
            if (YT == PSK_F32) {
              __stcs(reinterpret_cast<float4*>(yr) + (j >> 2), make_float4(ya.x, ya.y, yb.x, yb.y));
            } else {
              uint2 q;
              q.x = f32x2_to_bf16x2(ya.x, ya.y);
              q.y = f32x2_to_bf16x2(yb.x, yb.y);
              __stcs(reinterpret_cast<uint2*>(yr) + (j >> 2), q);
            }
          }
        }
        continue;
      }
#pragma unroll
      for (int c4 = 0; c4 < PIPE_EPT / 4; ++c4) {
        const int j = c4 * (PIPE_TT * 4) + 4 * tt;
        if (j < cols) {
          const float4 e = *reinterpret_cast<const float4*>(Er + j);
          float o4[4] = {e.x, e.y, e.z, e.w};
          if (MASK && sm == 0.0f) {                          // a zero sum only in a row the mask empties
            o4[0] = o4[1] = o4[2] = o4[3] = 0.0f;
          } else {
            row_div_n<4>(o4, sm, rs, fast_ok);
          }
          if (YT == PSK_F32) {
            __stcs(reinterpret_cast<float4*>(yr) + (j >> 2), make_float4(o4[0], o4[1], o4[2], o4[3]));
          } else {
            uint2 q;
            q.x = f32x2_to_bf16x2(o4[0], o4[1]);
            q.y = f32x2_to_bf16x2(o4[2], o4[3]);
            __stcs(reinterpret_cast<uint2*>(yr) + (j >> 2), q);
          }
        }
      }
    }
  }
}

// ------------------------------------------------- streaming rows (> 4096)
struct StreamShared {
  float E[SM_CAP];
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
__global__ void __launch_bounds__(SM_THREADS) softmax_stream_kernel(const __grid_constant__ RegionParams P) {
  __shared__ __align__(16) StreamShared sh;
  const int t = threadIdx.x;
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
        sh.E[i] = region_exp<EXPM>(__fsub_rn(load_x1<XT>(xr, base + i), m));
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
      float e = region_exp<EXPM>(__fsub_rn(load_x1<XT>(xr, j), m));
      store_y1<YT>(yr, j, div_by_recip(e, s, rs));
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ host
template <int XT, int YT, int EXPM, bool VEC>
static int launch_batch(RegionParams P, cudaStream_t stream) {
  constexpr int NBMAX = (XT == PSK_BF16) ? 4 : 2;
  // row buffers padded so that lanes of different rows start in different
  // banks: buffer b begins at b * estride, estride = cols rounded to 32 plus
  // the partial count rounded up to 4
  const int pad = ((P.partials + 3) / 4) * 4;
  P.nb = NBMAX;
  P.estride = (int)(((P.cols + 31) / 32) * 32 + (pad % 32));
  const size_t smem = (size_t)(P.nb * P.estride + P.nb * P.partials + 64) * sizeof(float);
  static bool attr[PSK_MAX_DEVICES] = {};
  smem_limit_once((const void*)softmax_batch_kernel<XT, YT, EXPM, VEC>, 100 * 1024, attr);
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, softmax_batch_kernel<XT, YT, EXPM, VEC>, SM_THREADS, smem);
  if (per_sm < 1) per_sm = 1;
  const int64_t nbatch = (P.rows + P.nb - 1) / P.nb;
  const int64_t cap = (int64_t)device_sm_count() * per_sm;
  const unsigned grid = (unsigned)(nbatch < cap ? nbatch : cap);
  softmax_batch_kernel<XT, YT, EXPM, VEC><<<grid, SM_THREADS, smem, stream>>>(P);
  return check_launch("softmax region kernel");
}

template <int XT, int YT, int EXPM>
static int launch_stream(const RegionParams& P, cudaStream_t stream) {
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, softmax_stream_kernel<XT, YT, EXPM>, SM_THREADS, 0);
  if (per_sm < 1) per_sm = 1;
  const int64_t cap = (int64_t)device_sm_count() * per_sm;
  const unsigned grid = (unsigned)(P.rows < cap ? P.rows : cap);
  softmax_stream_kernel<XT, YT, EXPM><<<grid, SM_THREADS, 0, stream>>>(P);
  return check_launch("softmax region kernel (streaming rows)");
}

// Ring depths from the shared-memory budget.  The value ring holds SE =
// 4 (LAG + 1) rows, about 4 LAG of them in their chains, and a team waits for
// the sums of the rows it produced LAG iterations earlier: the deeper the
// value ring, the less the teams wait, for long chains (the sequential order
// over 4096 columns) and short ones alike (interleaved(8) over 4096 columns:
// 0.247 ms at LAG 1 with 8 x slots, 0.205 ms at LAG 2 with 4).  So the value
// ring comes first, the x ring keeping 4 slots (four rows ahead per SM cover
// HBM latency), and the x ring takes 8 only where that costs no value slot.
// Chain groups take G <= 4 consecutive rows (one per team).
template <int KIND, int XT, int YT, int EXPM, bool MASK = false>
static int launch_pipe(RegionParams P, cudaStream_t stream) {
  const int pad = P.partials < 4 ? 4 : ((P.partials + 3) / 4) * 4;
  P.estride = (int)(((P.cols + 31) / 32) * 32 + pad);
  const size_t xsz = XT == PSK_F32 ? 4 : 2;
  const size_t xrow = (size_t)((P.cols * xsz * (KIND == REGION_SOFTMAX_BWD ? 2 : 1) + 127) / 128) * 128;
  const size_t erow = (size_t)P.estride * sizeof(float);
  // the correctly rounded exp makes a team's row work long enough that with
  // short chains the sums are ready in time, and the x ring's depth pays
  // instead (interleaved(8): 0.466 ms with SX = 8, SE = 8; 0.500 with 4, 12),
  // as does the exp table in shared memory (0.337 ms against 0.362 without);
  // long chains want the value ring deep instead (sequential: 0.423 ms with
  // SE = 12 and the table in global memory, 0.502 with SE = 8 and the table
  // in shared memory)
  const int64_t chain = (P.cols + P.partials - 1) / P.partials;
  const bool stage_tab = KIND == REGION_SOFTMAX && EXPM == PSK_EXP_EXACT && chain < 1024;
  const size_t tab = stage_tab ? PIPE_EXP_TAB_BYTES : 0;
  const size_t budget = PIPE_SMEM_BUDGET - tab;
  int sx = (KIND == REGION_SOFTMAX && EXPM == PSK_EXP_EXACT && chain < 1024) ? PIPE_SX_DEEP : 4;
  int se = (int)((budget - sx * xrow) / (PIPE_TEAMS * erow)) * PIPE_TEAMS;
  if (se > PIPE_SE_MAX) se = PIPE_SE_MAX;
  // x slots stay a multiple of the team count, so that each slot serves one
  // team and its parity waits run in order
  if (sx < PIPE_SX_DEEP && PIPE_SX_DEEP * xrow + se * erow <= budget) sx = PIPE_SX_DEEP;
  // PSK_PIPE_RINGS="sx,se" in the environment overrides both depths (a tuning
  // aid; ignored unless both are multiples of the team count, se >= 2 teams,
  // sx within the barrier arrays and the rings within the budget)
  static const char* rings = getenv("PSK_PIPE_RINGS");
  if (rings) {
    int a = 0, b = 0;
    if (sscanf(rings, "%d,%d", &a, &b) == 2 && a >= PIPE_TEAMS && a <= PIPE_SX_MAX && a % PIPE_TEAMS == 0 &&
        b >= 2 * PIPE_TEAMS && b <= PIPE_SE_MAX && b % PIPE_TEAMS == 0 && a * xrow + b * erow <= budget) {
      sx = a;
      se = b;
    }
  }
  if (se < 2 * PIPE_TEAMS) {  // cannot happen for cols <= 4096; kept as a guard
    return fail(PSK_E_ARG, "row ring does not fit shared memory (cols %lld)", (long long)P.cols);
  }
  P.sx = sx;
  P.se = se;
  // chain group: G in {4, 2, 1} rows (a divisor of SE) of 32 / P lanes at
  // most (P partials, at most one per column)
  const int glanes = 32 / (P.partials < P.cols ? P.partials : (int)P.cols);
  P.nb = glanes >= 4 ? 4 : (glanes >= 2 ? 2 : 1);
  const size_t smem = sx * xrow + se * erow + tab;
  const int64_t sms = device_sm_count();
  const unsigned grid = (unsigned)(P.rows < sms ? P.rows : sms);
  if constexpr (KIND == REGION_SOFTMAX && EXPM == PSK_EXP_EXACT) {
    if (stage_tab) {
      static bool attr_tab[PSK_MAX_DEVICES] = {};
      smem_limit_once((const void*)region_pipe_kernel<KIND, XT, YT, EXPM, MASK, true>, (int)PIPE_SMEM_BUDGET,
                      attr_tab);
      region_pipe_kernel<KIND, XT, YT, EXPM, MASK, true><<<grid, PIPE_THREADS, smem, stream>>>(P);
      return check_launch("row region kernel (pipelined)");
    }
  }
  static bool attr[PSK_MAX_DEVICES] = {};
  smem_limit_once((const void*)region_pipe_kernel<KIND, XT, YT, EXPM, MASK>, (int)PIPE_SMEM_BUDGET, attr);
  region_pipe_kernel<KIND, XT, YT, EXPM, MASK><<<grid, PIPE_THREADS, smem, stream>>>(P);
  return check_launch("row region kernel (pipelined)");
}

template <int XT, int YT, int EXPM>
static int dispatch_exp(const RegionParams& P, bool vec, cudaStream_t s) {
  if (P.cols > SM_CAP) return launch_stream<XT, YT, EXPM>(P, s);
  if (XT == PSK_BF16 && YT == PSK_BF16 && vec) {   // many rows: a lane per row (lanes.cu)
    bool taken = false;
    const int rc = softmax_lanes(P, EXPM, s, &taken);
    if (taken) return rc;
  }
  if (XT == PSK_BF16 && vec && P.partials <= 32 && P.cols >= 8)
    return launch_pipe<REGION_SOFTMAX, PSK_BF16, YT, EXPM>(P, s);
  return vec ? launch_batch<XT, YT, EXPM, true>(P, s) : launch_batch<XT, YT, EXPM, false>(P, s);
}

template <int XT, int YT>
static int dispatch_softmax(const RegionParams& P, int exp_mode, bool vec, cudaStream_t s) {
  return exp_mode == PSK_EXP_EXACT ? dispatch_exp<XT, YT, PSK_EXP_EXACT>(P, vec, s)
                                   : dispatch_exp<XT, YT, PSK_EXP_FAST>(P, vec, s);
}

// ------------------------------------------------ row regions, any shape
// One row at a time per CTA (grid-stride over rows): the row's values in
// shared memory as f32 -- softmax: the (masked) scores, then e = exp(x - m);
// backward: RN(ct y); norms: x -- the chains run by warp 0 (lane l takes
// partials l and l + 32, so up to 64), the partials combined left to right by
// lane 0, then every thread writes its outputs (IEEE division).  For rows the
// pipelined kernel does not take: unaligned, f32 masked scores, wider than
// 4096 (up to 49152), more than 32 partials.
constexpr int ROW_MAX_COLS = 49152;                  // 192 KB of f32 row in shared memory

template <int T>
__device__ __forceinline__ float load1(const void* base, int64_t off) {
  if (T == PSK_F32) return __ldg((const float*)base + off);
  return bf16_bits_to_f32(__ldg((const uint16_t*)base + off));
}

__device__ __forceinline__ float load1_rt(const void* base, int dtype, int64_t off) {
  return dtype == PSK_F32 ? __ldg((const float*)base + off) : bf16_bits_to_f32(__ldg((const uint16_t*)base + off));
}

template <int KIND, int XT, int YT, int EXPM>
__global__ void __launch_bounds__(SM_THREADS) region_row_kernel(const __grid_constant__ RegionParams P) {
  extern __shared__ __align__(16) float row[];
  __shared__ float part[SM_MAX_PARTIALS];
  __shared__ float red[SM_THREADS / 32];
  __shared__ float stat[2];                          // norms: mu, d; softmax: s; backward: s
  const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
  const int cols = (int)P.cols;
  const int parts = P.partials < cols ? P.partials : cols;
  const float n_f = (float)cols;                     // exact: cols <= 49152
  for (int64_t r = blockIdx.x; r < P.rows; r += gridDim.x) {
    const int64_t xo = r * P.ldx;
    if (KIND == REGION_SOFTMAX) {
      // masked scores and their maximum; a row the mask empties gets m = 0
      const uint8_t* mrow = P.mask ? P.mask + r * P.ldm : nullptr;
      float m = -INFINITY;
      int any = 0;
      for (int j = t; j < cols; j += SM_THREADS) {
        float v = load1<XT>(P.x, xo + j);
        if (mrow) {
          const bool allow = mrow[j] != 0;
          any |= allow;
          if (!allow) v = -INFINITY;
        }
        row[j] = v;
        m = max_nan(m, v);
      }
      for (int off = 16; off > 0; off >>= 1) m = max_nan(m, __shfl_xor_sync(0xffffffffu, m, off));
      if (lane == 0) red[wid] = m;
      any = __syncthreads_or(any);
      m = red[0];
      for (int q = 1; q < SM_THREADS / 32; ++q) m = max_nan(m, red[q]);
      if (mrow && !any) m = 0.0f;
      for (int j = t; j < cols; j += SM_THREADS) row[j] = region_exp<EXPM>(__fsub_rn(row[j], m));
    } else if (KIND == REGION_SOFTMAX_BWD) {
      const int64_t co = r * P.ldc;
      for (int j = t; j < cols; j += SM_THREADS)
        row[j] = __fmul_rn(load1_rt(P.ct, P.ct_dtype, co + j), load1<XT>(P.x, xo + j));
    } else {
      for (int j = t; j < cols; j += SM_THREADS) row[j] = load1<XT>(P.x, xo + j);
    }
    __syncthreads();
    if (t < 32) {
      float mu = 0.0f;
      if (KIND == REGION_LAYER) {
        for (int pp = lane; pp < parts; pp += 32) part[pp] = run_chain(row, cols, pp, parts);
        __syncwarp();
        if (lane == 0) {
          float s1 = part[0];
          for (int q = 1; q < parts; ++q) s1 = __fadd_rn(s1, part[q]);
          stat[0] = __fdiv_rn(s1, n_f);
        }
        __syncwarp();
        mu = stat[0];
        for (int pp = lane; pp < parts; pp += 32)
          part[pp] = run_chain(row, cols, pp, parts, ChainCenteredSquare{mu});
      } else if (KIND == REGION_RMS) {
        for (int pp = lane; pp < parts; pp += 32) part[pp] = run_chain(row, cols, pp, parts, ChainSquare());
      } else {
        for (int pp = lane; pp < parts; pp += 32) part[pp] = run_chain(row, cols, pp, parts);
      }
      __syncwarp();
      if (lane == 0) {
        float ss = part[0];
        for (int q = 1; q < parts; ++q) ss = __fadd_rn(ss, part[q]);
        stat[0] = mu;
        stat[1] = (KIND == REGION_RMS || KIND == REGION_LAYER) ? __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, n_f), P.eps)) : ss;
      }
    }
    __syncthreads();
    const float mu = stat[0], d = stat[1];
    const int64_t yo = r * P.ldy;
    for (int j = t; j < cols; j += SM_THREADS) {
      float v = row[j];
      if (KIND == REGION_SOFTMAX) {
        v = d == 0.0f ? 0.0f : __fdiv_rn(v, d);       // a zero sum only in a row the mask empties
      } else if (KIND == REGION_SOFTMAX_BWD) {
        const float y = load1<XT>(P.x, xo + j), c = load1_rt(P.ct, P.ct_dtype, r * P.ldc + j);
        v = __fmul_rn(y, __fsub_rn(c, d));
      } else {
        if (KIND == REGION_LAYER) v = __fsub_rn(v, mu);
        v = __fdiv_rn(v, d);
        if (P.gamma) v = __fmul_rn(v, load1_rt(P.gamma, P.param_dtype, j));
        if (KIND == REGION_LAYER && P.beta) v = __fadd_rn(v, load1_rt(P.beta, P.param_dtype, j));
      }
      store_y1<YT>(P.y, yo + j, v);
    }
    __syncthreads();
  }
}

template <int KIND, int XT, int YT, int EXPM>
static int launch_region_rows(const RegionParams& P, cudaStream_t stream) {
  const size_t smem = (size_t)P.cols * sizeof(float);
  static bool attr[PSK_MAX_DEVICES] = {};
  smem_limit_once((const void*)region_row_kernel<KIND, XT, YT, EXPM>, (int)(ROW_MAX_COLS * sizeof(float)), attr);
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, region_row_kernel<KIND, XT, YT, EXPM>, SM_THREADS, smem);
  if (per_sm < 1) per_sm = 1;
  const int64_t cap = (int64_t)device_sm_count() * per_sm;
  const unsigned grid = (unsigned)(P.rows < cap ? P.rows : cap);
  region_row_kernel<KIND, XT, YT, EXPM><<<grid, SM_THREADS, smem, stream>>>(P);
  return check_launch("row region kernel (row at a time)");
}

template <int KIND, int XT, int YT>
static int dispatch_norm(const RegionParams& P, bool pipe, cudaStream_t s) {
  if (pipe) return launch_pipe<KIND, XT, YT, PSK_EXP_EXACT>(P, s);
  return launch_region_rows<KIND, XT, YT, PSK_EXP_EXACT>(P, s);
}

template <int KIND>
static int dispatch_norm_types(const RegionParams& P, int xt, int yt, bool pipe, cudaStream_t s) {
  if (xt == PSK_BF16 && yt == PSK_BF16) return dispatch_norm<KIND, PSK_BF16, PSK_BF16>(P, pipe, s);
  if (xt == PSK_BF16 && yt == PSK_F32) return dispatch_norm<KIND, PSK_BF16, PSK_F32>(P, pipe, s);
  if (xt == PSK_F32 && yt == PSK_BF16) return dispatch_norm<KIND, PSK_F32, PSK_BF16>(P, pipe, s);
  return dispatch_norm<KIND, PSK_F32, PSK_F32>(P, pipe, s);
}

// masked softmax: the pipelined kernel for bf16 scores with 4-byte aligned
// mask rows, the row kernel otherwise
template <int XT, int YT, int EXPM>
static int dispatch_masked_exp(const RegionParams& P, bool pipe, cudaStream_t s) {
  if (XT == PSK_BF16 && pipe) return launch_pipe<REGION_SOFTMAX, PSK_BF16, YT, EXPM, true>(P, s);
  return launch_region_rows<REGION_SOFTMAX, XT, YT, EXPM>(P, s);
}

template <int XT, int YT>
static int dispatch_masked(const RegionParams& P, int exp_mode, bool pipe, cudaStream_t s) {
  return exp_mode == PSK_EXP_EXACT ? dispatch_masked_exp<XT, YT, PSK_EXP_EXACT>(P, pipe, s)
                                   : dispatch_masked_exp<XT, YT, PSK_EXP_FAST>(P, pipe, s);
}

template <int XT, int YT>
static int dispatch_bwd(const RegionParams& P, bool pipe, cudaStream_t s) {
  if (XT == PSK_BF16 && YT == PSK_BF16 && pipe) {   // many rows, one chain: a lane per row (lanes.cu)
    bool taken = false;
    const int rc = softmax_bwd_lanes(P, s, &taken);
    if (taken) return rc;
  }
  if (pipe) return launch_pipe<REGION_SOFTMAX_BWD, XT, YT, PSK_EXP_EXACT>(P, s);
  return launch_region_rows<REGION_SOFTMAX_BWD, XT, YT, PSK_EXP_EXACT>(P, s);
}

}  // namespace psk

using namespace psk;

// Number of partial chains of a declared order, or a refusal (shared by both
// region entry points).
static int order_partials(const psk_order& order, int* partials) {
  *partials = 1;
  switch (order.kind) {
    case PSK_ORDER_SEQUENTIAL: return PSK_OK;
    case PSK_ORDER_BLOCKED:
      if (order.param < 1) return fail(PSK_E_ORDER, "blocked width %d < 1", order.param);
      return PSK_OK;
    case PSK_ORDER_INTERLEAVED:
      if (order.param < 1 || order.param > SM_MAX_PARTIALS)
        return fail(PSK_E_ORDER, "interleaved partials %d (1..%d)", order.param, SM_MAX_PARTIALS);
      *partials = order.param;
      return PSK_OK;
    default:
      return fail(PSK_E_ORDER, "order kind %d", order.kind);
  }
}

static bool overlaps(const void* a, size_t abytes, const void* b, size_t bbytes) {
  const char* a0 = (const char*)a;
  const char* b0 = (const char*)b;
  return a0 < b0 + bbytes && b0 < a0 + abytes;
}

extern "C" int psk_norm_region(const void* x, int32_t xt, void* y, int32_t yt, int64_t rows, int64_t cols,
                               int64_t ldx, int64_t ldy, int32_t kind, double eps, const void* gamma,
                               const void* beta, int32_t param_dtype, psk_order order, void* stream) {
  clear_error();
  if (!dtype_ok(xt)) return fail(PSK_E_DTYPE, "x dtype %d", xt);
  if (!dtype_ok(yt)) return fail(PSK_E_DTYPE, "y dtype %d", yt);
  if (kind != PSK_NORM_RMS && kind != PSK_NORM_LAYER) return fail(PSK_E_ARG, "norm kind %d", kind);
  if (!(eps == eps) || eps > 3.4e38 || eps < -3.4e38) return fail(PSK_E_ARG, "eps is not a finite f32 value");
  if (kind == PSK_NORM_RMS && beta) return fail(PSK_E_ARG, "RMSNorm takes no bias");
  if ((gamma || beta) && !dtype_ok(param_dtype)) return fail(PSK_E_DTYPE, "parameter dtype %d", param_dtype);
  if (rows < 0 || cols < 0) return fail(PSK_E_SHAPE, "rows %lld, cols %lld", (long long)rows, (long long)cols);
  int partials = 1;
  int rc = order_partials(order, &partials);
  if (rc) return rc;
  if (rows == 0 || cols == 0) return PSK_OK;
  if (cols > ROW_MAX_COLS) return fail(PSK_E_SHAPE, "cols %lld above %d", (long long)cols, ROW_MAX_COLS);
  if (!x || !y) return fail(PSK_E_NULL, "x or y is NULL");
  if (ldx < cols || ldy < cols) return fail(PSK_E_SHAPE, "leading dimension below cols");
  const size_t xbytes = (size_t)((rows - 1) * ldx + cols) * dtype_size(xt);
  const size_t ybytes = (size_t)((rows - 1) * ldy + cols) * dtype_size(yt);
  if (overlaps(x, xbytes, y, ybytes) && !(x == y && xt == yt && ldx == ldy))
    return fail(PSK_E_ALIAS, "y overlaps x and is not the same buffer");
  const size_t pbytes = (size_t)cols * dtype_size(param_dtype);
  if ((gamma && overlaps(gamma, pbytes, y, ybytes)) || (beta && overlaps(beta, pbytes, y, ybytes)))
    return fail(PSK_E_ALIAS, "y overlaps gamma or beta");
  RegionParams P{x, y, rows, cols, ldx, ldy, partials, 1, 0, 0, 0, gamma, beta, param_dtype, (float)eps};
  const bool pipe = cols <= SM_CAP && cols >= 8 && cols % 8 == 0 && ldx % 8 == 0 && ldy % 8 == 0 &&
                    partials <= 32 && (uintptr_t)x % 16 == 0 && (uintptr_t)y % 16 == 0 &&
                    (uintptr_t)gamma % 16 == 0 && (uintptr_t)beta % 16 == 0;
  cudaStream_t s = (cudaStream_t)stream;
  if (xt == PSK_BF16 && yt == PSK_BF16) {   // many rows: a lane per row (lanes.cu)
    bool taken = false;
    const int rc = norm_lanes(P, kind == PSK_NORM_RMS ? REGION_RMS : REGION_LAYER, s, &taken);
    if (taken) return rc;
  }
  return kind == PSK_NORM_RMS ? dispatch_norm_types<REGION_RMS>(P, xt, yt, pipe, s)
                              : dispatch_norm_types<REGION_LAYER>(P, xt, yt, pipe, s);
}

extern "C" int psk_test_drop_row(int64_t row) {
  clear_error();
  if (row < -1) return fail(PSK_E_ARG, "row %lld (-1 or a local row index)", (long long)row);
  const long long v = row;
  if (cudaMemcpyToSymbol(g_pipe_drop_row, &v, sizeof(v)) != cudaSuccess) return check_launch("test hook write");
  return lanes_set_drop_row(v);
}

namespace psk {
// The softmax region's fast exp, elementwise (the test hook below).
__global__ void fast_exp_kernel(const float* x, float* y, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    y[i] = exp_unit_nonpos(x[i]);
}
}  // namespace psk

extern "C" int psk_test_fast_exp(const float* x, float* y, int64_t n, void* stream) {
  clear_error();
  if (n < 0) return fail(PSK_E_SHAPE, "n %lld", (long long)n);
  if (n == 0) return PSK_OK;
  if (!x || !y) return fail(PSK_E_NULL, "x or y is NULL");
  const int64_t blocks = (n + 255) / 256;
  const int64_t cap = device_sm_count() * 8;
  fast_exp_kernel<<<(unsigned)(blocks < cap ? blocks : cap), 256, 0, (cudaStream_t)stream>>>(x, y, n);
  return check_launch("fast exp test kernel");
}

extern "C" int psk_device_status(uint32_t* status, int32_t reset) {
  clear_error();
  if (!status) return fail(PSK_E_NULL, "status is NULL");
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_pipe_status, sizeof(v)) != cudaSuccess) return check_launch("device status read");
  if (reset) {
    const unsigned int z = 0;
    if (cudaMemcpyToSymbol(g_pipe_status, &z, sizeof(z)) != cudaSuccess) return check_launch("device status reset");
  }
  unsigned int lv = 0;
  const int lrc = lanes_status(&lv, reset != 0);
  if (lrc) return lrc;
  *status = v | lv;
  return PSK_OK;
}

extern "C" int psk_softmax_region(const void* x, int32_t xt, void* y, int32_t yt, int64_t rows, int64_t cols,
                                  int64_t ldx, int64_t ldy, psk_order order, int32_t exp_mode, void* stream) {
  clear_error();
  if (!dtype_ok(xt)) return fail(PSK_E_DTYPE, "x dtype %d", xt);
  if (!dtype_ok(yt)) return fail(PSK_E_DTYPE, "y dtype %d", yt);
  if (rows < 0 || cols < 0) return fail(PSK_E_SHAPE, "rows %lld, cols %lld", (long long)rows, (long long)cols);
  if (cols > 0x7FFFFFFF) return fail(PSK_E_SHAPE, "cols %lld above 2^31-1", (long long)cols);
  if (exp_mode != PSK_EXP_EXACT && exp_mode != PSK_EXP_FAST) return fail(PSK_E_ARG, "exp_mode %d", exp_mode);
  int partials = 1;
  const int orc = order_partials(order, &partials);
  if (orc) return orc;
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
  RegionParams P{x, y, rows, cols, ldx, ldy, partials, 1, 0, 0, 0};
  const bool vec = (cols % 8 == 0) && (ldx % 8 == 0) && (ldy % 8 == 0) && ((uintptr_t)x % 16 == 0) &&
                   ((uintptr_t)y % 16 == 0);
  cudaStream_t s = (cudaStream_t)stream;
  if (xt == PSK_BF16 && yt == PSK_BF16) return dispatch_softmax<PSK_BF16, PSK_BF16>(P, exp_mode, vec, s);
  if (xt == PSK_BF16 && yt == PSK_F32) return dispatch_softmax<PSK_BF16, PSK_F32>(P, exp_mode, vec, s);
  if (xt == PSK_F32 && yt == PSK_BF16) return dispatch_softmax<PSK_F32, PSK_BF16>(P, exp_mode, vec, s);
  return dispatch_softmax<PSK_F32, PSK_F32>(P, exp_mode, vec, s);
}

extern "C" int psk_softmax_masked(const void* x, int32_t xt, void* y, int32_t yt, int64_t rows, int64_t cols,
                                  int64_t ldx, int64_t ldy, const uint8_t* mask, int64_t ldm, psk_order order,
                                  int32_t exp_mode, void* stream) {
  clear_error();
  if (!dtype_ok(xt)) return fail(PSK_E_DTYPE, "x dtype %d", xt);
  if (!dtype_ok(yt)) return fail(PSK_E_DTYPE, "y dtype %d", yt);
  if (rows < 0 || cols < 0) return fail(PSK_E_SHAPE, "rows %lld, cols %lld", (long long)rows, (long long)cols);
  if (exp_mode != PSK_EXP_EXACT && exp_mode != PSK_EXP_FAST) return fail(PSK_E_ARG, "exp_mode %d", exp_mode);
  int partials = 1;
  const int orc = order_partials(order, &partials);
  if (orc) return orc;
  if (rows == 0 || cols == 0) return PSK_OK;
  if (cols > ROW_MAX_COLS) return fail(PSK_E_SHAPE, "masked rows of %lld columns (max %d)", (long long)cols, ROW_MAX_COLS);
  if (!x || !y || !mask) return fail(PSK_E_NULL, "x, y or mask is NULL");
  if (ldx < cols || ldy < cols) return fail(PSK_E_SHAPE, "leading dimension below cols");
  if (ldm != 0 && ldm < cols) return fail(PSK_E_SHAPE, "mask leading dimension %lld (0 or >= cols)", (long long)ldm);
  const size_t xbytes = (size_t)((rows - 1) * ldx + cols) * dtype_size(xt);
  const size_t ybytes = (size_t)((rows - 1) * ldy + cols) * dtype_size(yt);
  const size_t mbytes = (size_t)(ldm == 0 ? cols : (rows - 1) * ldm + cols);
  if (overlaps(x, xbytes, y, ybytes) && !(x == y && xt == yt && ldx == ldy))
    return fail(PSK_E_ALIAS, "y overlaps x and is not the same buffer");
  if (overlaps(mask, mbytes, y, ybytes)) return fail(PSK_E_ALIAS, "y overlaps the mask");
  RegionParams P{x, y, rows, cols, ldx, ldy, partials, 1, 0, 0, 0};
  P.mask = mask;
  P.ldm = ldm;
  const bool pipe = cols <= SM_CAP && cols >= 8 && cols % 8 == 0 && ldx % 8 == 0 && ldy % 8 == 0 &&
                    partials <= 32 && (uintptr_t)x % 16 == 0 && (uintptr_t)y % 16 == 0 &&
                    (uintptr_t)mask % 4 == 0 && ldm % 4 == 0;
  cudaStream_t s = (cudaStream_t)stream;
  if (xt == PSK_BF16 && yt == PSK_BF16) return dispatch_masked<PSK_BF16, PSK_BF16>(P, exp_mode, pipe, s);
  if (xt == PSK_BF16 && yt == PSK_F32) return dispatch_masked<PSK_BF16, PSK_F32>(P, exp_mode, pipe, s);
  if (xt == PSK_F32 && yt == PSK_BF16) return dispatch_masked<PSK_F32, PSK_BF16>(P, exp_mode, pipe, s);
  return dispatch_masked<PSK_F32, PSK_F32>(P, exp_mode, pipe, s);
}

extern "C" int psk_softmax_backward(const void* y, int32_t yt, const void* ct, int32_t ct_t, void* dx, int32_t dxt,
                                    int64_t rows, int64_t cols, int64_t ldy, int64_t ldc, int64_t ldd,
                                    psk_order order, void* stream) {
  clear_error();
  if (!dtype_ok(yt) || !dtype_ok(ct_t) || !dtype_ok(dxt)) return fail(PSK_E_DTYPE, "storage type of y, ct or dx");
  if (rows < 0 || cols < 0) return fail(PSK_E_SHAPE, "rows %lld, cols %lld", (long long)rows, (long long)cols);
  int partials = 1;
  const int orc = order_partials(order, &partials);
  if (orc) return orc;
  if (rows == 0 || cols == 0) return PSK_OK;
  if (cols > ROW_MAX_COLS) return fail(PSK_E_SHAPE, "rows of %lld columns (max %d)", (long long)cols, ROW_MAX_COLS);
  if (!y || !ct || !dx) return fail(PSK_E_NULL, "y, ct or dx is NULL");
  if (ldy < cols || ldc < cols || ldd < cols) return fail(PSK_E_SHAPE, "leading dimension below cols");
  const size_t ybytes = (size_t)((rows - 1) * ldy + cols) * dtype_size(yt);
  const size_t cbytes = (size_t)((rows - 1) * ldc + cols) * dtype_size(ct_t);
  const size_t dbytes = (size_t)((rows - 1) * ldd + cols) * dtype_size(dxt);
  if (overlaps(dx, dbytes, y, ybytes) && !(dx == y && dxt == yt && ldd == ldy))
    return fail(PSK_E_ALIAS, "dx overlaps y and is not the same buffer");
  if (overlaps(dx, dbytes, ct, cbytes) && !(dx == ct && dxt == ct_t && ldd == ldc))
    return fail(PSK_E_ALIAS, "dx overlaps ct and is not the same buffer");
  RegionParams P{y, dx, rows, cols, ldy, ldd, partials, 1, 0, 0, 0};
  P.ct = ct;
  P.ldc = ldc;
  P.ct_dtype = ct_t;
  const bool pipe = ct_t == yt && cols <= SM_CAP && cols >= 8 && cols % 8 == 0 && ldy % 8 == 0 && ldc % 8 == 0 &&
                    ldd % 8 == 0 && partials <= 32 && (uintptr_t)y % 16 == 0 && (uintptr_t)ct % 16 == 0 &&
                    (uintptr_t)dx % 16 == 0;
  cudaStream_t s = (cudaStream_t)stream;
  if (yt == PSK_BF16 && dxt == PSK_BF16) return dispatch_bwd<PSK_BF16, PSK_BF16>(P, pipe, s);
  if (yt == PSK_BF16 && dxt == PSK_F32) return dispatch_bwd<PSK_BF16, PSK_F32>(P, pipe, s);
  if (yt == PSK_F32 && dxt == PSK_BF16) return dispatch_bwd<PSK_F32, PSK_BF16>(P, pipe, s);
  return dispatch_bwd<PSK_F32, PSK_F32>(P, pipe, s);
}
