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
#include "pipe.cuh"

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
  int32_t nb;           // rows per batch (resident kernel) / per chain group (pipelined)
  int32_t estride;      // floats between row buffers in shared memory
  int32_t sx, se;       // pipelined kernel: x and exp ring slots
};

// NaN-propagating max (exact; the order of a max reduction changes no bit
// except the sign of a zero maximum, which no exp(x - m) can see).
__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

template <int EXPM>
__device__ __forceinline__ float region_exp(float d) {
  if (EXPM == PSK_EXP_FAST) return exp_faithful_nonpos(d);
  return exp_cr(d, psk_exp_tab2);
}

// exp of eight values: the correctly rounded tier-1 cores run side by side
// (independent chains for the scheduler), the rare undecided lanes after.
template <int EXPM>
__device__ __forceinline__ void region_exp8(float* v) {
  if constexpr (EXPM == PSK_EXP_FAST) {
#pragma unroll
    for (int q = 0; q < 8; ++q) v[q] = exp_faithful_nonpos(v[q]);
  } else {
    float R[8], d[8];
    int n[8];
    bool inr[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      inr[q] = fabsf(v[q]) <= 87.0f;
      exp_tier1_core(inr[q] ? v[q] : 0.0f, psk_exp_tab2, R[q], d[q], n[q]);
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      float out = u2f((uint32_t)((int32_t)f2u(R[q]) + n[q] * (1 << 23)));
      if (!(inr[q] && tier1_decided(R[q], d[q]))) out = exp_tier2(v[q]);
      v[q] = out;
    }
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

// N quotients e_q / s at once: Markstein's correction for all, one test for
// the whole group, and the per-element path (IEEE division where the
// correction's operand range is left) only for a group that needs it.
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
    bad = bad || !(e >= 0x1p-100f);
  }
  if (bad) {
#pragma unroll
    for (int q = 0; q < N; ++q) y[q] = row_div(o[q], s, rs, fast_ok);
  }
#pragma unroll
  for (int q = 0; q < N; ++q) o[q] = y[q];
}

// One chain: acc over E[p], E[p+P], ... (n elements in the row), in index
// order.  The loads of the next block are issued before the dependent adds of
// the current one (registers double-buffered), so the chain runs at the add
// latency instead of add + shared-memory latency per block.
__device__ __forceinline__ float run_chain(const float* E, int n, int p, int P) {
  float acc = E[p];
  int j = p + P;
  if (P == 1) {
    for (; (j & 3) != 0 && j < n; ++j) acc = __fadd_rn(acc, E[j]);
    if (j + 15 < n) {
      float4 a = *(const float4*)&E[j], b = *(const float4*)&E[j + 4];
      float4 c = *(const float4*)&E[j + 8], d = *(const float4*)&E[j + 12];
      for (; j + 31 < n; j += 16) {
        const float4 na = *(const float4*)&E[j + 16], nb = *(const float4*)&E[j + 20];
        const float4 nc = *(const float4*)&E[j + 24], nd = *(const float4*)&E[j + 28];
        acc = __fadd_rn(acc, a.x); acc = __fadd_rn(acc, a.y); acc = __fadd_rn(acc, a.z); acc = __fadd_rn(acc, a.w);
        acc = __fadd_rn(acc, b.x); acc = __fadd_rn(acc, b.y); acc = __fadd_rn(acc, b.z); acc = __fadd_rn(acc, b.w);
        acc = __fadd_rn(acc, c.x); acc = __fadd_rn(acc, c.y); acc = __fadd_rn(acc, c.z); acc = __fadd_rn(acc, c.w);
        acc = __fadd_rn(acc, d.x); acc = __fadd_rn(acc, d.y); acc = __fadd_rn(acc, d.z); acc = __fadd_rn(acc, d.w);
        a = na; b = nb; c = nc; d = nd;
      }
      acc = __fadd_rn(acc, a.x); acc = __fadd_rn(acc, a.y); acc = __fadd_rn(acc, a.z); acc = __fadd_rn(acc, a.w);
      acc = __fadd_rn(acc, b.x); acc = __fadd_rn(acc, b.y); acc = __fadd_rn(acc, b.z); acc = __fadd_rn(acc, b.w);
      acc = __fadd_rn(acc, c.x); acc = __fadd_rn(acc, c.y); acc = __fadd_rn(acc, c.z); acc = __fadd_rn(acc, c.w);
      acc = __fadd_rn(acc, d.x); acc = __fadd_rn(acc, d.y); acc = __fadd_rn(acc, d.z); acc = __fadd_rn(acc, d.w);
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
      for (int i = 0; i < 8; ++i) acc = __fadd_rn(acc, v[i]);
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = nv[i];
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) acc = __fadd_rn(acc, v[i]);
    j += 8 * P;
  }
  for (; j < n; j += P) acc = __fadd_rn(acc, E[j]);
  return acc;
}

// --------------------------------------------------- resident rows (<= 4096)
template <int XT, int YT, int EXPM, bool VEC>
__global__ void __launch_bounds__(SM_THREADS, 3) softmax_batch_kernel(const __grid_constant__ SoftmaxParams P) {
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


// ------------------------------------- pipelined rows (bf16, <= 4096 columns)
// One persistent CTA per SM with three roles:
//   a producer warp streams this CTA's rows (bf16) into a shared ring of SX
//   slots with 1-D bulk copies (TMA) that complete on the slot's mbarrier;
//   4 teams of 4 compute warps each take every 4th row of the CTA (so four
//   rows are in the compute stage at once, each team synchronising only
//   within itself): the row's max (warp shuffles + a team barrier), e =
//   exp(x - m) into a shared ring of SE f32 rows, then -- LAG = SE/4 - 1 team
//   rows later, once the chain warps have published the row sum -- e / s,
//   stored with streaming stores;
//   3 chain warps each take groups of G consecutive rows: lane (row, p) adds
//   chain p of its row in index order, the partials are combined left to
//   right, and the row's sum and RN(1/s) are published on the row's mbarrier.
// A row's chain is a serial run of cols/P dependent adds, so about 4 LAG
// rows chain at once; long chains (sequential order) get a deeper exp ring
// and a shallower x ring.  Every wait is bounded (pipe.cuh).
constexpr int PIPE_TEAMS = 4;
constexpr int PIPE_TW = 4;                                   // warps per team
constexpr int PIPE_CW = PIPE_TEAMS * PIPE_TW;                // compute warps (16)
constexpr int PIPE_TT = PIPE_TW * 32;                        // threads per team (128)
constexpr int PIPE_EPT = SM_CAP / PIPE_TT;                   // row elements per team thread (32)
constexpr int PIPE_KW = 3;                                   // chain warps
constexpr int PIPE_THREADS = (PIPE_CW + PIPE_KW + 1) * 32;   // + producer warp
constexpr int PIPE_SX_MAX = 8;                               // x ring slots
constexpr int PIPE_SE_MAX = 16;                              // exp ring slots (a multiple of the teams)
constexpr size_t PIPE_SMEM_BUDGET = 225 * 1024;              // dynamic shared memory of one CTA

template <int YT, int EXPM>
__global__ void __launch_bounds__(PIPE_THREADS, 1) softmax_pipe_kernel(const __grid_constant__ SoftmaxParams P) {
  extern __shared__ __align__(128) unsigned char pipe_smem[];
  __shared__ __align__(8) uint64_t xfull[PIPE_SX_MAX], xempty[PIPE_SX_MAX], efull[PIPE_SE_MAX], sready[PIPE_SE_MAX];
  __shared__ float rowsum[PIPE_SE_MAX], rowrcp[PIPE_SE_MAX];
  __shared__ float red[PIPE_TEAMS][2][PIPE_TW];
  __shared__ volatile int abort_flag;

  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int cols = (int)P.cols;
  const uint32_t xbytes = (uint32_t)cols * 2u;
  const int xstr = (int)(((xbytes + 127u) / 128u) * 64u);    // ring slot stride in bf16 elements
  const int SX = P.sx, SE = P.se, LAG = P.se / PIPE_TEAMS - 1;
  uint16_t* X = reinterpret_cast<uint16_t*>(pipe_smem);
  float* E = reinterpret_cast<float*>(pipe_smem + (size_t)SX * xstr * 2);
  const int estride = P.estride;
  const int parts = P.partials < cols ? P.partials : cols;  // a partial beyond the row is empty
  const int G = P.nb;                                        // rows per chain group
  const int n_local = blockIdx.x < P.rows ? (int)((P.rows - 1 - blockIdx.x) / gridDim.x + 1) : 0;

  if (tid == 0) {
    for (int i = 0; i < SX; ++i) { mbar_init(&xfull[i], 1); mbar_init(&xempty[i], 1); }
    for (int i = 0; i < SE; ++i) { mbar_init(&efull[i], PIPE_TT); mbar_init(&sready[i], 1); }
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (w == PIPE_CW + PIPE_KW) {
    // ---------------- producer
    if (lane == 0) {
      int issued = 0;
      const uint16_t* src = (const uint16_t*)P.x + (int64_t)blockIdx.x * P.ldx;
      const int64_t step = (int64_t)gridDim.x * P.ldx;
      for (int i = 0; i < n_local; ++i) {
        const int s = i % SX;
        if (i >= SX && !mbar_wait(&xempty[s], (uint32_t)((i / SX) - 1) & 1u)) { abort_flag = 1; break; }
        if (abort_flag) break;
        mbar_arrive_expect_tx(&xfull[s], xbytes);
        bulk_copy_g2s(X + (size_t)s * xstr, src, xbytes, &xfull[s]);
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
    // pass at once), so every slot group of the exp ring (G consecutive
    // slots) belongs to one chain warp, which visits its phases in order.
    const int c = w - PIPE_CW;
    const int b = lane / parts, p = lane - (lane / parts) * parts;
    const int n_groups = SE / G;
    for (int g = 0; g * G < n_local; ++g) {
      if ((g % n_groups) % PIPE_KW != c) continue;
      if (abort_flag) break;
      const int j = g * G + b;
      const bool act = b < G && j < n_local;
      const int se = j % SE;
      bool ok = true;
      if (act) ok = mbar_wait(&efull[se], (uint32_t)(j / SE) & 1u);
      if (__any_sync(0xffffffffu, !ok)) { abort_flag = 1; break; }
      const float acc = act ? run_chain(E + (size_t)se * estride, cols, p, parts) : 0.0f;
      float sum = acc;
      for (int q = 1; q < parts; ++q) {
        const float o = __shfl_sync(0xffffffffu, acc, (lane - p + q) & 31);
        if (act) sum = __fadd_rn(sum, o);
      }
      if (act && p == 0) {
        rowsum[se] = sum;
        rowrcp[se] = __frcp_rn(sum);
        mbar_arrive(&sready[se]);
      }
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
  for (int k = 0;; ++k) {
    const int i = team + PIPE_TEAMS * k;                     // row produced in this team iteration
    const int o = i - PIPE_TEAMS * LAG;                      // row output in this team iteration
    if (o >= n_local) break;
    dead = dead || abort_flag;
    if (i < n_local) {
      const int s = i % SX;
      if (!dead && !mbar_wait(&xfull[s], (uint32_t)(i / SX) & 1u)) { abort_flag = 1; dead = true; }
      const uint16_t* xs = X + (size_t)s * xstr;
      float v[PIPE_EPT];
      float m = -INFINITY;
#pragma unroll
      for (int c4 = 0; c4 < PIPE_EPT / 4; ++c4) {
        const int j = c4 * (PIPE_TT * 4) + 4 * tt;
        if (j < cols && !dead) {
          const uint2 q = *reinterpret_cast<const uint2*>(xs + j);
          v[4 * c4 + 0] = __uint_as_float(q.x << 16);
          v[4 * c4 + 1] = __uint_as_float(q.x & 0xFFFF0000u);
          v[4 * c4 + 2] = __uint_as_float(q.y << 16);
          v[4 * c4 + 3] = __uint_as_float(q.y & 0xFFFF0000u);
        } else {
          v[4 * c4 + 0] = v[4 * c4 + 1] = v[4 * c4 + 2] = v[4 * c4 + 3] = -INFINITY;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) m = max_nan(m, v[4 * c4 + q]);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = max_nan(m, __shfl_xor_sync(0xffffffffu, m, off));
      if (lane == 0) red[team][k & 1][tw] = m;
      named_barrier(1 + team, PIPE_TT);
      m = red[team][k & 1][0];
#pragma unroll
      for (int q = 1; q < PIPE_TW; ++q) m = max_nan(m, red[team][k & 1][q]);
      if (tt == 0) mbar_arrive(&xempty[s]);              // every team thread has read x
      const int se = i % SE;
      float* Er = E + (size_t)se * estride;
      if (!dead) {
#pragma unroll
        for (int h = 0; h < PIPE_EPT / 8; ++h) {
          float u[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) u[q] = __fsub_rn(v[8 * h + q], m);
          region_exp8<EXPM>(u);
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const int j = (2 * h + kk) * (PIPE_TT * 4) + 4 * tt;
            if (j < cols)
              *reinterpret_cast<float4*>(Er + j) = make_float4(u[4 * kk], u[4 * kk + 1], u[4 * kk + 2], u[4 * kk + 3]);
          }
        }
      }
      mbar_arrive(&efull[se]);
    }
    if (o >= 0 && !dead) {
      const int se = o % SE;
      if (!mbar_wait(&sready[se], (uint32_t)(o / SE) & 1u)) { abort_flag = 1; dead = true; continue; }
      const float sm = rowsum[se], rs = rowrcp[se];
      const bool fast_ok = sm >= 1.0f && sm < 0x1p20f;
      const float* Er = E + (size_t)se * estride;
      char* yr = (char*)P.y + ((int64_t)blockIdx.x + (int64_t)o * gridDim.x) * P.ldy * ysz;
#pragma unroll
      for (int c4 = 0; c4 < PIPE_EPT / 4; ++c4) {
        const int j = c4 * (PIPE_TT * 4) + 4 * tt;
        if (j < cols) {
          const float4 e = *reinterpret_cast<const float4*>(Er + j);
          float o[4] = {e.x, e.y, e.z, e.w};
          row_div_n<4>(o, sm, rs, fast_ok);
          const float o0 = o[0], o1 = o[1], o2 = o[2], o3 = o[3];
          if (YT == PSK_F32) {
            __stcs(reinterpret_cast<float4*>(yr) + (j >> 2), make_float4(o0, o1, o2, o3));
          } else {
            uint2 q;
            q.x = f32x2_to_bf16x2(o0, o1);
            q.y = f32x2_to_bf16x2(o2, o3);
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
__global__ void __launch_bounds__(SM_THREADS) softmax_stream_kernel(const __grid_constant__ SoftmaxParams P) {
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
static int launch_batch(SoftmaxParams P, cudaStream_t stream) {
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
static int launch_stream(const SoftmaxParams& P, cudaStream_t stream) {
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, softmax_stream_kernel<XT, YT, EXPM>, SM_THREADS, 0);
  if (per_sm < 1) per_sm = 1;
  const int64_t cap = (int64_t)device_sm_count() * per_sm;
  const unsigned grid = (unsigned)(P.rows < cap ? P.rows : cap);
  softmax_stream_kernel<XT, YT, EXPM><<<grid, SM_THREADS, 0, stream>>>(P);
  return check_launch("softmax region kernel (streaming rows)");
}

// Ring depths from the shared-memory budget.  Eight bf16 rows in flight per
// SM cover HBM latency; the exp ring holds SE = 4 (LAG + 1) rows, about 4 LAG
// of them in their chains.  A long chain (cols / P >= 1024 adds, e.g. the
// sequential order over 4096 columns) is the bottleneck, so it gets the exp
// ring first (x ring down to 4 slots); otherwise the x ring comes first.
// Chain groups take G <= 4 consecutive rows (one per team).
template <int YT, int EXPM>
static int launch_pipe(SoftmaxParams P, cudaStream_t stream) {
  const int pad = P.partials < 4 ? 4 : ((P.partials + 3) / 4) * 4;
  P.estride = (int)(((P.cols + 31) / 32) * 32 + pad);
  const size_t xrow = (size_t)((P.cols * 2 + 127) / 128) * 128;
  const size_t erow = (size_t)P.estride * sizeof(float);
  const size_t budget = PIPE_SMEM_BUDGET;
  const bool long_chain = (P.cols + P.partials - 1) / P.partials >= 1024;
  int sx = long_chain ? 4 : PIPE_SX_MAX;
  int se = (int)((budget - sx * xrow) / (PIPE_TEAMS * erow)) * PIPE_TEAMS;
  if (se > PIPE_SE_MAX) se = PIPE_SE_MAX;
  // x slots stay a multiple of the team count, so that each slot serves one
  // team and its parity waits run in order
  if (sx < PIPE_SX_MAX && PIPE_SX_MAX * xrow + se * erow <= budget) sx = PIPE_SX_MAX;
  if (se < 2 * PIPE_TEAMS) {  // cannot happen for cols <= 4096; kept as a guard
    return fail(PSK_E_ARG, "softmax ring does not fit shared memory (cols %lld)", (long long)P.cols);
  }
  P.sx = sx;
  P.se = se;
  // chain group: G in {4, 2, 1} rows (a divisor of SE) of 32 / P lanes at
  // most (P partials, at most one per column)
  const int glanes = 32 / (P.partials < P.cols ? P.partials : (int)P.cols);
  P.nb = glanes >= 4 ? 4 : (glanes >= 2 ? 2 : 1);
  const size_t smem = sx * xrow + se * erow;
  static bool attr[PSK_MAX_DEVICES] = {};
  smem_limit_once((const void*)softmax_pipe_kernel<YT, EXPM>, (int)budget, attr);
  const int64_t sms = device_sm_count();
  const unsigned grid = (unsigned)(P.rows < sms ? P.rows : sms);
  softmax_pipe_kernel<YT, EXPM><<<grid, PIPE_THREADS, smem, stream>>>(P);
  return check_launch("softmax region kernel (pipelined)");
}

template <int XT, int YT, int EXPM>
static int dispatch_exp(const SoftmaxParams& P, bool vec, cudaStream_t s) {
  if (P.cols > SM_CAP) return launch_stream<XT, YT, EXPM>(P, s);
  if (XT == PSK_BF16 && vec && P.partials <= 32 && P.cols >= 8) return launch_pipe<YT, EXPM>(P, s);
  return vec ? launch_batch<XT, YT, EXPM, true>(P, s) : launch_batch<XT, YT, EXPM, false>(P, s);
}

template <int XT, int YT>
static int dispatch_softmax(const SoftmaxParams& P, int exp_mode, bool vec, cudaStream_t s) {
  return exp_mode == PSK_EXP_EXACT ? dispatch_exp<XT, YT, PSK_EXP_EXACT>(P, vec, s)
                                   : dispatch_exp<XT, YT, PSK_EXP_FAST>(P, vec, s);
}

}  // namespace psk

using namespace psk;

extern "C" int psk_device_status(uint32_t* status, int32_t reset) {
  clear_error();
  if (!status) return fail(PSK_E_NULL, "status is NULL");
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_pipe_status, sizeof(v)) != cudaSuccess) return check_launch("device status read");
  if (reset) {
    const unsigned int z = 0;
    if (cudaMemcpyToSymbol(g_pipe_status, &z, sizeof(z)) != cudaSuccess) return check_launch("device status reset");
  }
  *status = v;
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
  SoftmaxParams P{x, y, rows, cols, ldx, ldy, partials, 1, 0, 0, 0};
  const bool vec = (cols % 8 == 0) && (ldx % 8 == 0) && (ldy % 8 == 0) && ((uintptr_t)x % 16 == 0) &&
                   ((uintptr_t)y % 16 == 0);
  cudaStream_t s = (cudaStream_t)stream;
  if (xt == PSK_BF16 && yt == PSK_BF16) return dispatch_softmax<PSK_BF16, PSK_BF16>(P, exp_mode, vec, s);
  if (xt == PSK_BF16 && yt == PSK_F32) return dispatch_softmax<PSK_BF16, PSK_F32>(P, exp_mode, vec, s);
  if (xt == PSK_F32 && yt == PSK_BF16) return dispatch_softmax<PSK_F32, PSK_BF16>(P, exp_mode, vec, s);
  return dispatch_softmax<PSK_F32, PSK_F32>(P, exp_mode, vec, s);
}
