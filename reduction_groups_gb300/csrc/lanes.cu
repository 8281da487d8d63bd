// Lane-per-row row regions over bf16 rows (poot "Fusion and Planning",
// Reduction-rooted regions): the softmax, Reduce(Max) -> Sub -> Exp ->
// Reduce(Sum) -> Div, and the norms, RMSNorm's Reduce(Sum of x^2) and
// LayerNorm's Reduce(Sum) then Reduce(Sum of (x - mu)^2), each followed by its
// divide (presk PSK-Realize, "What it removes"); every sum in the declared
// order's bracketing tree (presk "Native execution", the realization's order;
// metrale "The LKB in Mathematics", section 2): the sequential and blocked(w)
// orders, one chain ((f0 + f1) + f2) + ... per row.
//
// Each lane of a warp owns one row of the warp's batch (nb <= 32 consecutive
// rows) and runs every pass over it itself:
//   softmax:   m = max over the row (on the stored bf16 pairs, exact); the
//              chain of e_j = exp(x_j - m); the output pass, e_j recomputed
//              (the same operations on the same values: the same bits) and
//              y_j = bf16_rn(e_j / s);
//   RMSNorm:   the chain of RN(x_j^2); the output pass x_j / d, * gamma;
//   LayerNorm: the chain of x_j (the mean), the chain of RN(RN(x_j - mu)^2);
//              the output pass (x_j - mu) / d, * gamma, + beta.
// The rows are never held whole on chip: every pass streams the batch
// through a ring of tiles of 64 columns x nb rows in shared memory, each one
// 2-D tensor copy (TMA), and the outputs leave through a ring of output tiles
// with 2-D tensor stores.  The chains run over the tiles left to right (their
// index order), the other passes right to left, so that a pass that can
// starts on the tiles the one before it read last, which L2 still holds
// (evict-last hints until the last pass, evict-first after).  Tiles use the
// 128-byte swizzle, so a lane's 16-byte reads and writes of its own row never
// share a bank group with the seven lanes beside it.  Rows past the tensor's
// end read as zeros and are never stored.
//
// Against the pipelined kernel (regions.cu), which keeps each row's values
// once in a shared f32 row and leaves the sums to a few chain lanes, this
// reads every row once per pass (and, for the softmax, evaluates the exp
// twice) but keeps up to 32 rows in their chains per warp (eight warps per
// SM, two per scheduler) instead of about eight per SM: a one-chain order's
// 4096 dependent adds per row are no longer the bound.  The softmax takes
// only its fast realization (the fast exp on f32 pairs) here; with the
// correctly rounded exp the doubled exp work costs more than the chains save.
//
// Every wait is bounded (pipe.cuh); a timeout is recorded in the status word
// and the warp winds down after its copies in flight have landed.

#include "common.cuh"
#include "crmath.cuh"
#include "pipe.cuh"
#include "pair.cuh"
#include "rowmath.cuh"

#include <cuda.h>
#include <stdlib.h>

namespace psk {

constexpr int LANE_WARPS = 8;                                  // warps per CTA (two per scheduler)
constexpr int LANE_TC = 64;                                    // columns of a tile (128 bytes of bf16)
constexpr int LANE_TILE = 32 * 128;                            // a tile's slot: up to 32 rows of 128 bytes
constexpr int LANE_NI = 6;                                     // input tiles per warp
constexpr int LANE_NO = 1;                                     // output tiles per warp
constexpr int LANE_WARP_SMEM = (LANE_NI + LANE_NO) * LANE_TILE;
constexpr int LANE_SMEM = LANE_WARPS * LANE_WARP_SMEM + 1024;  // + room to align the base to 1024 bytes
constexpr int LANE_MAX_COLS = 4096;

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 2-D tensor copy of the tile at (column c0, row r0) into shared memory,
// completing on `bar`, with an L2 cache policy.
__device__ __forceinline__ void tile_load(uint32_t dst, const CUtensorMap* map, int c0, int r0, uint64_t* bar,
                                          uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(map), "r"(c0), "r"(r0), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}

// 2-D tensor store of a shared-memory tile to (column c0, row r0), in the
// thread's current bulk async-group; elements outside the tensor are skipped.
__device__ __forceinline__ void tile_store(const CUtensorMap* map, int c0, int r0, uint32_t src, uint64_t pol) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group.L2::cache_hint [%0, {%1, %2}], [%3], %4;" ::
                   "l"(map),
               "r"(c0), "r"(r0), "r"(src), "l"(pol)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N of the thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Order this thread's shared-memory accesses before its later bulk copies.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// The eight exp values of a 16-byte group of bf16 x (element 2k in the low
// half of word k): x + (-m) and the fast exp on f32 pairs -- the same
// operations as the pipelined kernel's fast realization, so the same bits.
__device__ __forceinline__ void lane_exp8(const uint4 wv, float m, float* e) {
  const uint32_t wd[4] = {wv.x, wv.y, wv.z, wv.w};
  const f2 nm = f2_splat(-m);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const f2 r = exp2_unit_nonpos(f2_add(f2{__uint_as_float(wd[k] << 16), __uint_as_float(wd[k] & 0xFFFF0000u)}, nm));
    e[2 * k] = r.x;
    e[2 * k + 1] = r.y;
  }
}

// ------------------------------------------------------------ tile pieces
// A lane's eight 16-byte groups of one tile (its row's 64 columns), loaded
// together so that the work on them overlaps.
__device__ __forceinline__ void lane_load8(const unsigned char* tile, uint32_t lrow, uint32_t sw, uint4* v) {
#pragma unroll
  for (int k = 0; k < 8; ++k) v[k] = *reinterpret_cast<const uint4*>(tile + lrow + (((uint32_t)k ^ sw) << 4));
}

__device__ __forceinline__ void widen8(const uint4 w, float* v) {
  const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    v[2 * k] = __uint_as_float(wd[k] << 16);
    v[2 * k + 1] = __uint_as_float(wd[k] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint4 pack8(const float* o) {
  return make_uint4(f32x2_to_bf16x2(o[0], o[1]), f32x2_to_bf16x2(o[2], o[3]), f32x2_to_bf16x2(o[4], o[5]),
                    f32x2_to_bf16x2(o[6], o[7]));
}

// Eight consecutive norm parameters from global memory (the same address in
// every lane: one broadcast load).
template <int PT>
__device__ __forceinline__ void load_param8(const void* base, int j, float* v) {
  if (PT == PSK_BF16) {
    widen8(__ldg(reinterpret_cast<const uint4*>((const uint16_t*)base + j)), v);
  } else {
    const float4 a = __ldg(reinterpret_cast<const float4*>((const float*)base + j));
    const float4 b = __ldg(reinterpret_cast<const float4*>((const float*)base + j) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
}

// What a row carries from pass to pass.
struct LaneRow {
  float m = 0.0f;                     // softmax: the max
  float s = 1.0f, rs = 1.0f;          // softmax: the sum and RN(1 / s)
  bool fast_ok = true;
  f2 rs2 = {1.0f, 1.0f}, ns2 = {-1.0f, -1.0f};
  float mu = 0.0f;                    // LayerNorm: the mean
  RowDivisor D;                       // norms: the divisor sqrt(var + eps)
};

// Passes per region kind, and their direction: the chains run left to right
// (their index order); the other passes right to left, so that each pass
// starts on the tiles the one before it read last.
template <int KIND>
__host__ __device__ constexpr int lane_passes() { return KIND == REGION_RMS || KIND == REGION_SOFTMAX_BWD ? 2 : 3; }
template <int KIND>
__host__ __device__ constexpr bool lane_rev(int pass) {
  return KIND == REGION_SOFTMAX ? pass != 1 : pass == lane_passes<KIND>() - 1;
}

// The values a chain pass adds for a group of eight stored elements:
// softmax e = exp(x - m) (fast realization); RMSNorm RN(x^2); LayerNorm x,
// then RN(RN(x - mu)^2); softmax backward RN(ct y) (w the stored y, cw ct).
template <int KIND>
__device__ __forceinline__ void chain_values8(const uint4 w, const uint4 cw, int pass, const LaneRow& R, float* f) {
  if constexpr (KIND == REGION_SOFTMAX) {
    lane_exp8(w, R.m, f);
  } else if constexpr (KIND == REGION_SOFTMAX_BWD) {
    float c[8];
    widen8(w, f);
    widen8(cw, c);
#pragma unroll
    for (int q = 0; q < 8; ++q) f[q] = __fmul_rn(c[q], f[q]);
  } else {
    widen8(w, f);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (KIND == REGION_RMS) {
        f[q] = __fmul_rn(f[q], f[q]);
      } else if (pass == 1) {
        const float c = __fsub_rn(f[q], R.mu);
        f[q] = __fmul_rn(c, c);
      }
    }
  }
}

// The outputs of a group of eight stored elements at column j, rounded to
// bf16 pairs: softmax e / s (the pipelined kernel's fast realization); norms
// (x - mu) / d, * gamma, + beta; softmax backward RN(y RN(ct - s)) (w the
// stored y, cw ct).  PRE: the norms' bf16 gamma and beta of the group come
// in pg / pb (loaded before the tile's wait) instead of from global memory.
template <int KIND, int PT, bool PRE = false>
__device__ __forceinline__ uint4 out_group8(const uint4 w, const uint4 cw, int j, const LaneRow& R,
                                            const RegionParams& P, const uint4 pg = uint4{}, const uint4 pb = uint4{}) {
  float o[8];
  if constexpr (KIND == REGION_SOFTMAX_BWD) {
    float c[8];
    widen8(w, o);
    widen8(cw, c);
#pragma unroll
    for (int q = 0; q < 8; ++q) o[q] = __fmul_rn(o[q], __fsub_rn(c[q], R.s));
  } else if constexpr (KIND == REGION_SOFTMAX) {
    lane_exp8(w, R.m, o);
    if (R.fast_ok) {
      // Markstein's correction two at a time (no per-element range test)
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const f2 ea{o[2 * h], o[2 * h + 1]};
        const f2 qa = f2_mul(ea, R.rs2);
        const f2 ya = f2_fma(f2_fma(qa, R.ns2, ea), R.rs2, qa);
        o[2 * h] = ya.x;
        o[2 * h + 1] = ya.y;
      }
    } else {
      row_div_n<8>(o, R.s, R.rs, false);
    }
  } else {
    widen8(w, o);
    if (KIND == REGION_LAYER) {
#pragma unroll
      for (int q = 0; q < 8; ++q) o[q] = __fsub_rn(o[q], R.mu);
    }
    divide_n<8>(o, R.D);
    if (P.gamma) {
      float g[8];
      if (PRE) widen8(pg, g);
      else load_param8<PT>(P.gamma, j, g);
#pragma unroll
      for (int q = 0; q < 8; ++q) o[q] = __fmul_rn(o[q], g[q]);
    }
    if (KIND == REGION_LAYER && P.beta) {
      float bb[8];
      if (PRE) widen8(pb, bb);
      else load_param8<PT>(P.beta, j, bb);
#pragma unroll
      for (int q = 0; q < 8; ++q) o[q] = __fadd_rn(o[q], bb[q]);
    }
  }
  return pack8(o);
}

// ------------------------------------------------------------ the kernel
// KIND: the region; PP: the declared order's partial chains (element j feeds
// chain j mod PP; the entry points launch the one-chain orders, PP = 1); PT:
// the norms' parameter storage type; FULL: rows of exactly LANE_MAX_COLS
// columns (a compile-time row length: every tile whole).
// The request and consumption counters are 32-bit: a warp makes at most
// (2^31 rows / the grid's warps) batches x 3 passes x 64 tiles requests,
// far below 2^31.
// The softmax backward (KIND REGION_SOFTMAX_BWD; x is y, tct the cotangent's
// map, y is dx) loads a y tile and a ct tile per request: its ring slots are
// pairs of tiles, half as many.
template <int KIND, int PP, int PT, bool FULL = false>
__global__ void __launch_bounds__(LANE_WARPS * 32, 1)
    region_lane_kernel(const __grid_constant__ RegionParams P, const __grid_constant__ CUtensorMap tx,
                       const __grid_constant__ CUtensorMap ty, const __grid_constant__ CUtensorMap tct) {
  constexpr int NP = lane_passes<KIND>();
  constexpr bool BWD = KIND == REGION_SOFTMAX_BWD;
  constexpr int TPR = BWD ? 2 : 1;                             // tiles per request
  constexpr int NI = LANE_NI / TPR;                            // request slots
  constexpr bool PRE = (KIND == REGION_RMS || KIND == REGION_LAYER) && PT == PSK_BF16;
  extern __shared__ unsigned char lane_smem_raw[];
  __shared__ __align__(8) uint64_t full[LANE_WARPS][LANE_NI];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cols = FULL ? LANE_MAX_COLS : (int)P.cols;
  const int nch = (cols + LANE_TC - 1) / LANE_TC;             // tiles per pass
  const int nb = P.nb;                                         // rows per batch (a tile's height)
  const int64_t nbatch_all = (P.rows + nb - 1) / nb;
  const int64_t gw = (int64_t)blockIdx.x * LANE_WARPS + w;
  const int64_t wtot = (int64_t)gridDim.x * LANE_WARPS;
  const int my_batches = gw < nbatch_all ? (int)((nbatch_all - 1 - gw) / wtot + 1) : 0;
  const int total = my_batches * NP * nch;                   // tile requests of this warp
  // tiles start on 1024-byte boundaries (the period of the 128-byte swizzle)
  const uint32_t raw = smem_addr(lane_smem_raw);
  unsigned char* wp = lane_smem_raw + (((raw + 1023u) & ~1023u) - raw) + (size_t)w * LANE_WARP_SMEM;
  const uint32_t wa = smem_addr(wp);
  unsigned char* op = wp + (size_t)LANE_NI * LANE_TILE;
  // the lane's row in a tile; its k-th 16-byte group sits at group k ^ (lane % 8)
  const uint32_t lrow = (uint32_t)lane * 128u, sw = (uint32_t)(lane & 7);
  uint64_t* bars = full[w];
  const uint64_t pol_keep = policy_evict_last(), pol_drop = policy_evict_first();
  const long long drop = g_pipe_drop_row;
  const float n_f = (float)cols;                               // exact: cols <= 4096

  // fill the warp's tiles with bf16 ones: rows beyond the batch are never
  // copied in, and their lanes then compute on benign values that take no
  // slow path in any region (rows past the tensor's end read as zeros)
  for (int o = lane * 16; o < LANE_WARP_SMEM; o += 32 * 16)
    *reinterpret_cast<uint4*>(wp + o) = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
  fence_proxy_async_smem();
  if (lane == 0) {
    for (int i = 0; i < LANE_NI; ++i) mbar_init(&bars[i], 1);
    fence_barrier_init();
  }
  __syncwarp();

  // ---- requests (lane 0): q = ((batch * NP) + pass) * nch + tile, into slot
  // q % NI; the request state is kept by every lane alike
  int rq = 0;
  int rb = 0, rp = 0, rc = 0;
  int64_t rrow = gw * nb;                                    // the first row of the request's batch
  int withheld = -1;                                         // test hook: the request never made
  auto issue = [&]() {
    const int slot = rq % NI;
    const int tc = lane_rev<KIND>(rp) ? nch - 1 - rc : rc;   // the pass's tile order
    if (rp == 0 && rc == 0 && drop >= (long long)rb * nb && drop < (long long)rb * nb + nb) {
      withheld = rq;                                         // as if this copy were lost
    } else if (lane == 0) {
      mbar_arrive_expect_tx(&bars[slot], (uint32_t)(nb * 128 * TPR));
      tile_load(wa + (uint32_t)(slot * TPR) * LANE_TILE, &tx, tc * LANE_TC, (int)rrow, &bars[slot],
                rp < NP - 1 ? pol_keep : pol_drop);
      if (BWD)
        tile_load(wa + (uint32_t)(slot * TPR + 1) * LANE_TILE, &tct, tc * LANE_TC, (int)rrow, &bars[slot],
                  rp < NP - 1 ? pol_keep : pol_drop);
    }
    ++rq;
    if (++rc == nch) {
      rc = 0;
      if (++rp == NP) {
        rp = 0;
        ++rb;
        rrow += wtot * nb;
      }
    }
  };
  for (int i = 0; i < NI && rq < total; ++i) issue();

  // ---- consumption in request order
  int cq = 0;
  bool dead = false;
  auto take = [&]() -> bool {
    const bool ok = mbar_wait(&bars[cq % NI], (uint32_t)(cq / NI) & 1u);
    return !__any_sync(0xffffffffu, !ok);
  };
  auto release = [&]() {                                     // every lane has read the tile: refill its slot
    __syncwarp();
    ++cq;
    if (lane == 0) fence_proxy_async_smem();
    if (rq < total) issue();
  };
  int oq = 0;                                                // output tiles written

  for (int b = 0; b < my_batches && !dead; ++b) {
    const int64_t r0 = (gw + (int64_t)b * wtot) * nb;
    LaneRow R;
    for (int pass = 0; pass < NP && !dead; ++pass) {
      const bool rev = lane_rev<KIND>(pass);
      const bool out_pass = pass == NP - 1;
      const bool max_pass = KIND == REGION_SOFTMAX && pass == 0;
      uint32_t mb = 0xFF80FF80u;                            // softmax max: (-inf, -inf)
      float acc[PP];
#pragma unroll
      for (int p = 0; p < PP; ++p) acc[p] = -0.0f;          // -0 + f = f for every f: the chain starts at f(x_p)
      for (int t = 0; t < nch; ++t) {
        const int c = rev ? nch - 1 - t : t;
        // the norms' output pass over a whole tile: its bf16 gamma and beta
        // (the same in every lane) are loaded before the wait for the tile
        uint4 gq[PRE ? 8 : 1], bq[PRE ? 8 : 1];
        if (PRE && out_pass && cols - c * LANE_TC >= LANE_TC) {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int j = c * LANE_TC + 8 * k;
            gq[PRE ? k : 0] = P.gamma ? __ldg(reinterpret_cast<const uint4*>((const uint16_t*)P.gamma + j)) : uint4{};
            bq[PRE ? k : 0] = KIND == REGION_LAYER && P.beta ? __ldg(reinterpret_cast<const uint4*>((const uint16_t*)P.beta + j))
                                                              : uint4{};
          }
        }
        if (!take()) { dead = true; break; }
        const int ng = (cols - c * LANE_TC) / 8 < 8 ? (cols - c * LANE_TC) / 8 : 8;
        const unsigned char* tile = wp + (size_t)((cq % NI) * TPR) * LANE_TILE;
        const unsigned char* ctile = tile + LANE_TILE;            // the backward's ct tile
        if (out_pass) {
          if (lane == 0) bulk_wait_read<LANE_NO - 1>();     // the store that last used this slot has read it
          __syncwarp();
          unsigned char* ot = op + (size_t)(oq % LANE_NO) * LANE_TILE;
          if (ng == 8) {
            uint4 v[8], cv[8], o8[8];
            lane_load8(tile, lrow, sw, v);
            if (BWD) lane_load8(ctile, lrow, sw, cv);
#pragma unroll
            for (int k = 0; k < 8; ++k)
              o8[k] = out_group8<KIND, PT, PRE>(v[k], BWD ? cv[k] : v[k], c * LANE_TC + 8 * k, R, P, gq[PRE ? k : 0],
                                                bq[PRE ? k : 0]);
#pragma unroll
            for (int k = 0; k < 8; ++k) *reinterpret_cast<uint4*>(ot + lrow + (((uint32_t)k ^ sw) << 4)) = o8[k];
          } else {
            for (int k = 0; k < ng; ++k) {
              const uint4 v = *reinterpret_cast<const uint4*>(tile + lrow + (((uint32_t)k ^ sw) << 4));
              const uint4 cv = BWD ? *reinterpret_cast<const uint4*>(ctile + lrow + (((uint32_t)k ^ sw) << 4)) : v;
              *reinterpret_cast<uint4*>(ot + lrow + (((uint32_t)k ^ sw) << 4)) =
                  out_group8<KIND, PT>(v, cv, c * LANE_TC + 8 * k, R, P);
            }
          }
          fence_proxy_async_smem();                          // this lane's writes, before the async store
          __syncwarp();
          if (lane == 0) {
            tile_store(&ty, c * LANE_TC, (int)r0, smem_addr(ot), pol_drop);
            bulk_commit();
          }
          ++oq;
        } else if (max_pass) {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            if (k < ng) {
              const uint4 v = *reinterpret_cast<const uint4*>(tile + lrow + (((uint32_t)k ^ sw) << 4));
              mb = bf16x2_max_nan(mb, bf16x2_max_nan(v.x, v.y));
              mb = bf16x2_max_nan(mb, bf16x2_max_nan(v.z, v.w));
            }
          }
        } else if (ng == 8) {
          // a chain pass over a full tile: element 8 k + q feeds chain q mod P
          uint4 v[8], cv[8];
          lane_load8(tile, lrow, sw, v);
          if (BWD) lane_load8(ctile, lrow, sw, cv);
          float f[64];
#pragma unroll
          for (int k = 0; k < 8; ++k) chain_values8<KIND>(v[k], BWD ? cv[k] : v[k], pass, R, f + 8 * k);
#pragma unroll
          for (int j = 0; j < 64; ++j) acc[j % PP] = __fadd_rn(acc[j % PP], f[j]);
        } else {
          for (int k = 0; k < ng; ++k) {
            float f[8];
            const uint4 v = *reinterpret_cast<const uint4*>(tile + lrow + (((uint32_t)k ^ sw) << 4));
            const uint4 cv = BWD ? *reinterpret_cast<const uint4*>(ctile + lrow + (((uint32_t)k ^ sw) << 4)) : v;
            chain_values8<KIND>(v, cv, pass, R, f);
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q % PP] = __fadd_rn(acc[q % PP], f[q]);
          }
        }
        release();
      }
      if (dead) break;
      // what the pass leaves for the next ones
      float sum = acc[0];
#pragma unroll
      for (int p = 1; p < PP; ++p) sum = __fadd_rn(sum, acc[p]);   // partials left to right
      if (BWD) {
        R.s = sum;                                           // s = the sum of RN(ct y)
      } else if (KIND == REGION_SOFTMAX) {
        if (pass == 0) {
          R.m = max_nan(__uint_as_float(mb << 16), __uint_as_float(mb & 0xFFFF0000u));
        } else if (pass == 1) {
          R.s = sum;
          R.rs = __frcp_rn(sum);
          R.fast_ok = sum >= 1.0f && sum < 0x1p20f;
          R.rs2 = f2_splat(R.rs);
          R.ns2 = f2_splat(-sum);
        }
      } else if (KIND == REGION_LAYER && pass == 0) {
        R.mu = __fdiv_rn(sum, n_f);
      } else if (!out_pass) {                                // the sum of squares: the divisor
        R.D = make_divisor(__fsqrt_rn(__fadd_rn(__fdiv_rn(sum, n_f), P.eps)));
      }
    }
  }

  if (dead) {
    // a withheld copy (the test hook) is arrived for now, so that its phase
    // completes; then every request made is waited for (bounded) before the
    // warp leaves
    if (lane == 0 && withheld >= cq) mbar_arrive(&bars[withheld % NI]);
    __syncwarp();
    for (int q = cq; q < rq; ++q) mbar_wait(&bars[q % NI], (uint32_t)(q / NI) & 1u);
  }
  if (lane == 0) bulk_wait_all();
}

// ------------------------------------------------------------------ host

// cuTensorMapEncodeTiled, from the driver through the runtime (no link
// against the driver library), resolved once.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled() {
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return (EncodeTiledFn)p;
  }();
  return fn;
}

// The tensor map of bf16 rows [rows, cols] with row stride ld elements, in
// tiles of 64 columns x nb rows, 128-byte swizzled, zeros outside.
static int encode_rows(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int64_t ld, int nb) {
  const EncodeTiledFn fn = encode_tiled();
  if (!fn) return fail(PSK_E_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)ld * 2u};
  const cuuint32_t box[2] = {(cuuint32_t)LANE_TC, (cuuint32_t)nb};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PSK_E_CUDA, "tensor map encoding failed (CUresult %d)", (int)r);
  return PSK_OK;
}

// Rows per batch: the fewest batches of at most 32 rows that cover a warp's
// share, split evenly (32768 rows on 1216 warps: one batch of 27).
static int lane_batch_rows(int64_t rows, int64_t wtot) {
  const int64_t rpw = (rows + wtot - 1) / wtot;
  const int64_t nbat = (rpw + 31) / 32;
  return (int)((rpw + nbat - 1) / nbat);
}

template <int KIND, int PP, int PT>
static int launch_lanes(const RegionParams& P, const CUtensorMap& tx, const CUtensorMap& ty, const CUtensorMap& tct,
                        int64_t sms, cudaStream_t stream) {
  const int64_t nbatch = (P.rows + P.nb - 1) / P.nb;
  const int64_t need = (nbatch + LANE_WARPS - 1) / LANE_WARPS;
  const unsigned grid = (unsigned)(need < sms ? need : sms);
  if constexpr (KIND == REGION_SOFTMAX) {   // the softmax over full rows: the full-row variant
    if (P.cols == LANE_MAX_COLS) {
      static bool attr_full[PSK_MAX_DEVICES] = {};
      smem_limit_once((const void*)region_lane_kernel<KIND, PP, PT, true>, LANE_SMEM, attr_full);
      region_lane_kernel<KIND, PP, PT, true><<<grid, LANE_WARPS * 32, LANE_SMEM, stream>>>(P, tx, ty, tct);
      return check_launch("row region kernel (lane per row)");
    }
  }
  static bool attr[PSK_MAX_DEVICES] = {};
  smem_limit_once((const void*)region_lane_kernel<KIND, PP, PT>, LANE_SMEM, attr);
  region_lane_kernel<KIND, PP, PT><<<grid, LANE_WARPS * 32, LANE_SMEM, stream>>>(P, tx, ty, tct);
  return check_launch("row region kernel (lane per row)");
}

// The rows every lane-kernel region takes: bf16 x and y (checked by the
// callers) of 64 <= cols <= 4096 columns, cols a multiple of 8, rows on
// 16-byte boundaries, at least 8 rows per warp of a full grid (fewer rows
// leave most lanes idle; the pipelined kernel spreads each row over a team
// instead).  On success P carries the batch height and tx / ty the maps.
// Tuning aids, read once: PSK_LANES=0 turns the kernel off,
// PSK_LANE_MIN_ROWS sets the row threshold, PSK_LANE_NB (1..32) the rows per
// batch.
static bool lanes_take(RegionParams& P, CUtensorMap& tx, CUtensorMap& ty, int64_t& sms, int& rc) {
  rc = PSK_OK;
  static const char* off = getenv("PSK_LANES");
  if (off && off[0] == '0') return false;
  if (P.cols < LANE_TC || P.cols > LANE_MAX_COLS || P.cols % 8 != 0 || P.ldx % 8 != 0 || P.ldy % 8 != 0 ||
      (uintptr_t)P.x % 16 != 0 || (uintptr_t)P.y % 16 != 0 || P.rows >= ((int64_t)1 << 31))
    return false;
  sms = device_sm_count();
  const int64_t wtot = sms * LANE_WARPS;
  static const char* min_env = getenv("PSK_LANE_MIN_ROWS");
  const int64_t min_rows = min_env ? atoll(min_env) : 8 * wtot;
  if (P.rows < min_rows) return false;
  P.nb = lane_batch_rows(P.rows, wtot);
  static const char* nb_env = getenv("PSK_LANE_NB");
  if (nb_env) {
    const int v = atoi(nb_env);
    if (v >= 1 && v <= 32) P.nb = v;
  }
  if (P.nb > P.rows) P.nb = (int)P.rows;
  if ((rc = encode_rows(&tx, P.x, P.rows, P.cols, P.ldx, P.nb))) return true;
  rc = encode_rows(&ty, P.y, P.rows, P.cols, P.ldy, P.nb);
  return true;
}

// The softmax region: the fast realization of the one-chain orders
// (sequential, blocked).  Interleaved orders stay with the pipelined kernel:
// their chains are short there, and the second exp per element would cost
// more than the lane kernel saves; so does the correctly rounded exp.
int softmax_lanes(const RegionParams& P0, int exp_mode, cudaStream_t stream, bool* taken) {
  *taken = false;
  if (exp_mode != PSK_EXP_FAST || P0.partials != 1) return PSK_OK;
  RegionParams P = P0;
  CUtensorMap tx, ty;
  int64_t sms = 0;
  int rc = PSK_OK;
  if (!lanes_take(P, tx, ty, sms, rc)) return PSK_OK;
  *taken = true;
  if (rc) return rc;
  return launch_lanes<REGION_SOFTMAX, 1, PSK_F32>(P, tx, ty, tx, sms, stream);
}

// RMSNorm and LayerNorm: the one-chain orders too (interleaved orders run
// faster on the pipelined kernel, whose chains are short there); scale and
// bias (if any) on 16-byte boundaries.
int norm_lanes(const RegionParams& P0, int kind, cudaStream_t stream, bool* taken) {
  *taken = false;
  if (P0.partials != 1) return PSK_OK;
  if ((uintptr_t)P0.gamma % 16 != 0 || (uintptr_t)P0.beta % 16 != 0) return PSK_OK;
  RegionParams P = P0;
  CUtensorMap tx, ty;
  int64_t sms = 0;
  int rc = PSK_OK;
  if (!lanes_take(P, tx, ty, sms, rc)) return PSK_OK;
  *taken = true;
  if (rc) return rc;
  const bool bf = P.param_dtype == PSK_BF16;
  if (kind == REGION_RMS)
    return bf ? launch_lanes<REGION_RMS, 1, PSK_BF16>(P, tx, ty, tx, sms, stream)
              : launch_lanes<REGION_RMS, 1, PSK_F32>(P, tx, ty, tx, sms, stream);
  return bf ? launch_lanes<REGION_LAYER, 1, PSK_BF16>(P, tx, ty, tx, sms, stream)
            : launch_lanes<REGION_LAYER, 1, PSK_F32>(P, tx, ty, tx, sms, stream);
}

// The softmax backward: the one-chain orders over bf16 y, ct and dx (the
// chain of RN(ct y), then dx = RN(y RN(ct - s))), ct on 16-byte boundaries.
int softmax_bwd_lanes(const RegionParams& P0, cudaStream_t stream, bool* taken) {
  *taken = false;
  if (P0.partials != 1 || P0.ct_dtype != PSK_BF16 || (uintptr_t)P0.ct % 16 != 0 || P0.ldc % 8 != 0) return PSK_OK;
  RegionParams P = P0;
  CUtensorMap tx, ty, tct;
  int64_t sms = 0;
  int rc = PSK_OK;
  if (!lanes_take(P, tx, ty, sms, rc)) return PSK_OK;
  *taken = true;
  if (rc) return rc;
  if ((rc = encode_rows(&tct, P.ct, P.rows, P.cols, P.ldc, P.nb))) return rc;
  return launch_lanes<REGION_SOFTMAX_BWD, 1, PSK_F32>(P, tx, ty, tct, sms, stream);
}

// The status word and test hook of this translation unit's kernels (pipe.cuh
// keeps one copy per unit): read / reset and set by the entry points in
// regions.cu.
int lanes_status(unsigned int* v, bool reset) {
  if (cudaMemcpyFromSymbol(v, g_pipe_status, sizeof(*v)) != cudaSuccess) return check_launch("device status read");
  if (reset) {
    const unsigned int z = 0;
    if (cudaMemcpyToSymbol(g_pipe_status, &z, sizeof(z)) != cudaSuccess) return check_launch("device status reset");
  }
  return PSK_OK;
}

int lanes_set_drop_row(long long row) {
  if (cudaMemcpyToSymbol(g_pipe_drop_row, &row, sizeof(row)) != cudaSuccess) return check_launch("test hook write");
  return PSK_OK;
}

}  // namespace psk
