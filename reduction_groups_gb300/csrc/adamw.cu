// psk_adamw_tree: the AdamW step as one parameter-tree group, mapped over
// every leaf of the tree in one launch (PSK-Realize, Parameter trees: the
// optimizer step is one long elementwise chain over every parameter; presk
// "The language", The optimizer: AdamW as PyTorch defines it, t from 1).
//
// The leaf table (pointers, sizes, the first chunk of each leaf) travels in a
// __grid_constant__ kernel parameter.  The concatenated parameters are cut
// into chunks of 4096 elements that never straddle two leaves; a persistent
// grid walks the chunks, finds each chunk's leaf by binary search over the
// table (uniform across the CTA), and streams theta, m, v (f32, read and
// written) and the gradient (f32 or bf16, read) with 16-byte vector accesses
// and evict-first cache hints: 28 or 26 bytes per parameter, nothing else.
// Unaligned leaves and ragged tails take a scalar path with the same
// arithmetic.  Each operation is one IEEE f32 rounding, in the order of the
// definition, so every parameter is bit-identical to the unfused chain.
//
// psk_adamw_tree_ex adds the pages' schedules and global-norm clipping (the
// same passage: grad_clip = c scales g by min(1, c / (||g||_2 + 1e-6));
// constant / linear / cosine schedules with warmup).  The scheduled lr is
// computed on the host exactly (rational arithmetic on binary64 pairs, cos in
// double-double) and rounded once.  Clipping takes three short launches
// before the update, in the caller's workspace: ||g||^2 in f32 over a declared
// tree -- RN(g^2) summed in blocks of 1024 consecutive elements of a leaf (one
// thread per block), the block sums in groups of 64 and the group sums of a
// leaf (one CTA per leaf), the leaf sums in tree order (one thread) -- then
// scale = min(q, 1), q = RN(c / RN(sqrt(||g||^2) + RN(1e-6))), which the
// update kernel reads and applies as RN(g * scale).

#include <math.h>
#include <string.h>

#include <mutex>

#include <cuda.h>

#include "common.cuh"

namespace psk {

constexpr int AW_THREADS = 256;
constexpr int AW_CHUNK = 4096;                 // elements per chunk
constexpr int AW_VPT = AW_CHUNK / (AW_THREADS * 4);   // float4 vectors per thread per chunk

struct LeafDesc {
  void* th;
  void* m;
  void* v;
  const void* g;
  int64_t numel;
  int64_t chunk_begin;   // first chunk of this leaf in the launch
  int8_t gdt;            // storage type of the gradient
  int8_t pdt;            // storage type of theta, m, v
  int8_t vec;            // theta/m/v and grad aligned for 16-byte (f32) or 8-byte (bf16) vectors
};
static_assert(sizeof(LeafDesc) == 56, "512 leaf descriptors must fit the 32 KB kernel parameter space");

// Four consecutive stored values at element i, widened / rounded back.
__device__ __forceinline__ float4 load4_any(const void* p, int32_t dt, int64_t i) {
  if (dt == PSK_F32) return __ldcs((const float4*)((const float*)p + i));
  const uint2 q = __ldcs((const uint2*)((const unsigned short*)p + i));
  return make_float4(__uint_as_float(q.x << 16), __uint_as_float(q.x & 0xFFFF0000u),
                     __uint_as_float(q.y << 16), __uint_as_float(q.y & 0xFFFF0000u));
}
__device__ __forceinline__ void store4_any(void* p, int32_t dt, int64_t i, float4 v) {
  if (dt == PSK_F32) {
    __stcs((float4*)((float*)p + i), v);
  } else {
    uint2 q;
    q.x = f32x2_to_bf16x2(v.x, v.y);
    q.y = f32x2_to_bf16x2(v.z, v.w);
    __stcs((uint2*)((unsigned short*)p + i), q);
  }
}
__device__ __forceinline__ float load1_any(const void* p, int32_t dt, int64_t i) {
  if (dt == PSK_F32) return ((const float*)p)[i];
  return bf16_bits_to_f32(((const unsigned short*)p)[i]);
}
__device__ __forceinline__ void store1_any(void* p, int32_t dt, int64_t i, float v) {
  if (dt == PSK_F32) ((float*)p)[i] = v;
  else ((unsigned short*)p)[i] = f32_to_bf16_bits(v);
}

struct AdamScalars { float b1, b2, omb1, omb2, bc1, bc2, lr, eps, wd; };

struct AdamParams {
  AdamScalars s;
  int32_t n_leaves;
  int64_t n_chunks;
  LeafDesc leaf[PSK_ADAMW_MAX_LEAVES];
};

__device__ __forceinline__ void adamw_one(const AdamScalars& s, float& th, float& m, float& v, float g) {
  float m1 = __fadd_rn(__fmul_rn(s.b1, m), __fmul_rn(s.omb1, g));
  float v1 = __fadd_rn(__fmul_rn(s.b2, v), __fmul_rn(s.omb2, __fmul_rn(g, g)));
  float mh = __fdiv_rn(m1, s.bc1);
  float vh = __fdiv_rn(v1, s.bc2);
  float q = __fdiv_rn(mh, __fadd_rn(__fsqrt_rn(vh), s.eps));
  float u = __fadd_rn(q, __fmul_rn(s.wd, th));
  th = __fsub_rn(th, __fmul_rn(s.lr, u));
  m = m1;
  v = v1;
}

__device__ __forceinline__ float load_grad(const void* g, int32_t gdt, int64_t i) {
  if (gdt == PSK_F32) return __ldcs((const float*)g + i);
  return bf16_bits_to_f32(__ldcs((const unsigned short*)g + i));
}

// theta, m, v stored as PDT (a template parameter: the host launches the f32
// leaves and the bf16 leaves of a tree separately, so each kernel keeps one
// load and store path); the gradient's type is a per-chunk uniform branch.
template <bool CLIP, int PDT>
__global__ void __launch_bounds__(AW_THREADS) adamw_kernel(const __grid_constant__ AdamParams P, const float* clip) {
  const int t = threadIdx.x;
  const float scale = CLIP ? *clip : 1.0f;
  for (int64_t c = blockIdx.x; c < P.n_chunks; c += gridDim.x) {
    // the leaf holding chunk c: last leaf with chunk_begin <= c
    int lo = 0, hi = P.n_leaves - 1;
    while (lo < hi) {
      int mid = (lo + hi + 1) >> 1;
      if (P.leaf[mid].chunk_begin <= c) lo = mid; else hi = mid - 1;
    }
    const LeafDesc& L = P.leaf[lo];
    const int64_t base = (c - L.chunk_begin) * AW_CHUNK;
    const int64_t n = (L.numel - base) < AW_CHUNK ? (L.numel - base) : AW_CHUNK;
    if (L.vec && n == AW_CHUNK) {
      float4 th[AW_VPT], m[AW_VPT], v[AW_VPT], g[AW_VPT];
#pragma unroll
      for (int k = 0; k < AW_VPT; ++k) {
        const int64_t i = base + (int64_t)(k * AW_THREADS + t) * 4;
        th[k] = load4_any(L.th, PDT, i);
        m[k] = load4_any(L.m, PDT, i);
        v[k] = load4_any(L.v, PDT, i);
        if (L.gdt == PSK_F32) {
          g[k] = __ldcs((const float4*)((const float*)L.g + i));
        } else {
          uint2 q = __ldcs((const uint2*)((const unsigned short*)L.g + i));
          g[k] = make_float4(__uint_as_float(q.x << 16), __uint_as_float(q.x & 0xFFFF0000u),
                             __uint_as_float(q.y << 16), __uint_as_float(q.y & 0xFFFF0000u));
        }
      }
      // every load of the chunk is in flight before the first use of one
#pragma unroll
      for (int k = 0; k < AW_VPT; ++k) {
        if (CLIP) {
          g[k].x = __fmul_rn(g[k].x, scale); g[k].y = __fmul_rn(g[k].y, scale);
          g[k].z = __fmul_rn(g[k].z, scale); g[k].w = __fmul_rn(g[k].w, scale);
        }
        adamw_one(P.s, th[k].x, m[k].x, v[k].x, g[k].x);
        adamw_one(P.s, th[k].y, m[k].y, v[k].y, g[k].y);
        adamw_one(P.s, th[k].z, m[k].z, v[k].z, g[k].z);
        adamw_one(P.s, th[k].w, m[k].w, v[k].w, g[k].w);
        const int64_t i = base + (int64_t)(k * AW_THREADS + t) * 4;
        store4_any(L.th, PDT, i, th[k]);
        store4_any(L.m, PDT, i, m[k]);
        store4_any(L.v, PDT, i, v[k]);
      }
    } else {
      for (int64_t j = t; j < n; j += AW_THREADS) {
        const int64_t i = base + j;
        float th = load1_any(L.th, PDT, i), m = load1_any(L.m, PDT, i), v = load1_any(L.v, PDT, i);
        float g = load_grad(L.g, L.gdt, i);
        if (CLIP) g = __fmul_rn(g, scale);
        adamw_one(P.s, th, m, v, g);
        store1_any(L.th, PDT, i, th);
        store1_any(L.m, PDT, i, m);
        store1_any(L.v, PDT, i, v);
      }
    }
  }
}

// ------------------------------------------------- clipping: ||g||^2 tree
constexpr int SQ_BLOCK = 1024;                 // elements per block (one chain)
constexpr int SQ_GROUP = 64;                   // blocks per group
constexpr int SQ_THREADS = 256;

struct SqLeaf {
  const void* g;
  int64_t numel;
  int64_t block_begin;   // first block of the leaf in the launch's block array
  int64_t group_begin;   // first group of the leaf in the launch's group array
  int32_t gdt;
  int32_t leaf_index;    // position of the leaf in the whole tree (its leaf-sum slot)
};

struct SqParams {
  int32_t n_leaves;
  int64_t n_blocks;
  float* block_sums;     // workspace
  float* group_sums;     // workspace
  float* leaf_sums;      // workspace, one per leaf of the tree
  SqLeaf leaf[PSK_ADAMW_MAX_LEAVES];
};

// RN(g^2) added in index order over one block's (up to 1024) elements by
// one thread, read 8 (bf16) or 4 (f32) at a time when aligned: blocks that
// are short or unaligned, and warps holding any such block.
__device__ float block_sq_lane(const SqLeaf& L, int64_t base, int n) {
  float acc = 0.0f;
  int j = 0;
  if (L.gdt == PSK_BF16) {
    const uint16_t* g = (const uint16_t*)L.g + base;
    if (((uintptr_t)g & 15u) == 0) {
      // four 16-byte loads in flight per thread; the adds keep index order
      for (; j + 32 <= n; j += 32) {
        uint4 q[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) q[u] = __ldcs(reinterpret_cast<const uint4*>(g + j) + u);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t w[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float a = __uint_as_float(w[k] << 16), c = __uint_as_float(w[k] & 0xFFFF0000u);
            acc = __fadd_rn(acc, __fmul_rn(a, a));
            acc = __fadd_rn(acc, __fmul_rn(c, c));
          }
        }
      }
      for (; j + 8 <= n; j += 8) {
        const uint4 q = __ldcs(reinterpret_cast<const uint4*>(g + j));
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float a = __uint_as_float(w[k] << 16), c = __uint_as_float(w[k] & 0xFFFF0000u);
          acc = __fadd_rn(acc, __fmul_rn(a, a));
          acc = __fadd_rn(acc, __fmul_rn(c, c));
        }
      }
    }
    for (; j < n; ++j) {
      const float a = bf16_bits_to_f32(__ldcs(g + j));
      acc = __fadd_rn(acc, __fmul_rn(a, a));
    }
  } else {
    const float* g = (const float*)L.g + base;
    if (((uintptr_t)g & 15u) == 0) {
      for (; j + 16 <= n; j += 16) {
        float4 q[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) q[u] = __ldcs(reinterpret_cast<const float4*>(g + j) + u);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          acc = __fadd_rn(acc, __fmul_rn(q[u].x, q[u].x));
          acc = __fadd_rn(acc, __fmul_rn(q[u].y, q[u].y));
          acc = __fadd_rn(acc, __fmul_rn(q[u].z, q[u].z));
          acc = __fadd_rn(acc, __fmul_rn(q[u].w, q[u].w));
        }
      }
      for (; j + 4 <= n; j += 4) {
        const float4 q = __ldcs(reinterpret_cast<const float4*>(g + j));
        acc = __fadd_rn(acc, __fmul_rn(q.x, q.x));
        acc = __fadd_rn(acc, __fmul_rn(q.y, q.y));
        acc = __fadd_rn(acc, __fmul_rn(q.z, q.z));
        acc = __fadd_rn(acc, __fmul_rn(q.w, q.w));
      }
    }
    for (; j < n; ++j) {
      const float a = __ldcs(g + j);
      acc = __fadd_rn(acc, __fmul_rn(a, a));
    }
  }
  return acc;   // 0 + x = x: the chain starting from 0 is the chain starting from the first square
}

// Full, 16-byte aligned blocks: the warp's 32 blocks (lane l owns block
// b0 + l) are fetched cooperatively in stages of 32 elements per block --
// each 16-byte piece by one lane, `cp.async` into shared memory, the pieces of
// one block adjacent so a warp instruction reads whole 32-byte sectors -- and
// each lane then adds its own block's squares in index order from shared
// memory.  One lane per block reading its own 2 KB would issue 32 separate
// sectors per warp instruction and run at the L1's one wavefront per cycle.
constexpr int SQ_CH = 32;                                  // elements per block per stage
constexpr int SQ_STAGES = 3;
constexpr int SQ_SLOT = 144;                               // bytes per block per stage (128 + 16: no bank conflict)
constexpr int SQ_BLK_THREADS = 128;
constexpr int SQ_WARP_SMEM = SQ_STAGES * 32 * SQ_SLOT;
constexpr int SQ_BLK_SMEM = (SQ_BLK_THREADS / 32) * SQ_WARP_SMEM;

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem)), "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_2() { asm volatile("cp.async.wait_group 2;" ::: "memory"); }

__device__ float block_sq_warp(const unsigned char* g, int gdt, unsigned char* S) {
  const int lane = threadIdx.x & 31, q = lane & 7;
  const uint64_t gp = (uint64_t)(uintptr_t)g;
  const int esz = gdt == PSK_BF16 ? 2 : 4;
  // lane copies piece q of blocks 4 i + lane / 8, i = 0..7 (a bf16 stage of a
  // block is 4 pieces, an f32 one 8)
  const unsigned char* src[8];
  int step[8];
  bool ok[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int sb = 4 * i + (lane >> 3);
    const uint32_t lo = __shfl_sync(0xffffffffu, (uint32_t)gp, sb);
    const uint32_t hi = __shfl_sync(0xffffffffu, (uint32_t)(gp >> 32), sb);
    const int e = __shfl_sync(0xffffffffu, esz, sb);
    src[i] = (const unsigned char*)(uintptr_t)(((uint64_t)hi << 32) | lo) + q * 16;
    step[i] = SQ_CH * e;
    ok[i] = q * 16 < SQ_CH * e;
  }
  auto issue = [&](int it) {
    unsigned char* st = S + (it % SQ_STAGES) * (32 * SQ_SLOT);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (ok[i]) cp_async16(st + (4 * i + (lane >> 3)) * SQ_SLOT + q * 16, src[i] + (size_t)it * step[i]);
    cp_async_commit();
  };
  constexpr int NIT = SQ_BLOCK / SQ_CH;
  issue(0);
  issue(1);
  float acc = 0.0f;
  for (int it = 0; it < NIT; ++it) {
    if (it + 2 < NIT) issue(it + 2);
    else cp_async_commit();                                // an empty group keeps the count
    cp_async_wait_2();                                     // this lane's copies of stage `it` landed
    __syncwarp();                                          // ... and every other lane's
    const unsigned char* mine = S + (it % SQ_STAGES) * (32 * SQ_SLOT) + lane * SQ_SLOT;
    if (gdt == PSK_BF16) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint4 w4 = *reinterpret_cast<const uint4*>(mine + 16 * u);
        const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float a = __uint_as_float(w[k] << 16), c = __uint_as_float(w[k] & 0xFFFF0000u);
          acc = __fadd_rn(acc, __fmul_rn(a, a));
          acc = __fadd_rn(acc, __fmul_rn(c, c));
        }
      }
    } else {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float4 f = *reinterpret_cast<const float4*>(mine + 16 * u);
        acc = __fadd_rn(acc, __fmul_rn(f.x, f.x));
        acc = __fadd_rn(acc, __fmul_rn(f.y, f.y));
        acc = __fadd_rn(acc, __fmul_rn(f.z, f.z));
        acc = __fadd_rn(acc, __fmul_rn(f.w, f.w));
      }
    }
    __syncwarp();                                          // stage read before a later copy reuses it
  }
  return acc;
}

// One thread per block (SQ_BLK_THREADS blocks per CTA): the warp-cooperative
// path when all 32 blocks of a warp are full and 16-byte aligned, else each
// lane alone.
__global__ void __launch_bounds__(SQ_BLK_THREADS) sq_blocks_kernel(const __grid_constant__ SqParams P) {
  extern __shared__ __align__(16) unsigned char sq_smem[];
  const int64_t b = (int64_t)blockIdx.x * SQ_BLK_THREADS + threadIdx.x;
  const bool have = b < P.n_blocks;
  int lo = 0;
  if (have) {
    int hi = P.n_leaves - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (P.leaf[mid].block_begin <= b) lo = mid; else hi = mid - 1;
    }
  }
  const SqLeaf& L = P.leaf[lo];
  const int64_t base = have ? (b - L.block_begin) * SQ_BLOCK : 0;
  const int n = have ? (int)((L.numel - base) < SQ_BLOCK ? (L.numel - base) : SQ_BLOCK) : 0;
  const unsigned char* g = have ? (const unsigned char*)L.g + base * (L.gdt == PSK_BF16 ? 2 : 4) : nullptr;
  const bool full = have && n == SQ_BLOCK && ((uintptr_t)g & 15u) == 0;
  float acc;
  if (__all_sync(0xffffffffu, full)) acc = block_sq_warp(g, L.gdt, sq_smem + (threadIdx.x >> 5) * SQ_WARP_SMEM);
  else acc = have ? block_sq_lane(L, base, n) : 0.0f;
  if (have) P.block_sums[b] = acc;
}

// One CTA per leaf: its groups (64 consecutive blocks each, added in order) by
// the CTA's threads, then the leaf's sum of its group sums in order.
__global__ void __launch_bounds__(SQ_THREADS) sq_leaves_kernel(const __grid_constant__ SqParams P) {
  const SqLeaf& L = P.leaf[blockIdx.x];
  const int64_t nb = (L.numel + SQ_BLOCK - 1) / SQ_BLOCK;
  const int64_t ng = (nb + SQ_GROUP - 1) / SQ_GROUP;
  for (int64_t gi = threadIdx.x; gi < ng; gi += SQ_THREADS) {
    const int64_t b0 = gi * SQ_GROUP;
    const int64_t b1 = b0 + SQ_GROUP < nb ? b0 + SQ_GROUP : nb;
    const float* bs = P.block_sums + L.block_begin;
    float acc = bs[b0];
    for (int64_t b = b0 + 1; b < b1; ++b) acc = __fadd_rn(acc, bs[b]);
    P.group_sums[L.group_begin + gi] = acc;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const float* gs = P.group_sums + L.group_begin;
    float acc = gs[0];
    for (int64_t gi = 1; gi < ng; ++gi) acc = __fadd_rn(acc, gs[gi]);
    P.leaf_sums[L.leaf_index] = acc;
  }
}

// One thread: the leaf sums in tree order, then the clip scale.
__global__ void sq_scale_kernel(const float* leaf_sums, int32_t n_leaves, float clip, float* scale) {
  float acc = 0.0f;
  for (int i = 0; i < n_leaves; ++i) acc = i == 0 ? leaf_sums[0] : __fadd_rn(acc, leaf_sums[i]);
  const float norm = __fsqrt_rn(acc);
  const float den = __fadd_rn(norm, 1e-6f);
  const float q = __fdiv_rn(clip, den);
  *scale = q < 1.0f ? q : 1.0f;
}

// ------------------------------------------------- host: scalar injection
// Exact arithmetic on binary64 pairs (hi + lo) for 1 - beta and 1 - beta^t,
// then one rounding to binary32.
struct HD { double hi, lo; };

static HD hd_two_sum(double a, double b) {
  double s = a + b, bb = s - a;
  return HD{s, (a - (s - bb)) + (b - bb)};
}
static HD hd_norm(double a, double b) {  // |a| >= |b|
  double s = a + b;
  return HD{s, b - (s - a)};
}
static HD hd_mul(HD a, HD b) {
  double p = a.hi * b.hi;
  double e = fma(a.hi, b.hi, -p);
  e = fma(a.hi, b.lo, e);
  e = fma(a.lo, b.hi, e);
  return hd_norm(p, e);
}
static HD hd_pow(double x, int64_t t) {
  HD r{1.0, 0.0}, b{x, 0.0};
  while (t > 0) {
    if (t & 1) r = hd_mul(r, b);
    b = hd_mul(b, b);
    t >>= 1;
  }
  return r;
}
static HD hd_one_minus(HD a) {
  HD s = hd_two_sum(1.0, -a.hi);
  HD u = hd_two_sum(s.lo, -a.lo);
  return hd_norm(s.hi, u.hi + u.lo);
}
// nearest binary32 to hi + lo (|lo| <= ulp(hi)/2), ties to even
static float hd_to_f32(HD v) {
  float r = (float)v.hi;
  if ((double)r == v.hi || isinf(r)) return r;
  double a = fabs(v.hi), l = v.hi < 0 ? -v.lo : v.lo;
  float ar = fabsf(r);
  double other = (double)ar > a ? (double)nextafterf(ar, 0.0f) : (double)nextafterf(ar, INFINITY);
  double mid = 0.5 * ((double)ar + other);
  if (a != mid || l == 0.0) return r;
  float pick = ((l > 0) == (other > (double)ar)) ? (float)other : ar;
  return v.hi < 0 ? -pick : pick;
}

// ------------------------------------------------- host: lr schedules
static HD hd_div(HD a, double b) {      // a / b for an exact binary64 b
  const double q1 = a.hi / b;
  const double p = q1 * b, pe = fma(q1, b, -p);
  const double r = ((a.hi - p) - pe) + a.lo;
  return hd_norm(q1, r / b);
}
static HD hd_add(HD a, HD b) {
  HD s = hd_two_sum(a.hi, b.hi);
  return hd_norm(s.hi, s.lo + a.lo + b.lo);
}
static const HD HD_PI = {0x1.921fb54442d18p+1, 0x1.1a62633145c07p-53};

// cos(x), 0 <= x <= pi, in double-double (Taylor series after folding x to
// [0, pi/2]; error far below 2^-100).
static HD hd_cos(HD x) {
  bool neg = false;
  if (x.hi > 0.5 * HD_PI.hi) {
    x = hd_add(HD_PI, HD{-x.hi, -x.lo});
    neg = true;
  }
  const HD x2 = hd_mul(x, x);
  HD term{1.0, 0.0}, sum{1.0, 0.0};
  for (int k = 1; k < 30; ++k) {
    term = hd_div(hd_mul(term, x2), (double)((2 * k - 1) * (2 * k)));
    sum = hd_add(sum, (k & 1) ? HD{-term.hi, -term.lo} : term);
    if (fabs(term.hi) < 0x1p-110) break;
  }
  return neg ? HD{-sum.hi, -sum.lo} : sum;
}

// Exact comparison of two normalised double-double values.
static int hd_cmp(HD a, HD b) {
  if (a.hi != b.hi) return a.hi < b.hi ? -1 : 1;
  if (a.lo != b.lo) return a.lo < b.lo ? -1 : 1;
  return 0;
}
static HD hd_prod(double a, double b) {  // exact
  const double p = a * b;
  return hd_norm(p, fma(a, b, -p));
}

// RN_f32(lr * num / den) exactly, for num, den < 2^53 (lr * num and every
// candidate midpoint * den are exact double-double products).
static float rn_f32_rational(double lr, double num, double den) {
  if (num == 0.0 || lr == 0.0) return 0.0f * (float)lr;
  const HD a = hd_prod(lr, num);                 // exact
  const HD q = hd_div(a, den);
  const float c = (float)q.hi;
  const int side = hd_cmp(a, hd_prod((double)c, den));       // true value vs c
  if (side == 0) return c;
  const float nb = nextafterf(c, side > 0 ? INFINITY : -INFINITY);
  const double mid = 0.5 * ((double)c + (double)nb);        // exact
  const int m = hd_cmp(a, hd_prod(mid, den)) * (side > 0 ? 1 : -1);   // > 0: beyond the midpoint
  if (m > 0) return nb;
  if (m < 0) return c;
  uint32_t cb;
  memcpy(&cb, &c, 4);
  return (cb & 1u) ? nb : c;                                 // a tie: the even one
}

// The scheduled learning rate at step t, rounded once to f32.
static int scheduled_lr(const psk_adamw_hparams* hp, const psk_adamw_schedule* sc, float& out) {
  const int64_t t = hp->t, w = sc ? sc->warmup : 0, T = sc ? sc->total : 1;
  const int kind = sc ? sc->kind : PSK_LR_CONSTANT;
  if (kind == PSK_LR_CONSTANT) { out = (float)hp->lr; return PSK_OK; }
  if (kind != PSK_LR_LINEAR && kind != PSK_LR_COSINE) return fail(PSK_E_ARG, "schedule kind %d", kind);
  if (!(w >= 0 && w < T) || T > (int64_t(1) << 52))
    return fail(PSK_E_ARG, "schedule needs 0 <= warmup < total < 2^52 (warmup %lld, total %lld)", (long long)w,
                (long long)T);
  if (w > 0 && t <= w) { out = rn_f32_rational(hp->lr, (double)t, (double)w); return PSK_OK; }
  if (t >= T) { out = 0.0f; return PSK_OK; }
  const int64_t num = t - w, den = T - w;       // r = num / den in (0, 1)
  if (kind == PSK_LR_LINEAR) { out = rn_f32_rational(hp->lr, (double)(den - num), (double)den); return PSK_OK; }
  // cosine: rational where cos(pi r) is (r = 1/3, 1/2, 2/3), else via double-double
  if (3 * num == den) { out = rn_f32_rational(hp->lr, 3.0, 4.0); return PSK_OK; }
  if (2 * num == den) { out = rn_f32_rational(hp->lr, 1.0, 2.0); return PSK_OK; }
  if (3 * num == 2 * den) { out = rn_f32_rational(hp->lr, 1.0, 4.0); return PSK_OK; }
  const HD r = hd_div(HD{(double)num, 0.0}, (double)den);
  const HD c = hd_cos(hd_mul(HD_PI, r));
  const HD f = hd_mul(hd_add(HD{1.0, 0.0}, c), HD{0.5, 0.0});
  out = hd_to_f32(hd_mul(HD{hp->lr, 0.0}, f));
  return PSK_OK;
}

static int make_scalars(const psk_adamw_hparams* hp, AdamScalars& s) {
  if (!hp) return fail(PSK_E_NULL, "hyperparameters are NULL");
  if (hp->t < 1) return fail(PSK_E_ARG, "t = %lld: steps count from 1", (long long)hp->t);
  if (!(hp->beta1 > 0.0 && hp->beta1 < 1.0) || !(hp->beta2 > 0.0 && hp->beta2 < 1.0))
    return fail(PSK_E_ARG, "betas must lie in (0, 1)");
  if (!isfinite(hp->lr) || !isfinite(hp->eps) || !isfinite(hp->weight_decay))
    return fail(PSK_E_ARG, "lr, eps and weight_decay must be finite");
  s.b1 = (float)hp->beta1;
  s.b2 = (float)hp->beta2;
  s.omb1 = hd_to_f32(hd_one_minus(HD{hp->beta1, 0.0}));
  s.omb2 = hd_to_f32(hd_one_minus(HD{hp->beta2, 0.0}));
  s.bc1 = hd_to_f32(hd_one_minus(hd_pow(hp->beta1, hp->t)));
  s.bc2 = hd_to_f32(hd_one_minus(hd_pow(hp->beta2, hp->t)));
  s.lr = (float)hp->lr;
  s.eps = (float)hp->eps;
  s.wd = (float)hp->weight_decay;
  return PSK_OK;
}

// Workspace of the clipped step: the scale, then the block, group and leaf
// sums of the squared-norm tree, each 16-byte aligned.
struct Workspace {
  uint64_t scale_off, blocks_off, groups_off, leaves_off, bytes;
  int64_t n_blocks, n_groups, n_leaves;
};

static uint64_t align16(uint64_t v) { return (v + 15) & ~uint64_t(15); }

static Workspace plan_workspace(const psk_leaf* leaves, int32_t n_leaves, bool clip) {
  Workspace W{};
  if (!clip) return W;
  for (int i = 0; i < n_leaves; ++i) {
    if (leaves[i].numel <= 0) continue;
    const int64_t nb = (leaves[i].numel + SQ_BLOCK - 1) / SQ_BLOCK;
    W.n_blocks += nb;
    W.n_groups += (nb + SQ_GROUP - 1) / SQ_GROUP;
    W.n_leaves += 1;
  }
  W.scale_off = 0;
  W.blocks_off = 16;
  W.groups_off = align16(W.blocks_off + 4 * (uint64_t)W.n_blocks);
  W.leaves_off = align16(W.groups_off + 4 * (uint64_t)W.n_groups);
  W.bytes = align16(W.leaves_off + 4 * (uint64_t)W.n_leaves);
  return W;
}

static int check_leaves(const psk_leaf* leaves, int32_t n_leaves) {
  if (n_leaves < 0) return fail(PSK_E_ARG, "n_leaves %d", n_leaves);
  if (n_leaves > 0 && !leaves) return fail(PSK_E_NULL, "leaf table is NULL");
  for (int i = 0; i < n_leaves; ++i) {
    const psk_leaf& L = leaves[i];
    if (L.numel < 0) return fail(PSK_E_SHAPE, "leaf %d: numel %lld", i, (long long)L.numel);
    if (!dtype_ok(L.grad_dtype)) return fail(PSK_E_DTYPE, "leaf %d: grad dtype %d", i, L.grad_dtype);
    if (!dtype_ok(L.param_dtype)) return fail(PSK_E_DTYPE, "leaf %d: parameter dtype %d", i, L.param_dtype);
    if (L.numel > 0 && (!L.theta || !L.m || !L.v || !L.grad)) return fail(PSK_E_NULL, "leaf %d: NULL pointer", i);
  }
  return PSK_OK;
}

static int check_schedule(const psk_adamw_schedule* sc) {
  if (!sc) return PSK_OK;
  if (!(sc->grad_clip >= 0.0) || !isfinite(sc->grad_clip)) return fail(PSK_E_ARG, "grad_clip must be finite and >= 0");
  if (sc->kind != PSK_LR_CONSTANT && sc->kind != PSK_LR_LINEAR && sc->kind != PSK_LR_COSINE)
    return fail(PSK_E_ARG, "schedule kind %d", sc->kind);
  return PSK_OK;
}

// The block and group stages of the ||g||^2 tree (launches only): the group
// sums of the leaves in order into `groups_out` (NULL: the workspace's), the
// leaf sums into the workspace.
static int launch_sq_groups(const psk_leaf* leaves, int32_t n_leaves, const Workspace& W, char* ws,
                            float* groups_out, cudaStream_t stream, SqParams* staging) {
  SqParams* P = staging ? staging : new SqParams;
  float* blocks = (float*)(ws + W.blocks_off);
  float* groups = groups_out ? groups_out : (float*)(ws + W.groups_off);
  float* leaf_sums = (float*)(ws + W.leaves_off);
  int rc = PSK_OK, i = 0, leaf_index = 0;
  int64_t block0 = 0, group0 = 0;
  while (i < n_leaves && rc == PSK_OK) {
    int cnt = 0;
    int64_t nb_batch = 0, ng_batch = 0;
    for (; i < n_leaves && cnt < PSK_ADAMW_MAX_LEAVES; ++i) {
      const psk_leaf& L = leaves[i];
      if (L.numel == 0) continue;
      SqLeaf& d = P->leaf[cnt++];
      d.g = L.grad;
      d.numel = L.numel;
      d.gdt = L.grad_dtype;
      d.block_begin = nb_batch;
      d.group_begin = ng_batch;
      d.leaf_index = leaf_index++;
      const int64_t nb = (L.numel + SQ_BLOCK - 1) / SQ_BLOCK;
      nb_batch += nb;
      ng_batch += (nb + SQ_GROUP - 1) / SQ_GROUP;
    }
    if (cnt == 0) continue;
    P->n_leaves = cnt;
    P->n_blocks = nb_batch;
    P->block_sums = blocks + block0;
    P->group_sums = groups + group0;
    P->leaf_sums = leaf_sums;
    static bool smem_set[PSK_MAX_DEVICES];
    smem_limit_once((const void*)sq_blocks_kernel, SQ_BLK_SMEM, smem_set);
    sq_blocks_kernel<<<(unsigned)((nb_batch + SQ_BLK_THREADS - 1) / SQ_BLK_THREADS), SQ_BLK_THREADS, SQ_BLK_SMEM,
                       stream>>>(*P);
    rc = check_launch("squared-norm blocks kernel");
    if (rc) break;
    sq_leaves_kernel<<<cnt, SQ_THREADS, 0, stream>>>(*P);
    rc = check_launch("squared-norm leaves kernel");
    block0 += nb_batch;
    group0 += ng_batch;
  }
  if (!staging) delete P;
  return rc;
}

// ||g||^2 tree and the clip scale into the workspace (launches only).
static int launch_clip(const psk_leaf* leaves, int32_t n_leaves, const Workspace& W, char* ws, float clip,
                       cudaStream_t stream, SqParams* staging) {
  const int rc = launch_sq_groups(leaves, n_leaves, W, ws, nullptr, stream, staging);
  if (rc) return rc;
  sq_scale_kernel<<<1, 1, 0, stream>>>((const float*)(ws + W.leaves_off), (int32_t)W.n_leaves, clip,
                                       (float*)(ws + W.scale_off));
  return check_launch("clip scale kernel");
}

// The clip scale from a whole tree's group sums (the groups of its leaves in
// leaf order; leaf l owns groups [begin[l], begin[l + 1])): each leaf's sum
// of its groups in order, by one thread each, then the sum of the non-empty
// leaves' sums in order and the scale, by thread 0 -- the tree and the
// operations of the one-call step.
struct ClipFromGroups {
  int32_t n_leaves;
  float clip;
  int64_t begin[PSK_ADAMW_MAX_LEAVES + 1];
};

__global__ void __launch_bounds__(SQ_THREADS) clip_from_groups_kernel(const float* group_sums,
                                                                      const __grid_constant__ ClipFromGroups P,
                                                                      float* scale) {
  __shared__ float leaf_sum[PSK_ADAMW_MAX_LEAVES];
  for (int l = threadIdx.x; l < P.n_leaves; l += SQ_THREADS) {
    const int64_t g0 = P.begin[l], g1 = P.begin[l + 1];
    float acc = g1 > g0 ? group_sums[g0] : 0.0f;
    for (int64_t g = g0 + 1; g < g1; ++g) acc = __fadd_rn(acc, group_sums[g]);
    leaf_sum[l] = acc;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float acc = 0.0f;
    bool first = true;
    for (int l = 0; l < P.n_leaves; ++l) {
      if (P.begin[l + 1] == P.begin[l]) continue;            // an empty leaf has no groups
      acc = first ? leaf_sum[l] : __fadd_rn(acc, leaf_sum[l]);
      first = false;
    }
    const float norm = __fsqrt_rn(acc);
    const float den = __fadd_rn(norm, 1e-6f);
    const float q = __fdiv_rn(P.clip, den);
    *scale = q < 1.0f ? q : 1.0f;
  }
}

// Host staging of the kernel parameters (the leaf tables, about 28 KB and 20
// KB): from the heap per call, or the caller's (the allocation-free entry
// point passes thread-local ones).
struct HostStaging {
  AdamParams adam;
  SqParams sq;
};

// ext_scale: a clip scale already on the device (the sharded step's), used
// in place of the tree's own clipping.
static int adamw_run(const psk_leaf* leaves, int32_t n_leaves, const psk_adamw_hparams* hp,
                     const psk_adamw_schedule* sc, void* workspace, uint64_t workspace_bytes, void* stream,
                     HostStaging* staging = nullptr, const float* ext_scale = nullptr) {
  int rc = check_leaves(leaves, n_leaves);
  if (rc) return rc;
  rc = check_schedule(sc);
  if (rc) return rc;
  AdamParams* P = staging ? &staging->adam : new AdamParams;   // host staging of the kernel parameter
  rc = make_scalars(hp, P->s);
  if (rc == PSK_OK) rc = scheduled_lr(hp, sc, P->s.lr);
  const bool own_clip = !ext_scale && sc && sc->grad_clip > 0.0;
  const bool clip = own_clip || ext_scale;
  const Workspace W = plan_workspace(leaves, n_leaves, own_clip);
  if (rc == PSK_OK && own_clip) {
    if (!workspace) rc = fail(PSK_E_NULL, "clipping needs a workspace of %llu bytes", (unsigned long long)W.bytes);
    else if (workspace_bytes < W.bytes)
      rc = fail(PSK_E_ARG, "workspace of %llu bytes, clipping needs %llu", (unsigned long long)workspace_bytes,
                (unsigned long long)W.bytes);
    else if ((uintptr_t)workspace % 16 != 0) rc = fail(PSK_E_ARG, "workspace must be 16-byte aligned");
  }
  int sms = 1, per_sm = 1, dev = 0;
  if (rc == PSK_OK) {
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, adamw_kernel<false, PSK_F32>, AW_THREADS, 0);
    if (per_sm < 1) per_sm = 1;
  }
  cudaStream_t s = (cudaStream_t)stream;
  const float* scale = ext_scale ? ext_scale : (own_clip ? (const float*)((char*)workspace + W.scale_off) : nullptr);
  if (rc == PSK_OK && own_clip && W.n_leaves > 0) rc = launch_clip(leaves, n_leaves, W, (char*)workspace,
                                                               (float)sc->grad_clip, s,
                                                               staging ? &staging->sq : nullptr);
  // one launch per PSK_ADAMW_MAX_LEAVES non-empty leaves of each parameter
  // storage type (one launch for the trees here)
  for (int pdt = PSK_F32; pdt <= PSK_BF16 && rc == PSK_OK; ++pdt) {
  int i = 0;
  while (i < n_leaves && rc == PSK_OK) {
    int cnt = 0;
    int64_t chunks = 0;
    for (; i < n_leaves && cnt < PSK_ADAMW_MAX_LEAVES; ++i) {
      const psk_leaf& L = leaves[i];
      if (L.numel == 0 || L.param_dtype != pdt) continue;
      LeafDesc& d = P->leaf[cnt++];
      d.th = L.theta; d.m = L.m; d.v = L.v; d.g = L.grad;
      d.numel = L.numel;
      d.chunk_begin = chunks;
      d.gdt = (int8_t)L.grad_dtype;
      d.pdt = (int8_t)L.param_dtype;
      const uintptr_t ga = L.grad_dtype == PSK_F32 ? 16 : 8, pa = L.param_dtype == PSK_F32 ? 16 : 8;
      d.vec = (int8_t)(((uintptr_t)L.theta % pa == 0) && ((uintptr_t)L.m % pa == 0) && ((uintptr_t)L.v % pa == 0) &&
                       ((uintptr_t)L.grad % ga == 0));
      chunks += (L.numel + AW_CHUNK - 1) / AW_CHUNK;
    }
    if (cnt == 0) continue;
    P->n_leaves = cnt;
    P->n_chunks = chunks;
    int64_t cap = (int64_t)sms * per_sm;
    unsigned grid = (unsigned)(chunks < cap ? chunks : cap);
    if (pdt == PSK_F32) {
      if (clip) adamw_kernel<true, PSK_F32><<<grid, AW_THREADS, 0, s>>>(*P, scale);
      else adamw_kernel<false, PSK_F32><<<grid, AW_THREADS, 0, s>>>(*P, nullptr);
    } else {
      if (clip) adamw_kernel<true, PSK_BF16><<<grid, AW_THREADS, 0, s>>>(*P, scale);
      else adamw_kernel<false, PSK_BF16><<<grid, AW_THREADS, 0, s>>>(*P, nullptr);
    }
    rc = check_launch("adamw tree kernel");
  }
  }
  if (!staging) delete P;
  return rc;
}

// Scratch of psk_adamw_tree_static: one fixed buffer in the library's module
// per device, reserved when the module loads.  Host code must not hand the
// symbol itself to a kernel (on the host it names a host-side stand-in); its
// device address comes from cudaGetSymbolAddress, with the device current,
// once per device and CUDA context (a context created anew, after a device
// reset for instance, gets the address again).  Every value in it is written
// before it is read, so nothing is cleared.
static __device__ __align__(256) unsigned char g_adamw_static_ws[PSK_ADAMW_STATIC_WORKSPACE];

static int static_workspace(void** ptr) {
  struct Entry { CUcontext ctx; void* addr; };
  static Entry cache[PSK_MAX_DEVICES] = {};
  static std::mutex mu;
  static CUresult (*ctx_get_current)(CUcontext*) = [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      fn = nullptr;
    return (CUresult(*)(CUcontext*))fn;
  }();
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= PSK_MAX_DEVICES)
    return fail(PSK_E_CUDA, "no current CUDA device below %d", PSK_MAX_DEVICES);
  if (!ctx_get_current) return fail(PSK_E_CUDA, "cuCtxGetCurrent is not available from the driver");
  std::lock_guard<std::mutex> lock(mu);
  CUcontext ctx = nullptr;
  if (ctx_get_current(&ctx) != CUDA_SUCCESS) ctx = nullptr;
  Entry& e = cache[dev];
  if (!ctx || ctx != e.ctx || !e.addr) {
    void* addr = nullptr;   // cudaGetSymbolAddress also makes the device's primary context current
    if (cudaGetSymbolAddress(&addr, g_adamw_static_ws) != cudaSuccess || !addr) {
      e = Entry{nullptr, nullptr};
      return check_launch("static workspace address");
    }
    if (ctx_get_current(&ctx) != CUDA_SUCCESS) ctx = nullptr;
    e = Entry{ctx, addr};
  }
  *ptr = e.addr;
  return PSK_OK;
}

}  // namespace psk

using namespace psk;

extern "C" int psk_adamw_tree_static(const psk_leaf* leaves, int32_t n_leaves, const psk_adamw_hparams* hp,
                                     const psk_adamw_schedule* sched, void* stream) {
  clear_error();
  static thread_local HostStaging staging;   // no heap allocation per call
  const bool clip = sched && sched->grad_clip > 0.0;
  if (!clip) return adamw_run(leaves, n_leaves, hp, sched, nullptr, 0, stream, &staging);
  int rc = check_leaves(leaves, n_leaves);
  if (rc == PSK_OK) rc = check_schedule(sched);
  if (rc) return rc;
  const Workspace W = plan_workspace(leaves, n_leaves, true);
  if (W.bytes > (uint64_t)PSK_ADAMW_STATIC_WORKSPACE)
    return fail(PSK_E_ARG, "clipping this tree needs %llu bytes of scratch, the fixed buffer holds %llu",
                (unsigned long long)W.bytes, (unsigned long long)PSK_ADAMW_STATIC_WORKSPACE);
  void* ws = nullptr;
  rc = static_workspace(&ws);
  if (rc) return rc;
  return adamw_run(leaves, n_leaves, hp, sched, ws, PSK_ADAMW_STATIC_WORKSPACE, stream, &staging);
}

extern "C" int psk_adamw_scalars(const psk_adamw_hparams* hp, float out[9]) {
  clear_error();
  if (!out) return fail(PSK_E_NULL, "output array is NULL");
  AdamScalars s;
  int rc = make_scalars(hp, s);
  if (rc) return rc;
  float v[9] = {s.b1, s.b2, s.omb1, s.omb2, s.bc1, s.bc2, s.lr, s.eps, s.wd};
  memcpy(out, v, sizeof(v));
  return PSK_OK;
}

extern "C" int psk_adamw_lr(const psk_adamw_hparams* hp, const psk_adamw_schedule* sched, float* lr) {
  clear_error();
  if (!lr) return fail(PSK_E_NULL, "output is NULL");
  AdamScalars s;
  int rc = make_scalars(hp, s);
  if (rc == PSK_OK) rc = check_schedule(sched);
  if (rc == PSK_OK) rc = scheduled_lr(hp, sched, *lr);
  return rc;
}

extern "C" int psk_adamw_workspace(const psk_leaf* leaves, int32_t n_leaves, const psk_adamw_schedule* sched,
                                   uint64_t* bytes) {
  clear_error();
  if (!bytes) return fail(PSK_E_NULL, "output is NULL");
  int rc = check_leaves(leaves, n_leaves);
  if (rc == PSK_OK) rc = check_schedule(sched);
  if (rc) return rc;
  *bytes = plan_workspace(leaves, n_leaves, sched && sched->grad_clip > 0.0).bytes;
  return PSK_OK;
}

extern "C" int psk_adamw_tree(const psk_leaf* leaves, int32_t n_leaves, const psk_adamw_hparams* hp, void* stream) {
  clear_error();
  return adamw_run(leaves, n_leaves, hp, nullptr, nullptr, 0, stream);
}

extern "C" int psk_adamw_tree_ex(const psk_leaf* leaves, int32_t n_leaves, const psk_adamw_hparams* hp,
                                 const psk_adamw_schedule* sched, void* workspace, uint64_t workspace_bytes,
                                 void* stream) {
  clear_error();
  return adamw_run(leaves, n_leaves, hp, sched, workspace, workspace_bytes, stream);
}

extern "C" int psk_adamw_group_sqsums(const psk_leaf* leaves, int32_t n_leaves, float* group_sums, void* workspace,
                                      uint64_t workspace_bytes, void* stream) {
  clear_error();
  int rc = check_leaves(leaves, n_leaves);
  if (rc) return rc;
  const Workspace W = plan_workspace(leaves, n_leaves, true);
  if (W.n_groups == 0) return PSK_OK;
  if (!group_sums) return fail(PSK_E_NULL, "group_sums is NULL");
  if (!workspace) return fail(PSK_E_NULL, "the group sums need a workspace of %llu bytes", (unsigned long long)W.bytes);
  if (workspace_bytes < W.bytes)
    return fail(PSK_E_ARG, "workspace of %llu bytes, the group sums need %llu", (unsigned long long)workspace_bytes,
                (unsigned long long)W.bytes);
  if ((uintptr_t)workspace % 16 != 0) return fail(PSK_E_ARG, "workspace must be 16-byte aligned");
  return launch_sq_groups(leaves, n_leaves, W, (char*)workspace, group_sums, (cudaStream_t)stream, nullptr);
}

extern "C" int psk_adamw_clip_scale(const float* group_sums, const int64_t* groups_per_leaf, int32_t n_leaves,
                                    double grad_clip, float* scale, void* stream) {
  clear_error();
  if (n_leaves < 0 || n_leaves > PSK_ADAMW_MAX_LEAVES)
    return fail(PSK_E_ARG, "n_leaves %d (at most %d)", n_leaves, PSK_ADAMW_MAX_LEAVES);
  if (!(grad_clip > 0.0) || !isfinite(grad_clip)) return fail(PSK_E_ARG, "grad_clip must be finite and > 0");
  if (!scale) return fail(PSK_E_NULL, "scale is NULL");
  if (n_leaves > 0 && !groups_per_leaf) return fail(PSK_E_NULL, "groups_per_leaf is NULL");
  ClipFromGroups P;
  P.n_leaves = n_leaves;
  P.clip = (float)grad_clip;
  P.begin[0] = 0;
  for (int l = 0; l < n_leaves; ++l) {
    if (groups_per_leaf[l] < 0) return fail(PSK_E_ARG, "groups_per_leaf[%d] = %lld", l, (long long)groups_per_leaf[l]);
    P.begin[l + 1] = P.begin[l] + groups_per_leaf[l];
  }
  if (P.begin[n_leaves] > 0 && !group_sums) return fail(PSK_E_NULL, "group_sums is NULL");
  clip_from_groups_kernel<<<1, SQ_THREADS, 0, (cudaStream_t)stream>>>(group_sums, P, scale);
  return check_launch("clip scale from group sums");
}

extern "C" int psk_adamw_tree_scaled(const psk_leaf* leaves, int32_t n_leaves, const psk_adamw_hparams* hp,
                                     const psk_adamw_schedule* sched, const float* scale, void* stream) {
  clear_error();
  if (!scale) return fail(PSK_E_NULL, "scale is NULL");
  return adamw_run(leaves, n_leaves, hp, sched, nullptr, 0, stream, nullptr, scale);
}
