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

#include <math.h>
#include <string.h>

#include "common.cuh"

namespace psk {

constexpr int AW_THREADS = 256;
constexpr int AW_CHUNK = 4096;                 // elements per chunk
constexpr int AW_VPT = AW_CHUNK / (AW_THREADS * 4);   // float4 vectors per thread per chunk

struct LeafDesc {
  float* th;
  float* m;
  float* v;
  const void* g;
  int64_t numel;
  int64_t chunk_begin;   // first chunk of this leaf in the launch
  int32_t gdt;
  int32_t vec;           // 16-byte aligned theta/m/v and 8/16-byte aligned grad
};

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

__global__ void __launch_bounds__(AW_THREADS) adamw_kernel(const __grid_constant__ AdamParams P) {
  const int t = threadIdx.x;
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
        th[k] = __ldcs((const float4*)(L.th + i));
        m[k] = __ldcs((const float4*)(L.m + i));
        v[k] = __ldcs((const float4*)(L.v + i));
        if (L.gdt == PSK_F32) {
          g[k] = __ldcs((const float4*)((const float*)L.g + i));
        } else {
          uint2 q = __ldcs((const uint2*)((const unsigned short*)L.g + i));
          g[k] = make_float4(__uint_as_float(q.x << 16), __uint_as_float(q.x & 0xFFFF0000u),
                             __uint_as_float(q.y << 16), __uint_as_float(q.y & 0xFFFF0000u));
        }
      }
#pragma unroll
      for (int k = 0; k < AW_VPT; ++k) {
        adamw_one(P.s, th[k].x, m[k].x, v[k].x, g[k].x);
        adamw_one(P.s, th[k].y, m[k].y, v[k].y, g[k].y);
        adamw_one(P.s, th[k].z, m[k].z, v[k].z, g[k].z);
        adamw_one(P.s, th[k].w, m[k].w, v[k].w, g[k].w);
        const int64_t i = base + (int64_t)(k * AW_THREADS + t) * 4;
        __stcs((float4*)(L.th + i), th[k]);
        __stcs((float4*)(L.m + i), m[k]);
        __stcs((float4*)(L.v + i), v[k]);
      }
    } else {
      for (int64_t j = t; j < n; j += AW_THREADS) {
        const int64_t i = base + j;
        float th = L.th[i], m = L.m[i], v = L.v[i];
        float g = load_grad(L.g, L.gdt, i);
        adamw_one(P.s, th, m, v, g);
        L.th[i] = th;
        L.m[i] = m;
        L.v[i] = v;
      }
    }
  }
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

}  // namespace psk

using namespace psk;

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

extern "C" int psk_adamw_tree(const psk_leaf* leaves, int32_t n_leaves, const psk_adamw_hparams* hp, void* stream) {
  clear_error();
  if (n_leaves < 0) return fail(PSK_E_ARG, "n_leaves %d", n_leaves);
  if (n_leaves > 0 && !leaves) return fail(PSK_E_NULL, "leaf table is NULL");
  AdamParams* P = new AdamParams;   // host staging of the kernel parameter
  int rc = make_scalars(hp, P->s);
  for (int i = 0; i < n_leaves && rc == PSK_OK; ++i) {
    const psk_leaf& L = leaves[i];
    if (L.numel < 0) rc = fail(PSK_E_SHAPE, "leaf %d: numel %lld", i, (long long)L.numel);
    else if (!dtype_ok(L.grad_dtype)) rc = fail(PSK_E_DTYPE, "leaf %d: grad dtype %d", i, L.grad_dtype);
    else if (L.numel > 0 && (!L.theta || !L.m || !L.v || !L.grad)) rc = fail(PSK_E_NULL, "leaf %d: NULL pointer", i);
  }
  int sms = 1, per_sm = 1, dev = 0;
  if (rc == PSK_OK) {
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, adamw_kernel, AW_THREADS, 0);
    if (per_sm < 1) per_sm = 1;
  }
  // one launch per PSK_ADAMW_MAX_LEAVES non-empty leaves (one launch for the trees here)
  int i = 0;
  while (i < n_leaves && rc == PSK_OK) {
    int cnt = 0;
    int64_t chunks = 0;
    for (; i < n_leaves && cnt < PSK_ADAMW_MAX_LEAVES; ++i) {
      const psk_leaf& L = leaves[i];
      if (L.numel == 0) continue;
      LeafDesc& d = P->leaf[cnt++];
      d.th = L.theta; d.m = L.m; d.v = L.v; d.g = L.grad;
      d.numel = L.numel;
      d.chunk_begin = chunks;
      d.gdt = L.grad_dtype;
      const uintptr_t ga = L.grad_dtype == PSK_F32 ? 16 : 8;
      d.vec = ((uintptr_t)L.theta % 16 == 0) && ((uintptr_t)L.m % 16 == 0) && ((uintptr_t)L.v % 16 == 0) &&
              ((uintptr_t)L.grad % ga == 0);
      chunks += (L.numel + AW_CHUNK - 1) / AW_CHUNK;
    }
    if (cnt == 0) continue;
    P->n_leaves = cnt;
    P->n_chunks = chunks;
    int64_t cap = (int64_t)sms * per_sm;
    unsigned grid = (unsigned)(chunks < cap ? chunks : cap);
    adamw_kernel<<<grid, AW_THREADS, 0, (cudaStream_t)stream>>>(*P);
    rc = check_launch("adamw tree kernel");
  }
  delete P;
  return rc;
}
