// Device helpers shared by the library's kernels and by the group kernels
// compiled at run time: nothing here needs a host header.
#pragma once

#if !defined(__CUDACC_RTC__)
#include <stdint.h>
#endif

namespace psk {

// q = n / d for 32-bit n and a fixed d >= 1, by a multiply-high and shifts
// (the round-up method of Granlund and Montgomery).
struct FastDiv {
  uint32_t d, m, s;
  __host__ __device__ FastDiv() : d(1), m(0), s(0) {}
  __host__ __device__ explicit FastDiv(uint32_t div) : d(div), m(0), s(0) {
    if (d <= 1) { d = 1; return; }
    uint32_t l = 0;
    while ((1ull << l) < d) ++l;                       // l = ceil(log2 d) >= 1
    m = (uint32_t)((((1ull << l) - d) << 32) / d + 1);
    s = l;
  }
  __host__ __device__ __forceinline__ uint32_t div(uint32_t n) const {
    if (s == 0) return n;
#if defined(__CUDA_ARCH__)
    uint32_t t = __umulhi(n, m);
#else
    uint32_t t = (uint32_t)(((uint64_t)n * m) >> 32);
#endif
    return (t + ((n - t) >> 1)) >> (s - 1);
  }
};

// bf16 storage: widen by a shift; narrow by one round to nearest even.
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) { return __uint_as_float(b16 << 16); }

__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(x));
  return r;
}

}  // namespace psk
