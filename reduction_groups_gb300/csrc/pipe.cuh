// Shared-memory pipeline primitives for sm_100-class GPUs (inline PTX):
// mbarriers with bounded waits and 1-D bulk copies (TMA) from global memory
// into shared memory that complete on an mbarrier.
//
// Every wait is a try_wait loop with an iteration limit; when the limit is
// reached the caller gets false, the kernel records a timeout in a status
// word and winds down (no wait in this library can spin forever).
#pragma once

#include <stdint.h>

namespace psk {

// Status word of the pipelined kernels: 0 = no timeout seen.  One copy per
// translation unit that includes this header (each is its own device module);
// psk_device_status() reads and resets every copy.
static __device__ unsigned int g_pipe_status;

// Test hook (psk_test_drop_row): the local row at which every pipelined
// region CTA's producer stops, as if that row's copy were lost, so that the
// bounded waits run out; -1 (the default) never.  One copy per translation
// unit, like the status word; psk_test_drop_row() sets every copy.
static __device__ long long g_pipe_drop_row = -1;

constexpr unsigned int PIPE_TIMEOUT = 1u;
constexpr long long PIPE_WAIT_CYCLES = 4000000000LL;   // ~2 s at 2 GHz: far beyond any legitimate wait

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.release.cta.shared::cta.b64 st, [%0];\n\t}" ::"r"(
                   smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.release.cta.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
          smem_addr(bar)),
      "r"(bytes)
      : "memory");
}

// One probe of the phase with this parity; the thread may be suspended for
// up to about a microsecond while the phase is still open.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(1000u)
      : "memory");
  return ok != 0;
}

// Wait until the phase with this parity has completed; false (and the
// timeout recorded) after PIPE_WAIT_CYCLES of clock.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (clock64() - t0 < PIPE_WAIT_CYCLES)
    if (mbar_try_wait(bar, parity)) return true;
  atomicOr(&g_pipe_status, PIPE_TIMEOUT);
  return false;
}

// Make mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// 1-D bulk copy global -> shared of `bytes` (a multiple of 16, both addresses
// 16-byte aligned), completing `bytes` of transaction count on `bar`.
__device__ __forceinline__ void bulk_copy_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Named barrier among `nthreads` threads (a multiple of 32) with id `id` (1..15).
__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

}  // namespace psk
