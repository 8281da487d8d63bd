// Refusal bookkeeping of the C ABI: a thread-local message per refusal.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>

#include "../../include/psk.h"
#include "host.h"

namespace psk {

static thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

void clear_error() { g_err[0] = '\0'; }

int check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(PSK_E_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return PSK_OK;
}

static int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) dev = 0;
  return dev;
}

int device_sm_count() {
  static int cache[PSK_MAX_DEVICES] = {};
  const int dev = current_device();
  int n = dev < PSK_MAX_DEVICES ? cache[dev] : 0;
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    if (dev < PSK_MAX_DEVICES) cache[dev] = n;
  }
  return n;
}

void smem_limit_once(const void* kernel, int bytes, bool* done) {
  const int dev = current_device();
  if (dev < PSK_MAX_DEVICES && done[dev]) return;
  cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (dev < PSK_MAX_DEVICES) done[dev] = true;
}

}  // namespace psk

extern "C" const char* psk_last_error(void) { return psk::g_err; }
