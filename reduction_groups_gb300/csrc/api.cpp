// Refusal bookkeeping of the C ABI: a thread-local message per refusal.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>

#include "../../include/psk.h"

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

}  // namespace psk

extern "C" const char* psk_last_error(void) { return psk::g_err; }
