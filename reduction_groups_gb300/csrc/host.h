// Host-side bookkeeping shared by the library's translation units (defined
// in api.cpp): refusals with a thread-local message, launch-error mapping and
// per-device attribute caches.
#pragma once

namespace psk {

// Record a refusal for psk_last_error() and return its code.
int fail(int code, const char* fmt, ...);
void clear_error();
// Map a CUDA runtime error after a launch to PSK_E_CUDA with its name.
int check_launch(const char* what);

// Device attributes, cached per device (the current device of the calling
// thread).
constexpr int PSK_MAX_DEVICES = 64;
int device_sm_count();
// Raise `kernel`'s dynamic shared-memory limit to `bytes` on the current
// device, once per device; `done` is the call site's per-device flag array.
void smem_limit_once(const void* kernel, int bytes, bool* done);

}  // namespace psk
