// Shared helpers of the library's translation units: refusals with a
// thread-local message, storage conversions, fast 32-bit division.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdarg.h>

#include "../../include/psk.h"

#include "host.h"
#include "devcommon.cuh"

namespace psk {

inline int dtype_size(int32_t dt) { return dt == PSK_BF16 ? 2 : 4; }
inline bool dtype_ok(int32_t dt) { return dt == PSK_F32 || dt == PSK_BF16; }

}  // namespace psk
