// Host-side helpers shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>

#include "pa.h"

namespace pa {

// Remember a CUDA failure for pa_last_cuda_error(); returns PA_ERR_CUDA.
pa_status cuda_fail(const char* where, cudaError_t e);
pa_status cuda_fail_msg(const char* where, const char* msg);

// Streaming multiprocessors of the current device (cached per device).
int num_sms();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace pa
