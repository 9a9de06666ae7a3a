// Host-side helpers shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "pa.h"

namespace pa {

// Remember a CUDA failure for pa_last_cuda_error(); returns PA_ERR_CUDA.
pa_status cuda_fail(const char* where, cudaError_t e);
pa_status cuda_fail_msg(const char* where, const char* msg);

// Streaming multiprocessors of the current device (cached per device).
int num_sms();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// TMA descriptor of a K or V pool viewed as rows of D elements of eb bytes
// (num_blocks * n_kv * block_size rows); a box is box_rows rows of 128 bytes
// (64 bf16 or 128 fp8 columns) with the 128-byte swizzle. try3d: for bf16
// with D = 128, try one 3-D view that fetches both 64-column halves in one
// copy (*map3d = 1 if built). Encoded maps are cached per thread.
pa_status make_pool_map(CUtensorMap* map, const void* pool, int D, int eb, int64_t rows,
                        int box_rows, bool try3d, int* map3d);

}  // namespace pa
