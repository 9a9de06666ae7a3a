// Status strings, the thread-local CUDA error text, device queries, and the
// check that the library's bounded waits give up.
#include <cstdio>
#include <mutex>
#include <string>

#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {

static thread_local std::string g_last_error;

pa_status cuda_fail(const char* where, cudaError_t e) {
  g_last_error = std::string(where) + ": " + cudaGetErrorName(e) + " (" +
                 cudaGetErrorString(e) + ")";
  return PA_ERR_CUDA;
}

pa_status cuda_fail_msg(const char* where, const char* msg) {
  g_last_error = std::string(where) + ": " + msg;
  return PA_ERR_CUDA;
}

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

}  // namespace pa

extern "C" const char* pa_status_string(pa_status s) {
  switch (s) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
  }
  return "PA_UNKNOWN_STATUS";
}

extern "C" const char* pa_last_cuda_error(void) { return pa::g_last_error.c_str(); }

namespace pa {

// One thread waits on an mbarrier that nothing arrives on, with the same
// bounded wait the decode and prefill kernels use, and reports the timeout
// through the error word: the wait gives up and the kernel returns.
__global__ void bounded_wait_check_kernel(int32_t* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  fence_mbarrier_init();
  if (!mbar_wait_bounded(b, 0, limit_ns)) report(err, PA_DEV_ERR_TIMEOUT);
}

}  // namespace pa

extern "C" pa_status pa_check_bounded_wait(int32_t* err_word, int64_t limit_ns,
                                           pa_stream_t stream) {
  if (!err_word || limit_ns <= 0 || limit_ns > 2000000000LL) return PA_ERR_INVALID_ARG;
  pa::bounded_wait_check_kernel<<<1, 1, 0, (cudaStream_t)stream>>>(err_word,
                                                                    (uint64_t)limit_ns);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? PA_OK : pa::cuda_fail("pa_check_bounded_wait launch", e);
}

