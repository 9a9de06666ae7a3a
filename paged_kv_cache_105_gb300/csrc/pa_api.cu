// Status strings, the thread-local CUDA error text and device queries.
#include <cstdio>
#include <mutex>
#include <string>

#include "pa_internal.h"

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
