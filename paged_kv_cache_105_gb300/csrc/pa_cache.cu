// Cache writes of one decode step: the new tokens' K/V into their slots, and
// copy-on-write block duplication. Both are bit copies in 16-byte vectors;
// a (block, kv head) run and a token's head row are contiguous, so every
// warp reads and writes whole 128-byte lines.
//
// Sources: "PagedAttention" (mlapandio.dev), "A DECODE STEP" diagram (the
// step writes the new K and V into the current block) and "COPY-ON-WRITE ON
// A SHARED PREFIX" diagram (copy the shared block, then write);
// "03 · PagedAttention", "Sharing: copy-on-write, straight from fork()".
#include <cuda_runtime.h>
#include <stdint.h>

#include <cmath>

#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {

// One thread per 16-byte chunk of one (token, kv head) row of K or V.
__global__ void __launch_bounds__(256)
reshape_and_cache_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                         uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                         const int32_t* __restrict__ slot_mapping, int num_tokens,
                         int num_blocks, int n_kv, int chunks_per_row, int block_size,
                         int32_t* err) {
  // A programmatic dependent of the preceding kernel: wait for it (it may
  // have produced the new K/V, the slots or a copied block), then let a
  // dependent decode start launching; its prologue reads only inputs that
  // were complete before this point.
  griddep_wait();
  griddep_launch_dependents();
  const int64_t per_tensor = (int64_t)num_tokens * n_kv * chunks_per_row;
  const int64_t total = 2 * per_tensor;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const bool is_v = i >= per_tensor;
    const int64_t r = is_v ? i - per_tensor : i;
    const int c = (int)(r % chunks_per_row);
    const int64_t th = r / chunks_per_row;  // token * n_kv + head
    const int h = (int)(th % n_kv);
    const int t = (int)(th / n_kv);
    // both loads are issued before either is needed
    const int64_t src = th * chunks_per_row + c;
    const uint4 val = is_v ? __ldg(&v[src]) : __ldg(&k[src]);
    const int32_t slot = __ldg(&slot_mapping[t]);
    if (slot < 0) continue;  // padding
    if ((int64_t)slot >= (int64_t)num_blocks * block_size) {
      if (c == 0 && h == 0 && !is_v) report(err, PA_DEV_ERR_SLOT);
      continue;
    }
    const int64_t blk = slot / block_size, off = slot % block_size;
    const int64_t dst = ((blk * n_kv + h) * block_size + off) * chunks_per_row + c;
    (is_v ? v_pool : k_pool)[dst] = val;
  }
}

// grid.y = pair; threads stride over the 16-byte chunks of one block of K
// followed by the same block of V.
__global__ void __launch_bounds__(256)
copy_blocks_kernel(uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                   const int32_t* __restrict__ pairs, int num_blocks, int64_t chunks_per_block,
                   int32_t* err) {
  griddep_wait();  // a programmatic dependent: the preceding kernel first
  griddep_launch_dependents();
  const int p = blockIdx.y;
  const int32_t src = __ldg(&pairs[2 * p]);
  const int32_t dst = __ldg(&pairs[2 * p + 1]);
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report(err, PA_DEV_ERR_PAIR);
    return;
  }
  const int64_t total = 2 * chunks_per_block;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const bool is_v = i >= chunks_per_block;
    const int64_t c = is_v ? i - chunks_per_block : i;
    uint4* pool = is_v ? v_pool : k_pool;
    pool[(int64_t)dst * chunks_per_block + c] = pool[(int64_t)src * chunks_per_block + c];
  }
}

// fp8 cache write: one thread per 16 codes (16 bytes of output, 32 bytes of
// bf16 input) of one (token, kv head) row of K or V. code = E4M3 of
// fp32(x) / scale, the division rounded to nearest, the conversion rounded
// to nearest even and saturated to +-448.
__global__ void __launch_bounds__(256)
reshape_and_cache_fp8_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                             uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                             const int32_t* __restrict__ slot_mapping, int num_tokens,
                             int num_blocks, int n_kv, int chunks_per_row, int block_size,
                             float k_scale, float v_scale, int32_t* err) {
  griddep_wait();  // as reshape_and_cache_kernel
  griddep_launch_dependents();
  const int64_t per_tensor = (int64_t)num_tokens * n_kv * chunks_per_row;
  const int64_t total = 2 * per_tensor;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const bool is_v = i >= per_tensor;
    const int64_t r = is_v ? i - per_tensor : i;
    const int c = (int)(r % chunks_per_row);
    const int64_t th = r / chunks_per_row;  // token * n_kv + head
    const int h = (int)(th % n_kv);
    const int t = (int)(th / n_kv);
    const int64_t src = 2 * (th * chunks_per_row + c);  // two 16-byte bf16 chunks
    const uint4* in = is_v ? v : k;
    const uint4 x0 = __ldg(&in[src]), x1 = __ldg(&in[src + 1]);
    const int32_t slot = __ldg(&slot_mapping[t]);
    if (slot < 0) continue;
    if ((int64_t)slot >= (int64_t)num_blocks * block_size) {
      if (c == 0 && h == 0 && !is_v) report(err, PA_DEV_ERR_SLOT);
      continue;
    }
    const float sc = is_v ? v_scale : k_scale;
    const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      // two bf16 words = 4 values -> 4 codes (one 32-bit word)
      const uint32_t a = w[2 * j], b = w[2 * j + 1];
      const uint32_t lo = f32x2_to_e4m3x2(__fdiv_rn(__uint_as_float(a << 16), sc),
                                          __fdiv_rn(__uint_as_float(a & 0xffff0000u), sc));
      const uint32_t hi = f32x2_to_e4m3x2(__fdiv_rn(__uint_as_float(b << 16), sc),
                                          __fdiv_rn(__uint_as_float(b & 0xffff0000u), sc));
      o[j] = lo | (hi << 16);
    }
    const int64_t blk = slot / block_size, off = slot % block_size;
    const int64_t dst = ((blk * n_kv + h) * block_size + off) * chunks_per_row + c;
    (is_v ? v_pool : k_pool)[dst] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// Swap: grid.y strides over pairs; threads stride over the 16-byte chunks of
// the K block then the V block. Either side may be host memory the device
// addresses directly (pinned and mapped), so the copy runs over the
// chip-to-chip link without staging or one copy call per block.
__global__ void __launch_bounds__(256)
swap_blocks_kernel(uint4* __restrict__ dst_k, uint4* __restrict__ dst_v,
                   const uint4* __restrict__ src_k, const uint4* __restrict__ src_v,
                   const int32_t* __restrict__ pairs, int n_pairs, int src_num_blocks,
                   int dst_num_blocks, int64_t chunks_per_block, int32_t* err) {
  for (int p = blockIdx.y; p < n_pairs; p += gridDim.y) {
    const int32_t src = pairs[2 * p];
    const int32_t dst = pairs[2 * p + 1];
    if (src < 0 || src >= src_num_blocks || dst < 0 || dst >= dst_num_blocks) {
      if (blockIdx.x == 0 && threadIdx.x == 0) report(err, PA_DEV_ERR_PAIR);
      continue;
    }
    const int64_t total = 2 * chunks_per_block;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
      const bool is_v = i >= chunks_per_block;
      const int64_t c = is_v ? i - chunks_per_block : i;
      const uint4 val = (is_v ? src_v : src_k)[(int64_t)src * chunks_per_block + c];
      (is_v ? dst_v : dst_k)[(int64_t)dst * chunks_per_block + c] = val;
    }
  }
}

// A plain copy of n16 16-byte chunks where either side may be page-locked
// host memory the device addresses directly: the SMs move a step's small
// inputs and outputs over the chip-to-chip link on the same stream as the
// step's kernels, with no copy-engine hand-off between them.
__global__ void __launch_bounds__(256)
host_copy_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src, int64_t n16) {
  griddep_wait();  // a programmatic dependent: the preceding kernel first
  griddep_launch_dependents();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n16; i += 4 * stride) {  // four loads in flight per thread
    const uint4 a = src[i], b = src[i + stride], c = src[i + 2 * stride], d = src[i + 3 * stride];
    dst[i] = a;
    dst[i + stride] = b;
    dst[i + 2 * stride] = c;
    dst[i + 3 * stride] = d;
  }
  for (; i < n16; i += stride) dst[i] = src[i];
}

// The address through which the current device reaches `p`: device or
// managed memory of this device as is, page-locked host memory through its
// mapped device pointer. Anything else (pageable host memory, another
// device's memory) is refused before a kernel could touch it.
static bool device_view(const void* p, const void** out) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();  // clear the error the failed query recorded
    return false;
  }
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  switch (at.type) {
    case cudaMemoryTypeDevice:
      if (at.device != dev) return false;
      *out = p;
      return true;
    case cudaMemoryTypeManaged:
      *out = p;
      return true;
    case cudaMemoryTypeHost:
      if (at.devicePointer == nullptr) return false;
      *out = at.devicePointer;
      return true;
    default:
      return false;
  }
}

// Launch as a programmatic dependent of the preceding kernel on `stream`:
// the launch overlaps that kernel's tail, and the kernel waits for it
// (griddep_wait) before touching memory.
template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block,
                              cudaStream_t stream, Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

static bool supported_dims(int head_dim, int block_size) {
  return (head_dim == 64 || head_dim == 128) &&
         (block_size == 8 || block_size == 16 || block_size == 32);
}

}  // namespace pa

using namespace pa;

extern "C" pa_status pa_reshape_and_cache(const void* k, const void* v, void* k_pool,
                                          void* v_pool, const int32_t* slot_mapping,
                                          int num_tokens, int num_blocks, int n_kv_heads,
                                          int head_dim, int block_size, int32_t* err_word,
                                          pa_stream_t stream) {
  if (num_tokens < 0 || num_blocks <= 0 || n_kv_heads <= 0) return PA_ERR_INVALID_ARG;
  if (!supported_dims(head_dim, block_size)) return PA_ERR_UNSUPPORTED;
  if ((int64_t)num_blocks * n_kv_heads * block_size >= (int64_t)1 << 31)
    return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !k_pool || !v_pool || !slot_mapping) return PA_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_pool) || !aligned16(v_pool))
    return PA_ERR_INVALID_ARG;
  const int chunks = head_dim * 2 / 16;
  const int64_t total = 2LL * num_tokens * n_kv_heads * chunks;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = (int64_t)num_sms() * 8;
  if (blocks > cap) blocks = cap;
  cudaError_t e = launch_pdl(reshape_and_cache_kernel, dim3((unsigned)blocks), dim3(threads),
                             (cudaStream_t)stream, (const uint4*)k, (const uint4*)v,
                             (uint4*)k_pool, (uint4*)v_pool, slot_mapping, num_tokens,
                             num_blocks, n_kv_heads, chunks, block_size, err_word);
  return e == cudaSuccess ? PA_OK : cuda_fail("pa_reshape_and_cache launch", e);
}

extern "C" pa_status pa_copy_blocks(void* k_pool, void* v_pool, const int32_t* pairs,
                                    int n_pairs, int n_kv_heads, int head_dim, int block_size,
                                    int num_blocks, int32_t* err_word, pa_stream_t stream) {
  if (n_pairs < 0 || num_blocks <= 0 || n_kv_heads <= 0) return PA_ERR_INVALID_ARG;
  if (!supported_dims(head_dim, block_size)) return PA_ERR_UNSUPPORTED;
  if (n_pairs > 65535) return PA_ERR_INVALID_ARG;
  if (n_pairs == 0) return PA_OK;
  if (!k_pool || !v_pool || !pairs) return PA_ERR_INVALID_ARG;
  if (!aligned16(k_pool) || !aligned16(v_pool)) return PA_ERR_INVALID_ARG;
  const int64_t chunks = (int64_t)n_kv_heads * block_size * head_dim * 2 / 16;
  const int threads = 256;
  int64_t bx = (2 * chunks + threads - 1) / threads;
  if (bx > 64) bx = 64;
  dim3 grid((unsigned)bx, (unsigned)n_pairs);
  cudaError_t e = launch_pdl(copy_blocks_kernel, grid, dim3(threads), (cudaStream_t)stream,
                             (uint4*)k_pool, (uint4*)v_pool, pairs, num_blocks, chunks,
                             err_word);
  return e == cudaSuccess ? PA_OK : cuda_fail("pa_copy_blocks launch", e);
}

extern "C" pa_status pa_reshape_and_cache_fp8(const void* k, const void* v, void* k_pool,
                                              void* v_pool, const int32_t* slot_mapping,
                                              int num_tokens, int num_blocks, int n_kv_heads,
                                              int head_dim, int block_size, float k_scale,
                                              float v_scale, int32_t* err_word,
                                              pa_stream_t stream) {
  if (num_tokens < 0 || num_blocks <= 0 || n_kv_heads <= 0) return PA_ERR_INVALID_ARG;
  if (!supported_dims(head_dim, block_size)) return PA_ERR_UNSUPPORTED;
  if (!(k_scale > 0.f && v_scale > 0.f && k_scale < INFINITY && v_scale < INFINITY))
    return PA_ERR_INVALID_ARG;
  if ((int64_t)num_blocks * n_kv_heads * block_size >= (int64_t)1 << 31)
    return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !k_pool || !v_pool || !slot_mapping) return PA_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_pool) || !aligned16(v_pool))
    return PA_ERR_INVALID_ARG;
  const int chunks = head_dim / 16;  // 16 codes per output chunk
  const int64_t total = 2LL * num_tokens * n_kv_heads * chunks;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = (int64_t)num_sms() * 8;
  if (blocks > cap) blocks = cap;
  cudaError_t e = launch_pdl(reshape_and_cache_fp8_kernel, dim3((unsigned)blocks),
                             dim3(threads), (cudaStream_t)stream, (const uint4*)k,
                             (const uint4*)v, (uint4*)k_pool, (uint4*)v_pool, slot_mapping,
                             num_tokens, num_blocks, n_kv_heads, chunks, block_size, k_scale,
                             v_scale, err_word);
  return e == cudaSuccess ? PA_OK : cuda_fail("pa_reshape_and_cache_fp8 launch", e);
}

extern "C" pa_status pa_copy_blocks_fp8(void* k_pool, void* v_pool, const int32_t* pairs,
                                        int n_pairs, int n_kv_heads, int head_dim,
                                        int block_size, int num_blocks, int32_t* err_word,
                                        pa_stream_t stream) {
  if (n_pairs < 0 || num_blocks <= 0 || n_kv_heads <= 0) return PA_ERR_INVALID_ARG;
  if (!supported_dims(head_dim, block_size)) return PA_ERR_UNSUPPORTED;
  if (n_pairs > 65535) return PA_ERR_INVALID_ARG;
  if (n_pairs == 0) return PA_OK;
  if (!k_pool || !v_pool || !pairs) return PA_ERR_INVALID_ARG;
  if (!aligned16(k_pool) || !aligned16(v_pool)) return PA_ERR_INVALID_ARG;
  const int64_t chunks = (int64_t)n_kv_heads * block_size * head_dim / 16;  // 1-byte codes
  const int threads = 256;
  int64_t bx = (2 * chunks + threads - 1) / threads;
  if (bx > 64) bx = 64;
  dim3 grid((unsigned)bx, (unsigned)n_pairs);
  cudaError_t e = launch_pdl(copy_blocks_kernel, grid, dim3(threads), (cudaStream_t)stream,
                             (uint4*)k_pool, (uint4*)v_pool, pairs, num_blocks, chunks,
                             err_word);
  return e == cudaSuccess ? PA_OK : cuda_fail("pa_copy_blocks_fp8 launch", e);
}

extern "C" pa_status pa_swap_blocks(void* dst_k, void* dst_v, const void* src_k,
                                    const void* src_v, const int32_t* pairs, int n_pairs,
                                    size_t block_bytes, int src_num_blocks, int dst_num_blocks,
                                    int32_t* err_word, pa_stream_t stream) {
  if (n_pairs < 0 || src_num_blocks <= 0 || dst_num_blocks <= 0) return PA_ERR_INVALID_ARG;
  if (block_bytes == 0 || block_bytes % 16 != 0) return PA_ERR_INVALID_ARG;
  if (n_pairs == 0) return PA_OK;
  if (!dst_k || !dst_v || !src_k || !src_v || !pairs) return PA_ERR_INVALID_ARG;
  const void* ptr[5] = {dst_k, dst_v, src_k, src_v, pairs};
  const void* dv[5];
  for (int i = 0; i < 5; ++i)
    if (!device_view(ptr[i], &dv[i])) return PA_ERR_INVALID_ARG;
  if (err_word) {
    const void* ew;
    if (!device_view(err_word, &ew)) return PA_ERR_INVALID_ARG;
    err_word = const_cast<int32_t*>(static_cast<const int32_t*>(ew));
  }
  for (int i = 0; i < 4; ++i)
    if (!aligned16(dv[i])) return PA_ERR_INVALID_ARG;
  const int64_t chunks = (int64_t)(block_bytes / 16);
  const int threads = 256;
  int64_t bx = (2 * chunks + threads - 1) / threads;
  if (bx > 16) bx = 16;
  const unsigned gy = (unsigned)(n_pairs < 65535 ? n_pairs : 65535);
  swap_blocks_kernel<<<dim3((unsigned)bx, gy), threads, 0, (cudaStream_t)stream>>>(
      (uint4*)dv[0], (uint4*)dv[1], (const uint4*)dv[2], (const uint4*)dv[3],
      (const int32_t*)dv[4], n_pairs, src_num_blocks, dst_num_blocks, chunks, err_word);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? PA_OK : cuda_fail("pa_swap_blocks launch", e);
}

extern "C" pa_status pa_copy_host(void* dst, const void* src, size_t nbytes, pa_stream_t stream) {
  if (nbytes == 0) return PA_OK;
  if (!dst || !src || nbytes % 16 != 0) return PA_ERR_INVALID_ARG;
  const void* dd;
  const void* ds;
  if (!device_view(dst, &dd) || !device_view(src, &ds)) return PA_ERR_INVALID_ARG;
  if (!aligned16(dd) || !aligned16(ds)) return PA_ERR_INVALID_ARG;
  const int64_t n16 = (int64_t)(nbytes / 16);
  const int threads = 256;
  int64_t blocks = (n16 + threads - 1) / threads;
  const int64_t cap = (int64_t)num_sms() * 2;
  if (blocks > cap) blocks = cap;
  cudaError_t e = launch_pdl(host_copy_kernel, dim3((unsigned)blocks), dim3(threads),
                             (cudaStream_t)stream, (uint4*)dd, (const uint4*)ds, n16);
  return e == cudaSuccess ? PA_OK : cuda_fail("pa_copy_host launch", e);
}

