// Paged chunked-prefill attention for sm_103a.
//
// What it computes ("Serving: vLLM and PagedAttention", section 2.4, chunked
// prefill; "03 · PagedAttention", the kernel gathers K/V through the block
// table): a sequence's last c tokens (its chunk, already written to the pool)
// each attend causally to every cached position up to their own, the pool
// reached through the block table exactly as in decode.
//
// Design: one CTA per (query tile, sequence, kv head). The tile's rows are
// (token, query head) pairs of the G query heads sharing the kv head, 64 rows
// (64 / G tokens), 16 per warp, so every K/V unit staged in shared memory
// serves all G heads. 16-token K/V units stream through a 4-stage ring filled
// by TMA (128-byte swizzle, the same boxes as decode) and shared by the four
// warps. Per unit and warp: S = Q K^T with Q in registers and K^T fragments
// from ldmatrix, causal and length masking, online softmax in base 2 with a
// lazily moved reference, then O += P V with P reused from the score
// registers (as a bf16 hi + lo pair) and V^T fragments from ldmatrix.trans;
// bf16 mma.sync m16n8k16, fp32 accumulation. Tiles are numbered so the longest (latest) tiles of a
// sequence start first.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace {

constexpr int kPWarps = 4;
constexpr int kPThreads = kPWarps * 32;
constexpr int kPRows = kPWarps * 16;  // (token, head) rows per tile
constexpr int kPUnit = 16;            // K/V tokens per stage
constexpr int kPStages = 4;
constexpr uint64_t kPWaitNs = 2000000000ull;      // 2 s: a wait that long is a fault
constexpr uint64_t kPWaitAfterFaultNs = 1000000ull;
constexpr float kPLazyLog2 = 8.f;
constexpr float kPLog2e = 1.4426950408889634f;

struct PrefillArgs {
  __nv_bfloat16* out;
  const __nv_bfloat16* q;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const int32_t* cu_q;
  int32_t* err;
  int num_seqs, max_blocks, num_blocks, n_q, n_kv, group;
  int tile_tokens;  // query tokens per tile: 64 / G, rounded down
  int n_tiles;      // grid.x: tiles of the longest chunk
  int map3d;
  float scale_log2;
};

template <int D, int BS>
struct PCfg {
  static constexpr int ROWS = BS < kPUnit ? BS : kPUnit;  // rows per TMA box
  static constexpr int BOXES = kPUnit / ROWS;
  static constexpr int KH = D / 64;                       // 128-byte halves of a row
  static constexpr int BOX_BYTES = KH * ROWS * 128;
  static constexpr int KV_BYTES = BOXES * BOX_BYTES;      // 16 rows of K (or V)
  static constexpr int STAGE = 2 * KV_BYTES;
  static constexpr int BAR_OFF = kPStages * STAGE;
  static constexpr int MASK_OFF = BAR_OFF + kPStages * 8;
  static constexpr int FAULT_OFF = MASK_OFF + kPStages * 4;
  static constexpr size_t SMEM = 1024 + FAULT_OFF + 16;
};

// Shared-memory address of 16-byte chunk `ch` of K/V row `r` (0..15) of a
// unit staged at `base` (boxes of ROWS rows, 128-byte halves, swizzled).
template <int D, int BS>
__device__ __forceinline__ uint32_t unit_addr(uint32_t base, int r, int ch) {
  using C = PCfg<D, BS>;
  return base + (r / C::ROWS) * C::BOX_BYTES + (ch >> 3) * C::ROWS * 128 +
         (r % C::ROWS) * 128 + (((ch & 7) ^ (r & 7)) << 4);
}

template <int D, int BS>
__global__ void __launch_bounds__(kPThreads)
prefill_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
               const PrefillArgs a) {
  using C = PCfg<D, BS>;
  constexpr int KS = D / 16;  // k-steps of Q K^T
  constexpr int DT = D / 8;   // n-tiles of the output
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  int* smask = reinterpret_cast<int*>(smem + C::MASK_OFF);
  volatile int* fault = reinterpret_cast<int*>(smem + C::FAULT_OFF);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, cq = lane & 3;

  griddep_wait();  // the chunk's K/V come from the preceding cache write

  const int s = blockIdx.y, g = blockIdx.z;
  const int qt = a.n_tiles - 1 - (int)blockIdx.x;  // the latest tiles first
  const int cq0 = __ldg(&a.cu_q[s]);
  const int c = __ldg(&a.cu_q[s + 1]) - cq0;
  const int G = a.group, TQ = a.tile_tokens;
  const int t0 = qt * TQ;
  // a chunk longer than max_q_len: the rows beyond the grid stay unwritten
  if (blockIdx.x == 0 && g == 0 && tid == 0 && c > a.n_tiles * TQ)
    report(a.err, PA_DEV_ERR_SEQ_LEN);
  if (c <= 0 || t0 >= c) return;
  int L = __ldg(&a.seq_lens[s]);
  const int cap = a.max_blocks * BS;
  if (L > cap || L < c) {  // clamped / nothing visible: flagged, rows not written if L < c
    if (tid == 0 && blockIdx.x == 0 && g == 0) report(a.err, PA_DEV_ERR_SEQ_LEN);
    if (L > cap) L = cap;
  }
  const int nt = min(TQ, c - t0);  // query tokens in this tile

  // ---- this thread's two rows (gq and gq + 8 of the warp's 16)
  int pos[2];
  int64_t orow[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = warp * 16 + gq + 8 * h;
    const int t = r / G, n = r - (r / G) * G;
    const bool ok = r < TQ * G && t < nt && L >= c;
    pos[h] = ok ? L - c + t0 + t : -1;  // -1: no key is visible, the row is not written
    orow[h] = ok ? ((int64_t)(cq0 + t0 + t) * a.n_q + (int64_t)g * G + n) : -1;
  }
  // ---- Q fragments (A operand, rows x head_dim)
  uint32_t qa[KS][4];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t* qr = reinterpret_cast<const uint32_t*>(a.q + (orow[h] < 0 ? 0 : orow[h]) * D);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qa[ks][h] = orow[h] < 0 ? 0u : __ldg(&qr[ks * 8 + cq]);
      qa[ks][2 + h] = orow[h] < 0 ? 0u : __ldg(&qr[ks * 8 + 4 + cq]);
    }
  }

  const int pmax = L - c + t0 + nt - 1;  // the tile's last position
  const int n_units = pmax < 0 ? 0 : pmax / kPUnit + 1;
  const int32_t* table = a.block_tables + (int64_t)s * a.max_blocks;

  if (tid == 0) {
    for (int i = 0; i < kPStages; ++i) mbar_init(sbase + C::BAR_OFF + 8 * i, 1);
    *fault = 0;
    fence_mbarrier_init();
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
  }
  __syncthreads();

  // Unit u's pool blocks (one per box), raw; checked where they are used.
  auto unit_ids = [&](int u, int (&ids)[C::BOXES]) {
#pragma unroll
    for (int b = 0; b < C::BOXES; ++b) {
      const int tok = u * kPUnit + b * C::ROWS;
      ids[b] = tok < L ? __ldg(&table[tok / BS]) : -1;
    }
  };
  // Thread 0: load unit u into stage st (absent or invalid boxes skipped).
  auto issue = [&](int u, int st, const int (&ids)[C::BOXES]) {
    const uint32_t fb = sbase + C::BAR_OFF + 8 * st;
    int mask = 0, nload = 0;
#pragma unroll
    for (int b = 0; b < C::BOXES; ++b) {
      const int tok = u * kPUnit + b * C::ROWS;
      if (tok >= L) continue;
      if (ids[b] >= 0 && ids[b] < a.num_blocks) {
        mask |= 1 << b;
        ++nload;
      } else {
        report(a.err, PA_DEV_ERR_BLOCK_ID);
      }
    }
    smask[st] = mask;
    if (nload == 0) {
      mbar_arrive(fb);
      return;
    }
    mbar_arrive_expect_tx(fb, (uint32_t)nload * 2 * C::BOX_BYTES);
    const uint32_t kdst = sbase + st * C::STAGE, vdst = kdst + C::KV_BYTES;
#pragma unroll
    for (int b = 0; b < C::BOXES; ++b) {
      if (!(mask >> b & 1)) continue;
      const int tok_in_block = (u * kPUnit) % BS + b * C::ROWS;
      const int32_t y = (ids[b] * a.n_kv + g) * BS + (BS > kPUnit ? tok_in_block : 0);
      if (C::KH == 2 && a.map3d) {
        tma_load_3d(kdst + b * C::BOX_BYTES, &tmk, 0, y, 0, fb);
        tma_load_3d(vdst + b * C::BOX_BYTES, &tmv, 0, y, 0, fb);
      } else {
#pragma unroll
        for (int h = 0; h < C::KH; ++h) {
          tma_load_2d(kdst + b * C::BOX_BYTES + h * C::ROWS * 128, &tmk, h * 64, y, fb);
          tma_load_2d(vdst + b * C::BOX_BYTES + h * C::ROWS * 128, &tmv, h * 64, y, fb);
        }
      }
    }
  };

  int ids_next[C::BOXES];
  if (tid == 0) {
    for (int u = 0; u < n_units && u < kPStages; ++u) {
      int ids[C::BOXES];
      unit_ids(u, ids);
      issue(u, u, ids);
    }
  }

  float acc[DT][4];
#pragma unroll
  for (int dt = 0; dt < DT; ++dt) acc[dt][0] = acc[dt][1] = acc[dt][2] = acc[dt][3] = 0.f;
  float mrun[2] = {-INFINITY, -INFINITY}, lrun[2] = {0.f, 0.f};

  // ldmatrix lane roles: matrix mi = lane / 8, its row lane % 8
  const int mi = lane >> 3;
  const int k_row = (lane & 7) + 8 * (mi >> 1), k_ch = mi & 1;  // K: x4 = 2 token groups x 2 chunks
  const int v_row = (lane & 7) + 8 * (mi & 1), v_ch = mi >> 1;  // V^T: x4 = 2 chunks x 2 token groups

#pragma unroll 1
  for (int u = 0; u < n_units; ++u) {
    const int st = u % kPStages;
    if (tid == 0 && u + kPStages < n_units) unit_ids(u + kPStages, ids_next);
    {
      const uint64_t limit = *fault ? kPWaitAfterFaultNs : kPWaitNs;
      if (!mbar_wait_bounded(sbase + C::BAR_OFF + 8 * st, (u / kPStages) & 1, limit)) {
        report(a.err, PA_DEV_ERR_TIMEOUT);
        *fault = 1;
      }
    }
    const int mask = smask[st];
    const int j0 = u * kPUnit;
    const int nvalid = min(kPUnit, L - j0);
    const uint32_t kb = sbase + st * C::STAGE, vb = kb + C::KV_BYTES;
    bool all_ok = nvalid == kPUnit;
#pragma unroll
    for (int b = 0; b < C::BOXES; ++b)
      if (b * C::ROWS < nvalid && !(mask >> b & 1)) all_ok = false;
    if (!all_ok) {
      // rows of absent tokens may hold anything (even NaN): zero their V so a
      // zero weight times the row stays zero
      for (int i = tid; i < kPUnit * C::KH * 8; i += kPThreads) {
        const int r = i / (C::KH * 8), ch = i % (C::KH * 8);
        if (r >= nvalid || !(mask >> (r / C::ROWS) & 1))
          *reinterpret_cast<uint4*>(smem + (unit_addr<D, BS>(vb, r, ch) - sbase)) =
              make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();  // before the stage is refilled by TMA
      __syncthreads();
    }

    // ---- S = Q K^T, 16 rows x 16 tokens per warp
    float sc[2][4];
#pragma unroll
    for (int i = 0; i < 2; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4(unit_addr<D, BS>(kb, k_row, 2 * ks + k_ch), b0, b1, b2, b3);
      mma_bf16_16816(sc[0], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
      mma_bf16_16816(sc[1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
    }
    // ---- causal / length / block masks, online softmax (lazy reference)
    float x[2][4];
    float rmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int jl = i * 8 + 2 * cq + (e & 1);  // token within the unit
        const int h = e >> 1;                     // row gq or gq + 8
        const bool ok = jl < nvalid && (mask >> (jl / C::ROWS) & 1) && j0 + jl <= pos[h];
        x[i][e] = ok ? sc[i][e] * a.scale_log2 : -INFINITY;
        rmax[h] = fmaxf(rmax[h], x[i][e]);
      }
    const bool need = rmax[0] > mrun[0] + kPLazyLog2 || rmax[1] > mrun[1] + kPLazyLog2;
    if (__any_sync(0xffffffffu, need)) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float mx = rmax[h];
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(mrun[h], mx);
        const float alpha = fast_exp2(mrun[h] - (m_new == -INFINITY ? 0.f : m_new));
        lrun[h] *= alpha;
#pragma unroll
        for (int dt = 0; dt < DT; ++dt) {
          acc[dt][2 * h] *= alpha;
          acc[dt][2 * h + 1] *= alpha;
        }
        mrun[h] = m_new;
      }
    }
    float p[2][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int h = e >> 1;
        p[i][e] = fast_exp2(x[i][e] - (mrun[h] == -INFINITY ? 0.f : mrun[h]));
        lrun[h] += p[i][e];
      }
    // P as a bf16 pair hi + lo (hi = bf16(p), lo = bf16(p - hi)): a lone
    // bf16 weight is off by up to 2^-9 relative, which on rows that see only
    // a few keys (the start of a prompt) is as large as the whole output
    // tolerance; the pair is good to about 2^-17.
    uint32_t ph[4], pl[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float lo_in = p[k >> 1][(k & 1) * 2], hi_in = p[k >> 1][(k & 1) * 2 + 1];
      ph[k] = pack_bf16x2(lo_in, hi_in);
      pl[k] = pack_bf16x2(lo_in - __uint_as_float(ph[k] << 16),
                          hi_in - __uint_as_float(ph[k] & 0xffff0000u));
    }
    // ---- O += P V
#pragma unroll
    for (int dp = 0; dp < DT / 2; ++dp) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4_trans(unit_addr<D, BS>(vb, v_row, 2 * dp + v_ch), b0, b1, b2, b3);
      mma_bf16_16816(acc[2 * dp], ph[0], ph[1], ph[2], ph[3], b0, b1);
      mma_bf16_16816(acc[2 * dp + 1], ph[0], ph[1], ph[2], ph[3], b2, b3);
      mma_bf16_16816(acc[2 * dp], pl[0], pl[1], pl[2], pl[3], b0, b1);
      mma_bf16_16816(acc[2 * dp + 1], pl[0], pl[1], pl[2], pl[3], b2, b3);
    }
    __syncthreads();  // every warp is done with stage st
    if (tid == 0 && u + kPStages < n_units) issue(u + kPStages, st, ids_next);
  }

  // ---- normalise and write the rows
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float l = lrun[h];
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    if (orow[h] < 0) continue;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    __nv_bfloat162* o = reinterpret_cast<__nv_bfloat162*>(a.out + orow[h] * D);
#pragma unroll
    for (int dt = 0; dt < DT; ++dt)
      o[dt * 4 + cq] = __floats2bfloat162_rn(acc[dt][2 * h] * inv, acc[dt][2 * h + 1] * inv);
  }
}

template <int D, int BS>
pa_status launch_prefill(PrefillArgs a, const void* k_pool, const void* v_pool,
                         cudaStream_t stream) {
  using C = PCfg<D, BS>;
  const int64_t rows = (int64_t)a.num_blocks * a.n_kv * BS;
  CUtensorMap tmk, tmv;
  int k3 = 0, v3 = 0;
  pa_status st = make_pool_map(&tmk, k_pool, D, 2, rows, C::ROWS, true, &k3);
  if (st != PA_OK) return st;
  st = make_pool_map(&tmv, v_pool, D, 2, rows, C::ROWS, k3 == 1, &v3);
  if (st != PA_OK) return st;
  if (k3 != v3) {
    st = make_pool_map(&tmk, k_pool, D, 2, rows, C::ROWS, false, &k3);
    if (st != PA_OK) return st;
  }
  a.map3d = k3 && v3;
  auto kern = prefill_kernel<D, BS>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
    if (e != cudaSuccess) return cuda_fail("pa_prefill smem attribute", e);
    configured = true;
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.n_tiles, (unsigned)a.num_seqs, (unsigned)a.n_kv);
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tmk, tmv, a);
  return e == cudaSuccess ? PA_OK : cuda_fail("pa_prefill launch", e);
}

template <int D>
pa_status prefill_bs(int bs, const PrefillArgs& a, const void* kp, const void* vp,
                     cudaStream_t st) {
  switch (bs) {
    case 8: return launch_prefill<D, 8>(a, kp, vp, st);
    case 16: return launch_prefill<D, 16>(a, kp, vp, st);
    default: return launch_prefill<D, 32>(a, kp, vp, st);
  }
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" pa_status pa_prefill(void* out, const void* q, const void* k_pool, const void* v_pool,
                                const int32_t* block_tables, const int32_t* seq_lens,
                                const int32_t* cu_q, int num_seqs, int max_blocks_per_seq,
                                int num_blocks, int n_q_heads, int n_kv_heads, int head_dim,
                                int block_size, float scale, int max_q_len, int32_t* err_word,
                                pa_stream_t stream) {
  if (num_seqs < 0 || num_seqs > 65535 || max_blocks_per_seq < 1 || num_blocks < 1 ||
      n_q_heads < 1 || n_kv_heads < 1 || n_kv_heads > 65535 || max_q_len < 0)
    return PA_ERR_INVALID_ARG;
  if (n_q_heads % n_kv_heads != 0) return PA_ERR_INVALID_ARG;
  const int G = n_q_heads / n_kv_heads;
  if ((head_dim != 64 && head_dim != 128) ||
      (block_size != 8 && block_size != 16 && block_size != 32) || G > kPRows)
    return PA_ERR_UNSUPPORTED;
  if ((int64_t)num_blocks * n_kv_heads * block_size >= (int64_t)1 << 31)
    return PA_ERR_INVALID_ARG;
  if (num_seqs == 0 || max_q_len == 0) return PA_OK;
  if (!out || !q || !k_pool || !v_pool || !block_tables || !seq_lens || !cu_q)
    return PA_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool))
    return PA_ERR_INVALID_ARG;
  PrefillArgs a;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.block_tables = block_tables;
  a.seq_lens = seq_lens;
  a.cu_q = cu_q;
  a.err = err_word;
  a.num_seqs = num_seqs;
  a.max_blocks = max_blocks_per_seq;
  a.num_blocks = num_blocks;
  a.n_q = n_q_heads;
  a.n_kv = n_kv_heads;
  a.group = G;
  a.tile_tokens = kPRows / G;
  const int64_t tiles = ((int64_t)max_q_len + a.tile_tokens - 1) / a.tile_tokens;
  if (tiles > 2147483647) return PA_ERR_INVALID_ARG;
  a.n_tiles = (int)tiles;
  a.map3d = 0;
  a.scale_log2 = scale * kPLog2e;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (head_dim == 64) return prefill_bs<64>(block_size, a, k_pool, v_pool, st);
  return prefill_bs<128>(block_size, a, k_pool, v_pool, st);
}
