// Paged decode attention for sm_103a.
//
// What it computes ("03 · PagedAttention", "The part the analogy hides: the
// kernel"; "PagedAttention" (mlapandio.dev), "A DECODE STEP" diagram): for
// each sequence, one query token per query head attends over every cached
// token, whose K/V are gathered from scattered pool blocks through the
// sequence's block table. The pages describe no kernel design; everything
// below is this library's.
//
// Design (one GPU, HBM-bound: every step reads all cached K/V once):
//  * Work items are (sequence, kv head, partition of P tokens). Items are
//    numbered sequence-major from per-sequence prefix sums that every CTA
//    builds in shared memory; persistent CTAs (a few per SM) take them from
//    a global counter, so no CTA is launched for empty work.
//  * A CTA has 4 warps. The item's 16-token units (a 16-token block, two
//    8-token blocks, or one 32-token block) are dealt round-robin to the
//    warps. Each warp runs its own STAGES-deep pipeline: one lane looks up
//    the unit's physical block(s) and issues 2-D TMA tile loads of the K and
//    V rows, 128-byte swizzled, completing on a per-stage mbarrier.
//  * The GQA group (the G query heads sharing the kv head) is the N side of
//    bf16 mma.sync m16n8k16 with the tokens on M: S^T = K Q^T, then
//    O^T += V^T P^T. movmatrix turns the score fragment into the P^T operand
//    in registers. Online softmax in fp32 (base-2, running max per head).
//  * Warps merge through shared memory; a one-partition sequence writes its
//    bf16 output directly, otherwise the partition's (O, m, l) goes to the
//    workspace and the last CTA to finish a (sequence, kv head) — decided by
//    an atomic ticket, nobody waits — merges the partitions with
//    log-sum-exp weights and writes the output.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <climits>
#include <mutex>

#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: a wait that long is a fault
constexpr int kMaxParts = 1024;
constexpr int kMaxSeqs = 65536;
constexpr float kLog2e = 1.4426950408889634f;

struct DecodeArgs {
  __nv_bfloat16* out;
  const __nv_bfloat16* q;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  float* ws_o;               // [S][Hq][max_parts][D]  un-normalised partial outputs
  float2* ws_ml;             // [S][Hq][max_parts]     (running max, sum) in log2 units
  int32_t* tickets;          // [S][Hkv]               partitions finished
  int32_t* work;             // [2]: items handed out beyond the first wave, CTAs done
  int32_t* err;
  int num_seqs, max_blocks, num_blocks, n_q, n_kv, group;
  int part_tokens, max_parts, len_cap;
  float scale_log2;
};

template <int D, int BS, int NT>
struct Cfg {
  static constexpr int ST = BS < 16 ? 16 : BS;  // tokens per pipeline stage (one unit)
  static constexpr int BPU = ST / BS;           // pool blocks per unit
  static constexpr int KH = D / 64;             // 128-byte halves of a K/V row
  static constexpr int TILE = ST * 128;         // bytes of one half of K or V for a unit
  static constexpr int STAGE = 2 * KH * TILE;   // K + V bytes of a unit
  static constexpr int STAGES_RAW = 24576 / STAGE;
  static constexpr int STAGES = STAGES_RAW < 2 ? 2 : (STAGES_RAW > 8 ? 8 : STAGES_RAW);
  static constexpr int PIPE = kWarps * STAGES * STAGE;
  static constexpr int MSTRIDE = D + 4;  // padded row of the cross-warp merge buffer
  static constexpr int HEADS = NT * 8;
  static constexpr int MERGE = kWarps * HEADS * (MSTRIDE + 2) * 4;
  static_assert(MERGE <= PIPE, "merge buffer must fit in the pipeline buffers");
  static constexpr int BAR_OFF = PIPE;
  static constexpr int MISC_OFF = BAR_OFF + kWarps * STAGES * 8;
  static constexpr int PREFIX_OFF = MISC_OFF + 16;
  static size_t smem_bytes(int num_seqs) {
    return 1024 /* alignment slack */ + PREFIX_OFF + sizeof(int) * (size_t)(num_seqs + 1);
  }
};

__device__ __forceinline__ int clamp_len(int len, int cap) {
  return len < 0 ? 0 : (len > cap ? cap : len);
}

__device__ __forceinline__ int parts_of(int len, int P) {
  return len <= 0 ? 1 : (len + P - 1) / P;
}

__device__ __forceinline__ float warp_max_xor4(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
  return v;
}

__device__ __forceinline__ float warp_sum_xor4(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 4);
  v += __shfl_xor_sync(0xffffffffu, v, 8);
  v += __shfl_xor_sync(0xffffffffu, v, 16);
  return v;
}

// Exclusive prefix over sequences of the item count n_kv * parts(len).
__device__ void build_prefix(int* prefix, const DecodeArgs& a, int* warp_tot) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (a.num_seqs + kThreads - 1) / kThreads;
  const int b = min(a.num_seqs, tid * per), e = min(a.num_seqs, b + per);
  int sum = 0;
  for (int s = b; s < e; ++s) {
    const int raw = __ldg(&a.seq_lens[s]);
    const int len = clamp_len(raw, a.len_cap);
    if (raw != len && blockIdx.x == 0) report(a.err, PA_DEV_ERR_SEQ_LEN);
    sum += a.n_kv * parts_of(len, a.part_tokens);
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int base = 0;
  for (int w = 0; w < warp; ++w) base += warp_tot[w];
  int run = base + incl - sum;
  for (int s = b; s < e; ++s) {
    prefix[s] = run;
    run += a.n_kv * parts_of(clamp_len(__ldg(&a.seq_lens[s]), a.len_cap), a.part_tokens);
  }
  if (tid == kThreads - 1) prefix[a.num_seqs] = base + incl;
}

template <int D, int BS, int NT>
__global__ void __launch_bounds__(kThreads)
decode_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
              const DecodeArgs a) {
  using C = Cfg<D, BS, NT>;
  constexpr int ST = C::ST, BPU = C::BPU, KH = C::KH, STAGES = C::STAGES;
  constexpr int KS = D / 16;  // 16-wide steps along head_dim

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t bar_base = smem_base + C::BAR_OFF;
  int* misc = reinterpret_cast<int*>(smem + C::MISC_OFF);  // [0] next item [1] last [2] abort
  int* prefix = reinterpret_cast<int*>(smem + C::PREFIX_OFF);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int i = 0; i < kWarps * STAGES; ++i) mbar_init(bar_base + 8 * i, 1);
    misc[2] = 0;
    fence_mbarrier_init();
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
  }
  {
    // warp totals borrow the merge area (not yet in use)
    int* warp_tot = reinterpret_cast<int*>(smem);
    build_prefix(prefix, a, warp_tot);
  }
  __syncthreads();
  const int total = prefix[a.num_seqs];

  const uint32_t warp_pipe = smem_base + warp * STAGES * C::STAGE;
  const uint32_t warp_bar = bar_base + warp * STAGES * 8;
  uint32_t used = 0;  // stages this warp has consumed so far (same on all lanes)
  int item = blockIdx.x;
  uint32_t drain_from = 0, drain_to = 0;  // stages still in flight after a timeout

  while (item < total) {
    int next = 0;
    if (tid == 0) next = atomicAdd(&a.work[0], 1) + (int)gridDim.x;

    // ---- locate the item: sequence s, kv head g, partition p
    int lo = 0, hi = a.num_seqs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (prefix[mid] <= item) lo = mid; else hi = mid - 1;
    }
    const int s = lo;
    const int nparts = (prefix[s + 1] - prefix[s]) / a.n_kv;
    const int local = item - prefix[s];
    const int g = local / nparts, p = local - g * nparts;
    const int len = clamp_len(__ldg(&a.seq_lens[s]), a.len_cap);
    const int tok_begin = p * a.part_tokens;
    const int tok_end = min(len, tok_begin + a.part_tokens);
    const int u_begin = tok_begin / ST;
    const int n_units = tok_end > tok_begin ? (tok_end + ST - 1) / ST - u_begin : 0;
    const int n_w = n_units > warp ? (n_units - warp + kWarps - 1) / kWarps : 0;
    const int32_t* table = a.block_tables + (int64_t)s * a.max_blocks;

    // ---- lane k holds the physical block(s) of this warp's k-th unit
    int ids[BPU];
#pragma unroll
    for (int b = 0; b < BPU; ++b) ids[b] = -2;  // -2: no tokens there
    if (lane < n_w) {
      const int u = u_begin + warp + lane * kWarps;
#pragma unroll
      for (int b = 0; b < BPU; ++b) {
        const int j = u * BPU + b;
        if (j * BS < tok_end) {
          int id = __ldg(&table[j]);
          if (id < 0 || id >= a.num_blocks) {
            report(a.err, PA_DEV_ERR_BLOCK_ID);
            id = -1;  // tokens of this block are treated as absent
          }
          ids[b] = id;
        }
      }
    }

    auto issue = [&](int k) {
      int bid[BPU];
#pragma unroll
      for (int b = 0; b < BPU; ++b) bid[b] = __shfl_sync(0xffffffffu, ids[b], k);
      if (lane == 0) {
        const uint32_t stage = (used + k) % STAGES;
        const uint32_t bar = warp_bar + 8 * stage;
        const uint32_t kdst = warp_pipe + stage * C::STAGE;
        const uint32_t vdst = kdst + KH * C::TILE;
        int nload = 0;
#pragma unroll
        for (int b = 0; b < BPU; ++b) nload += bid[b] >= 0;
        if (nload == 0) {
          mbar_arrive(bar);
        } else {
          mbar_arrive_expect_tx(bar, (uint32_t)nload * 2 * KH * BS * 128);
#pragma unroll
          for (int b = 0; b < BPU; ++b) {
            if (bid[b] < 0) continue;
            const int32_t y = (bid[b] * a.n_kv + g) * BS;
#pragma unroll
            for (int h = 0; h < KH; ++h) {
              tma_load_2d(kdst + h * C::TILE + b * BS * 128, &tmk, h * 64, y, bar);
              tma_load_2d(vdst + h * C::TILE + b * BS * 128, &tmv, h * 64, y, bar);
            }
          }
        }
      }
    };

#pragma unroll 1
    for (int k = 0; k < STAGES; ++k)
      if (k < n_w) issue(k);

    // ---- query fragments (B operand: head_dim x heads, column-major = q rows)
    uint32_t qf[NT][KS][2];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int n = t * 8 + (lane >> 2);
      const bool real = n < a.group;
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
          a.q + ((int64_t)s * a.n_q + g * a.group + (real ? n : 0)) * D);
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qf[t][ks][0] = real ? __ldg(&qrow[ks * 8 + (lane & 3)]) : 0u;
        qf[t][ks][1] = real ? __ldg(&qrow[ks * 8 + 4 + (lane & 3)]) : 0u;
      }
    }

    float acc[NT][KS][4];
    float mrun[NT][2], lrun[NT][2];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
#pragma unroll
      for (int dt = 0; dt < KS; ++dt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[t][dt][i] = 0.f;
      mrun[t][0] = mrun[t][1] = -INFINITY;
      lrun[t][0] = lrun[t][1] = 0.f;
    }

#pragma unroll 1
    for (int k = 0; k < n_w; ++k) {
      const uint32_t idx = used + k;
      const uint32_t stage = idx % STAGES;
      if (!mbar_wait_bounded(warp_bar + 8 * stage, (idx / STAGES) & 1u, kWaitLimitNs)) {
        if (lane == 0) {
          report(a.err, PA_DEV_ERR_TIMEOUT);
          misc[2] = 1;
        }
        drain_from = used + k;
        drain_to = used + min(n_w, k + STAGES);
        break;
      }
      const int u = u_begin + warp + k * kWarps;
      const int nv = min(ST, tok_end - u * ST);  // valid tokens in this unit
      int bid[BPU];
      bool all_ok = nv == ST;
#pragma unroll
      for (int b = 0; b < BPU; ++b) {
        bid[b] = __shfl_sync(0xffffffffu, ids[b], k);
        if (b * BS < nv && bid[b] < 0) all_ok = false;
      }
      const uint32_t kb = warp_pipe + stage * C::STAGE;
      const uint32_t vb = kb + KH * C::TILE;
      if (!all_ok) {
        // Rows of absent tokens may hold anything (even NaN): zero their V so
        // that a zero weight times the row stays zero.
        uint8_t* vgen = smem + (vb - smem_base);
        for (int i = lane; i < ST * KH * 8; i += 32) {
          const int r = i / (KH * 8), rest = i % (KH * 8);
          const int h = rest / 8, c = rest % 8;
          if (r >= nv || bid[r / BS] < 0)
            *reinterpret_cast<uint4*>(vgen + h * C::TILE + r * 128 + c * 16) =
                make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }

#pragma unroll
      for (int mt = 0; mt < ST / 16; ++mt) {
        if (mt * 16 >= nv) break;
        // ---- S^T = K Q^T for 16 tokens x 8 heads (per n-tile)
        float sc[NT][4];
#pragma unroll
        for (int t = 0; t < NT; ++t) sc[t][0] = sc[t][1] = sc[t][2] = sc[t][3] = 0.f;
        {
          const int r = mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            const int h = ks >> 2;
            const int c = ((ks & 3) << 1) + (lane >> 4);
            const uint32_t addr = kb + h * C::TILE + r * 128 + ((c ^ (r & 7)) << 4);
            uint32_t a0, a1, a2, a3;
            ldsm_x4(addr, a0, a1, a2, a3);
#pragma unroll
            for (int t = 0; t < NT; ++t)
              mma_bf16_16816(sc[t], a0, a1, a2, a3, qf[t][ks][0], qf[t][ks][1]);
          }
        }
        // ---- mask, online softmax (base 2), P^T fragments
        const int tA = mt * 16 + (lane >> 2), tB = tA + 8;
        const bool okA = tA < nv && bid[tA / BS] >= 0;
        const bool okB = tB < nv && bid[tB / BS] >= 0;
        uint32_t pb[NT][2];
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          float pv[4];
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const float xa = okA ? sc[t][j] * a.scale_log2 : -INFINITY;
            const float xb = okB ? sc[t][j + 2] * a.scale_log2 : -INFINITY;
            const float mx = warp_max_xor4(fmaxf(xa, xb));
            const float m_new = fmaxf(mrun[t][j], mx);
            const float base = m_new == -INFINITY ? 0.f : m_new;
            const float alpha = fast_exp2(mrun[t][j] - base);
            pv[j] = fast_exp2(xa - base);
            pv[j + 2] = fast_exp2(xb - base);
            lrun[t][j] = lrun[t][j] * alpha + pv[j] + pv[j + 2];
            mrun[t][j] = m_new;
#pragma unroll
            for (int dt = 0; dt < KS; ++dt) {
              acc[t][dt][j] *= alpha;
              acc[t][dt][j + 2] *= alpha;
            }
          }
          pb[t][0] = movmatrix_trans(pack_bf16x2(pv[0], pv[1]));
          pb[t][1] = movmatrix_trans(pack_bf16x2(pv[2], pv[3]));
        }
        // ---- O^T += V^T P^T
        {
          const int mi = lane >> 3;
          const int r = mt * 16 + (lane & 7) + (mi >> 1) * 8;
#pragma unroll
          for (int dt = 0; dt < KS; ++dt) {
            const int h = dt >> 2;
            const int c = ((dt & 3) << 1) + (mi & 1);
            const uint32_t addr = vb + h * C::TILE + r * 128 + ((c ^ (r & 7)) << 4);
            uint32_t a0, a1, a2, a3;
            ldsm_x4_trans(addr, a0, a1, a2, a3);
#pragma unroll
            for (int t = 0; t < NT; ++t)
              mma_bf16_16816(acc[t][dt], a0, a1, a2, a3, pb[t][0], pb[t][1]);
          }
        }
      }
      __syncwarp();
      if (k + STAGES < n_w) issue(k + STAGES);
    }
    used += n_w;

#pragma unroll
    for (int t = 0; t < NT; ++t) {
      lrun[t][0] = warp_sum_xor4(lrun[t][0]);
      lrun[t][1] = warp_sum_xor4(lrun[t][1]);
    }

    __syncthreads();  // every warp is done with its stages; the buffers are free
    if (misc[2]) break;

    // ---- cross-warp merge through shared memory
    float* macc = reinterpret_cast<float*>(smem);
    float* mm = macc + kWarps * C::HEADS * C::MSTRIDE;
    float* ml = mm + kWarps * C::HEADS;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
#pragma unroll
      for (int dt = 0; dt < KS; ++dt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int n = t * 8 + 2 * (lane & 3) + (i & 1);
          const int d = dt * 16 + (lane >> 2) + 8 * (i >> 1);
          macc[(warp * C::HEADS + n) * C::MSTRIDE + d] = acc[t][dt][i];
        }
      if (lane < 4) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          mm[warp * C::HEADS + t * 8 + 2 * lane + j] = mrun[t][j];
          ml[warp * C::HEADS + t * 8 + 2 * lane + j] = lrun[t][j];
        }
      }
    }
    __syncthreads();

    const int G = a.group;
    const int64_t row0 = (int64_t)s * a.n_q + (int64_t)g * G;
    for (int i = tid; i < G * D; i += kThreads) {
      const int n = i / D, d = i - n * D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mm[w * C::HEADS + n]);
      float L = 0.f, O = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float mw = mm[w * C::HEADS + n];
        const float e = mw == -INFINITY ? 0.f : fast_exp2(mw - M);
        L += e * ml[w * C::HEADS + n];
        O += e * macc[(w * C::HEADS + n) * C::MSTRIDE + d];
      }
      if (nparts == 1) {
        a.out[(row0 + n) * D + d] = __float2bfloat16_rn(L > 0.f ? O / L : 0.f);
      } else {
        const int64_t wr = (row0 + n) * a.max_parts + p;
        a.ws_o[wr * D + d] = O;
        if (d == 0) a.ws_ml[wr] = make_float2(M, L);
      }
    }

    if (nparts > 1) {
      __threadfence();
      __syncthreads();
      if (tid == 0) {
        int32_t* tk = &a.tickets[(int64_t)s * a.n_kv + g];
        const int done = atomicAdd(tk, 1);
        const int last = done == nparts - 1;
        if (last) atomicExch(tk, 0);  // every partition has checked in: reset
        misc[1] = last;
      }
      __syncthreads();
      if (misc[1]) {
        __threadfence();
        // log-sum-exp weights per head and partition: w_p = 2^(m_p - M) / L
        float* wts = reinterpret_cast<float*>(smem);
        for (int n = warp; n < G; n += kWarps) {
          const float2* mlp = a.ws_ml + (row0 + n) * a.max_parts;
          float M = -INFINITY;
          for (int q = lane; q < nparts; q += 32) M = fmaxf(M, __ldcg(&mlp[q]).x);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
          float L = 0.f;
          for (int q = lane; q < nparts; q += 32) {
            const float2 v = __ldcg(&mlp[q]);
            L += v.x == -INFINITY ? 0.f : fast_exp2(v.x - M) * v.y;
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
          const float inv = L > 0.f ? 1.f / L : 0.f;
          for (int q = lane; q < nparts; q += 32) {
            const float mq = __ldcg(&mlp[q]).x;
            wts[n * a.max_parts + q] = mq == -INFINITY ? 0.f : fast_exp2(mq - M) * inv;
          }
        }
        __syncthreads();
        for (int i = tid; i < G * D; i += kThreads) {
          const int n = i / D, d = i - n * D;
          const float* op = a.ws_o + (row0 + n) * a.max_parts * D + d;
          const float* wn = wts + n * a.max_parts;
          float O0 = 0.f, O1 = 0.f;
          int q = 0;
          for (; q + 1 < nparts; q += 2) {
            O0 += wn[q] * __ldcg(op + (int64_t)q * D);
            O1 += wn[q + 1] * __ldcg(op + (int64_t)(q + 1) * D);
          }
          if (q < nparts) O0 += wn[q] * __ldcg(op + (int64_t)q * D);
          a.out[(row0 + n) * D + d] = __float2bfloat16_rn(O0 + O1);
        }
      }
    }

    fence_proxy_async_smem();  // generic writes above precede the next TMA loads
    if (tid == 0) misc[0] = next;
    __syncthreads();
    item = misc[0];
  }

  // After a timeout, let this warp's copies still in flight land (bounded)
  // before the CTA exits.
  for (uint32_t i = drain_from; i < drain_to; ++i)
    mbar_wait_bounded(warp_bar + 8 * (i % STAGES), (i / STAGES) & 1u, 100000000ull);
  if (tid == 0) {
    const int fin = atomicAdd(&a.work[1], 1);
    if (fin == (int)gridDim.x - 1) {  // the last CTA resets the shared counters
      atomicExch(&a.work[0], 0);
      atomicExch(&a.work[1], 0);
    }
  }
}

// ------------------------------------------------------------------ host

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// The pool as a 2-D bf16 tensor [num_blocks * n_kv * bs rows][D columns];
// one box is 64 columns (128 bytes, the swizzle span) by block_size rows.
static pa_status make_pool_map(CUtensorMap* map, const void* pool, int D, int64_t rows, int bs) {
  auto fn = encode_fn();
  if (!fn) return cuda_fail_msg("pa_decode", "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)bs};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(pool), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail_msg("pa_decode", "cuTensorMapEncodeTiled failed");
  return PA_OK;
}

template <int D, int BS, int NT>
static pa_status launch(const DecodeArgs& a, const void* k_pool, const void* v_pool,
                        int64_t items_upper, cudaStream_t stream) {
  using C = Cfg<D, BS, NT>;
  auto kern = decode_kernel<D, BS, NT>;
  const int64_t rows = (int64_t)a.num_blocks * a.n_kv * BS;
  CUtensorMap tmk, tmv;
  pa_status st = make_pool_map(&tmk, k_pool, D, rows, BS);
  if (st != PA_OK) return st;
  st = make_pool_map(&tmv, v_pool, D, rows, BS);
  if (st != PA_OK) return st;

  const size_t smem = C::smem_bytes(a.num_seqs);
  static int configured = 0;  // largest dynamic smem size already allowed
  static int occ_for_smem[2] = {-1, 0};
  if ((int)smem > configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return cuda_fail("pa_decode smem attribute", e);
    configured = (int)smem;
  }
  int occ = 0;
  if (occ_for_smem[0] == (int)smem) {
    occ = occ_for_smem[1];
  } else {
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, smem);
    if (e != cudaSuccess) return cuda_fail("pa_decode occupancy", e);
    if (occ < 1) return cuda_fail_msg("pa_decode", "kernel does not fit on an SM");
    occ_for_smem[0] = (int)smem;
    occ_for_smem[1] = occ;
  }
  int64_t grid = (int64_t)num_sms() * occ;
  if (grid > items_upper) grid = items_upper;
  if (grid < 1) grid = 1;
  kern<<<(unsigned)grid, kThreads, smem, stream>>>(tmk, tmv, a);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? PA_OK : cuda_fail("pa_decode launch", e);
}

template <int D, int BS>
static pa_status dispatch_nt(const DecodeArgs& a, const void* kp, const void* vp, int64_t ub,
                             cudaStream_t st) {
  if (a.group <= 8) return launch<D, BS, 1>(a, kp, vp, ub, st);
  return launch<D, BS, 2>(a, kp, vp, ub, st);
}

template <int D>
static pa_status dispatch_bs(int bs, const DecodeArgs& a, const void* kp, const void* vp,
                             int64_t ub, cudaStream_t st) {
  switch (bs) {
    case 8: return dispatch_nt<D, 8>(a, kp, vp, ub, st);
    case 16: return dispatch_nt<D, 16>(a, kp, vp, ub, st);
    default: return dispatch_nt<D, 32>(a, kp, vp, ub, st);
  }
}

static int stage_tokens(int block_size) { return block_size < 16 ? 16 : block_size; }

// Partition size: explicit, or the largest of 512/256/128/64 tokens that
// still gives the persistent grid (about 2 CTAs on each of ~150 SMs) several
// items each, estimating the mean length as half the maximum.
static int resolve_partition(int num_seqs, int n_kv, int block_size, int max_seq_len,
                             int partition_tokens) {
  const int st = stage_tokens(block_size);
  if (partition_tokens != 0) {
    if (partition_tokens < st || partition_tokens % st != 0 || partition_tokens > 128 * st)
      return -1;
    return partition_tokens;
  }
  const int64_t slots = 2 * 152;
  const int64_t half = max_seq_len > 1 ? (max_seq_len + 1) / 2 : 1;
  int P = 512;
  while (P > 64) {
    const int64_t items = (int64_t)num_seqs * n_kv * ((half + P - 1) / P);
    if (items >= 4 * slots) break;
    P >>= 1;
  }
  if (P < st) P = st;
  return P;
}

struct WsLayout {
  size_t o_off, ml_off, tick_off, work_off, total;
  int max_parts;
};

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

static bool layout(int num_seqs, int n_q, int n_kv, int D, int P, int max_seq_len, WsLayout* w) {
  const int64_t mp = max_seq_len <= 0 ? 1 : ((int64_t)max_seq_len + P - 1) / P;
  if (mp > kMaxParts) return false;
  w->max_parts = (int)mp;
  const size_t rows = (size_t)num_seqs * n_q * mp;
  w->o_off = 0;
  w->ml_off = align256(rows * D * sizeof(float));
  w->tick_off = w->ml_off + align256(rows * sizeof(float2));
  w->work_off = w->tick_off + align256((size_t)num_seqs * n_kv * sizeof(int32_t));
  w->total = w->work_off + 256;
  return true;
}

static bool supported(int head_dim, int block_size, int n_q, int n_kv) {
  return (head_dim == 64 || head_dim == 128) &&
         (block_size == 8 || block_size == 16 || block_size == 32) && n_q / n_kv <= 16;
}

}  // namespace pa

using namespace pa;

extern "C" int pa_decode_partition_tokens(int num_seqs, int n_kv_heads, int block_size,
                                          int max_seq_len, int partition_tokens) {
  if (num_seqs < 0 || n_kv_heads <= 0 || max_seq_len < 0) return -1;
  if (block_size != 8 && block_size != 16 && block_size != 32) return -1;
  return resolve_partition(num_seqs, n_kv_heads, block_size, max_seq_len, partition_tokens);
}

extern "C" size_t pa_decode_workspace_bytes(int num_seqs, int n_q_heads, int n_kv_heads,
                                            int head_dim, int block_size, int max_seq_len,
                                            int partition_tokens) {
  if (num_seqs < 0 || n_q_heads <= 0 || n_kv_heads <= 0 || n_q_heads % n_kv_heads) return 0;
  if (!supported(head_dim, block_size, n_q_heads, n_kv_heads)) return 0;
  const int P =
      resolve_partition(num_seqs, n_kv_heads, block_size, max_seq_len, partition_tokens);
  if (P <= 0) return 0;
  WsLayout w;
  if (!layout(num_seqs, n_q_heads, n_kv_heads, head_dim, P, max_seq_len, &w)) return 0;
  return w.total;
}

extern "C" pa_status pa_decode(void* out, const void* q, const void* k_pool, const void* v_pool,
                               const int32_t* block_tables, const int32_t* seq_lens,
                               int num_seqs, int max_blocks_per_seq, int num_blocks,
                               int n_q_heads, int n_kv_heads, int head_dim, int block_size,
                               float scale, int partition_tokens, int max_seq_len,
                               void* workspace, size_t workspace_bytes, int32_t* err_word,
                               pa_stream_t stream) {
  if (num_seqs < 0 || num_seqs > kMaxSeqs || max_blocks_per_seq < 1 || num_blocks < 1 ||
      n_q_heads < 1 || n_kv_heads < 1 || max_seq_len < 0)
    return PA_ERR_INVALID_ARG;
  if (n_q_heads % n_kv_heads != 0) return PA_ERR_INVALID_ARG;
  if (!supported(head_dim, block_size, n_q_heads, n_kv_heads)) return PA_ERR_UNSUPPORTED;
  if ((int64_t)num_blocks * n_kv_heads * block_size >= (int64_t)1 << 31)
    return PA_ERR_INVALID_ARG;
  if ((int64_t)max_seq_len > (int64_t)max_blocks_per_seq * block_size) return PA_ERR_INVALID_ARG;
  const int P = resolve_partition(num_seqs, n_kv_heads, block_size, max_seq_len,
                                  partition_tokens);
  if (P <= 0) return PA_ERR_UNSUPPORTED;
  WsLayout w;
  if (!layout(num_seqs, n_q_heads, n_kv_heads, head_dim, P, max_seq_len, &w))
    return PA_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PA_OK;
  if (!out || !q || !k_pool || !v_pool || !block_tables || !seq_lens || !workspace)
    return PA_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return PA_ERR_INVALID_ARG;
  if (workspace_bytes < w.total) return PA_ERR_INVALID_ARG;

  DecodeArgs a;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.block_tables = block_tables;
  a.seq_lens = seq_lens;
  a.ws_o = reinterpret_cast<float*>(ws + w.o_off);
  a.ws_ml = reinterpret_cast<float2*>(ws + w.ml_off);
  a.tickets = reinterpret_cast<int32_t*>(ws + w.tick_off);
  a.work = reinterpret_cast<int32_t*>(ws + w.work_off);
  a.err = err_word;
  a.num_seqs = num_seqs;
  a.max_blocks = max_blocks_per_seq;
  a.num_blocks = num_blocks;
  a.n_q = n_q_heads;
  a.n_kv = n_kv_heads;
  a.group = n_q_heads / n_kv_heads;
  a.part_tokens = P;
  a.max_parts = w.max_parts;
  a.len_cap = max_seq_len;
  a.scale_log2 = scale * kLog2e;
  const int64_t items_upper = (int64_t)num_seqs * n_kv_heads * w.max_parts;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (head_dim == 64) return dispatch_bs<64>(block_size, a, k_pool, v_pool, items_upper, st);
  return dispatch_bs<128>(block_size, a, k_pool, v_pool, items_upper, st);
}

// ------------------------------------------------------------------ no-alloc

namespace pa {

// Scratch of pa_decode_noalloc: a fixed array in device memory that exists on
// every GPU that loads this library, from module load until the process
// exits. Host code must not use its name as an address; the device address is
// looked up once per device below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch on the current device (looked up on the
// first call per device, with that device current). nullptr on failure.
static void* noalloc_scratch(pa_status* st) {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    *st = cuda_fail("pa_decode_noalloc cudaGetDevice", e);
    return nullptr;
  }
  if (dev < 0 || dev >= 64) {
    *st = cuda_fail_msg("pa_decode_noalloc", "device index above 63");
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      *st = cuda_fail("pa_decode_noalloc cudaGetSymbolAddress", e);
      return nullptr;
    }
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace pa

extern "C" pa_status pa_decode_noalloc(void* out, const void* q, const void* k_pool,
                                       const void* v_pool, const int32_t* block_tables,
                                       const int32_t* seq_lens, int num_seqs,
                                       int max_blocks_per_seq, int num_blocks, int n_q_heads,
                                       int n_kv_heads, int head_dim, int block_size,
                                       float scale, int partition_tokens, int max_seq_len,
                                       int32_t* err_word, pa_stream_t stream) {
  const size_t need = pa_decode_workspace_bytes(num_seqs, n_q_heads, n_kv_heads, head_dim,
                                                block_size, max_seq_len, partition_tokens);
  if (need == 0 || num_seqs <= 0) {
    // Unsupported arguments or nothing to do: pa_decode returns the status
    // before it touches any memory.
    return pa_decode(out, q, k_pool, v_pool, block_tables, seq_lens, num_seqs,
                     max_blocks_per_seq, num_blocks, n_q_heads, n_kv_heads, head_dim,
                     block_size, scale, partition_tokens, max_seq_len, nullptr, 0, err_word,
                     stream);
  }
  if (need > (size_t)PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_INVALID_ARG;
  pa_status st = PA_OK;
  void* scratch = noalloc_scratch(&st);
  if (scratch == nullptr) return st;
  // The tickets and work counters must start at zero. A completed call
  // leaves them zeroed, but the array is shared by every call in the
  // process, so clear them here rather than trust the previous caller.
  const int P = resolve_partition(num_seqs, n_kv_heads, block_size, max_seq_len,
                                  partition_tokens);
  WsLayout w;
  if (P <= 0 || !layout(num_seqs, n_q_heads, n_kv_heads, head_dim, P, max_seq_len, &w))
    return PA_ERR_UNSUPPORTED;
  cudaError_t e = cudaMemsetAsync(static_cast<uint8_t*>(scratch) + w.tick_off, 0,
                                  w.total - w.tick_off, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail("pa_decode_noalloc memset", e);
  return pa_decode(out, q, k_pool, v_pool, block_tables, seq_lens, num_seqs,
                   max_blocks_per_seq, num_blocks, n_q_heads, n_kv_heads, head_dim, block_size,
                   scale, partition_tokens, max_seq_len, scratch, PA_NOALLOC_SCRATCH_BYTES,
                   err_word, stream);
}
