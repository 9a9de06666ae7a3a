// Paged chunked-prefill attention for sm_103a, on the fifth-generation tensor
// cores (tcgen05, accumulators in tensor memory).
//
// What it computes ("Serving: vLLM and PagedAttention", section 2.4, chunked
// prefill; "03 · PagedAttention", the kernel gathers K/V through the block
// table): a sequence's last c tokens (its chunk, already written to the pool)
// each attend causally to every cached position up to their own, the pool
// reached through the block table exactly as in decode.
//
// Design: one CTA (two warpgroups) per (query tile, sequence, kv head). The
// tile is 256 rows of (token, query head) pairs of the G query heads sharing
// the kv head (256 / G tokens), so every K/V tile in shared memory serves all
// G heads twice over; each warpgroup owns 128 rows (one MMA M), and row r of
// a warpgroup's accumulators is TMEM lane r, owned by its thread r: the
// softmax of a row runs in one thread with no shuffles.
//  * Q (2 x 128 x head_dim, bf16) is staged once in shared memory in the
//    128-byte-swizzled K-major layout the MMA reads.
//  * K/V stream in tiles of 64 tokens (four 16-token units, the decode's TMA
//    boxes, each 64-column half of a row stored as its own 64-row slab)
//    through 4-stage rings (K and V separately) filled by TMA.
//  * Per tile: S = Q K^T (M 128, N 64, both operands K-major) into TMEM;
//    every thread loads its row of S, masks it (causal, length, bad blocks),
//    runs the online softmax in base 2 with a lazily moved reference
//    (rescaling its row of O in TMEM in the rare case the reference moves),
//    and writes P to TMEM as a bf16 pair hi + lo; then O += P_hi V + P_lo V
//    (M 128, N head_dim, A = P from TMEM, V read MN-major) accumulates in
//    TMEM. S and P have TMEM buffers of their own: S of the next tile is
//    computed as soon as the threads have loaded this one, and P V of the
//    previous tile runs while they compute this softmax.
//  * O is normalised and written as bf16 after the last tile.
// Blocks take the tiles longest first (longest_first_tile): the hardware
// starts blocks in index order, so a list schedule that begins with the
// costliest tiles ends near the average load per SM.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <cstring>
#include <mutex>

#include "pa_internal.h"
#include "pa_ptx.cuh"
#include "pa_tc.cuh"

namespace pa {
namespace {

constexpr int kTWarpgroups = 2;             // each owns 128 rows (one MMA M)
constexpr int kTThreads = 128 * kTWarpgroups;  // softmax threads, one per row
// then three single-lane roles, each on its own warp scheduler: the MMA
// issuer of warpgroup 0, the TMA copies, the MMA issuer of warpgroup 1
constexpr int kTIssue0Warp = kTThreads / 32;
constexpr int kTLoadWarp = kTIssue0Warp + 1;
constexpr int kTIssue1Warp = kTIssue0Warp + 2;
constexpr int kTCtaThreads = kTThreads + 96;
constexpr int kTRows = 128;                 // M of every MMA: rows per warpgroup
constexpr int kTTileRows = kTRows * kTWarpgroups;  // (token, head) rows per CTA
constexpr int kTKv = 64;                    // K/V tokens per tile (N of S)
constexpr int kTUnit = 16;                  // tokens per TMA unit
constexpr int kTStages = 4;
// TMEM columns of warpgroup w: O at 256 w (head_dim fp32 columns), S at
// 256 w + 128 (64 fp32), P at 256 w + 192 (hi then lo: 32 + 32 bf16 pairs)
constexpr uint32_t kTmemCols = 512;
__host__ __device__ constexpr uint32_t tmem_o_col(int w) { return 256 * w; }
__host__ __device__ constexpr uint32_t tmem_s_col(int w) { return 256 * w + 128; }
__host__ __device__ constexpr uint32_t tmem_p_col(int w) { return 256 * w + 192; }
constexpr uint64_t kTWaitNs = 2000000000ull;      // 2 s: a wait that long is a fault
constexpr uint64_t kTWaitAfterFaultNs = 1000000ull;
constexpr float kTLazyLog2 = 8.f;
constexpr float kTLog2e = 1.4426950408889634f;
constexpr int kTRankSeqs = 256;  // longest-first order for batches up to this many sequences

struct PrefillArgs {
  __nv_bfloat16* out;
  const __nv_bfloat16* q;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const int32_t* cu_q;
  int32_t* err;
  int num_seqs, total_q, max_blocks, num_blocks, n_q, n_kv, group;
  int q_tma;        // 1: the copy warp loads Q by TMA (G a power of two), else the softmax warps
  int tile_tokens;  // query tokens per tile: 256 / G, rounded down
  int rank_tiles;   // 1: blocks take the tiles longest first (longest_first_tile)
  int n_tiles;      // grid.x: tiles of the longest chunk
  int max_q_len;    // host bound of the chunk lengths
  float scale_log2;
};

template <int D, int BS>
struct TCfg {
  static constexpr int ROWS = BS < kTUnit ? BS : kTUnit;  // rows per TMA box
  static constexpr int NB = kTKv / ROWS;                  // boxes (blocks) per tile
  static constexpr int KH = D / 64;                       // 64-column halves
  static constexpr int HALF = kTKv * 128;                 // one half of K (or V): 8 KB
  static constexpr int KV_BYTES = KH * HALF;
  static constexpr int QHALF = kTRows * 128;              // 16 KB
  static constexpr int QWG = KH * QHALF;                  // one warpgroup's Q
  static constexpr int Q_OFF = 0;
  // K stages [kTStages][KV_BYTES], then V stages: K of a tile is freed by its
  // S, well before its V is freed by its P V, so each streams on its own ring
  static constexpr int K_OFF = Q_OFF + kTWarpgroups * QWG;
  static constexpr int V_OFF = K_OFF + kTStages * KV_BYTES;
  // fullK, fullV, emptyK, emptyV (one per stage); per warpgroup: S full,
  // S free, P full, P V done; the one-time start signal of warpgroup 1; per
  // warpgroup, Q stored
  static constexpr int BAR_OFF = V_OFF + kTStages * KV_BYTES;
  static constexpr int NBARS = 4 * kTStages + 4 * kTWarpgroups + 1 + kTWarpgroups;
  static constexpr int TMEM_OFF = BAR_OFF + NBARS * 8;
  static constexpr int FAULT_OFF = TMEM_OFF + 8;  // fault flag, warpgroup 0's finished tiles
  static constexpr int SEL_OFF = FAULT_OFF + 8;  // the block's tile: s, qt, g, cq0, c, L
  static constexpr int ROWS_OFF = SEL_OFF + 24;  // its first output row
  static constexpr size_t SMEM = 1024 + ROWS_OFF + 16;
};

// Byte offset of bf16 element (r, c) of a [rows][64] half-tile with the
// 128-byte swizzle (8-row atoms of 1024 bytes; 16-byte chunks XOR row % 8).
__device__ __forceinline__ uint32_t swz128(int r, int c) {
  return r * 128 + ((((c >> 3) ^ r) & 7) << 4) + (c & 7) * 2;
}

// A tile is (sequence s, query tile qt, kv head g); its cost is the number of
// 64-token K/V tiles it streams, plus one. The tile's last query position is
// base_s + min((qt + 1) TQ, c_s) with base_s = L_s - c_s - 1, so the cost
// never falls as qt grows, and cost >= T (T >= 2) holds exactly when
// min((qt + 1) TQ, c_s) >= 64 (T - 2) - base_s. Returns the first such qt
// below Q (the sequence's tile count), or Q.
__device__ __forceinline__ int first_tile_at_least(int T, int c, int base, int Q, int TQ) {
  if (T <= 1) return 0;
  const long long R = (long long)kTKv * (T - 2) - base;
  if (R > c) return Q;
  if (R <= TQ) return 0;
  const int q = (int)(R - 1) / TQ;  // ceil(R / TQ) - 1, with TQ < R <= c
  return q < Q ? q : Q;
}

struct TileSel {
  int s, qt, g;  // s < 0: no tile for this block
  int cq0, c, L;  // its sequence's cu_q entry, chunk length, seq_lens entry (cq0 -1: not read)
};

// The tile of block `rank` in longest-first order. The kv heads of a
// (sequence, query tile) pair cost the same, so the order is that of the
// pairs, costliest first with ties in (s, qt) order, each pair repeated for
// g = 0 .. n_kv - 1: block `rank` takes pair rank / n_kv, head rank % n_kv.
// One warp; lane l holds sequences l, l + 32, ... (at most kTRankSeqs, and
// the host keeps the pair count below 2^31). A search over the cost finds
// the pair's cost class: up to 32 sequences, each lane tries its own cost
// and sums over every sequence (a 32-way split per round); beyond, a binary
// search with one warp reduction per step. Then a scan over the sequences
// finds the pair.
__device__ TileSel longest_first_tile(const PrefillArgs& a, int cap, long long rank, int lane) {
  constexpr int J = kTRankSeqs / 32;
  const int TQ = a.tile_tokens, S = a.num_seqs;
  int cc[J], qq[J], bb[J];
  int c00 = 0, l00 = 0;  // cu_q and seq_lens of sequence `lane`
  int pairs = 0, tmax = 0;
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int s = lane + 32 * j;
    cc[j] = 0;
    qq[j] = 0;
    bb[j] = 0;
    if (s < S) {
      const int q0 = __ldg(&a.cu_q[s]), lr = __ldg(&a.seq_lens[s]);
      if (j == 0) {
        c00 = q0;
        l00 = lr;
      }
      const int c = __ldg(&a.cu_q[s + 1]) - q0;
      // L outside [0, cap] costs as its clamp does: nothing is visible
      // below 0, and the kernel clamps above cap
      const int L = min(max(lr, 0), cap);
      const int Q = c <= 0 ? 0 : min((c - 1) / TQ + 1, a.n_tiles);
      cc[j] = c;
      qq[j] = Q;
      bb[j] = L - c - 1;
      if (Q > 0) {
        const long long pm = (long long)bb[j] + min((long long)Q * TQ, (long long)c);
        tmax = max(tmax, (int)(1 + (pm < 0 ? 0 : pm / kTKv + 1)));
        pairs += Q;
      }
    }
  }
  pairs = __reduce_add_sync(0xffffffffu, pairs);
  tmax = __reduce_max_sync(0xffffffffu, tmax);
  if (rank >= (long long)pairs * a.n_kv) return {-1, 0, 0, 0, 0, 0};
  const int pr = (int)(rank / a.n_kv), g = (int)(rank % a.n_kv);
  auto count_at_least = [&](int T) {  // pairs of cost >= T
    int n = 0;
#pragma unroll
    for (int j = 0; j < J; ++j)
      if (32 * j < S && qq[j] > 0) n += qq[j] - first_tile_at_least(T, cc[j], bb[j], qq[j], TQ);
    return (int)__reduce_add_sync(0xffffffffu, n);
  };
  int lo = 1, hi = tmax + 1;  // count_at_least(lo) > pr >= count_at_least(hi)
  if (S <= 32) {
#pragma unroll 1
    while (hi - lo > 1) {
      const int step = (hi - lo + 31) >> 5;
      const int T = lo + lane * step;
      int n = 0;
#pragma unroll 1
      for (int q = 0; q < S; ++q) {  // sequence q, from lane q
        const int cq = __shfl_sync(0xffffffffu, cc[0], q);
        const int nq = __shfl_sync(0xffffffffu, qq[0], q);
        const int bq = __shfl_sync(0xffffffffu, bb[0], q);
        if (nq > 0) n += nq - first_tile_at_least(T, cq, bq, nq, TQ);
      }
      // lanes below the first count <= pr: lane 0 (T = lo) always counts > pr
      const unsigned more = __ballot_sync(0xffffffffu, T < hi && n > pr);
      lo += (31 - __clz(more)) * step;
      hi = min(hi, lo + step);
    }
  } else {
#pragma unroll 1
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (count_at_least(mid) > pr) lo = mid;
      else hi = mid;
    }
  }
  int r = pr - count_at_least(lo + 1);  // the rank among the pairs of cost lo
#pragma unroll
  for (int j = 0; j < J; ++j) {
    if (32 * j >= S) break;
    int f0 = 0, n = 0;
    if (qq[j] > 0) {
      f0 = first_tile_at_least(lo, cc[j], bb[j], qq[j], TQ);
      n = first_tile_at_least(lo + 1, cc[j], bb[j], qq[j], TQ) - f0;
    }
    int inc = n;  // inclusive scan over the lanes, in sequence order
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += v;
    }
    const int here = __shfl_sync(0xffffffffu, inc, 31);
    if (r < here) {
      const int src = __ffs(__ballot_sync(0xffffffffu, r < inc)) - 1;
      const int before = __shfl_sync(0xffffffffu, inc - n, src);
      const int q0 = __shfl_sync(0xffffffffu, f0, src);
      const int cq = __shfl_sync(0xffffffffu, c00, src), lq = __shfl_sync(0xffffffffu, l00, src);
      const int cl = __shfl_sync(0xffffffffu, cc[0], src);
      // the sequence's cu_q and seq_lens entries when lane src holds them
      // (sequences below 32), else cq0 = -1: the caller reads them
      return {src + 32 * j, q0 + (r - before), g, j == 0 ? cq : -1, cl, lq};
    }
    r -= here;
  }
  return {-1, 0, 0, 0, 0, 0};  // not reached: the ranks below the total cover every pair
}

// Roles: eight softmax warps (one row per thread); lane 0 of one warp issues
// the MMAs of warpgroup 0, of another those of warpgroup 1, of a third the
// TMA copies (one warp scheduler each). Each warpgroup runs its own pipeline:
// the softmax of tile kt loads S(kt) and frees its buffer, so S(kt + 1) runs
// on the tensor cores while the threads compute; P(kt) is stored once
// P V(kt - 1) has read the P buffer. The warpgroups share only the K/V
// stages. The roles meet only at mbarriers, each arranged so that no waiter
// can fall two phases behind:
//   fullK/fullV[st]   copies landed             (loader -> both issuers)
//   emptyK/emptyV[st] S / P V of the tile done  (2 MMA commits -> loader)
// and, per warpgroup w,
//   s_full[w]         S_w(kt) in TMEM           (S commit -> softmax w)
//   s_free[w]         S_w(kt) loaded            (128 arrivals -> issuer w)
//   p_full[w]         P_w(kt) in TMEM           (128 arrivals -> issuer w)
//   pv_done[w]        P V_w(kt) done            (P V commit -> softmax w)
// S(kt + 1) is issued after s_free(kt), which follows s_full(kt); P V(kt)
// after p_full(kt), and P(kt + 1) is stored after pv_done(kt): each barrier
// completes a phase only after its waiter has seen the one before.
template <int D, int BS>
__global__ void __launch_bounds__(kTCtaThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv,
                  const __grid_constant__ CUtensorMap tmq, const PrefillArgs a) {
  using C = TCfg<D, BS>;
  constexpr int NB = C::NB;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  volatile int* fault = reinterpret_cast<int*>(smem + C::FAULT_OFF);
  const volatile uint32_t* tmem_slot =
      reinterpret_cast<const volatile uint32_t*>(smem + C::TMEM_OFF);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool softmax = warp < kTIssue0Warp;
  const int wg = (tid >> 7) & 1, lr = tid & 127;  // warpgroup; row within it = TMEM lane
  const uint32_t fullK = sbase + C::BAR_OFF, fullV = fullK + 8 * kTStages;
  const uint32_t emptyK = fullV + 8 * kTStages, emptyV = emptyK + 8 * kTStages;
  // per warpgroup w, 8 bytes each: s_full, s_free, p_full, pv_done at
  // s_full0 + 32 w + 0, 8, 16, 24
  const uint32_t s_full0 = emptyV + 8 * kTStages;
  const uint32_t go1 = s_full0 + 32 * kTWarpgroups;
  const uint32_t q_full0 = go1 + 8;  // per warpgroup: its Q rows stored

  griddep_wait();  // the chunk's K/V come from the preceding cache write

  // ---- this block's tile: longest first; past kTRankSeqs sequences (or
  // 2^31 (sequence, query tile) pairs) the grid's own order, a sequence's
  // latest tiles first
  const int cap = a.max_blocks * BS;
  int s, qt, g, cq0, c, L;
  if (a.rank_tiles) {
    int* sel = reinterpret_cast<int*>(smem + C::SEL_OFF);
    const long long rank =
        blockIdx.x + (long long)gridDim.x * (blockIdx.y + (long long)gridDim.y * blockIdx.z);
    // Up to 32 sequences and one (sequence, query tile) pair per thread, the
    // whole block ranks: thread p takes pair p (pairs in (s, qt) order) and
    // counts the pairs that go before it, costlier or as costly and earlier;
    // the one with as many as rank / n_kv before it is the block's. Else
    // warp 0 searches (longest_first_tile). Scratch in the Q region, which
    // is loaded only after this.
    int* scr = reinterpret_cast<int*>(smem + C::Q_OFF);
    int *qpre = scr, *sc = scr + 40, *sb = scr + 72, *sc0 = scr + 104, *slr = scr + 136;
    int *cost = scr + 168, *npairs = cost + kTCtaThreads;
    if (warp == 0) {
      if (a.num_seqs <= 32) {
        int Q = 0;
        if (lane < a.num_seqs) {
          const int q0 = __ldg(&a.cu_q[lane]), lraw = __ldg(&a.seq_lens[lane]);
          const int cl = __ldg(&a.cu_q[lane + 1]) - q0;
          Q = cl <= 0 ? 0 : min((cl - 1) / a.tile_tokens + 1, a.n_tiles);
          sc[lane] = cl;
          sb[lane] = min(max(lraw, 0), cap) - cl - 1;  // costs as the clamped length does
          sc0[lane] = q0;
          slr[lane] = lraw;
        }
        int inc = Q;  // inclusive scan: pairs of sequences 0 .. lane
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, inc, o);
          if (lane >= o) inc += v;
        }
        qpre[lane + 1] = inc;
        if (lane == 0) qpre[0] = 0;
        if (lane == 31) *npairs = inc;
      } else if (lane == 0) {
        *npairs = -1;
      }
    }
    __syncthreads();
    const int pairs = *npairs;
    if (pairs >= 0 && pairs <= kTCtaThreads) {
      const int pr = (int)(rank / a.n_kv);
      int my_cost = 0, my_s = 0;
      if (tid < pairs) {
        while (qpre[my_s + 1] <= tid) ++my_s;
        const int t0p = (tid - qpre[my_s]) * a.tile_tokens;
        const int pm = sb[my_s] + t0p + min(a.tile_tokens, sc[my_s] - t0p);  // last position
        my_cost = pm < 0 ? 0 : pm / kTKv + 1;
        cost[tid] = my_cost;
      }
      if (tid == 0 && rank >= (long long)pairs * a.n_kv) sel[0] = -1;  // no tile left
      __syncthreads();
      if (tid < pairs) {
        int before = 0;
#pragma unroll 4
        for (int u = 0; u < pairs; ++u) {
          const int cu = cost[u];
          before += (cu > my_cost) | ((cu == my_cost) & (u < tid));
        }
        if (before == pr && rank < (long long)pairs * a.n_kv) {
          sel[0] = my_s;
          sel[1] = tid - qpre[my_s];
          sel[2] = (int)(rank % a.n_kv);
          sel[3] = sc0[my_s];
          sel[4] = sc[my_s];
          sel[5] = slr[my_s];
        }
      }
    } else if (warp == 0) {
      const TileSel t = longest_first_tile(a, cap, rank, lane);
      if (lane == 0) {
        sel[0] = t.s;
        sel[1] = t.qt;
        sel[2] = t.g;
        sel[3] = t.cq0;
        sel[4] = t.c;
        sel[5] = t.L;
      }
    }
    __syncthreads();
    s = sel[0];
    qt = sel[1];
    g = sel[2];
    cq0 = sel[3];
    c = sel[4];
    L = sel[5];
    if (s < 0) return;
    if (cq0 < 0) {
      cq0 = __ldg(&a.cu_q[s]);
      c = __ldg(&a.cu_q[s + 1]) - cq0;
      L = __ldg(&a.seq_lens[s]);
    }
  } else {
    s = blockIdx.y;
    g = blockIdx.z;
    qt = a.n_tiles - 1 - (int)blockIdx.x;
    cq0 = __ldg(&a.cu_q[s]);
    c = __ldg(&a.cu_q[s + 1]) - cq0;
    L = __ldg(&a.seq_lens[s]);
  }
  const int G = a.group, TQ = a.tile_tokens;
  const int t0 = qt * TQ;
  // a chunk longer than max_q_len breaks the contract: flagged (rows beyond
  // the grid's n_tiles * TQ stay unwritten)
  if (qt == 0 && g == 0 && tid == 0 && c > a.max_q_len) report(a.err, PA_DEV_ERR_SEQ_LEN);
  if (c <= 0 || t0 >= c) return;
  // clamped / nothing visible (rows not written if L < c) / the chunk runs
  // past the rows of q and out (those rows are neither read nor written):
  // flagged
  if (L > cap || L < c || cq0 + c > a.total_q) {
    if (tid == 0 && qt == 0 && g == 0) report(a.err, PA_DEV_ERR_SEQ_LEN);
    if (L > cap) L = cap;
  }
  const int nt = min(TQ, c - t0);  // query tokens in this tile
  const int nt_rows = max(0, min(nt, a.total_q - (cq0 + t0)));  // of them inside q and out

  const int nrows = L >= c ? nt_rows * G : 0;  // rows present: every head of these tokens
  const bool row_ok = softmax && tid < nrows;  // this thread's row is row tid
  const int pos = row_ok ? L - c + t0 + tid / G : -1;  // -1: no key visible, row not written
  const int pmax = L - c + t0 + nt - 1;  // the tile's last position
  const int n_kv = pmax < 0 ? 0 : pmax / kTKv + 1;
  const int32_t* table = a.block_tables + (int64_t)s * a.max_blocks;
  if (tid == 0)  // the first output row, kept in shared memory for the output
    *reinterpret_cast<int64_t*>(smem + C::ROWS_OFF) = (int64_t)(cq0 + t0) * a.n_q + (int64_t)g * G;

  // ---- set-up; then the copy warp starts the first K/V tiles while the
  // softmax warps load Q (q_full tells each issuer its warpgroup's Q is in)
  if (warp == 0) tc_alloc(sbase + C::TMEM_OFF, kTmemCols);
  if (tid == 0) {
    for (int i = 0; i < C::NBARS; ++i) mbar_init(fullK + 8 * i, 1);
    for (int st = 0; st < kTStages; ++st) {  // one commit from each issuer
      mbar_init(emptyK + 8 * st, kTWarpgroups);
      mbar_init(emptyV + 8 * st, kTWarpgroups);
    }
    for (int w = 0; w < kTWarpgroups; ++w) {  // every thread of warpgroup w, once per tile
      mbar_init(s_full0 + 32 * w + 8, 128);
      mbar_init(s_full0 + 32 * w + 16, 128);
      mbar_init(q_full0 + 8 * w, a.q_tma ? 1 : 128);  // and once: Q stored
    }

    *fault = 0;
    fault[1] = 0;  // softmax tiles finished by warpgroup 0 (its thread 0)
    fence_mbarrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto wait = [&](uint32_t bar, uint32_t parity) {
    if (mbar_test_wait(bar, parity)) return;
    const uint64_t limit = *fault ? kTWaitAfterFaultNs : kTWaitNs;
    if (!mbar_wait_bounded(bar, parity, limit)) {
      report(a.err, PA_DEV_ERR_TIMEOUT);
      *fault = 1;
    }
  };
  // Tile kt's pool blocks, one per TMA box, raw (checked where used), and the
  // mask of its tokens present in the pool (inside the sequence, valid block).
  auto tile_ids = [&](int kt, int (&ids)[NB]) {
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      const int tok = kt * kTKv + i * C::ROWS;
      ids[i] = tok < L ? __ldg(&table[tok / BS]) : -1;
    }
  };
  auto tile_mask = [&](int kt, const int (&ids)[NB]) {
    uint64_t mask = 0;
#pragma unroll
    for (int i = 0; i < NB; ++i)
      if (ids[i] >= 0 && ids[i] < a.num_blocks)
        mask |= ((1ull << C::ROWS) - 1) << (i * C::ROWS);
    const int nvalid = min(kTKv, L - kt * kTKv);
    if (nvalid < kTKv) mask &= (1ull << nvalid) - 1;
    return mask;
  };

  if (warp == kTLoadWarp) {
    // ---- copies: K and V of every tile through their rings. Lane j below
    // NB * KH issues box j (block j / KH, 64-column half j % KH) of each
    // tile, so one warp instruction starts a tile's copies; the block ids of
    // the next tile are loaded while this one is copied.
    constexpr int NBOX = NB * C::KH;
    static_assert(2 * NBOX <= 32, "one box per lane");
    if (lane == 0) {
      prefetch_tensormap(&tmk);
      prefetch_tensormap(&tmv);
    }
    const int bi = lane / C::KH, bh = lane % C::KH;  // this lane's box: block, half
    // Q by TMA: warpgroup w's 128 rows are the G heads of tokens t0 + w 128/G
    // .. of the tile, one box (64 columns, G heads, 128/G tokens) per
    // 64-column half; rows past total_q read as zeros. Rows past the chunk
    // but inside q are read and never written out.
    if (a.q_tma && n_kv > 0 && lane == 0) {
      prefetch_tensormap(&tmq);
      for (int w = 0; w < kTWarpgroups; ++w) {
        const uint32_t qb = q_full0 + 8 * w;
        mbar_arrive_expect_tx(qb, C::QWG);
#pragma unroll
        for (int h = 0; h < C::KH; ++h)
          tma_load_3d(sbase + C::Q_OFF + w * C::QWG + h * C::QHALF, &tmq, h * 64, g * G,
                      cq0 + t0 + w * (kTRows / G), qb);
      }
    }
    auto box_id = [&](int kt) {
      const int tok = kt * kTKv + bi * C::ROWS;
      return (lane < NBOX && tok < L) ? __ldg(&table[tok / BS]) : -1;
    };
    int id_nxt = n_kv > 0 ? box_id(0) : -1;
#pragma unroll 1
    for (int kt = 0; kt < n_kv; ++kt) {
      const int st = kt % kTStages;
      const int id = id_nxt;
      if (kt + 1 < n_kv) id_nxt = box_id(kt + 1);
      const int tok = kt * kTKv + bi * C::ROWS;
      const bool present = lane < NBOX && tok < L;
      const bool ok = present && id >= 0 && id < a.num_blocks;
      if (present && !ok && bh == 0) report(a.err, PA_DEV_ERR_BLOCK_ID);
      const uint32_t bytes = (uint32_t)__popc(__ballot_sync(0xffffffffu, ok)) * C::ROWS * 128;
      const int32_t y = (id * a.n_kv + g) * BS + (BS > kTUnit ? tok % BS : 0);
      if (kt >= kTStages) {  // the stages' previous tile is done with them
        wait(emptyK + 8 * st, ((kt - kTStages) / kTStages) & 1);
        wait(emptyV + 8 * st, ((kt - kTStages) / kTStages) & 1);
      }
      if (lane == 0) {
        if (bytes == 0) {
          mbar_arrive(fullK + 8 * st);
          mbar_arrive(fullV + 8 * st);
        } else {
          mbar_arrive_expect_tx(fullK + 8 * st, bytes);
          mbar_arrive_expect_tx(fullV + 8 * st, bytes);
        }
      }
      __syncwarp();
      // lanes 0 .. NBOX-1 copy K, lanes NBOX .. 2 NBOX-1 the same boxes of V
      {
        const int src = lane < NBOX ? lane : lane - NBOX;  // box index
        const int okb = __shfl_sync(0xffffffffu, (int)ok, src & 31);
        const int yb = __shfl_sync(0xffffffffu, y, src & 31);
        const bool isv = lane >= NBOX;
        if (lane < 2 * NBOX && okb) {
          const int b_i = src / C::KH, b_h = src % C::KH;
          const uint32_t dst = sbase + (isv ? C::V_OFF : C::K_OFF) + st * C::KV_BYTES +
                               b_h * C::HALF + b_i * C::ROWS * 128;
          tma_load_2d(dst, isv ? &tmv : &tmk, b_h * 64, yb, (isv ? fullV : fullK) + 8 * st);
        }
      }
    }
    __syncwarp();
  } else if (warp == kTIssue0Warp || warp == kTIssue1Warp) {
    // ---- the MMAs of warpgroup w, issued by one lane: S_w(0), then per
    // tile S_w(kt + 1) (once the softmax has loaded S_w(kt)) and P V_w(kt)
    // (once it has stored P_w(kt)). S_w(kt) = Q_w K(kt)^T; O_w += P_hi V +
    // P_lo V. Operand descriptors: the start address sits in the low 14 bits
    // in 16-byte units (shared addresses stay below 2^18), so an offset into a
    // tile is added to the descriptor directly; they are formed before the
    // waits, so that each MMA issues on its own.
    const int w = warp == kTIssue0Warp ? 0 : 1;
    if (lane == 0) {
      const uint64_t dq = tc_desc_sw128(sbase + C::Q_OFF + w * C::QWG, 16, 1024);
      const uint64_t dk = tc_desc_sw128(sbase + C::K_OFF, 16, 1024);
      const uint64_t dv = tc_desc_sw128(sbase + C::V_OFF, C::HALF, 1024);
      constexpr uint32_t kIdS = tc_idesc_bf16(kTRows, kTKv, 0);
      constexpr uint32_t kIdPV = tc_idesc_bf16(kTRows, D, 1);
      const uint32_t s_full = s_full0 + 32 * w, s_free = s_full + 8;
      const uint32_t p_full = s_full + 16, pv_done = s_full + 24;
      const uint32_t tS = tmem + tmem_s_col(w), tP = tmem + tmem_p_col(w);
      const uint32_t tO = tmem + tmem_o_col(w);
      uint64_t dqs[D / 16];
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        dqs[ks] = dq + (((ks >> 2) * C::QHALF + (ks & 3) * 32) >> 4);
      auto issue_s = [&](int kt) {
        const int st = kt % kTStages;
        uint64_t dks[D / 16];
        const uint64_t dk_st = dk + ((st * C::KV_BYTES) >> 4);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          dks[ks] = dk_st + (((ks >> 2) * C::HALF + (ks & 3) * 32) >> 4);
        if (kt >= 1) wait(s_free, (kt - 1) & 1);  // the softmax has loaded S_w(kt - 1)
        wait(fullK + 8 * st, (kt / kTStages) & 1);
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) tc_mma_bf16(tS, dqs[ks], dks[ks], kIdS, ks > 0);
        tc_commit(s_full);
        tc_commit(emptyK + 8 * st);
      };
      auto issue_pv = [&](int kt) {
        const int st = kt % kTStages;
        uint64_t dvs[kTKv / 16];
        const uint64_t dv_st = dv + ((st * C::KV_BYTES) >> 4);
#pragma unroll
        for (int ks = 0; ks < kTKv / 16; ++ks) dvs[ks] = dv_st + ks * 128;
        const uint32_t first = kt == 0;
        wait(p_full, kt & 1);  // P_w(kt) stored (after P V_w(kt - 1) was done)
        wait(fullV + 8 * st, (kt / kTStages) & 1);
        tc_fence_after();
#pragma unroll
        for (int part = 0; part < 2; ++part)
#pragma unroll
          for (int ks = 0; ks < kTKv / 16; ++ks)
            tc_mma_bf16_ta64(tO, tP + part * 32 + ks * 8, dvs[ks], kIdPV,
                             (part | ks) ? 1u : !first);
        tc_commit(pv_done);
        tc_commit(emptyV + 8 * st);
      };
      // Warpgroup 1 starts once S_0(0) is done, so that the two warpgroups
      // run out of phase to begin with.
      if (w == 1 && n_kv > 0) wait(go1, 0);
      if (n_kv > 0) {
        wait(q_full0 + 8 * w, 0);  // this warpgroup's Q stored (used once)
        issue_s(0);
      }
      if (w == 0 && n_kv > 0) tc_commit(go1);  // used once: one phase
#pragma unroll 1
      for (int kt = 0; kt < n_kv; ++kt) {
        if (kt + 1 < n_kv) issue_s(kt + 1);
        issue_pv(kt);
      }
    }
    __syncwarp();
  } else {
    // ---- the softmax warps: one row per thread, on warpgroup wg's barriers.
    // First, for a group size that is not a power of two (its 128 rows are not
    // whole tokens, so not one box), this warpgroup's rows of Q into shared
    // memory (K-major, swizzled; absent rows zero): consecutive threads take
    // consecutive 16-byte pieces of a row, every load in flight before the
    // first store.
    if (!a.q_tma) {
      constexpr int CPR = D / 8;  // 16-byte pieces per row
      const int64_t orow0 = *reinterpret_cast<const int64_t*>(smem + C::ROWS_OFF);
      const float inv_g = 1.f / (float)G;  // r / G in floats: exact for r < 256, G <= 64
      uint4 v[CPR];
#pragma unroll
      for (int it = 0; it < CPR; ++it) {
        const int idx = it * kTRows + lr, r = wg * kTRows + idx / CPR, ch = idx % CPR;
        const int tr = (int)(((float)r + 0.5f) * inv_g);
        v[it] = r < nrows ? __ldg(reinterpret_cast<const uint4*>(
                                      a.q + (orow0 + (int64_t)tr * a.n_q + (r - tr * G)) * D) +
                                  ch)
                          : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int it = 0; it < CPR; ++it) {
        const int idx = it * kTRows + lr, rl = idx / CPR, ch = idx % CPR;
        *reinterpret_cast<uint4*>(smem + C::Q_OFF + wg * C::QWG + (ch >> 3) * C::QHALF +
                                  swz128(rl, (ch & 7) * 8)) = v[it];
      }
      fence_proxy_async_smem();  // generic writes before the MMAs read them
      mbar_arrive(q_full0 + 8 * wg);
    }
    const uint32_t tO = tmem + tmem_o_col(wg), tS = tmem + tmem_s_col(wg);
    const uint32_t tP = tmem + tmem_p_col(wg);
    const uint32_t s_full = s_full0 + 32 * wg, s_free = s_full + 8;
    const uint32_t p_full = s_full + 16, pv_done = s_full + 24;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    float m = -INFINITY, l = 0.f;
    int ids_nxt[NB];
    if (n_kv > 0) tile_ids(0, ids_nxt);
#pragma unroll 1
    for (int kt = 0; kt < n_kv; ++kt) {
      const int st = kt % kTStages;
      const uint64_t tmask = tile_mask(kt, ids_nxt);
      if (kt + 1 < n_kv) tile_ids(kt + 1, ids_nxt);  // in flight during this tile
      if (wg == 1) {
        // Not ahead of warpgroup 0: a softmax starts after warpgroup 0's of the
        // same tile, so the two stay apart and each one's softmax overlaps the
        // other's MMAs (in step, both wait on the tensor cores together).
        if (lane == 0) {
          const uint64_t t_start = globaltimer_ns();
          const uint64_t limit = *fault ? kTWaitAfterFaultNs : kTWaitNs;
#pragma unroll 1
          for (uint32_t it = 0; fault[1] < kt + 1; ++it)
            if (it >= (1u << 28) || globaltimer_ns() - t_start > limit) {
              report(a.err, PA_DEV_ERR_TIMEOUT);
              *fault = 1;
              break;
            }
        }
        __syncwarp();
      }
      wait(s_full, kt & 1);  // S(kt) is in TMEM
      tc_fence_after();
      // masked, lazy online softmax of this thread's row. Scores stay in raw
      // units (the scale, > 0, goes into one FFMA per weight); masked
      // positions become -inf. On tiles the row sees whole, nothing is masked.
      uint32_t sr[2][32];
      tc_ld32(tS + lane_off, sr[0]);
      tc_ld32(tS + lane_off + 32, sr[1]);
      tc_wait_ld_bind(sr[0]);
      tc_wait_ld_bind(sr[1]);
      tc_fence_before();
      mbar_arrive(s_free);  // the S buffer may take the next tile
      const int lim = min(kTKv - 1, pos - kt * kTKv);  // last position this row may see
      const uint64_t vis = lim < 0 ? 0ull : tmask & (lim >= 63 ? ~0ull : ((2ull << lim) - 1));
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // independent chains
      if (vis == ~0ull) {
#pragma unroll
        for (int j = 0; j < kTKv; ++j)
          mx4[j & 3] = fmaxf(mx4[j & 3], __uint_as_float(sr[j >> 5][j & 31]));
      } else {
#pragma unroll
        for (int j = 0; j < kTKv; ++j) {
          const float x = (vis >> j & 1) ? __uint_as_float(sr[j >> 5][j & 31]) : -INFINITY;
          sr[j >> 5][j & 31] = __float_as_uint(x);
          mx4[j & 3] = fmaxf(mx4[j & 3], x);
        }
      }
      const float rmax = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * a.scale_log2;
      const bool need = rmax > m + kTLazyLog2;
      const bool warp_need = __any_sync(0xffffffffu, need);
      float alpha = 1.f;
      if (need) {
        const float m_new = fmaxf(m, rmax);
        alpha = fast_exp2(m - (m_new == -INFINITY ? 0.f : m_new));
        m = m_new;
      }
      const float nbase = m == -INFINITY ? 0.f : -m;
      const float sl2 = a.scale_log2;
      float l4[4] = {0.f, 0.f, 0.f, 0.f};  // independent chains
      // P as a bf16 pair hi + lo (hi = bf16(p), lo = bf16(p - hi)): a lone
      // bf16 weight is off by up to 2^-9 relative, which on rows that see only
      // a few keys (the start of a prompt) is as large as the whole tolerance.
      uint32_t pk[2][32];
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const float p0 =
            fast_exp2(fmaf(__uint_as_float(sr[(2 * k) >> 5][(2 * k) & 31]), sl2, nbase));
        const float p1 =
            fast_exp2(fmaf(__uint_as_float(sr[(2 * k + 1) >> 5][(2 * k + 1) & 31]), sl2, nbase));
        l4[k & 3] += p0 + p1;
        pk[0][k] = pack_bf16x2(p0, p1);
        pk[1][k] = pack_bf16x2(p0 - __uint_as_float(pk[0][k] << 16),
                               p1 - __uint_as_float(pk[0][k] & 0xffff0000u));
      }
      l = l * alpha + ((l4[0] + l4[1]) + (l4[2] + l4[3]));
      // P(kt) goes to the P buffer once P V(kt - 1) has read it. O then holds
      // earlier tiles only: rescale this warp's rows (alpha = 1 for the
      // others) if the reference moved.
      if (kt > 0) {
        wait(pv_done, (kt - 1) & 1);
        tc_fence_after();
        if (warp_need) {
#pragma unroll
          for (int cc = 0; cc < D; cc += 32) {
            uint32_t o[32];
            tc_ld32(tO + lane_off + cc, o);
            tc_wait_ld_bind(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tc_st32(tO + lane_off + cc, o);
          }
        }
      }
      tc_st32(tP + lane_off, pk[0]);  // this thread's lane, hi then lo
      tc_st32(tP + lane_off + 32, pk[1]);
      tc_wait_st();
      if (tmask != ~0ull) {
        // V rows with no token of the sequence may hold anything (even NaN):
        // zero them so that a zero weight times them stays zero (rare: the
        // sequence's last tile or a bad block). Each warpgroup zeroes every
        // such row itself, since its P V waits only for its own threads (the
        // other warpgroup writes the same zeros).
        wait(fullV + 8 * st, (kt / kTStages) & 1);
        uint8_t* vb = smem + C::V_OFF + st * C::KV_BYTES;
        for (int i = lr; i < kTKv * C::KH * 8; i += 128) {
          const int r = i / (C::KH * 8), rest = i % (C::KH * 8), h = rest / 8, ch = rest % 8;
          if (!(tmask >> r & 1))
            *reinterpret_cast<uint4*>(vb + h * C::HALF + r * 128 + ch * 16) =
                make_uint4(0, 0, 0, 0);
        }
      }
      if (tmask != ~0ull) fence_proxy_async_smem();  // zeroed rows before the MMA reads them
      tc_fence_before();
      mbar_arrive(p_full);
      if (tid == 0) fault[1] = kt + 1;
    }

    // ---- normalise and write the rows
    if (n_kv > 0) {
      // The last P V (and with it every earlier one): the phase after the
      // one this thread saw before storing P(n - 1).
      wait(pv_done, (n_kv - 1) & 1);
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const int64_t orow = row_ok ? *reinterpret_cast<const int64_t*>(smem + C::ROWS_OFF) +
                                        (int64_t)(tid / G) * a.n_q + (tid % G)
                                  : -1;
#pragma unroll
      for (int cc = 0; cc < D; cc += 32) {
        uint32_t o[32];
        tc_ld32(tO + lane_off + cc, o);
        tc_wait_ld_bind(o);
        if (orow >= 0) {
          uint4* dst = reinterpret_cast<uint4*>(a.out + orow * D + cc);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
              w[k] = pack_bf16x2(__uint_as_float(o[v * 8 + 2 * k]) * inv,
                                 __uint_as_float(o[v * 8 + 2 * k + 1]) * inv);
            dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tc_dealloc(tmem, kTmemCols);
}

static PFN_cuTensorMapEncodeTiled_v12000 q_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult r;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &r) == cudaSuccess &&
        r == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// q [total_q][n_q][D] in boxes of one warpgroup's 128 rows: 64 columns (128
// bytes, the swizzle span), the G heads of a kv head, 128 / G tokens.
static pa_status make_q_map(CUtensorMap* map, const void* q, int D, int n_q, int total_q, int G) {
  auto fn = q_encode_fn();
  if (!fn) return cuda_fail_msg("pa_prefill", "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)n_q, (cuuint64_t)total_q};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)n_q * D * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)(kTRows / G)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : cuda_fail_msg("pa_prefill", "cuTensorMapEncodeTiled failed");
}

template <int D, int BS>
pa_status launch_prefill(PrefillArgs a, const void* k_pool, const void* v_pool,
                         cudaStream_t stream) {
  using C = TCfg<D, BS>;
  const int64_t rows = (int64_t)a.num_blocks * a.n_kv * BS;
  CUtensorMap tmk, tmv, tmq;
  int k3 = 0, v3 = 0;  // 2-D maps: each 64-column half lands in its own slab
  pa_status st = make_pool_map(&tmk, k_pool, D, 2, rows, C::ROWS, false, &k3);
  if (st != PA_OK) return st;
  st = make_pool_map(&tmv, v_pool, D, 2, rows, C::ROWS, false, &v3);
  if (st != PA_OK) return st;
  memset(&tmq, 0, sizeof(tmq));
  if (a.q_tma) {
    st = make_q_map(&tmq, a.q, D, a.n_q, a.total_q, a.group);
    if (st != PA_OK) return st;
  }
  auto kern = prefill_tc_kernel<D, BS>;
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
  cfg.blockDim = dim3(kTCtaThreads);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tmk, tmv, tmq, a);
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
                                const int32_t* cu_q, int num_seqs, int total_q,
                                int max_blocks_per_seq, int num_blocks, int n_q_heads,
                                int n_kv_heads, int head_dim, int block_size, float scale,
                                int max_q_len, int32_t* err_word, pa_stream_t stream) {
  if (num_seqs < 0 || num_seqs > 65535 || total_q < 0 || max_blocks_per_seq < 1 ||
      num_blocks < 1 ||
      n_q_heads < 1 || n_kv_heads < 1 || n_kv_heads > 65535 || max_q_len < 0)
    return PA_ERR_INVALID_ARG;
  if (n_q_heads % n_kv_heads != 0) return PA_ERR_INVALID_ARG;
  const int G = n_q_heads / n_kv_heads;
  if ((head_dim != 64 && head_dim != 128) ||
      (block_size != 8 && block_size != 16 && block_size != 32) || G > 64)
    return PA_ERR_UNSUPPORTED;
  if ((int64_t)num_blocks * n_kv_heads * block_size >= (int64_t)1 << 31)
    return PA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || scale == INFINITY) return PA_ERR_INVALID_ARG;
  if (num_seqs == 0 || max_q_len == 0 || total_q == 0) return PA_OK;
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
  a.total_q = total_q;
  a.max_blocks = max_blocks_per_seq;
  a.num_blocks = num_blocks;
  a.n_q = n_q_heads;
  a.n_kv = n_kv_heads;
  a.group = G;
  a.tile_tokens = kTTileRows / G;
  const int64_t tiles = ((int64_t)max_q_len + a.tile_tokens - 1) / a.tile_tokens;
  if (tiles > 2147483647) return PA_ERR_INVALID_ARG;
  a.n_tiles = (int)tiles;
  a.max_q_len = max_q_len;
  a.rank_tiles = num_seqs <= kTRankSeqs && tiles * num_seqs < ((int64_t)1 << 31);
  a.q_tma = (G & (G - 1)) == 0;  // 128 rows are 128 / G whole tokens
  a.scale_log2 = scale * kTLog2e;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (head_dim == 64) return prefill_bs<64>(block_size, a, k_pool, v_pool, st);
  return prefill_bs<128>(block_size, a, k_pool, v_pool, st);
}
