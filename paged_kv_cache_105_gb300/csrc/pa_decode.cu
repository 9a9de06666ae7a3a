// Paged decode attention for sm_103a.
//
// What it computes ("03 · PagedAttention", "The part the analogy hides: the
// kernel"; "PagedAttention" (mlapandio.dev), "A DECODE STEP" diagram): for
// each sequence, one query token per query head attends over every cached
// token, whose K/V are gathered from scattered pool blocks through the
// sequence's block table. The pages describe no kernel design; everything
// below is this library's.
//
// Design (one GPU, HBM-bound: every step reads all cached K/V once). The
// unit of streaming is 16 tokens of one (sequence, kv head): one 16-token
// block, two 8-token blocks or half a 32-token block. Two kernels split the
// work; both end in the same merge.
//  * Balanced split (split_kernel, the default): the (sequence, kv head)
//    pairs, in order, form one stream of units (plus a small cost per pair),
//    cut into equal contiguous shares, one per warp of a persistent grid (3
//    CTAs of 4 warps per SM). A warp walks its share in chunks of up to 32
//    units through its own stage ring (lane 0 issues the TMA tile loads,
//    128-byte swizzle, one mbarrier per stage) with no barrier and no
//    cross-warp exchange; the ring runs across chunk and pair boundaries. A
//    pair wholly inside a share is written straight from the warp's
//    registers; a cut pair leaves a partial in one of the warp's two slots.
//  * Fixed partitions (decode_kernel): items are (sequence, kv head,
//    partition of P tokens), numbered sequence-major from per-sequence prefix
//    sums that every CTA builds in shared memory. Persistent CTAs take items
//    from a global counter and learn their next-but-one item through a
//    shared-memory mailbox while they work; an item's units are dealt
//    round-robin to the CTA's 4 warps, whose states meet in shared memory in
//    two rounds (warps 2, 3 -> 0, 1, then 1 -> 0).
//  * Math: the GQA group (the G query heads sharing the kv head) is the N
//    side of bf16 mma.sync m16n8k16 with the tokens on M: S^T = K Q^T, then
//    O^T += V^T P^T; movmatrix turns the score fragment into the P^T operand
//    in registers. Online softmax in fp32, base 2; the running maximum is
//    moved (and the state rescaled) only when a score exceeds it by 2^8. The
//    fp8 variant converts E4M3 codes to f16 in registers after the byte load.
//  * Merge: a second, small kernel combines the partials with log-sum-exp
//    weights (a warp per query row, or a CTA per row when rows are few). It
//    is a programmatic dependent launch that waits on the grid dependency
//    before reading.
//  * The decode grid itself is a programmatic dependent of whatever precedes
//    it on the stream (normally the cache write), so its launch overlaps that
//    kernel; it waits on the dependency before reading the pools.
//  * Every mbarrier wait is bounded; on timeout the kernel flags
//    PA_DEV_ERR_TIMEOUT and keeps its control flow, so it always terminates.
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
constexpr int kUnit = 16;                           // tokens per pipeline stage
constexpr int kMaxUnitsPerPart = 128;               // lane-held table entries: 32 per warp
constexpr uint64_t kWaitLimitNs = 2000000000ull;    // 2 s: a wait that long is a fault
constexpr uint64_t kWaitAfterFaultNs = 1000000ull;  // 1 ms once something has timed out
constexpr int kMaxParts = 1024;
constexpr int kMaxSeqs = 8192;
constexpr int kMaxGrid = 512;                       // persistent CTAs at most
constexpr int kMaxWorkers = kMaxGrid * 4;           // balanced split: one worker per warp
constexpr int kMinUnitsPerWorker = 8;  // balanced split: work per warp at least
// Balanced split: each (sequence, kv head) pair also costs this many units in
// the stream being cut (its merge and bookkeeping), so a warp whose share holds
// many short pairs gets fewer units.
constexpr int kPairCost = 4;
constexpr float kLog2e = 1.4426950408889634f;

struct DecodeArgs {
  __nv_bfloat16* out;
  const __nv_bfloat16* q;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  // Partials. Fixed partitions: [S][Hq][max_parts] rows. Balanced split:
  // [kMaxWorkers warps][2 slots][G heads] rows. O rows have D floats, (m, l)
  // in log2 units.
  float* ws_o;
  float2* ws_ml;
  int32_t* work;             // [2]: items handed out dynamically, CTAs done
  int4* pair_info;           // balanced: [S][Hkv] (first worker, parts, first slot, -)
  int32_t* err;
  int num_seqs, max_blocks, num_blocks, n_q, n_kv, group;
  int part_tokens, max_parts, len_cap;
  int balanced;              // 1: even split of all units across warps
  int map3d;                 // 1: one TMA op loads both 64-column halves of a row
  float scale_log2;          // softmax scale (times the K scale for fp8) times log2(e)
  float v_scale;             // fp8: the V scale; 1 for bf16
};

// EB: bytes per cached element (2: bf16, 1: fp8 E4M3).
template <int D, int BS, int NT, int EB = 2>
struct Cfg {
  static constexpr int ROWS = BS < kUnit ? BS : kUnit;  // rows per TMA box
  static constexpr int BOXES = kUnit / ROWS;            // boxes (blocks) per unit
  static constexpr int KH = D * EB / 128;               // 128-byte pieces of a row
  static_assert(KH >= 1, "a cached row must span at least one 128-byte swizzle span");
  static constexpr int BOX_BYTES = KH * ROWS * 128;     // one box of K (or V), all halves
  static constexpr int KV_BYTES = BOXES * BOX_BYTES;    // K (or V) of a unit = 16 * D * 2
  static constexpr int STAGE = 2 * KV_BYTES;
  static constexpr int BUDGET = 16384;  // pipeline bytes per warp
  static constexpr int STAGES_RAW = BUDGET / STAGE;
  static constexpr int STAGES = STAGES_RAW < 2 ? 2 : (STAGES_RAW > 8 ? 8 : STAGES_RAW);
  static constexpr int HEADS = NT * 8;
  static constexpr int KS = D / 16;
  static constexpr int MSTRIDE = D + 4;  // padded row of the merge buffer
  static constexpr int PIPE_OFF = 0;
  static constexpr int BAR_OFF = kWarps * STAGES * STAGE;
  static constexpr int NBARS = kWarps * STAGES + 4;  // stage barriers + mailbox
  static constexpr int MAIL_OFF = BAR_OFF + NBARS * 8;
  static constexpr int MISC_OFF = MAIL_OFF + 16;
  static constexpr int FIN_OFF = MISC_OFF + 32;      // 2 x 16 floats
  static constexpr int ML_OFF = FIN_OFF + 2 * 16 * 4;  // 2 slots x HEADS x (m, l)
  static constexpr int MERGE_OFF = ML_OFF + 2 * HEADS * 2 * 4;
  // Merge buffer: 2 slots x G heads x MSTRIDE floats; then the prefix table.
  __host__ __device__ static int prefix_off(int group) {
    return MERGE_OFF + 2 * group * MSTRIDE * 4;
  }
  // prefix[num_seqs + 1] then the clamped lengths lens[num_seqs]
  static size_t smem_bytes(int num_seqs, int group) {
    return 1024 /* alignment slack */ + prefix_off(group) +
           sizeof(int) * (size_t)(2 * num_seqs + 1);
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

// Balanced split: a pair's length in the stream (its units plus the pair cost;
// an empty sequence takes no room).
__device__ __forceinline__ int stream_len(int len) {
  return len > 0 ? (len + kUnit - 1) / kUnit + kPairCost : 0;
}

// Exclusive prefix over sequences of the per-sequence count - items
// n_kv * parts(len) for fixed partitions, 16-token units for the balanced
// split - and the clamped lengths, both kept in shared memory.
__device__ void build_prefix(int* prefix, int* lens, const DecodeArgs& a, int* warp_tot) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (a.num_seqs + kThreads - 1) / kThreads;
  const int b = min(a.num_seqs, tid * per), e = min(a.num_seqs, b + per);
  int sum = 0;
  for (int s = b; s < e; ++s) {
    const int raw = __ldg(&a.seq_lens[s]);
    const int len = clamp_len(raw, a.len_cap);
    if (raw != len && blockIdx.x == 0) report(a.err, PA_DEV_ERR_SEQ_LEN);
    lens[s] = len;
    sum += a.balanced ? stream_len(len) : a.n_kv * parts_of(len, a.part_tokens);
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
    run += a.balanced ? stream_len(lens[s]) : a.n_kv * parts_of(lens[s], a.part_tokens);
  }
  if (tid == kThreads - 1) prefix[a.num_seqs] = base + incl;
}

// Bounded wait that flags a timeout (and shortens later waits) instead of
// hanging; control flow continues either way.
__device__ __forceinline__ void wait_or_flag(uint32_t bar, uint32_t parity, const DecodeArgs& a,
                                             volatile int* fault) {
  const uint64_t limit = *fault ? kWaitAfterFaultNs : kWaitLimitNs;
  if (!mbar_wait_bounded(bar, parity, limit)) {
    report(a.err, PA_DEV_ERR_TIMEOUT);
    *fault = 1;
  }
}

// A chunk of work: up to 128 units of one (sequence, kv head). `part` says
// where the result goes (-1: the output itself; fixed partitions: the
// partition index; balanced split: this warp's partial slot 0 or 1). A
// segment (one warp's share of one (sequence, kv head)) may span several
// chunks: the softmax state is reset at `first` and written at `last`.
struct Item {
  int s, g, tok_end, u_begin, n_units, part;
  bool first, last;
  bool holds_first;  // balanced split: the segment contains the pair's first unit
  long long end;  // balanced split: unit position after this chunk
};

__device__ __forceinline__ Item decode_item(int item, const int* prefix, const int* lens,
                                            const DecodeArgs& a) {
  int lo = 0, hi = a.num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= item) lo = mid; else hi = mid - 1;
  }
  Item it;
  it.s = lo;
  const int nparts = (prefix[lo + 1] - prefix[lo]) / a.n_kv;
  const int local = item - prefix[lo];
  it.g = local / nparts;
  const int p = local - it.g * nparts;
  const int len = lens[lo];
  const int tok_begin = p * a.part_tokens;
  it.tok_end = min(len, tok_begin + a.part_tokens);
  it.u_begin = tok_begin / kUnit;
  it.n_units = it.tok_end > tok_begin ? (it.tok_end + kUnit - 1) / kUnit - it.u_begin : 0;
  it.part = nparts == 1 ? -1 : p;
  it.first = it.last = true;
  it.holds_first = false;
  it.end = 0;
  return it;
}

// Balanced split: the (sequence, kv head) pairs in order (sequence-major)
// form one stream; pair (s, g) occupies [A, B) = kPairCost positions of
// bookkeeping then its 16-token units [A + kPairCost, B). Warp c owns
// positions [c W / n, (c+1) W / n) of the W-long stream. The chunk that
// starts at or after position `pos` inside the warp's range [lo, hi): up to
// max_units units of one pair. Returns false if the range holds no more units.
__device__ __forceinline__ bool decode_chunk(long long pos, long long lo, long long hi,
                                             const int* prefix, const int* lens,
                                             const DecodeArgs& a, Item& it,
                                             int max_units = kMaxUnitsPerPart) {
#pragma unroll 1
  while (pos < hi) {
    int l = 0, h = a.num_seqs - 1;  // last sequence starting at or before pos
    while (l < h) {
      const int mid = (l + h + 1) >> 1;
      if ((long long)a.n_kv * prefix[mid] <= pos) l = mid; else h = mid - 1;
    }
    const int w = prefix[l + 1] - prefix[l];  // > 0: empty sequences start nowhere
    const long long base = (long long)a.n_kv * prefix[l];
    const int g = (int)((pos - base) / w);
    const long long A = base + (long long)g * w, B = A + w, R = A + kPairCost;
    const long long seg_lo = R > lo ? R : lo, seg_hi = B < hi ? B : hi;
    if (pos < seg_lo) pos = seg_lo;
    if (pos >= seg_hi) {  // no units of this pair in the range: next pair
      pos = B;
      continue;
    }
    long long end = pos + max_units;
    if (end > seg_hi) end = seg_hi;
    it.s = l;
    it.g = g;
    it.u_begin = (int)(pos - R);
    it.n_units = (int)(end - pos);
    it.tok_end = min(lens[l], (int)(end - R) * kUnit);
    it.first = pos == seg_lo;
    it.last = end == seg_hi;
    it.part = (lo <= R && B <= hi) ? -1 : (lo >= A ? 0 : 1);
    it.holds_first = seg_lo == R;
    it.end = end == seg_hi ? B : end;  // where the next chunk search starts
    return true;
  }
  return false;
}

__device__ __forceinline__ int units_of_warp(const Item& it, int warp) {
  return it.n_units > warp ? (it.n_units - warp + kWarps - 1) / kWarps : 0;
}

// Lane j gets the pool blocks of this warp's j-th unit of the item (one per
// TMA box), raw: they are checked where they are used, so that nothing
// waits on these loads until the unit is issued.
template <int BS, int BOXES, int ROWS>
__device__ __forceinline__ void load_ids(int (&ids)[BOXES], const Item& it, int warp, int lane,
                                         const DecodeArgs& a) {
  const int32_t* table = a.block_tables + (int64_t)it.s * a.max_blocks;
  const int u = it.u_begin + warp + lane * kWarps;
  const bool mine = lane < units_of_warp(it, warp);
#pragma unroll
  for (int b = 0; b < BOXES; ++b) {
    const int tok = u * kUnit + b * ROWS;
    ids[b] = (mine && tok < it.tok_end) ? __ldg(&table[tok / BS]) : 0;
  }
}

// Valid-box mask of a unit: box b holds tokens (b * ROWS < nv) and its block
// id lies inside the pool.
template <int BOXES, int ROWS>
__device__ __forceinline__ int box_mask(const int (&bid)[BOXES], int nv, int num_blocks) {
  int mask = 0;
#pragma unroll
  for (int b = 0; b < BOXES; ++b)
    if (b * ROWS < nv && bid[b] >= 0 && bid[b] < num_blocks) mask |= 1 << b;
  return mask;
}

// B-operand fragments of the item's queries (head_dim x heads, column-major
// = the q rows); heads past the group are zero.
template <int D, int NT>
__device__ __forceinline__ void load_q(uint32_t (&qf)[NT][D / 16][2], const Item& it, int lane,
                                       const DecodeArgs& a) {
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const int n = t * 8 + (lane >> 2);
    const bool real = n < a.group;
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
        a.q + ((int64_t)it.s * a.n_q + (int64_t)it.g * a.group + (real ? n : 0)) * D);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      qf[t][ks][0] = real ? __ldg(&qrow[ks * 8 + (lane & 3)]) : 0u;
      qf[t][ks][1] = real ? __ldg(&qrow[ks * 8 + 4 + (lane & 3)]) : 0u;
    }
  }
}

// Online softmax of one unit's scores, base 2, with a lazily moved
// reference: m (per query head) only moves when some score exceeds it by
// more than kLazyLog2, and then the accumulators and sums are rescaled to the
// new maximum; otherwise the weights 2^(x - m) are used as they are. They
// stay below 2^kLazyLog2, which the fp32 sums and the 16-bit P operand hold
// exactly as well as weights below 1. (m, l) keep their meaning: l is the sum
// of 2^(x - m) and O the matching weighted sum, whatever m is. sc holds the
// raw scores of tokens tA = g (sc[..][0..1]) and tB = g + 8 (sc[..][2..3]);
// masked tokens weigh zero. P^T fragments come back in pb (f16 or bf16) as a
// pair: pb[..][0..1] the rounded weights, pb[..][2..3] what rounding left
// (split_pair); both go through the P V product.
constexpr float kLazyLog2 = 8.f;

// Two weights as a 16-bit pair hi + lo: hi = p rounded to the operand type,
// lo = (p - hi) rounded, so hi + lo carries p to about 2^-16 relative. A lone
// 16-bit weight is off by up to 2^-8 (bf16) or 2^-11 (f16) relative, which
// is too coarse for an output element that is a near-cancelling sum of
// larger terms (short contexts): there the error of the weights, not of the
// element, sets the element's error. p - hi is exact in fp32.
template <bool F16P>
__device__ __forceinline__ void split_pair(float p0, float p1, uint32_t& hi, uint32_t& lo) {
  if constexpr (F16P) {
    hi = pack_f16x2(p0, p1);
    const float2 h = unpack_f16x2(hi);
    lo = pack_f16x2(p0 - h.x, p1 - h.y);
  } else {
    hi = pack_bf16x2(p0, p1);
    lo = pack_bf16x2(p0 - __uint_as_float(hi << 16), p1 - __uint_as_float(hi & 0xffff0000u));
  }
}

template <int NT, int KS, bool F16P>
__device__ __forceinline__ void softmax_unit(const float (&sc)[NT][4], bool okA, bool okB,
                                             float scale_log2, float (&acc)[NT][KS][4],
                                             float (&mrun)[NT][2], float (&lrun)[NT][2],
                                             uint32_t (&pb)[NT][4]) {
  float x[NT][4];
  bool need = false;
#pragma unroll
  for (int t = 0; t < NT; ++t) {
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      x[t][jj] = okA ? sc[t][jj] * scale_log2 : -INFINITY;
      x[t][jj + 2] = okB ? sc[t][jj + 2] * scale_log2 : -INFINITY;
      need |= fmaxf(x[t][jj], x[t][jj + 2]) > mrun[t][jj] + kLazyLog2;
    }
  }
  if (__any_sync(0xffffffffu, need)) {  // warp-uniform: move the reference
#pragma unroll
    for (int t = 0; t < NT; ++t) {
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const float mx = warp_max_xor4(fmaxf(x[t][jj], x[t][jj + 2]));
        const float m_new = fmaxf(mrun[t][jj], mx);
        const float alpha = fast_exp2(mrun[t][jj] - (m_new == -INFINITY ? 0.f : m_new));
        lrun[t][jj] *= alpha;
#pragma unroll
        for (int dt = 0; dt < KS; ++dt) {
          acc[t][dt][jj] *= alpha;
          acc[t][dt][jj + 2] *= alpha;
        }
        mrun[t][jj] = m_new;
      }
    }
  }
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    float pv[4];
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const float base = mrun[t][jj] == -INFINITY ? 0.f : mrun[t][jj];
      pv[jj] = fast_exp2(x[t][jj] - base);
      pv[jj + 2] = fast_exp2(x[t][jj + 2] - base);
      lrun[t][jj] += pv[jj] + pv[jj + 2];
    }
    uint32_t hA, lA, hB, lB;
    split_pair<F16P>(pv[0], pv[1], hA, lA);
    split_pair<F16P>(pv[2], pv[3], hB, lB);
    pb[t][0] = movmatrix_trans(hA);
    pb[t][1] = movmatrix_trans(hB);
    pb[t][2] = movmatrix_trans(lA);
    pb[t][3] = movmatrix_trans(lB);
  }
}

// One 16-token unit of attention for the warp, online softmax in base 2.
// K and V rows sit in shared memory (128-byte swizzled tiles, one box of
// ROWS rows per block); tokens >= nv or in a box whose bit is clear in
// `mask` are absent. S^T = K Q^T (tokens on M, the query heads of the group
// on N), then O^T += V^T P^T, with P^T made from the score fragment by
// movmatrix.
template <int D, int ROWS, int NT>
__device__ __forceinline__ void attend_unit(uint32_t kb, uint32_t vb, int lane, int nv, int mask,
                                            float scale_log2,
                                            const uint32_t (&qf)[NT][D / 16][2],
                                            float (&acc)[NT][D / 16][4], float (&mrun)[NT][2],
                                            float (&lrun)[NT][2]) {
  constexpr int KS = D / 16;
  constexpr int BOX_BYTES = (D / 64) * ROWS * 128;
    // ---- S^T = K Q^T for 16 tokens x 8 heads (per n-tile)
    float sc[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t) sc[t][0] = sc[t][1] = sc[t][2] = sc[t][3] = 0.f;
    {
      const int r = (lane & 7) + ((lane >> 3) & 1) * 8;
      const uint32_t row = kb + (r / ROWS) * BOX_BYTES + (r % ROWS) * 128;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const int h = ks >> 2;
        const int c = ((ks & 3) << 1) + (lane >> 4);
        uint32_t a0, a1, a2, a3;
        ldsm_x4(row + h * ROWS * 128 + ((c ^ (r & 7)) << 4), a0, a1, a2, a3);
#pragma unroll
        for (int t = 0; t < NT; ++t)
          mma_bf16_16816(sc[t], a0, a1, a2, a3, qf[t][ks][0], qf[t][ks][1]);
      }
    }
    // ---- mask, online softmax (base 2), P^T fragments
    const int tA = lane >> 2, tB = tA + 8;
    const bool okA = tA < nv && (mask >> (tA / ROWS) & 1);
    const bool okB = tB < nv && (mask >> (tB / ROWS) & 1);
    uint32_t pb[NT][4];
    softmax_unit<NT, KS, false>(sc, okA, okB, scale_log2, acc, mrun, lrun, pb);
    // ---- O^T += V^T P^T
    {
      const int mi = lane >> 3;
      const int r = (lane & 7) + (mi >> 1) * 8;
      const uint32_t row = vb + (r / ROWS) * BOX_BYTES + (r % ROWS) * 128;
#pragma unroll
      for (int dt = 0; dt < KS; ++dt) {
        const int h = dt >> 2;
        const int c = ((dt & 3) << 1) + (mi & 1);
        uint32_t a0, a1, a2, a3;
        ldsm_x4_trans(row + h * ROWS * 128 + ((c ^ (r & 7)) << 4), a0, a1, a2, a3);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          mma_bf16_16816(acc[t][dt], a0, a1, a2, a3, pb[t][0], pb[t][1]);
          mma_bf16_16816(acc[t][dt], a0, a1, a2, a3, pb[t][2], pb[t][3]);
        }
      }
    }
}

// ------------------------------------------------------------ fp8 (E4M3) K/V
//
// The fp8 cache holds E4M3 codes; a code times the tensor's fp32 scale is the
// value. Codes are exact in f16, so the contractions run as f16 mma.sync on
// the codes (scores S = codes . q, the K scale folded into the softmax scale;
// the V scale applied to the output). A row of D = 128 codes is one 128-byte
// swizzle span. ldmatrix on byte data gives each lane 4 consecutive codes of
// one row per 8x8 b16 matrix; that fixes the order in which the k (and, for
// V^T, the m) index of a 16-wide slice is walked:
//   K (A of S^T = K Q^T): lane (g, c) holds d = 4c .. 4c+3 of a 16-column
//     chunk; k-slots (2c, 2c+1) take d (4c, 4c+1) and (2c+8, 2c+9) take
//     d (4c+2, 4c+3). Q (the B operand) is loaded in the same order.
//   V (A of O^T += V^T P^T): the codes of 8 tokens x 16 d, converted, are two
//     8x8 f16 matrices M1 (d = 4j'+{0,1}) and M2 (d = 4j'+{2,3}); movmatrix
//     transposes each into the (d, token) layout, so rows 0-7 of a 16-row
//     A tile are the d of M1 and rows 8-15 those of M2 (see fp8_out_d).

// B-operand fragments of the query heads in f16, k-slots in the order above.
template <int D, int NT>
__device__ __forceinline__ void load_q_f16(uint32_t (&qf)[NT][D / 16][2], const Item& it,
                                           int lane, const DecodeArgs& a) {
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const int n = t * 8 + (lane >> 2);
    const bool real = n < a.group;
    const uint2* qrow = reinterpret_cast<const uint2*>(
        a.q + ((int64_t)it.s * a.n_q + (int64_t)it.g * a.group + (real ? n : 0)) * D);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const uint2 v = real ? __ldg(&qrow[ks * 4 + (lane & 3)]) : make_uint2(0u, 0u);
      // bf16 -> f32 is a shift; f32 -> f16 rounds to nearest
      qf[t][ks][0] = pack_f16x2(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u));
      qf[t][ks][1] = pack_f16x2(__uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
    }
  }
}

// Head-dim column of accumulator row `r` (0..15) of 16-column chunk dt.
__device__ __forceinline__ int fp8_out_d(int dt, int r) {
  const int j = r & 7;
  return dt * 16 + 4 * (j >> 1) + (j & 1) + (r >> 3) * 2;
}

// attend_unit over fp8 codes: one 16-token unit, 128-byte rows.
template <int D, int ROWS, int NT>
__device__ __forceinline__ void attend_unit_fp8(uint32_t kb, uint32_t vb, int lane, int nv,
                                                int mask, float scale_log2,
                                                const uint32_t (&qf)[NT][D / 16][2],
                                                float (&acc)[NT][D / 16][4],
                                                float (&mrun)[NT][2], float (&lrun)[NT][2]) {
  constexpr int KS = D / 16;
  constexpr int BOX_BYTES = ROWS * 128;
  static_assert(D == 128, "fp8 rows are one 128-byte span");
  // lanes 8i..8i+7 address matrix i: tokens (i & 1) * 8 + 0..7 of chunk 2p + (i >> 1)
  const int mi = lane >> 3;
  const int r = (lane & 7) + (mi & 1) * 8;
  const int rsw = r & 7;
  const uint32_t roff = (r / ROWS) * BOX_BYTES + (r % ROWS) * 128;
  // ---- S^T = K Q^T
  float sc[NT][4];
#pragma unroll
  for (int t = 0; t < NT; ++t) sc[t][0] = sc[t][1] = sc[t][2] = sc[t][3] = 0.f;
#pragma unroll
  for (int p = 0; p < KS / 2; ++p) {
    const int c = 2 * p + (mi >> 1);
    uint32_t x[4];
    ldsm_x4(kb + roff + ((c ^ rsw) << 4), x[0], x[1], x[2], x[3]);
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      uint32_t a0, a1, a2, a3;
      e4m3x4_to_f16x2x2(x[2 * hf], a0, a2);      // token g
      e4m3x4_to_f16x2x2(x[2 * hf + 1], a1, a3);  // token g + 8
#pragma unroll
      for (int t = 0; t < NT; ++t)
        mma_f16_16816(sc[t], a0, a1, a2, a3, qf[t][2 * p + hf][0], qf[t][2 * p + hf][1]);
    }
  }
  // ---- mask, online softmax (base 2), P^T fragments
  const int tA = lane >> 2, tB = tA + 8;
  const bool okA = tA < nv && (mask >> (tA / ROWS) & 1);
  const bool okB = tB < nv && (mask >> (tB / ROWS) & 1);
  uint32_t pb[NT][4];
  softmax_unit<NT, KS, true>(sc, okA, okB, scale_log2, acc, mrun, lrun, pb);
  // ---- O^T += V^T P^T
#pragma unroll
  for (int p = 0; p < KS / 2; ++p) {
    const int c = 2 * p + (mi >> 1);
    uint32_t y[4];
    ldsm_x4(vb + roff + ((c ^ rsw) << 4), y[0], y[1], y[2], y[3]);
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      uint32_t m1a, m2a, m1b, m2b;
      e4m3x4_to_f16x2x2(y[2 * hf], m1a, m2a);      // tokens 0-7
      e4m3x4_to_f16x2x2(y[2 * hf + 1], m1b, m2b);  // tokens 8-15
      const uint32_t a0 = movmatrix_trans(m1a), a1 = movmatrix_trans(m2a);
      const uint32_t a2 = movmatrix_trans(m1b), a3 = movmatrix_trans(m2b);
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        mma_f16_16816(acc[t][2 * p + hf], a0, a1, a2, a3, pb[t][0], pb[t][1]);
        mma_f16_16816(acc[t][2 * p + hf], a0, a1, a2, a3, pb[t][2], pb[t][3]);
      }
    }
  }
}

template <int D, int BS, int NT>
__global__ void __launch_bounds__(kThreads)
decode_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
              const DecodeArgs a) {
  using C = Cfg<D, BS, NT>;
  constexpr int ROWS = C::ROWS, BOXES = C::BOXES, KH = C::KH, STAGES = C::STAGES;
  constexpr int KS = C::KS;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  int* mail = reinterpret_cast<int*>(smem + C::MAIL_OFF);
  int* misc = reinterpret_cast<int*>(smem + C::MISC_OFF);  // [1] fault flag
  float* fin = reinterpret_cast<float*>(smem + C::FIN_OFF);
  float* mlb = reinterpret_cast<float*>(smem + C::ML_OFF);
  float* macc = reinterpret_cast<float*>(smem + C::MERGE_OFF);
  int* prefix = reinterpret_cast<int*>(smem + C::prefix_off(a.group));
  int* lens = prefix + a.num_seqs + 1;
  volatile int* fault = misc + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t my_pipe = sbase + C::PIPE_OFF + warp * STAGES * C::STAGE;
  const uint32_t my_bar = sbase + C::BAR_OFF + warp * STAGES * 8;
  const uint32_t mail_bar = sbase + C::BAR_OFF + kWarps * STAGES * 8;

  if (tid == 0) {
    for (int i = 0; i < C::NBARS; ++i) mbar_init(sbase + C::BAR_OFF + 8 * i, 1);
    misc[0] = 0;
    misc[1] = 0;
    fence_mbarrier_init();
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
  }
  // The prologue below reads only q, the tables and the lengths; under a
  // programmatic launch it overlaps the preceding kernel (the cache write),
  // and everything that touches the pools or the outputs waits for it.
  build_prefix(prefix, lens, a, reinterpret_cast<int*>(smem + C::ML_OFF));
  __syncthreads();
  const int total = prefix[a.num_seqs];
  const int G = a.group;

  // This CTA's items are blockIdx.x, blockIdx.x + gridDim.x, then one per
  // dynamic fetch (2 * gridDim.x + counter).
  int item = blockIdx.x;
  Item cur{}, nxt{};
  int ids_cur[BOXES], ids_nxt[BOXES];
  uint32_t qf_cur[NT][KS][2], qf_nxt[NT][KS][2];
  bool have_cur, have_nxt = false;
  have_cur = item < total;
  if (have_cur) {
    cur = decode_item(item, prefix, lens, a);
    const int item1 = item + (int)gridDim.x;
    have_nxt = item1 < total;
    if (have_nxt) nxt = decode_item(item1, prefix, lens, a);
  }
  if (have_cur) {
    load_ids<BS, BOXES, ROWS>(ids_cur, cur, warp, lane, a);
    load_q<D, NT>(qf_cur, cur, lane, a);
    if (have_nxt) {
      load_ids<BS, BOXES, ROWS>(ids_nxt, nxt, warp, lane, a);
      load_q<D, NT>(qf_nxt, nxt, lane, a);
    }
  }
  griddep_wait();  // from here on: pool reads, output and workspace writes

  float acc[NT][KS][4];               // this warp's softmax state for the segment
  float mrun[NT][2], lrun[NT][2];
  uint32_t issued = 0, consumed = 0;  // units of this warp (same on all lanes)
  int issue_in_next = 0, issue_j = 0;  // issue cursor: (current or next item, unit)

  // Issue TMA loads into free stages, running from the current item into the
  // next one. Warp-collective.
  auto fill = [&]() {
#pragma unroll 1
    while (issued - consumed < (uint32_t)STAGES) {
      const int nm = issue_in_next ? units_of_warp(nxt, warp) : units_of_warp(cur, warp);
      if (issue_j >= nm) {
        if (!issue_in_next && have_nxt) {
          issue_in_next = 1;
          issue_j = 0;
          continue;
        }
        break;
      }
      int bid[BOXES];
#pragma unroll
      for (int b = 0; b < BOXES; ++b)
        bid[b] = __shfl_sync(0xffffffffu, issue_in_next ? ids_nxt[b] : ids_cur[b], issue_j);
      const int g = issue_in_next ? nxt.g : cur.g;
      if (lane == 0) {
        const uint32_t st = issued % STAGES;
        const uint32_t fb = my_bar + 8 * st;
        const int iu = (issue_in_next ? nxt.u_begin : cur.u_begin) + warp + issue_j * kWarps;
        const int inv = min(kUnit, (issue_in_next ? nxt.tok_end : cur.tok_end) - iu * kUnit);
        const int mask = box_mask<BOXES, ROWS>(bid, inv, a.num_blocks);
        int nload = 0;
#pragma unroll
        for (int b = 0; b < BOXES; ++b) {
          nload += mask >> b & 1;
          if (b * ROWS < inv && !(mask >> b & 1)) report(a.err, PA_DEV_ERR_BLOCK_ID);
        }
        if (nload == 0) {
          mbar_arrive(fb);
        } else {
          mbar_arrive_expect_tx(fb, (uint32_t)nload * 2 * C::BOX_BYTES);
          const uint32_t kdst = my_pipe + st * C::STAGE;
          const uint32_t vdst = kdst + C::KV_BYTES;
#pragma unroll
          for (int b = 0; b < BOXES; ++b) {
            if (!(mask >> b & 1)) continue;
            // first row of this box: block row base plus the 16-token
            // window's offset inside a 32-token block
            const int tok_in_block = ((issue_in_next ? nxt.u_begin : cur.u_begin) +
                                      warp + issue_j * kWarps) * kUnit % BS + b * ROWS;
            const int32_t y = (bid[b] * a.n_kv + g) * BS + (BS > kUnit ? tok_in_block : 0);
            if (KH == 2 && a.map3d) {
              tma_load_3d(kdst + b * C::BOX_BYTES, &tmk, 0, y, 0, fb);
              tma_load_3d(vdst + b * C::BOX_BYTES, &tmv, 0, y, 0, fb);
            } else {
#pragma unroll
              for (int h = 0; h < KH; ++h) {
                tma_load_2d(kdst + b * C::BOX_BYTES + h * ROWS * 128, &tmk, h * 64, y, fb);
                tma_load_2d(vdst + b * C::BOX_BYTES + h * ROWS * 128, &tmv, h * 64, y, fb);
              }
            }
          }
        }
      }
      ++issued;
      ++issue_j;
    }
  };

#pragma unroll 1
  for (int k = 0; have_cur; ++k) {
    // ---- fetch item k + 2 of this CTA; the value is only needed after the
    // merge, so it is published then and its latency hides behind the units
    int fetched = INT_MAX;
    if (tid == 0 && have_nxt) fetched = 2 * (int)gridDim.x + atomicAdd(&a.work[0], 1);

    // ---- stream this warp's units of the current chunk
    if (cur.first) {
#pragma unroll
      for (int t = 0; t < NT; ++t) {
#pragma unroll
        for (int dt = 0; dt < KS; ++dt)
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[t][dt][i] = 0.f;
        mrun[t][0] = mrun[t][1] = -INFINITY;
        lrun[t][0] = lrun[t][1] = 0.f;
      }
    }
    const int n_mine = units_of_warp(cur, warp);
#pragma unroll 1
    for (int j = 0; j < n_mine; ++j) {
      fill();
      const uint32_t st = consumed % STAGES;
      wait_or_flag(my_bar + 8 * st, (consumed / STAGES) & 1u, a, fault);
      const int nv = min(kUnit, cur.tok_end - (cur.u_begin + warp + j * kWarps) * kUnit);
      int cbid[BOXES];
#pragma unroll
      for (int b = 0; b < BOXES; ++b) cbid[b] = __shfl_sync(0xffffffffu, ids_cur[b], j);
      const int mask = box_mask<BOXES, ROWS>(cbid, nv, a.num_blocks);
      const uint32_t kb = my_pipe + st * C::STAGE;
      const uint32_t vb = kb + C::KV_BYTES;
      bool all_ok = nv == kUnit;
#pragma unroll
      for (int b = 0; b < BOXES; ++b)
        if (b * ROWS < nv && !(mask >> b & 1)) all_ok = false;
      if (!all_ok) {
        // Rows of absent tokens may hold anything (even NaN): zero their V
        // so that a zero weight times the row stays zero.
        uint8_t* vgen = smem + (vb - sbase);
        for (int i = lane; i < kUnit * KH * 8; i += 32) {
          const int r = i / (KH * 8), rest = i % (KH * 8);
          const int h = rest / 8, c = rest % 8;
          if (r >= nv || !(mask >> (r / ROWS) & 1))
            *reinterpret_cast<uint4*>(vgen + (r / ROWS) * C::BOX_BYTES + h * ROWS * 128 +
                                      (r % ROWS) * 128 + c * 16) = make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
      }

      attend_unit<D, ROWS, NT>(kb, vb, lane, nv, mask, a.scale_log2, qf_cur, acc, mrun, lrun);
      // The stage is refilled by this warp's next fill(); generic writes to
      // it (the zeroed rows) must be ordered before that TMA.
      if (!all_ok) fence_proxy_async_smem();
      __syncwarp();
      ++consumed;
    }
    fill();  // the next item's first units fly while the CTA merges
    if (tid == 0) {
      mail[k & 3] = fetched;
      mbar_arrive(mail_bar + 8 * (k & 3));
    }

    if (cur.last) {
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      lrun[t][0] = warp_sum_xor4(lrun[t][0]);
      lrun[t][1] = warp_sum_xor4(lrun[t][1]);
    }

    // ---- merge: the four warps' states meet in two rounds through two
    // shared-memory slots (warps 2, 3 -> 0, 1, then 1 -> 0), so that the
    // buffer holds two warps' rows, not three
    auto put = [&](int slot) {
      float* buf = macc + slot * G * C::MSTRIDE;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
#pragma unroll
        for (int dt = 0; dt < KS; ++dt)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int n = t * 8 + 2 * (lane & 3) + (i & 1);
            const int d = dt * 16 + (lane >> 2) + 8 * (i >> 1);
            if (n < G) buf[n * C::MSTRIDE + d] = acc[t][dt][i];
          }
        if (lane < 4) {
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            const int n = t * 8 + 2 * lane + jj;
            mlb[(slot * C::HEADS + n) * 2] = mrun[t][jj];
            mlb[(slot * C::HEADS + n) * 2 + 1] = lrun[t][jj];
          }
        }
      }
    };
    auto take = [&](int slot) {
      const float* buf = macc + slot * G * C::MSTRIDE;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          const int n = t * 8 + 2 * (lane & 3) + jj;
          if (n >= G) continue;
          const float mo = mlb[(slot * C::HEADS + n) * 2];
          const float lo = mlb[(slot * C::HEADS + n) * 2 + 1];
          const float M = fmaxf(mrun[t][jj], mo);
          const float es = mrun[t][jj] == -INFINITY ? 0.f : fast_exp2(mrun[t][jj] - M);
          const float eo = mo == -INFINITY ? 0.f : fast_exp2(mo - M);
          lrun[t][jj] = es * lrun[t][jj] + eo * lo;
          mrun[t][jj] = M;
#pragma unroll
          for (int dt = 0; dt < KS; ++dt) {
            const int d = dt * 16 + (lane >> 2);
            acc[t][dt][jj] = es * acc[t][dt][jj] + eo * buf[n * C::MSTRIDE + d];
            acc[t][dt][jj + 2] = es * acc[t][dt][jj + 2] + eo * buf[n * C::MSTRIDE + d + 8];
          }
        }
      }
    };
    if (warp >= 2) put(warp - 2);
    __syncthreads();
    if (warp < 2) take(warp);
    __syncthreads();
    if (warp == 1) put(0);
    __syncthreads();
    if (warp == 0) {
      take(0);
      // the CTA's result for the item, back into buffer 0 for coalesced writes
      float* buf = macc;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
#pragma unroll
        for (int dt = 0; dt < KS; ++dt)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int n = t * 8 + 2 * (lane & 3) + (i & 1);
            const int d = dt * 16 + (lane >> 2) + 8 * (i >> 1);
            if (n < G) buf[n * C::MSTRIDE + d] = acc[t][dt][i];
          }
        if (lane < 4) {
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            fin[t * 8 + 2 * lane + jj] = mrun[t][jj];
            fin[16 + t * 8 + 2 * lane + jj] = lrun[t][jj];
          }
        }
      }
    }
    __syncthreads();

    const int64_t row0 = (int64_t)cur.s * a.n_q + (int64_t)cur.g * G;
    for (int i = tid; i < G * D; i += kThreads) {
      const int n = i / D, d = i - n * D;
      const float O = macc[n * C::MSTRIDE + d];
      const float M = fin[n], L = fin[16 + n];
      if (cur.part < 0) {
        a.out[(row0 + n) * D + d] = __float2bfloat16_rn(L > 0.f ? O / L : 0.f);
      } else {
        const int64_t wr = (row0 + n) * a.max_parts + cur.part;
        a.ws_o[wr * D + d] = O;
        if (d == 0) a.ws_ml[wr] = make_float2(M, L);
      }
    }

    __syncthreads();  // merge buffer, fin and misc are free again
    }  // cur.last

    // ---- advance: the next item becomes current; learn the one after it
    have_cur = have_nxt;
    if (!have_cur) break;
    cur = nxt;
#pragma unroll
    for (int b = 0; b < BOXES; ++b) ids_cur[b] = ids_nxt[b];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qf_cur[t][ks][0] = qf_nxt[t][ks][0];
        qf_cur[t][ks][1] = qf_nxt[t][ks][1];
      }
    if (issue_in_next) {
      issue_in_next = 0;  // the issue cursor already runs inside the new current item
    } else {
      issue_j = 0;
    }
    {
      // the new next item is this CTA's item k + 2, fetched at the top of
      // this iteration into mailbox slot k mod 4
      const int slot = k & 3;
      wait_or_flag(mail_bar + 8 * slot, (k >> 2) & 1u, a, fault);
      const int item_n = mail[slot];
      have_nxt = item_n < total;
      if (have_nxt) nxt = decode_item(item_n, prefix, lens, a);
    }
    if (have_nxt) {
      load_ids<BS, BOXES, ROWS>(ids_nxt, nxt, warp, lane, a);
      load_q<D, NT>(qf_nxt, nxt, lane, a);
    }
  }

  __syncthreads();
  griddep_launch_dependents();  // the partition merge may start launching
  if (tid == 0) {
    const int fin_ctas = atomicAdd(&a.work[1], 1);
    if (fin_ctas == (int)gridDim.x - 1) {  // the last CTA resets the shared counters
      atomicExch(&a.work[0], 0);
      atomicExch(&a.work[1], 0);
    }
  }
}

// Stage-ring bytes per warp of the balanced split: two stages of 16 tokens
// of K and V (bf16: 2 x 8 KB at head_dim 128; E4M3: 2 x 4 KB).
constexpr int kSplitRingBytes = 16384;
constexpr int kSplitRingBytesFp8 = 8192;

// Shared-memory layout of the balanced-split kernel: per-warp stage rings,
// their mbarriers, a fault flag, then the prefix and length tables.
template <int D, int BS, int NT, bool FP8 = false>
struct SplitCfg {
  using C = Cfg<D, BS, NT, FP8 ? 1 : 2>;
  static constexpr int STAGE = C::STAGE;
  static constexpr int STAGES_RAW = (FP8 ? kSplitRingBytesFp8 : kSplitRingBytes) / STAGE;
  static constexpr int STAGES = STAGES_RAW < 2 ? 2 : (STAGES_RAW > 8 ? 8 : STAGES_RAW);
  static constexpr int BAR_OFF = kWarps * STAGES * STAGE;
  static constexpr int MISC_OFF = BAR_OFF + kWarps * STAGES * 8;
  static constexpr int PREFIX_OFF = MISC_OFF + 64;  // [0..15] ints: fault flag, scan scratch
  static size_t smem_bytes(int num_seqs) {
    return 1024 + PREFIX_OFF + sizeof(int) * (size_t)(2 * num_seqs + 1);
  }
};

// Balanced split at warp granularity: every warp is a worker that owns an
// equal contiguous share of the unit stream (see decode_chunk) and streams
// it alone through its own stage ring, writing each pair it completes
// straight from its registers (or, for a pair cut at its share's edges, one
// of its two partial slots). No barrier and no cross-warp merge in the main
// loop; the merge kernel combines the cut pairs. FP8: the pools hold E4M3
// codes (attend_unit_fp8).
template <int D, int BS, int NT, bool FP8 = false>
__global__ void __launch_bounds__(kThreads)
split_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
             const DecodeArgs a) {
  using C = Cfg<D, BS, NT, FP8 ? 1 : 2>;
  using SC = SplitCfg<D, BS, NT, FP8>;
  constexpr int ROWS = C::ROWS, BOXES = C::BOXES, KH = C::KH, STAGES = SC::STAGES;
  constexpr int KS = C::KS;
  constexpr int kChunk = 32;  // units per chunk: one table entry per lane

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  int* misc = reinterpret_cast<int*>(smem + SC::MISC_OFF);
  int* prefix = reinterpret_cast<int*>(smem + SC::PREFIX_OFF);
  int* lens = prefix + a.num_seqs + 1;
  volatile int* fault = misc;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t my_pipe = sbase + warp * STAGES * SC::STAGE;
  const uint32_t my_bar = sbase + SC::BAR_OFF + warp * STAGES * 8;

  if (tid == 0) {
    for (int i = 0; i < kWarps * STAGES; ++i) mbar_init(sbase + SC::BAR_OFF + 8 * i, 1);
    misc[0] = 0;
    fence_mbarrier_init();
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
  }
  build_prefix(prefix, lens, a, misc + 8);
  __syncthreads();
  const int G = a.group;
  const long long U = (long long)a.n_kv * prefix[a.num_seqs];  // stream length
  long long n_workers = (U + kMinUnitsPerWorker - 1) / kMinUnitsPerWorker;
  if (n_workers > (long long)gridDim.x * kWarps) n_workers = (long long)gridDim.x * kWarps;
  if (n_workers < 1) n_workers = 1;
  const long long worker = (long long)blockIdx.x * kWarps + warp;
  const long long lo = worker * U / n_workers, hi = (worker + 1) * U / n_workers;

  Item cur{}, nxt{};
  int ids_cur[BOXES], ids_nxt[BOXES];
  uint32_t qf_cur[NT][KS][2], qf_nxt[NT][KS][2];
  bool have_cur = worker < n_workers && decode_chunk(lo, lo, hi, prefix, lens, a, cur, kChunk);
  bool have_nxt = have_cur && decode_chunk(cur.end, lo, hi, prefix, lens, a, nxt, kChunk);

  // lane j: the pool blocks of unit j of the chunk (raw; checked where used)
  auto load_ids_w = [&](int (&ids)[BOXES], const Item& it) {
    const int32_t* table = a.block_tables + (int64_t)it.s * a.max_blocks;
#pragma unroll
    for (int b = 0; b < BOXES; ++b) {
      const int tok = (it.u_begin + lane) * kUnit + b * ROWS;
      ids[b] = (lane < it.n_units && tok < it.tok_end) ? __ldg(&table[tok / BS]) : 0;
    }
  };
  auto load_qf = [&](uint32_t (&qf)[NT][KS][2], const Item& it) {
    if constexpr (FP8) load_q_f16<D, NT>(qf, it, lane, a);
    else load_q<D, NT>(qf, it, lane, a);
  };
  if (have_cur) {
    load_ids_w(ids_cur, cur);
    load_qf(qf_cur, cur);
    if (have_nxt) {
      load_ids_w(ids_nxt, nxt);
      load_qf(qf_nxt, nxt);
    }
  }
  griddep_wait();  // from here on: pool reads, output and workspace writes
  // sequences with no tokens own no units: their outputs are zero
  for (int sq = blockIdx.x; sq < a.num_seqs; sq += gridDim.x)
    if (lens[sq] == 0)
      for (int i = tid; i < a.n_q * D; i += kThreads)
        a.out[(int64_t)sq * a.n_q * D + i] = __float2bfloat16_rn(0.f);

  float acc[NT][KS][4];
  float mrun[NT][2], lrun[NT][2];
  uint32_t issued = 0, consumed = 0;
  int issue_in_next = 0, issue_j = 0;

  auto fill = [&]() {
#pragma unroll 1
    while (issued - consumed < (uint32_t)STAGES) {
      const int nm = issue_in_next ? nxt.n_units : cur.n_units;
      if (issue_j >= nm) {
        if (!issue_in_next && have_nxt) {
          issue_in_next = 1;
          issue_j = 0;
          continue;
        }
        break;
      }
      int bid[BOXES];
#pragma unroll
      for (int b = 0; b < BOXES; ++b)
        bid[b] = __shfl_sync(0xffffffffu, issue_in_next ? ids_nxt[b] : ids_cur[b], issue_j);
      if (lane == 0) {
        const Item& it = issue_in_next ? nxt : cur;
        const uint32_t st = issued % STAGES;
        const uint32_t fb = my_bar + 8 * st;
        const int iu = it.u_begin + issue_j;
        const int inv = min(kUnit, it.tok_end - iu * kUnit);
        const int mask = box_mask<BOXES, ROWS>(bid, inv, a.num_blocks);
        int nload = 0;
#pragma unroll
        for (int b = 0; b < BOXES; ++b) {
          nload += mask >> b & 1;
          if (b * ROWS < inv && !(mask >> b & 1)) report(a.err, PA_DEV_ERR_BLOCK_ID);
        }
        if (nload == 0) {
          mbar_arrive(fb);
        } else {
          mbar_arrive_expect_tx(fb, (uint32_t)nload * 2 * C::BOX_BYTES);
          const uint32_t kdst = my_pipe + st * SC::STAGE;
          const uint32_t vdst = kdst + C::KV_BYTES;
#pragma unroll
          for (int b = 0; b < BOXES; ++b) {
            if (!(mask >> b & 1)) continue;
            const int tok_in_block = (iu * kUnit) % BS + b * ROWS;
            const int32_t y = (bid[b] * a.n_kv + it.g) * BS + (BS > kUnit ? tok_in_block : 0);
            if (KH == 2 && a.map3d) {
              tma_load_3d(kdst + b * C::BOX_BYTES, &tmk, 0, y, 0, fb);
              tma_load_3d(vdst + b * C::BOX_BYTES, &tmv, 0, y, 0, fb);
            } else {
#pragma unroll
              for (int h = 0; h < KH; ++h) {
                constexpr int kCols = FP8 ? 128 : 64;  // elements per 128-byte piece
                tma_load_2d(kdst + b * C::BOX_BYTES + h * ROWS * 128, &tmk, h * kCols, y, fb);
                tma_load_2d(vdst + b * C::BOX_BYTES + h * ROWS * 128, &tmv, h * kCols, y, fb);
              }
            }
          }
        }
      }
      ++issued;
      ++issue_j;
    }
  };

#pragma unroll 1
  while (have_cur) {
    if (cur.first) {
#pragma unroll
      for (int t = 0; t < NT; ++t) {
#pragma unroll
        for (int dt = 0; dt < KS; ++dt)
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[t][dt][i] = 0.f;
        mrun[t][0] = mrun[t][1] = -INFINITY;
        lrun[t][0] = lrun[t][1] = 0.f;
      }
    }
#pragma unroll 1
    for (int j = 0; j < cur.n_units; ++j) {
      fill();
      const uint32_t st = consumed % STAGES;
      wait_or_flag(my_bar + 8 * st, (consumed / STAGES) & 1u, a, fault);
      const int nv = min(kUnit, cur.tok_end - (cur.u_begin + j) * kUnit);
      int cbid[BOXES];
#pragma unroll
      for (int b = 0; b < BOXES; ++b) cbid[b] = __shfl_sync(0xffffffffu, ids_cur[b], j);
      const int mask = box_mask<BOXES, ROWS>(cbid, nv, a.num_blocks);
      const uint32_t kb = my_pipe + st * SC::STAGE;
      const uint32_t vb = kb + C::KV_BYTES;
      bool all_ok = nv == kUnit;
#pragma unroll
      for (int b = 0; b < BOXES; ++b)
        if (b * ROWS < nv && !(mask >> b & 1)) all_ok = false;
      if (!all_ok) {
        // Rows of absent tokens may hold anything (even NaN): zero their V
        // so that a zero weight times the row stays zero.
        uint8_t* vgen = smem + (vb - sbase);
        for (int i = lane; i < kUnit * KH * 8; i += 32) {
          const int r = i / (KH * 8), rest = i % (KH * 8);
          const int h = rest / 8, c = rest % 8;
          if (r >= nv || !(mask >> (r / ROWS) & 1))
            *reinterpret_cast<uint4*>(vgen + (r / ROWS) * C::BOX_BYTES + h * ROWS * 128 +
                                      (r % ROWS) * 128 + c * 16) = make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
      }
      if constexpr (FP8)
        attend_unit_fp8<D, ROWS, NT>(kb, vb, lane, nv, mask, a.scale_log2, qf_cur, acc, mrun,
                                     lrun);
      else
        attend_unit<D, ROWS, NT>(kb, vb, lane, nv, mask, a.scale_log2, qf_cur, acc, mrun, lrun);
      // The stage is refilled by this warp's next fill(); generic writes to
      // it (the zeroed rows) must be ordered before that TMA.
      if (!all_ok) fence_proxy_async_smem();
      __syncwarp();
      ++consumed;
    }
    fill();  // keep the ring full across the write below

    if (cur.last) {
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        lrun[t][0] = warp_sum_xor4(lrun[t][0]);
        lrun[t][1] = warp_sum_xor4(lrun[t][1]);
      }
      const int64_t row0 = (int64_t)cur.s * a.n_q + (int64_t)cur.g * G;
      const long long prow = (worker * 2 + (cur.part < 0 ? 0 : cur.part)) * G;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int n = t * 8 + 2 * (lane & 3) + (i & 1);
          if (n >= G) continue;
          const float l = lrun[t][i & 1];
          // fp8: the V scale rides on the output (and on the partials)
          const float inv = (l > 0.f ? 1.f / l : 0.f) * (FP8 ? a.v_scale : 1.f);
          const float pscale = FP8 ? a.v_scale : 1.f;
#pragma unroll
          for (int dt = 0; dt < KS; ++dt) {
            const int r = (lane >> 2) + 8 * (i >> 1);
            const int d = FP8 ? fp8_out_d(dt, r) : dt * 16 + r;
            if (cur.part < 0)
              a.out[(row0 + n) * D + d] = __float2bfloat16_rn(acc[t][dt][i] * inv);
            else
              a.ws_o[(prow + n) * D + d] = acc[t][dt][i] * pscale;
          }
        }
        if (cur.part >= 0 && lane < 4) {
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            const int n = t * 8 + 2 * lane + jj;
            if (n < G) a.ws_ml[prow + n] = make_float2(mrun[t][jj], lrun[t][jj]);
          }
        }
      }
      if (lane == 0 && cur.holds_first) {
        // this worker holds the pair's first unit: tell the merge where its parts are
        const int w = prefix[cur.s + 1] - prefix[cur.s];
        const long long B = (long long)a.n_kv * prefix[cur.s] + (long long)(cur.g + 1) * w;
        const long long c1 = (B * n_workers - 1) / U;
        a.pair_info[(int64_t)cur.s * a.n_kv + cur.g] =
            make_int4((int)worker, (int)(c1 - worker + 1), cur.part < 0 ? 0 : cur.part, 0);
      }
    }

    // ---- advance
    have_cur = have_nxt;
    if (!have_cur) break;
    cur = nxt;
#pragma unroll
    for (int b = 0; b < BOXES; ++b) ids_cur[b] = ids_nxt[b];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qf_cur[t][ks][0] = qf_nxt[t][ks][0];
        qf_cur[t][ks][1] = qf_nxt[t][ks][1];
      }
    if (issue_in_next) issue_in_next = 0; else issue_j = 0;
    have_nxt = decode_chunk(cur.end, lo, hi, prefix, lens, a, nxt, kChunk);
    if (have_nxt) {
      load_ids_w(ids_nxt, nxt);
      load_qf(qf_nxt, nxt);
    }
  }

  __syncthreads();
  griddep_launch_dependents();  // the merge may start launching
}

// Merge of fixed split-KV partitions: one warp per (sequence, query head)
// row with more than one partition; lanes own head_dim columns. With m_p,
// l_p the running max (log2 units) and sum of partition p and O_p its
// unnormalised output: out = sum_p 2^(m_p - M) O_p / sum_p 2^(m_p - M) l_p,
// M = max_p m_p. Fixed partitions: the parts of a row are its partitions.
// Balanced split: the parts are the warps whose shares cut the row's
// (sequence, kv head) pair, as recorded by the warp holding its first unit.
struct MergeArgs {
  __nv_bfloat16* out;
  const float* ws_o;
  const float2* ws_ml;
  const int32_t* seq_lens;
  const int4* pair_info;
  int num_seqs, n_q, n_kv, group, part_tokens, max_parts, len_cap, balanced;
  int coop;  // 1: one CTA per row, its warps sharing the row's parts (few rows)
};

constexpr int kMergeWarps = 8;
constexpr int kMergePre = 8;       // parts a merge warp reads with the statistics, then per round
constexpr int kCoopRowsPerSm = 2;  // a CTA per merge row up to this many rows per SM

// The parts of merge row `row`: part q lives in partial row
// q == 0 ? rfirst : rbase + q * rstep. Returns their number (0 or 1: the
// decode kernel wrote the output itself).
__device__ __forceinline__ int merge_row_parts(const MergeArgs& m, int row, long long& rfirst,
                                               long long& rbase, long long& rstep) {
  const int s = row / m.n_q;
  const int len = clamp_len(__ldg(&m.seq_lens[s]), m.len_cap);
  if (m.balanced) {
    // Balanced split: parts are warps c0 .. c0 + n - 1; warp c keeps slot
    // (2c + slot) * G + head; only c0 may use slot 1.
    const int h = row - s * m.n_q, g = h / m.group, n = h - g * m.group;
    const int4 pi = __ldcg(&m.pair_info[(int64_t)s * m.n_kv + g]);
    rfirst = ((long long)pi.x * 2 + pi.z) * m.group + n;
    rbase = (long long)pi.x * 2 * m.group + n;
    rstep = 2LL * m.group;
    return len > 0 ? pi.y : 0;
  }
  rbase = rfirst = (long long)row * m.max_parts;
  rstep = 1;
  return parts_of(len, m.part_tokens);
}

// One row merged by a whole CTA (launched when there are few rows, e.g. one
// long sequence whose pairs are cut into hundreds of parts): warp w folds
// parts w, w + 8, ... into a running (max, sum, O), kB parts per round trip;
// warp 0 then combines the eight with the same identity.
template <int D>
__device__ __forceinline__ void merge_row_coop(const MergeArgs& m, int row) {
  constexpr int PER = D / 32, kB = 4;
  __shared__ float s_acc[kMergeWarps][D];
  __shared__ float2 s_ml[kMergeWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  long long rfirst, rbase, rstep;
  const int nparts = merge_row_parts(m, row, rfirst, rbase, rstep);
  if (nparts <= 1) return;  // the same on every thread of the CTA
  auto rowq = [&](int q) -> long long { return q == 0 ? rfirst : rbase + q * rstep; };
  float M = -INFINITY, L = 0.f, acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  for (int q0 = warp; q0 < nparts; q0 += kMergeWarps * kB) {
    float2 ml[kB];
    float ov[kB][PER];
#pragma unroll
    for (int b = 0; b < kB; ++b) {
      const int q = q0 + b * kMergeWarps;
      const bool in = q < nparts;
      const long long r = rowq(in ? q : 0);
      ml[b] = in ? __ldcg(&m.ws_ml[r]) : make_float2(-INFINITY, 0.f);
#pragma unroll
      for (int i = 0; i < PER; ++i) ov[b][i] = in ? __ldcg(m.ws_o + r * D + lane + 32 * i) : 0.f;
    }
#pragma unroll
    for (int b = 0; b < kB; ++b) {
      if (ml[b].x == -INFINITY) continue;  // absent, or a part that saw only masked tokens
      const float mx = fmaxf(M, ml[b].x);
      const float sc = M == -INFINITY ? 0.f : fast_exp2(M - mx);
      const float w = fast_exp2(ml[b].x - mx);
      L = L * sc + w * ml[b].y;
#pragma unroll
      for (int i = 0; i < PER; ++i) acc[i] = acc[i] * sc + w * ov[b][i];
      M = mx;
    }
  }
#pragma unroll
  for (int i = 0; i < PER; ++i) s_acc[warp][lane + 32 * i] = acc[i];
  if (lane == 0) s_ml[warp] = make_float2(M, L);
  __syncthreads();
  if (warp != 0) return;
  float Mx = -INFINITY;
#pragma unroll
  for (int w = 0; w < kMergeWarps; ++w) Mx = fmaxf(Mx, s_ml[w].x);
  float Lt = 0.f, out[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) out[i] = 0.f;
#pragma unroll
  for (int w = 0; w < kMergeWarps; ++w) {
    const float2 v = s_ml[w];
    const float wt = v.x == -INFINITY ? 0.f : fast_exp2(v.x - Mx);
    Lt += wt * v.y;
#pragma unroll
    for (int i = 0; i < PER; ++i) out[i] += wt * s_acc[w][lane + 32 * i];
  }
  const float inv = Lt > 0.f ? 1.f / Lt : 0.f;
#pragma unroll
  for (int i = 0; i < PER; ++i)
    m.out[(int64_t)row * D + lane + 32 * i] = __float2bfloat16_rn(out[i] * inv);
}

template <int D>
__global__ void __launch_bounds__(kMergeWarps * 32) merge_kernel(const MergeArgs m) {
  griddep_wait();  // the partials come from the decode grid
  griddep_launch_dependents();  // a dependent (which waits for this grid) may launch
  if (m.coop) {  // grid = rows
    merge_row_coop<D>(m, blockIdx.x);
    return;
  }
  constexpr int PER = D / 32;
  const int lane = threadIdx.x & 31;
  const int rows = m.num_seqs * m.n_q;
  for (int row = blockIdx.x * kMergeWarps + (threadIdx.x >> 5); row < rows;
       row += gridDim.x * kMergeWarps) {
    long long rbase, rfirst, rstep;  // row of part q: q == 0 ? rfirst : rbase + q * rstep
    const int nparts = merge_row_parts(m, row, rfirst, rbase, rstep);
    if (nparts <= 1) continue;  // written directly by the decode kernel
    auto rowq = [&](int q) -> long long { return q == 0 ? rfirst : rbase + q * rstep; };
    // One round trip for the statistics (lane q holds part q) and the first
    // kPre parts' rows; the rest stream kPre at a time.
    constexpr int kPre = kMergePre;
    float2 st = make_float2(-INFINITY, 0.f);
    if (lane < nparts) st = __ldcg(&m.ws_ml[rowq(lane)]);
    float pre[kPre][PER];
#pragma unroll
    for (int q = 0; q < kPre; ++q)
#pragma unroll
      for (int i = 0; i < PER; ++i)
        pre[q][i] = q < nparts ? __ldcg(m.ws_o + rowq(q) * D + lane + 32 * i) : 0.f;
    float M = st.x;
    for (int q = lane + 32; q < nparts; q += 32) M = fmaxf(M, __ldcg(&m.ws_ml[rowq(q)]).x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float wl = st.x == -INFINITY ? 0.f : fast_exp2(st.x - M);  // weight of part `lane`
    float L = wl * st.y;
    for (int q = lane + 32; q < nparts; q += 32) {
      const float2 v = __ldcg(&m.ws_ml[rowq(q)]);
      L += v.x == -INFINITY ? 0.f : fast_exp2(v.x - M) * v.y;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    const float inv = L > 0.f ? 1.f / L : 0.f;
    float acc[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = 0.f;
#pragma unroll
    for (int q = 0; q < kPre; ++q) {
      const float w = __shfl_sync(0xffffffffu, wl, q);  // zero for q >= nparts
#pragma unroll
      for (int i = 0; i < PER; ++i) acc[i] += w * pre[q][i];
    }
    for (int q0 = kPre; q0 < nparts; q0 += kPre) {  // kPre parts in flight at a time
      float mv[kPre], ov[kPre][PER];
#pragma unroll
      for (int q = 0; q < kPre; ++q) {
        const bool in = q0 + q < nparts;
        const long long r = rowq(in ? q0 + q : 0);
        mv[q] = in ? __ldcg(&m.ws_ml[r]).x : -INFINITY;
#pragma unroll
        for (int i = 0; i < PER; ++i) ov[q][i] = in ? __ldcg(m.ws_o + r * D + lane + 32 * i) : 0.f;
      }
#pragma unroll
      for (int q = 0; q < kPre; ++q) {
        const float w = mv[q] == -INFINITY ? 0.f : fast_exp2(mv[q] - M);
#pragma unroll
        for (int i = 0; i < PER; ++i) acc[i] += w * ov[q][i];
      }
    }
#pragma unroll
    for (int i = 0; i < PER; ++i)
      m.out[(int64_t)row * D + lane + 32 * i] = __float2bfloat16_rn(acc[i] * inv);
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

// The pool as rows of D elements of eb bytes (num_blocks * n_kv * bs rows);
// a box is `box_rows` rows of 128 bytes (the swizzle span): 64 bf16 columns
// or 128 fp8 codes. For bf16 with D = 128 a 3-D view (64 columns, rows, 2
// halves 128 bytes apart) lets one copy fetch both halves of the rows;
// *map3d says which view was built.
static pa_status encode_pool_map(CUtensorMap* map, const void* pool, int D, int eb,
                                 int64_t rows, int box_rows, bool try3d, int* map3d);

// Encoding a tensor map costs host time on every call; a decode loop reuses
// the same pools, so keep the last few per thread.
pa_status make_pool_map(CUtensorMap* map, const void* pool, int D, int eb, int64_t rows,
                        int box_rows, bool try3d, int* map3d) {
  struct Entry {
    const void* pool;
    int D, eb, box_rows, try3d, map3d;
    int64_t rows;
    CUtensorMap map;
  };
  static thread_local Entry cache[8];
  static thread_local int used = 0, next = 0;
  for (int i = 0; i < used; ++i) {
    const Entry& e = cache[i];
    if (e.pool == pool && e.D == D && e.eb == eb && e.rows == rows &&
        e.box_rows == box_rows && e.try3d == (int)try3d) {
      *map = e.map;
      *map3d = e.map3d;
      return PA_OK;
    }
  }
  pa_status st = encode_pool_map(map, pool, D, eb, rows, box_rows, try3d, map3d);
  if (st != PA_OK) return st;
  Entry& e = cache[next];
  e.pool = pool;
  e.D = D;
  e.eb = eb;
  e.rows = rows;
  e.box_rows = box_rows;
  e.try3d = (int)try3d;
  e.map3d = *map3d;
  e.map = *map;
  next = (next + 1) % 8;
  if (used < 8) ++used;
  return PA_OK;
}

static pa_status encode_pool_map(CUtensorMap* map, const void* pool, int D, int eb,
                                 int64_t rows, int box_rows, bool try3d, int* map3d) {
  auto fn = encode_fn();
  if (!fn) return cuda_fail_msg("pa_decode", "cuTensorMapEncodeTiled unavailable");
  if (eb == 1) {  // fp8 codes: one 128-byte row per token and head
    cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)D};
    cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(pool), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cuda_fail_msg("pa_decode", "cuTensorMapEncodeTiled failed");
    *map3d = 0;
    return PA_OK;
  }
  if (try3d && D == 128) {
    cuuint64_t dims[3] = {64, (cuuint64_t)rows, 2};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, 128};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(pool), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r == CUDA_SUCCESS) {
      *map3d = 1;
      return PA_OK;
    }
  }
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(pool), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail_msg("pa_decode", "cuTensorMapEncodeTiled failed");
  *map3d = 0;
  return PA_OK;
}

// FP8: E4M3 pools, balanced split only (a.balanced must be 1).
template <int D, int BS, int NT, bool FP8 = false>
static pa_status launch(DecodeArgs a, const void* k_pool, const void* v_pool,
                        int64_t items_upper, cudaStream_t stream) {
  using C = Cfg<D, BS, NT>;
  auto kern = decode_kernel<D, BS, NT>;
  const int64_t rows = (int64_t)a.num_blocks * a.n_kv * BS;
  constexpr int EB = FP8 ? 1 : 2;
  CUtensorMap tmk, tmv;
  int k3 = 0, v3 = 0;
  pa_status st = make_pool_map(&tmk, k_pool, D, EB, rows, C::ROWS, !FP8, &k3);
  if (st != PA_OK) return st;
  st = make_pool_map(&tmv, v_pool, D, EB, rows, C::ROWS, k3 == 1, &v3);
  if (st != PA_OK) return st;
  if (k3 != v3) {  // both views must agree
    st = make_pool_map(&tmk, k_pool, D, EB, rows, C::ROWS, false, &k3);
    if (st != PA_OK) return st;
  }
  a.map3d = k3 && v3;

  // Allow the dynamic shared memory and find the CTAs per SM, once per
  // (kernel, size).
  auto prepare = [](auto fn, size_t smem, int* configured, int* occ_cache, int* occ) {
    if ((int)smem > *configured) {
      cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
      if (e != cudaSuccess) return cuda_fail("pa_decode smem attribute", e);
      *configured = (int)smem;
    }
    if (occ_cache[0] == (int)smem) {
      *occ = occ_cache[1];
      return PA_OK;
    }
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, fn, kThreads, smem);
    if (e != cudaSuccess) return cuda_fail("pa_decode occupancy", e);
    if (*occ < 1) return cuda_fail_msg("pa_decode", "kernel does not fit on an SM");
    occ_cache[0] = (int)smem;
    occ_cache[1] = *occ;
    return PA_OK;
  };
  static int cfg_item = 0, cfg_split = 0;
  static int occ_item[2] = {-1, 0}, occ_split[2] = {-1, 0};
  auto skern = split_kernel<D, BS, NT, FP8>;
  const size_t smem = a.balanced ? SplitCfg<D, BS, NT, FP8>::smem_bytes(a.num_seqs)
                                 : C::smem_bytes(a.num_seqs, a.group);
  int occ = 0;
  st = a.balanced ? prepare(skern, smem, &cfg_split, occ_split, &occ)
                  : prepare(kern, smem, &cfg_item, occ_item, &occ);
  if (st != PA_OK) return st;
  int64_t grid = (int64_t)num_sms() * occ;
  if (!a.balanced && grid > items_upper) grid = items_upper;
  if (grid > kMaxGrid) grid = kMaxGrid;
  if (grid < 1) grid = 1;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = a.balanced ? cudaLaunchKernelEx(&cfg, skern, tmk, tmv, a)
                              : cudaLaunchKernelEx(&cfg, kern, tmk, tmv, a);
  if (e != cudaSuccess) return cuda_fail("pa_decode launch", e);
  if (a.balanced || a.max_parts > 1) {
    MergeArgs m;
    m.out = a.out;
    m.ws_o = a.ws_o;
    m.ws_ml = a.ws_ml;
    m.seq_lens = a.seq_lens;
    m.pair_info = a.pair_info;
    m.n_kv = a.n_kv;
    m.group = a.group;
    m.balanced = a.balanced;
    m.num_seqs = a.num_seqs;
    m.n_q = a.n_q;
    m.part_tokens = a.part_tokens;
    m.max_parts = a.max_parts;
    m.len_cap = a.len_cap;
    const int64_t rows = (int64_t)a.num_seqs * a.n_q;
    // Few rows (up to two per SM): a CTA per row, so that a row cut into many
    // parts is merged by eight warps; otherwise a warp per row.
    m.coop = rows <= (long long)kCoopRowsPerSm * num_sms();
    int64_t mgrid = m.coop ? rows : (rows + kMergeWarps - 1) / kMergeWarps;
    const int64_t mcap = (int64_t)num_sms() * 8;
    if (!m.coop && mgrid > mcap) mgrid = mcap;
    cudaLaunchConfig_t mc = {};
    mc.gridDim = dim3((unsigned)mgrid);
    mc.blockDim = dim3(kMergeWarps * 32);
    mc.dynamicSmemBytes = 0;
    mc.stream = stream;
    mc.attrs = attr;
    mc.numAttrs = 1;
    e = cudaLaunchKernelEx(&mc, merge_kernel<D>, m);
    if (e != cudaSuccess) return cuda_fail("pa_decode merge launch", e);
  }
  return PA_OK;
}

template <int D, int BS, bool FP8>
static pa_status dispatch_nt(const DecodeArgs& a, const void* kp, const void* vp, int64_t ub,
                             cudaStream_t st) {
  if (a.group <= 8) return launch<D, BS, 1, FP8>(a, kp, vp, ub, st);
  return launch<D, BS, 2, FP8>(a, kp, vp, ub, st);
}

template <int D, bool FP8 = false>
static pa_status dispatch_bs(int bs, const DecodeArgs& a, const void* kp, const void* vp,
                             int64_t ub, cudaStream_t st) {
  switch (bs) {
    case 8: return dispatch_nt<D, 8, FP8>(a, kp, vp, ub, st);
    case 16: return dispatch_nt<D, 16, FP8>(a, kp, vp, ub, st);
    default: return dispatch_nt<D, 32, FP8>(a, kp, vp, ub, st);
  }
}

// Partition size: explicit (a multiple of the 16-token unit, at most 2048:
// fixed partitions, dynamically scheduled), or 0 for the balanced split
// (every CTA gets the same number of units of the whole batch).
static int resolve_partition(int num_seqs, int n_kv, int block_size, int max_seq_len,
                             int partition_tokens) {
  (void)num_seqs;
  (void)n_kv;
  (void)block_size;
  (void)max_seq_len;
  if (partition_tokens == 0) return 0;
  if (partition_tokens < kUnit || partition_tokens % kUnit != 0 ||
      partition_tokens > kMaxUnitsPerPart * kUnit)
    return -1;
  return partition_tokens;
}

struct WsLayout {
  size_t o_off, ml_off, work_off, tick_off, total;
  int max_parts;
};

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

static bool layout(int num_seqs, int n_q, int n_kv, int D, int P, int max_seq_len, WsLayout* w) {
  size_t rows;
  if (P == 0) {  // balanced split: two partial slots per worker (warp)
    w->max_parts = 0;
    rows = (size_t)kMaxWorkers * 2 * (n_q / n_kv);
    // the unit stream must be addressable: num_seqs * units per sequence
    if ((int64_t)num_seqs * (((int64_t)max_seq_len + kUnit - 1) / kUnit) >= ((int64_t)1 << 31))
      return false;
  } else {
    const int64_t mp = max_seq_len <= 0 ? 1 : ((int64_t)max_seq_len + P - 1) / P;
    if (mp > kMaxParts) return false;
    w->max_parts = (int)mp;
    rows = (size_t)num_seqs * n_q * mp;
  }
  w->o_off = 0;
  w->ml_off = align256(rows * D * sizeof(float));
  w->work_off = w->ml_off + align256(rows * sizeof(float2));
  w->tick_off = w->work_off + 256;
  w->total = w->tick_off + (P == 0 ? align256((size_t)num_seqs * n_kv * sizeof(int4)) : 0);
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
  if (P < 0) return 0;
  WsLayout w;
  if (!layout(num_seqs, n_q_heads, n_kv_heads, head_dim, P, max_seq_len, &w)) return 0;
  return w.total;
}

namespace pa {

// Checks and launch shared by pa_decode and pa_decode_fp8 (fp8: E4M3 pools,
// head_dim 128, balanced split; the K scale joins the softmax scale).
static pa_status decode_common(void* out, const void* q, const void* k_pool, const void* v_pool,
                               const int32_t* block_tables, const int32_t* seq_lens,
                               int num_seqs, int max_blocks_per_seq, int num_blocks,
                               int n_q_heads, int n_kv_heads, int head_dim, int block_size,
                               float scale, int partition_tokens, int max_seq_len,
                               void* workspace, size_t workspace_bytes, int32_t* err_word,
                               pa_stream_t stream, bool fp8, float k_scale, float v_scale,
                               bool clear_counters = false) {
  if (fp8 && head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (fp8 && !(k_scale > 0.f && v_scale > 0.f && k_scale < INFINITY && v_scale < INFINITY))
    return PA_ERR_INVALID_ARG;
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
  if (P < 0) return PA_ERR_UNSUPPORTED;
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
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (clear_counters) {
    // A workspace shared with earlier calls: its work counters and pair
    // descriptors must start at zero. Every check above has passed, so a
    // call that is refused launches nothing.
    cudaError_t e = cudaMemsetAsync(static_cast<uint8_t*>(workspace) + w.work_off, 0,
                                    w.total - w.work_off, st);
    if (e != cudaSuccess) return cuda_fail("pa_decode_noalloc memset", e);
  }

  DecodeArgs a;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.block_tables = block_tables;
  a.seq_lens = seq_lens;
  a.ws_o = reinterpret_cast<float*>(ws + w.o_off);
  a.ws_ml = reinterpret_cast<float2*>(ws + w.ml_off);
  a.work = reinterpret_cast<int32_t*>(ws + w.work_off);
  a.pair_info = reinterpret_cast<int4*>(ws + w.tick_off);
  a.balanced = P == 0;
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
  a.scale_log2 = scale * (fp8 ? k_scale : 1.f) * kLog2e;
  a.v_scale = fp8 ? v_scale : 1.f;
  a.map3d = 0;
  const int64_t items_upper = (int64_t)num_seqs * n_kv_heads * (w.max_parts > 0 ? w.max_parts : 1);
  if (fp8) return dispatch_bs<128, true>(block_size, a, k_pool, v_pool, items_upper, st);
  if (head_dim == 64) return dispatch_bs<64>(block_size, a, k_pool, v_pool, items_upper, st);
  return dispatch_bs<128>(block_size, a, k_pool, v_pool, items_upper, st);
}

}  // namespace pa

extern "C" pa_status pa_decode(void* out, const void* q, const void* k_pool, const void* v_pool,
                               const int32_t* block_tables, const int32_t* seq_lens,
                               int num_seqs, int max_blocks_per_seq, int num_blocks,
                               int n_q_heads, int n_kv_heads, int head_dim, int block_size,
                               float scale, int partition_tokens, int max_seq_len,
                               void* workspace, size_t workspace_bytes, int32_t* err_word,
                               pa_stream_t stream) {
  return decode_common(out, q, k_pool, v_pool, block_tables, seq_lens, num_seqs,
                       max_blocks_per_seq, num_blocks, n_q_heads, n_kv_heads, head_dim,
                       block_size, scale, partition_tokens, max_seq_len, workspace,
                       workspace_bytes, err_word, stream, false, 1.f, 1.f);
}

extern "C" pa_status pa_decode_fp8(void* out, const void* q, const void* k_pool,
                                   const void* v_pool, const int32_t* block_tables,
                                   const int32_t* seq_lens, int num_seqs,
                                   int max_blocks_per_seq, int num_blocks, int n_q_heads,
                                   int n_kv_heads, int head_dim, int block_size, float scale,
                                   float k_scale, float v_scale, int max_seq_len,
                                   void* workspace, size_t workspace_bytes, int32_t* err_word,
                                   pa_stream_t stream) {
  return decode_common(out, q, k_pool, v_pool, block_tables, seq_lens, num_seqs,
                       max_blocks_per_seq, num_blocks, n_q_heads, n_kv_heads, head_dim,
                       block_size, scale, 0, max_seq_len, workspace, workspace_bytes, err_word,
                       stream, true, k_scale, v_scale);
}

// ------------------------------------------------------------------ no-alloc

namespace pa {

// Scratch of pa_decode_noalloc: a fixed array in device memory that exists on
// every GPU that loads this library, from module load until the process
// exits. Host code must not use its name as an address; the device address is
// looked up once per device below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch in the calling thread's current
// context. The address belongs to a context, not to a device index: it is
// looked up (cudaGetSymbolAddress, with that context current) on the first
// call from each context and cached under the context's process-unique id,
// so that a context made after a device reset, or one the caller created
// itself, gets its own lookup instead of a stale address. nullptr on failure.
static void* noalloc_scratch(pa_status* st) {
  static std::mutex mu;
  static PFN_cuCtxGetCurrent_v4000 get_ctx = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_ctx = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  if (!get_ctx || !get_id) {
    *st = cuda_fail_msg("pa_decode_noalloc", "context queries unavailable");
    return nullptr;
  }
  // The context the kernel will run in. Without a current context the
  // runtime makes the device's primary context current on its first call;
  // the symbol lookup below is such a call, so look the context up after it.
  auto current_id = [&](unsigned long long* id) {
    CUcontext ctx = nullptr;
    if (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
  };
  constexpr int kSlots = 64;
  static unsigned long long ids[kSlots];
  static void* addrs[kSlots];
  static int used = 0, next = 0;
  std::lock_guard<std::mutex> lock(mu);
  unsigned long long id = 0;
  if (current_id(&id))
    for (int i = 0; i < used; ++i)
      if (ids[i] == id) return addrs[i];
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess || p == nullptr) {
    *st = cuda_fail("pa_decode_noalloc cudaGetSymbolAddress", e);
    return nullptr;
  }
  if (current_id(&id)) {  // cache it (the oldest entry gives way when full)
    const int i = used < kSlots ? used++ : (next++ % kSlots);
    ids[i] = id;
    addrs[i] = p;
  }
  return p;
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
  // The array is shared by every call in the process: its counters are
  // cleared on `stream` once every argument check has passed.
  return decode_common(out, q, k_pool, v_pool, block_tables, seq_lens, num_seqs,
                       max_blocks_per_seq, num_blocks, n_q_heads, n_kv_heads, head_dim,
                       block_size, scale, partition_tokens, max_seq_len, scratch,
                       PA_NOALLOC_SCRATCH_BYTES, err_word, stream, false, 1.f, 1.f, true);
}
