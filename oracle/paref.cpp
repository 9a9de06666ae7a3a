// paref — CPU oracle for paged KV-cache decode attention.
//
// TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
// CPU-baseline leg of the benchmark, never by the GPU library. Plain loops,
// fp64 arithmetic, no blocking, no fusion. See paref.h for the contract of
// every function and for the page each one follows.
#include "paref.h"

#include <cmath>
#include <cstring>
#include <vector>

// ---------------------------------------------------------------------------
// Accounting. [P1] "Try It" (three allocators on one length mix) and
// [P1] "Why this eliminates the waste, precisely": a sequence of L tokens
// takes ceil(L / block_size) blocks, so at most block_size - 1 slots are
// empty. [P3] worked example: the same rounding per request, and capacity as
// the pool divided by the mean allocation per request, rounded down.
// ---------------------------------------------------------------------------

extern "C" int paref_blocks_for(int len, int block_size) {
  if (len <= 0) return 0;
  return (len + block_size - 1) / block_size;
}

extern "C" int paref_tail_waste(int len, int block_size) {
  return paref_blocks_for(len, block_size) * block_size - (len > 0 ? len : 0);
}

extern "C" int64_t paref_paged_slots(const int32_t* lens, int n, int block_size) {
  int64_t total = 0;
  for (int i = 0; i < n; ++i)
    total += (int64_t)paref_blocks_for(lens[i], block_size) * block_size;
  return total;
}

extern "C" int64_t paref_used_tokens(const int32_t* lens, int n) {
  int64_t total = 0;
  for (int i = 0; i < n; ++i) total += lens[i];
  return total;
}

extern "C" int64_t paref_naive_slots(int n, int max_len) { return (int64_t)n * max_len; }

extern "C" int64_t paref_capacity(int64_t pool_slots, int64_t alloc_slots, int n) {
  // floor(pool / (alloc / n)) == floor(pool * n / alloc) for positive values.
  if (alloc_slots <= 0 || n <= 0) return 0;
  return (pool_slots * (int64_t)n) / alloc_slots;
}

// ---------------------------------------------------------------------------
// Block allocator. [P1] "Blocks and block tables": a block is taken only when
// the previous one is full. [P2] "Pros": the blocks are uniform, so a plain
// free list serves. [P1] "Sharing: copy-on-write" and [P2] copy-on-write
// diagram: blocks carry a reference count; a writer into a block with count
// above one copies it, points its own table at the copy, and the original's
// count drops by one.
// ---------------------------------------------------------------------------

struct paref_alloc {
  int block_size;
  std::vector<int> refcount;           // per physical block
  std::vector<int32_t> free_stack;     // top of stack = back()
  std::vector<std::vector<int32_t>> tables;
  std::vector<int> lens;
  std::vector<char> alive;
};

extern "C" paref_alloc* paref_alloc_new(int num_blocks, int block_size, const int32_t* free_order) {
  if (num_blocks < 0 || block_size <= 0) return nullptr;
  paref_alloc* a = new paref_alloc;
  a->block_size = block_size;
  a->refcount.assign(num_blocks, 0);
  // free_order[0] must be popped first, so it goes on top of the stack.
  a->free_stack.resize(num_blocks);
  for (int i = 0; i < num_blocks; ++i) {
    int id = free_order ? free_order[i] : i;
    a->free_stack[num_blocks - 1 - i] = id;
  }
  return a;
}

extern "C" void paref_alloc_delete(paref_alloc* a) { delete a; }

extern "C" int paref_alloc_add_seq(paref_alloc* a) {
  a->tables.emplace_back();
  a->lens.push_back(0);
  a->alive.push_back(1);
  return (int)a->tables.size() - 1;
}

static bool seq_ok(const paref_alloc* a, int seq) {
  return seq >= 0 && seq < (int)a->tables.size() && a->alive[seq];
}

extern "C" int paref_alloc_append(paref_alloc* a, int seq, int32_t* slot, int32_t* cow_src,
                                  int32_t* cow_dst) {
  if (!seq_ok(a, seq)) return -2;
  const int bs = a->block_size;
  const int pos = a->lens[seq];
  std::vector<int32_t>& table = a->tables[seq];
  int32_t src = -1, dst = -1;
  if (pos % bs == 0) {
    // The previous block (if any) is full: this token opens a new block.
    if (a->free_stack.empty()) return -1;
    int32_t b = a->free_stack.back();
    a->free_stack.pop_back();
    a->refcount[b] = 1;
    table.push_back(b);
  } else {
    int32_t last = table[pos / bs];
    if (a->refcount[last] > 1) {
      // Copy-on-write: the block is shared, so this writer takes a copy.
      if (a->free_stack.empty()) return -1;
      int32_t b = a->free_stack.back();
      a->free_stack.pop_back();
      a->refcount[last] -= 1;
      a->refcount[b] = 1;
      table[pos / bs] = b;
      src = last;
      dst = b;
    }
  }
  if (slot) *slot = table[pos / bs] * bs + pos % bs;
  if (cow_src) *cow_src = src;
  if (cow_dst) *cow_dst = dst;
  a->lens[seq] = pos + 1;
  return 0;
}

extern "C" int paref_alloc_fork(paref_alloc* a, int seq) {
  if (!seq_ok(a, seq)) return -2;
  std::vector<int32_t> copy = a->tables[seq];
  int len = a->lens[seq];
  for (int32_t b : copy) a->refcount[b] += 1;
  a->tables.push_back(copy);
  a->lens.push_back(len);
  a->alive.push_back(1);
  return (int)a->tables.size() - 1;
}

extern "C" int paref_alloc_free_seq(paref_alloc* a, int seq) {
  if (!seq_ok(a, seq)) return -2;
  std::vector<int32_t>& table = a->tables[seq];
  int returned = 0;
  for (int j = (int)table.size() - 1; j >= 0; --j) {
    int32_t b = table[j];
    a->refcount[b] -= 1;
    if (a->refcount[b] == 0) {
      a->free_stack.push_back(b);
      ++returned;
    }
  }
  table.clear();
  a->lens[seq] = 0;
  a->alive[seq] = 0;
  return returned;
}

// Usage of the live pool ("03 · PagedAttention", Try It: stored tokens over
// allocated slots; "PagedAttention" (mlapandio.dev), closing advice: watch the
// share of the pool in use). A block in use holds as many tokens as the
// furthest any sequence mapping it has written into it; sharers of a block
// hold the same tokens there, since a write into a shared block copies it
// first, so a shared block counts once.
extern "C" void paref_alloc_usage(const paref_alloc* a, int64_t* tokens, int64_t* slots,
                                  int64_t* blocks_in_use) {
  const int bs = a->block_size;
  std::vector<int> fill(a->refcount.size(), 0);
  for (size_t s = 0; s < a->tables.size(); ++s) {
    if (!a->alive[s]) continue;
    const std::vector<int32_t>& t = a->tables[s];
    for (size_t j = 0; j < t.size(); ++j) {
      int64_t in_block = (int64_t)a->lens[s] - (int64_t)j * bs;
      int n = in_block >= bs ? bs : (int)in_block;
      if (n > fill[t[j]]) fill[t[j]] = n;
    }
  }
  int64_t tok = 0, used = 0;
  for (size_t b = 0; b < a->refcount.size(); ++b) {
    if (a->refcount[b] > 0) {
      ++used;
      tok += fill[b];
    }
  }
  if (tokens) *tokens = tok;
  if (slots) *slots = used * bs;
  if (blocks_in_use) *blocks_in_use = used;
}

extern "C" int paref_alloc_num_free(const paref_alloc* a) { return (int)a->free_stack.size(); }
extern "C" int paref_alloc_num_blocks(const paref_alloc* a) { return (int)a->refcount.size(); }

extern "C" int paref_alloc_refcount(const paref_alloc* a, int block) {
  if (block < 0 || block >= (int)a->refcount.size()) return -1;
  return a->refcount[block];
}

extern "C" int paref_alloc_seq_len(const paref_alloc* a, int seq) {
  if (seq < 0 || seq >= (int)a->tables.size()) return -1;
  return a->lens[seq];
}

extern "C" int paref_alloc_seq_nblocks(const paref_alloc* a, int seq) {
  if (seq < 0 || seq >= (int)a->tables.size()) return -1;
  return (int)a->tables[seq].size();
}

extern "C" int paref_alloc_seq_alive(const paref_alloc* a, int seq) {
  if (seq < 0 || seq >= (int)a->tables.size()) return 0;
  return a->alive[seq];
}

extern "C" int paref_alloc_table(const paref_alloc* a, int seq, int32_t* out, int cap) {
  if (seq < 0 || seq >= (int)a->tables.size()) return -1;
  const std::vector<int32_t>& t = a->tables[seq];
  for (int j = 0; j < (int)t.size() && j < cap; ++j) out[j] = t[j];
  return (int)t.size();
}

extern "C" int paref_alloc_free_list(const paref_alloc* a, int32_t* out, int cap) {
  int n = (int)a->free_stack.size();
  for (int i = 0; i < n && i < cap; ++i) out[i] = a->free_stack[n - 1 - i];
  return n;
}

// ---------------------------------------------------------------------------
// Attention in fp64. [P1] "The part the analogy hides: the kernel": the
// kernel takes the block table and gathers K/V from the scattered blocks.
// [P2] decode-step diagram: one query per sequence is scored against every
// cached key. [P2] "Pros": the result is not an approximation, and [P3]:
// same K/V, same output. So this is plain softmax attention over the
// gathered keys, the maximum subtracted before exponentiating.
// ---------------------------------------------------------------------------

static double bf16_to_double(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return (double)f;
}

// One row of attention given already-gathered pointers to each key/value.
static void attend_row(double* out, const uint16_t* q, const std::vector<const uint16_t*>& keys,
                       const std::vector<const uint16_t*>& vals, int head_dim, double scale) {
  const int n = (int)keys.size();
  for (int d = 0; d < head_dim; ++d) out[d] = 0.0;
  if (n == 0) return;
  std::vector<double> x(n);
  for (int i = 0; i < n; ++i) {
    double dot = 0.0;
    for (int d = 0; d < head_dim; ++d) dot += bf16_to_double(q[d]) * bf16_to_double(keys[i][d]);
    x[i] = scale * dot;
  }
  double m = x[0];
  for (int i = 1; i < n; ++i)
    if (x[i] > m) m = x[i];
  double denom = 0.0;
  std::vector<double> w(n);
  for (int i = 0; i < n; ++i) {
    w[i] = std::exp(x[i] - m);
    denom += w[i];
  }
  for (int i = 0; i < n; ++i) {
    const double wi = w[i] / denom;
    for (int d = 0; d < head_dim; ++d) out[d] += wi * bf16_to_double(vals[i][d]);
  }
}

extern "C" int paref_attention_paged(double* out, const uint16_t* q, const uint16_t* k_pool,
                                     const uint16_t* v_pool, const int32_t* block_tables,
                                     const int32_t* seq_lens, int num_seqs, int max_blocks,
                                     int num_blocks, int n_q_heads, int n_kv_heads, int head_dim,
                                     int block_size, double scale, const int32_t* rows,
                                     int n_rows) {
  if (n_kv_heads <= 0 || n_q_heads % n_kv_heads != 0) return -1;
  const int group = n_q_heads / n_kv_heads;
  const int total = rows ? n_rows : num_seqs * n_q_heads;
  for (int r = 0; r < total; ++r) {
    const int s = rows ? rows[2 * r] : r / n_q_heads;
    const int h = rows ? rows[2 * r + 1] : r % n_q_heads;
    if (s < 0 || s >= num_seqs || h < 0 || h >= n_q_heads) return -1;
    const int len = seq_lens[s];
    if (len < 0 || (int64_t)len > (int64_t)max_blocks * block_size) return -1;
    const int g = h / group;
    std::vector<const uint16_t*> keys(len), vals(len);
    for (int i = 0; i < len; ++i) {
      const int32_t phys = block_tables[(int64_t)s * max_blocks + i / block_size];
      if (phys < 0 || phys >= num_blocks) return -1;
      const int64_t off =
          (((int64_t)phys * n_kv_heads + g) * block_size + i % block_size) * head_dim;
      keys[i] = k_pool + off;
      vals[i] = v_pool + off;
    }
    attend_row(out + (int64_t)r * head_dim, q + ((int64_t)s * n_q_heads + h) * head_dim, keys,
               vals, head_dim, scale);
  }
  return 0;
}

extern "C" int paref_prefill_paged(double* out, const uint16_t* q, const uint16_t* k_pool,
                                   const uint16_t* v_pool, const int32_t* block_tables,
                                   const int32_t* seq_lens, const int32_t* cu_q, int num_seqs,
                                   int max_blocks, int num_blocks, int n_q_heads, int n_kv_heads,
                                   int head_dim, int block_size, double scale,
                                   const int32_t* rows, int n_rows) {
  if (n_kv_heads <= 0 || n_q_heads % n_kv_heads != 0 || num_seqs < 0) return -1;
  const int group = n_q_heads / n_kv_heads;
  const int total_q = num_seqs > 0 ? cu_q[num_seqs] : 0;
  const int64_t total = rows ? n_rows : (int64_t)total_q * n_q_heads;
  for (int64_t r = 0; r < total; ++r) {
    const int row = rows ? rows[2 * r] : (int)(r / n_q_heads);
    const int h = rows ? rows[2 * r + 1] : (int)(r % n_q_heads);
    if (row < 0 || row >= total_q || h < 0 || h >= n_q_heads) return -1;
    int s = 0;  // the sequence whose chunk holds this query row
    while (s + 1 < num_seqs && cu_q[s + 1] <= row) ++s;
    const int c = cu_q[s + 1] - cu_q[s];
    const int len = seq_lens[s];
    if (c < 0 || len < c || (int64_t)len > (int64_t)max_blocks * block_size) return -1;
    const int pos = len - c + (row - cu_q[s]);  // this query token's position
    const int g = h / group;
    std::vector<const uint16_t*> keys(pos + 1), vals(pos + 1);
    for (int j = 0; j <= pos; ++j) {
      const int32_t phys = block_tables[(int64_t)s * max_blocks + j / block_size];
      if (phys < 0 || phys >= num_blocks) return -1;
      const int64_t off =
          (((int64_t)phys * n_kv_heads + g) * block_size + j % block_size) * head_dim;
      keys[j] = k_pool + off;
      vals[j] = v_pool + off;
    }
    attend_row(out + r * head_dim, q + ((int64_t)row * n_q_heads + h) * head_dim, keys, vals,
               head_dim, scale);
  }
  return 0;
}

extern "C" int paref_attention_contiguous(double* out, const uint16_t* q, const uint16_t* k,
                                          const uint16_t* v, int len, int n_q_heads,
                                          int n_kv_heads, int head_dim, double scale) {
  if (n_kv_heads <= 0 || n_q_heads % n_kv_heads != 0 || len < 0) return -1;
  const int group = n_q_heads / n_kv_heads;
  for (int h = 0; h < n_q_heads; ++h) {
    const int g = h / group;
    double* o = out + (int64_t)h * head_dim;
    for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
    if (len == 0) continue;
    // Scores, then a max-subtracted softmax, written out a second time on
    // purpose (no helper shared with the paged routine).
    std::vector<double> x(len);
    for (int i = 0; i < len; ++i) {
      const uint16_t* key = k + ((int64_t)i * n_kv_heads + g) * head_dim;
      double dot = 0.0;
      for (int d = 0; d < head_dim; ++d)
        dot += bf16_to_double(q[(int64_t)h * head_dim + d]) * bf16_to_double(key[d]);
      x[i] = scale * dot;
    }
    double m = x[0];
    for (int i = 1; i < len; ++i) m = x[i] > m ? x[i] : m;
    double denom = 0.0;
    for (int i = 0; i < len; ++i) denom += std::exp(x[i] - m);
    for (int i = 0; i < len; ++i) {
      const double wi = std::exp(x[i] - m) / denom;
      const uint16_t* val = v + ((int64_t)i * n_kv_heads + g) * head_dim;
      for (int d = 0; d < head_dim; ++d) o[d] += wi * bf16_to_double(val[d]);
    }
  }
  return 0;
}

// ---------------------------------------------------------------------------
// Cache writes. [P2] decode-step diagram: the new K and V are written into
// the sequence's current block. [P2] copy-on-write diagram: the runtime
// copies the shared block, then writes.
// ---------------------------------------------------------------------------

extern "C" int paref_reshape_and_cache(const uint16_t* k, const uint16_t* v, uint16_t* k_pool,
                                       uint16_t* v_pool, const int32_t* slot_mapping,
                                       int num_tokens, int num_blocks, int n_kv_heads,
                                       int head_dim, int block_size) {
  int skipped = 0;
  for (int t = 0; t < num_tokens; ++t) {
    const int32_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if ((int64_t)slot >= (int64_t)num_blocks * block_size) {
      ++skipped;
      continue;
    }
    const int32_t blk = slot / block_size;
    const int32_t off = slot % block_size;
    for (int h = 0; h < n_kv_heads; ++h) {
      const int64_t dst = (((int64_t)blk * n_kv_heads + h) * block_size + off) * head_dim;
      const int64_t src = ((int64_t)t * n_kv_heads + h) * head_dim;
      for (int d = 0; d < head_dim; ++d) {
        k_pool[dst + d] = k[src + d];
        v_pool[dst + d] = v[src + d];
      }
    }
  }
  return skipped;
}

extern "C" int paref_copy_blocks(uint16_t* k_pool, uint16_t* v_pool, const int32_t* pairs,
                                 int n_pairs, int n_kv_heads, int head_dim, int block_size,
                                 int num_blocks) {
  int skipped = 0;
  const int64_t block_elems = (int64_t)n_kv_heads * block_size * head_dim;
  for (int p = 0; p < n_pairs; ++p) {
    const int32_t src = pairs[2 * p], dst = pairs[2 * p + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
      ++skipped;
      continue;
    }
    for (int64_t e = 0; e < block_elems; ++e) {
      k_pool[dst * block_elems + e] = k_pool[src * block_elems + e];
      v_pool[dst * block_elems + e] = v_pool[src * block_elems + e];
    }
  }
  return skipped;
}

extern "C" int paref_swap_blocks(uint8_t* dst_k, uint8_t* dst_v, const uint8_t* src_k,
                                 const uint8_t* src_v, const int32_t* pairs, int n_pairs,
                                 int64_t block_bytes, int src_num_blocks, int dst_num_blocks) {
  int skipped = 0;
  for (int p = 0; p < n_pairs; ++p) {
    const int32_t src = pairs[2 * p], dst = pairs[2 * p + 1];
    if (src < 0 || src >= src_num_blocks || dst < 0 || dst >= dst_num_blocks) {
      ++skipped;
      continue;
    }
    for (int64_t b = 0; b < block_bytes; ++b) {
      dst_k[dst * block_bytes + b] = src_k[src * block_bytes + b];
      dst_v[dst * block_bytes + b] = src_v[src * block_bytes + b];
    }
  }
  return skipped;
}

// ---------------------------------------------------------------------------
// FP8 E4M3 (OCP FP8 formats): sign, 4 exponent bits with bias 7, 3 mantissa
// bits. Exponent field 0 is subnormal (value m * 2^-9); the all-ones
// exponent with all-ones mantissa is NaN; there is no infinity, so the
// largest finite value is 1.75 * 2^8 = 448.
// ---------------------------------------------------------------------------

extern "C" double paref_e4m3_decode(uint8_t code) {
  const int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) return std::nan("");
  double mag = e == 0 ? std::ldexp((double)m, -9) : std::ldexp(1.0 + m / 8.0, e - 7);
  return sign ? -mag : mag;
}

// Round a non-negative double to the nearest integer, ties to even.
static double round_half_even(double v) {
  double f = std::floor(v);
  double diff = v - f;
  if (diff > 0.5) return f + 1.0;
  if (diff < 0.5) return f;
  return std::fmod(f, 2.0) == 0.0 ? f : f + 1.0;
}

extern "C" uint8_t paref_e4m3_encode(double x) {
  if (std::isnan(x)) return 0x7F;
  const uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
  double a = std::fabs(x);
  if (a >= 448.0) return sign | 0x7E;  // saturate
  if (a < std::ldexp(1.0, -6)) {
    // subnormal range: multiples of 2^-9; 8 * 2^-9 is the smallest normal
    const int m = (int)round_half_even(std::ldexp(a, 9));
    return sign | (uint8_t)m;  // m == 8 encodes exponent 1, mantissa 0
  }
  int e = (int)std::floor(std::log2(a));
  if (std::ldexp(1.0, e) > a) --e;        // guard log2 rounding
  if (std::ldexp(1.0, e + 1) <= a) ++e;
  int m = (int)round_half_even((std::ldexp(a, -e) - 1.0) * 8.0);
  if (m == 8) {
    m = 0;
    ++e;
  }
  if (e > 8 || (e == 8 && m == 7)) return sign | 0x7E;  // rounded past 448
  return sign | (uint8_t)(((e + 7) << 3) | m);
}

extern "C" int paref_reshape_and_cache_fp8(const uint16_t* k, const uint16_t* v, uint8_t* k_pool,
                                           uint8_t* v_pool, const int32_t* slot_mapping,
                                           int num_tokens, int num_blocks, int n_kv_heads,
                                           int head_dim, int block_size, float k_scale,
                                           float v_scale) {
  int skipped = 0;
  for (int t = 0; t < num_tokens; ++t) {
    const int32_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if ((int64_t)slot >= (int64_t)num_blocks * block_size) {
      ++skipped;
      continue;
    }
    const int32_t blk = slot / block_size, off = slot % block_size;
    for (int h = 0; h < n_kv_heads; ++h) {
      const int64_t dst = (((int64_t)blk * n_kv_heads + h) * block_size + off) * head_dim;
      const int64_t src = ((int64_t)t * n_kv_heads + h) * head_dim;
      for (int d = 0; d < head_dim; ++d) {
        const float kq = (float)bf16_to_double(k[src + d]) / k_scale;  // fp32 division
        const float vq = (float)bf16_to_double(v[src + d]) / v_scale;
        k_pool[dst + d] = paref_e4m3_encode(kq);
        v_pool[dst + d] = paref_e4m3_encode(vq);
      }
    }
  }
  return skipped;
}

extern "C" int paref_attention_paged_fp8(double* out, const uint16_t* q, const uint8_t* k_pool,
                                         const uint8_t* v_pool, const int32_t* block_tables,
                                         const int32_t* seq_lens, int num_seqs, int max_blocks,
                                         int num_blocks, int n_q_heads, int n_kv_heads,
                                         int head_dim, int block_size, double scale,
                                         double k_scale, double v_scale, const int32_t* rows,
                                         int n_rows) {
  if (n_kv_heads <= 0 || n_q_heads % n_kv_heads != 0) return -1;
  const int group = n_q_heads / n_kv_heads;
  const int total = rows ? n_rows : num_seqs * n_q_heads;
  for (int r = 0; r < total; ++r) {
    const int s = rows ? rows[2 * r] : r / n_q_heads;
    const int h = rows ? rows[2 * r + 1] : r % n_q_heads;
    if (s < 0 || s >= num_seqs || h < 0 || h >= n_q_heads) return -1;
    const int len = seq_lens[s];
    if (len < 0 || (int64_t)len > (int64_t)max_blocks * block_size) return -1;
    const int g = h / group;
    double* o = out + (int64_t)r * head_dim;
    for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
    if (len == 0) continue;
    const uint16_t* qr = q + ((int64_t)s * n_q_heads + h) * head_dim;
    std::vector<double> x(len);
    std::vector<int64_t> off(len);
    for (int i = 0; i < len; ++i) {
      const int32_t phys = block_tables[(int64_t)s * max_blocks + i / block_size];
      if (phys < 0 || phys >= num_blocks) return -1;
      off[i] = (((int64_t)phys * n_kv_heads + g) * block_size + i % block_size) * head_dim;
      double dot = 0.0;
      for (int d = 0; d < head_dim; ++d)
        dot += bf16_to_double(qr[d]) * (paref_e4m3_decode(k_pool[off[i] + d]) * k_scale);
      x[i] = scale * dot;
    }
    double m = x[0];
    for (int i = 1; i < len; ++i) m = x[i] > m ? x[i] : m;
    double denom = 0.0;
    for (int i = 0; i < len; ++i) denom += std::exp(x[i] - m);
    for (int i = 0; i < len; ++i) {
      const double w = std::exp(x[i] - m) / denom;
      for (int d = 0; d < head_dim; ++d)
        o[d] += w * (paref_e4m3_decode(v_pool[off[i] + d]) * v_scale);
    }
  }
  return 0;
}
