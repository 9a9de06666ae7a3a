/*
 * paref — the CPU oracle for paged KV-cache decode attention.
 *
 * TEST INFRASTRUCTURE ONLY. This library is the plain, slow, obviously
 * correct statement of what the GPU path computes. Only the test suite,
 * the smoke check and the CPU-baseline leg of the benchmark load it. It
 * shares no code, header or table with the CUDA library, and the CUDA
 * library never calls it.
 *
 * Sources (web pages on PagedAttention):
 *   [P1] "03 · PagedAttention" (sunilkunchoor.github.io)
 *   [P2] "PagedAttention" (mlapandio.dev, daily terms)
 *   [P3] "paged-attention" course lesson (tbash.cc), the worked example
 *   [P4] "Serving: vLLM and PagedAttention" (henryfzh-note.com)
 *
 * Conventions the pages leave open (each is a stated reading):
 *   - pool layout  k_pool/v_pool[num_blocks][n_kv_heads][block_size][head_dim],
 *     bf16 stored as raw uint16 bit patterns;
 *   - kv head of query head h is h / (n_q_heads / n_kv_heads);
 *   - slot = physical_block * block_size + (position mod block_size);
 *   - block tables int32 [num_seqs][max_blocks_per_seq].
 */
#ifndef PAREF_H
#define PAREF_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------- accounting ([P1] "Try It", [P3] worked example) ------- */

/* blocks a sequence of len tokens occupies: ceil(len / block_size). */
int paref_blocks_for(int len, int block_size);
/* empty slots in the last block: block_size * ceil(len/bs) - len. */
int paref_tail_waste(int len, int block_size);
/* sum over sequences of block_size * ceil(len/bs). */
int64_t paref_paged_slots(const int32_t* lens, int n, int block_size);
/* sum of lengths (tokens actually stored). */
int64_t paref_used_tokens(const int32_t* lens, int n);
/* reserve-max allocation: n * max_len. */
int64_t paref_naive_slots(int n, int max_len);
/* how many requests of the observed mean allocation fit a pool:
   floor(pool_slots / (alloc_slots / n)) computed exactly. */
int64_t paref_capacity(int64_t pool_slots, int64_t alloc_slots, int n);

/* ---------------- block allocator ([P1] "Blocks and block tables",
   "Sharing: copy-on-write"; [P2] copy-on-write diagram, "Pros") -------- */

typedef struct paref_alloc paref_alloc;

/* A pool of num_blocks blocks. free_order (nullable; default 0..n-1) is the
   order in which never-used blocks are handed out: free_order[0] first. */
paref_alloc* paref_alloc_new(int num_blocks, int block_size, const int32_t* free_order);
void paref_alloc_delete(paref_alloc* a);

/* New empty sequence; returns its id (ids are 0, 1, 2, ... in call order). */
int paref_alloc_add_seq(paref_alloc* a);
/* Append one token to seq. On success returns 0 and writes the token's slot.
   If the token starts a new block, one block is popped from the free list.
   If it lands in a block that other sequences share (refcount > 1), the
   block is copied first: a fresh block is popped, (*cow_src,*cow_dst) get
   (old, new) and the table is repointed; otherwise *cow_src = *cow_dst = -1.
   Returns -1 (state unchanged) when a block is needed and none is free,
   -2 for a bad sequence id. */
int paref_alloc_append(paref_alloc* a, int seq, int32_t* slot, int32_t* cow_src, int32_t* cow_dst);
/* New sequence sharing all of seq's blocks (refcount + 1 each); returns id. */
int paref_alloc_fork(paref_alloc* a, int seq);
/* Release seq: every block's refcount drops by one; blocks reaching zero go
   back on the free list, walking the table from its last entry to its first.
   Returns the number of blocks returned to the free list. */
int paref_alloc_free_seq(paref_alloc* a, int seq);

/* Usage of the live pool: *tokens = tokens held, a block in use counting
   the furthest any sequence mapping it has written into it (a shared block
   counts once); *slots = blocks in use * block_size; *blocks_in_use = blocks
   with refcount > 0. Any output pointer may be NULL. */
void paref_alloc_usage(const paref_alloc* a, int64_t* tokens, int64_t* slots,
                       int64_t* blocks_in_use);
int paref_alloc_num_free(const paref_alloc* a);
int paref_alloc_num_blocks(const paref_alloc* a);
int paref_alloc_refcount(const paref_alloc* a, int block);
int paref_alloc_seq_len(const paref_alloc* a, int seq);
int paref_alloc_seq_nblocks(const paref_alloc* a, int seq);
int paref_alloc_seq_alive(const paref_alloc* a, int seq);
/* copy up to cap table entries of seq into out; returns the table length. */
int paref_alloc_table(const paref_alloc* a, int seq, int32_t* out, int cap);
/* copy the free list, next-to-be-popped first; returns its length. */
int paref_alloc_free_list(const paref_alloc* a, int32_t* out, int cap);

/* ---------------- attention in fp64 ([P1] "The part the analogy hides:
   the kernel"; [P2] decode-step diagram; [P3] "same K/V, same output") -- */

/* For each requested (seq, q_head) row r = rows[2i], rows[2i+1] (or every
   row, in (seq, head) order, when rows == NULL):
     x_i = scale * sum_d q[s,h,d] * K_i[d]   for i < seq_lens[s], with
     K_i = k_pool[block_tables[s][i / bs], h / G, i % bs, :]
     w   = softmax(x)
     out[r, :] = sum_i w_i * V_i
   out is [n_rows][head_dim] (rows == NULL: [num_seqs][n_q_heads][head_dim]).
   A row with seq_len == 0 is all zeros. Returns 0, or -1 on a block id
   outside [0, num_blocks) or a length beyond the table. */
int paref_attention_paged(double* out, const uint16_t* q, const uint16_t* k_pool,
                          const uint16_t* v_pool, const int32_t* block_tables,
                          const int32_t* seq_lens, int num_seqs, int max_blocks,
                          int num_blocks, int n_q_heads, int n_kv_heads, int head_dim,
                          int block_size, double scale, const int32_t* rows, int n_rows);

/* The same attention for ONE sequence whose K/V sit contiguously:
   k, v are [len][n_kv_heads][head_dim]; q is [n_q_heads][head_dim];
   out is [n_q_heads][head_dim]. Written separately from the paged routine
   so that "paged equals contiguous" is a check between two codes. */
int paref_attention_contiguous(double* out, const uint16_t* q, const uint16_t* k,
                               const uint16_t* v, int len, int n_q_heads, int n_kv_heads,
                               int head_dim, double scale);

/* ---------------- chunked prefill ("Serving: vLLM and PagedAttention",
   section 2.4, chunked prefill: a prompt is split into chunks that run
   beside decode steps; each chunk's tokens attend, causally, to everything
   cached before them and to the chunk's earlier tokens) ---------------- */

/* Sequence s contributes c_s = cu_q[s+1] - cu_q[s] query tokens (rows
   cu_q[s] .. cu_q[s+1]-1 of q and out, [total_q][n_q_heads][head_dim]),
   which are its LAST c_s tokens: seq_lens[s] counts everything cached,
   the chunk included. Query token i of s sits at position
   p = seq_lens[s] - c_s + i and attends to positions 0..p:
     out[cu_q[s]+i, h, :] = sum_{j<=p} softmax_j(scale * q . K_j) V_j
   with K_j, V_j gathered through the block table as for decode. When
   rows != NULL only the listed (query row, head) pairs are computed, into
   out[n_rows][head_dim]. Returns 0, or -1 on a bad table, length or
   c_s > seq_lens[s]. */
int paref_prefill_paged(double* out, const uint16_t* q, const uint16_t* k_pool,
                        const uint16_t* v_pool, const int32_t* block_tables,
                        const int32_t* seq_lens, const int32_t* cu_q, int num_seqs,
                        int max_blocks, int num_blocks, int n_q_heads, int n_kv_heads,
                        int head_dim, int block_size, double scale, const int32_t* rows,
                        int n_rows);

/* ---------------- cache writes ([P2] decode-step diagram: the new K and V
   go into the current block; copy-on-write diagram: copy, then write) ----- */

/* For token t with slot_mapping[t] >= 0: k_pool[slot/bs, h, slot%bs, :] =
   k[t, h, :] for every kv head h, and the same for v. Negative slots are
   skipped. Returns the number of slots >= num_blocks*bs that were skipped. */
int paref_reshape_and_cache(const uint16_t* k, const uint16_t* v, uint16_t* k_pool,
                            uint16_t* v_pool, const int32_t* slot_mapping, int num_tokens,
                            int num_blocks, int n_kv_heads, int head_dim, int block_size);

/* For each (src, dst) pair: block dst of both pools becomes a copy of block
   src (all kv heads). Returns the number of pairs skipped for an id outside
   [0, num_blocks). */
int paref_copy_blocks(uint16_t* k_pool, uint16_t* v_pool, const int32_t* pairs, int n_pairs,
                      int n_kv_heads, int head_dim, int block_size, int num_blocks);

/* ---------------- swap ("03 · PagedAttention", "Memory management, in
   brief": when memory runs out a sequence can be preempted by swapping its
   blocks out to CPU memory and back in later; "Serving: vLLM and
   PagedAttention", preemption by swapping) ---------------------------- */

/* For each (src, dst) pair: block dst of the destination pools becomes a
   byte copy of block src of the source pools (K and V), where a block is
   block_bytes bytes (n_kv_heads * block_size * head_dim * element size).
   The two sides are different pools (device and host memory in the GPU
   path). Returns the number of pairs skipped for an id outside the source
   or destination pool. */
int paref_swap_blocks(uint8_t* dst_k, uint8_t* dst_v, const uint8_t* src_k, const uint8_t* src_v,
                      const int32_t* pairs, int n_pairs, int64_t block_bytes,
                      int src_num_blocks, int dst_num_blocks);

/* ---------------- FP8 KV cache ("PagedAttention" (mlapandio.dev), Cons and
   honest limits, and "Serving: vLLM and PagedAttention" section 3.1: an fp8
   KV cache halves the cache and the bytes read per step). The format is
   OCP FP8 E4M3 (bias 7, no infinities, 0x7F/0xFF = NaN, max 448); a stored
   code times a per-tensor fp32 scale gives the value. ------------------- */

/* Value of an E4M3 code (NaN for 0x7F / 0xFF). */
double paref_e4m3_decode(uint8_t code);
/* E4M3 code nearest to x (ties to even), saturating to +-448; NaN -> 0x7F. */
uint8_t paref_e4m3_encode(double x);

/* Cache write into fp8 pools: code = e4m3(fp32(k) / k_scale), the division
   in fp32 (round to nearest), likewise for v. Pools are uint8
   [num_blocks][n_kv_heads][block_size][head_dim]. Returns skipped slots. */
int paref_reshape_and_cache_fp8(const uint16_t* k, const uint16_t* v, uint8_t* k_pool,
                                uint8_t* v_pool, const int32_t* slot_mapping, int num_tokens,
                                int num_blocks, int n_kv_heads, int head_dim, int block_size,
                                float k_scale, float v_scale);

/* paref_attention_paged over fp8 pools: K_i = decode(k code) * k_scale,
   V_i = decode(v code) * v_scale, in fp64. */
int paref_attention_paged_fp8(double* out, const uint16_t* q, const uint8_t* k_pool,
                              const uint8_t* v_pool, const int32_t* block_tables,
                              const int32_t* seq_lens, int num_seqs, int max_blocks,
                              int num_blocks, int n_q_heads, int n_kv_heads, int head_dim,
                              int block_size, double scale, double k_scale, double v_scale,
                              const int32_t* rows, int n_rows);

#ifdef __cplusplus
}
#endif

#endif /* PAREF_H */
