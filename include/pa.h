/*
 * pa.h — C ABI of the paged KV-cache decode library (libpa.so, sm_103a).
 *
 * The hot path of one decode step over a paged KV cache, as three calls:
 *   pa_copy_blocks        copy-on-write block duplication
 *   pa_reshape_and_cache  write each new token's K/V into its slot
 *   pa_decode             attention of one query per sequence over its
 *                         cached K/V, gathered through the block table
 * A step issues them in that order on one stream: copy, then write, then
 * attend (the new token attends to itself).
 *
 * Sources (web pages on PagedAttention):
 *   "03 · PagedAttention" (sunilkunchoor.github.io): "Blocks and block
 *     tables", "The part the analogy hides: the kernel", "Sharing:
 *     copy-on-write, straight from fork()".
 *   "PagedAttention" (mlapandio.dev daily terms): definition, the pool and
 *     block-table diagram, "A DECODE STEP" and "COPY-ON-WRITE ON A SHARED
 *     PREFIX" diagrams.
 *   "Serving: vLLM and PagedAttention" (henryfzh-note.com), section 2.2
 *     "Paging: the block table as virtual memory".
 *
 * Data layout (the pages fix only that a block holds block_size consecutive
 * tokens and is reached through a per-sequence table; the rest is this
 * library's convention):
 *   k_pool, v_pool  bf16 [num_blocks][n_kv_heads][block_size][head_dim]:
 *                   one (block, kv head) is a contiguous block_size*head_dim
 *                   run of bf16 (4 KiB at block 16, head_dim 128).
 *   block_tables    int32 [num_seqs][max_blocks_per_seq], row-major; entry j
 *                   of row s is the physical block of tokens
 *                   [j*block_size, (j+1)*block_size) of sequence s.
 *   seq_lens        int32 [num_seqs]: tokens to attend, new token included.
 *   q, out          bf16 [num_seqs][n_q_heads][head_dim].
 *   slot            physical_block * block_size + (position mod block_size).
 *   GQA             query head h reads kv head h / (n_q_heads / n_kv_heads).
 *
 * Ownership and execution: every pointer argument is DEVICE memory owned by
 * the caller (unless stated otherwise); the library keeps no device
 * allocation of its own. Every call is asynchronous on `stream` (0 = legacy
 * default stream) and returns after enqueueing. The return status covers
 * host-side argument checks and launch errors only. Problems only the device
 * can see (a block id or slot outside the pool, a length beyond the table)
 * never trap: the offending access is skipped and a bit is OR-ed into
 * *err_word (a device int32 the caller zeroes and reads; NULL = do not
 * report). Bad data never makes a kernel read or write outside the buffers
 * described by the arguments.
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* pa_stream_t; /* same handle as cudaStream_t */

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer,
                             n_q_heads % n_kv_heads != 0, workspace too small */
  PA_ERR_UNSUPPORTED = 2, /* head_dim not 64/128, block_size not 8/16/32,
                             n_q_heads / n_kv_heads > 16, partition size */
  PA_ERR_CUDA = 3         /* a CUDA runtime/driver call failed; see
                             pa_last_cuda_error() */
} pa_status;

/* Bits OR-ed into *err_word by the kernels. */
#define PA_DEV_ERR_BLOCK_ID 0x1 /* table entry outside [0, num_blocks): its
                                   tokens are treated as absent */
#define PA_DEV_ERR_SLOT 0x2     /* slot >= num_blocks*block_size: not written */
#define PA_DEV_ERR_PAIR 0x4     /* copy pair id outside the pool: skipped */
#define PA_DEV_ERR_SEQ_LEN 0x8  /* seq_len < 0, > max_blocks_per_seq*block_size
                                   or > max_seq_len: clamped into range */
#define PA_DEV_ERR_TIMEOUT 0x10 /* a bounded wait inside a kernel gave up; the
                                   output is undefined and the workspace must
                                   be zeroed again before the next pa_decode */

/* Human-readable name of a status. Never NULL. */
const char* pa_status_string(pa_status s);

/* Text of the last CUDA error seen by this library on the calling thread
   ("" if none). Valid until the next call on that thread. */
const char* pa_last_cuda_error(void);

/*
 * Partition size pa_decode uses, in tokens: `partition_tokens` itself when
 * non-zero (checked: a multiple of 16, at most 2048; a partition may start
 * inside a 32-token block), or 0 for the balanced split chosen by
 * `partition_tokens == 0` (see pa_decode). Returns a negative value for
 * unsupported arguments.
 */
int pa_decode_partition_tokens(int num_seqs, int n_kv_heads, int block_size, int max_seq_len,
                               int partition_tokens);

/*
 * Bytes of device workspace pa_decode needs for these arguments (same
 * meaning as in pa_decode). The workspace holds the split-KV partial
 * results and a few counters. It must be ZEROED before its first use
 * (cudaMemset / torch.zeros); pa_decode leaves it zeroed again when it
 * completes, so one workspace can serve any number of stream-ordered
 * calls. Calls that may run concurrently need separate workspaces.
 * Returns 0 for unsupported arguments.
 */
size_t pa_decode_workspace_bytes(int num_seqs, int n_q_heads, int n_kv_heads, int head_dim,
                                 int block_size, int max_seq_len, int partition_tokens);

/*
 * pa_decode — paged decode attention.
 * Defined by "03 · PagedAttention", "The part the analogy hides: the
 * kernel" (the kernel takes the block table and gathers K/V from scattered
 * blocks during attention) and the "A DECODE STEP" diagram of
 * "PagedAttention" (mlapandio.dev: one launch for the whole batch; each
 * sequence's query is scored against every key in its blocks).
 *
 * For every sequence s and query head h (kv head g = h / G,
 * G = n_q_heads / n_kv_heads), with K_i, V_i the rows of token i < len_s
 * gathered as k_pool[block_tables[s][i / block_size]][g][i % block_size]:
 *   out[s][h] = sum_i softmax_i(scale * <q[s][h], K_i>) * V_i
 * in fp32 arithmetic on bf16 inputs, rounded to bf16 (nearest even).
 * A sequence with len_s == 0 gets zeros.
 *
 * Split-KV: with partition_tokens > 0 every sequence's tokens are cut into
 * partitions of that many tokens, processed in parallel. With
 * partition_tokens == 0 (the default) the 16-token units of all (sequence,
 * kv head) pairs, taken in order, are cut into equal contiguous shares, one
 * per warp of a persistent grid, so every warp streams the same number of
 * bytes whatever the length mix. Either way partial results are merged with a log-sum-exp
 * reduction (the same value as unsplit attention, up to fp32 rounding). The call
 * launches the decode kernel and, when partials need merging, a merge kernel
 * after it. Both are programmatic dependent launches. The decode kernel may
 * start while the preceding kernel on the stream is still running if that
 * kernel signals programmatic completion early (pa_reshape_and_cache does);
 * it then reads q, block_tables and seq_lens right away, and waits for the
 * preceding kernel to complete before it reads the pools or writes anything.
 * So q, block_tables and seq_lens must not be written by a kernel that
 * signals early and directly precedes pa_decode; kernels that do not use
 * programmatic launch are always complete before pa_decode starts.
 *
 *   out                bf16 [num_seqs][n_q_heads][head_dim], 16-B aligned
 *   q                  bf16 [num_seqs][n_q_heads][head_dim], 16-B aligned
 *   k_pool, v_pool     bf16 [num_blocks][n_kv_heads][block_size][head_dim],
 *                      16-B aligned
 *   block_tables       int32 [num_seqs][max_blocks_per_seq]; only the first
 *                      ceil(len_s / block_size) entries of row s are read
 *   seq_lens           int32 [num_seqs]
 *   num_seqs           >= 0 (0: nothing is launched), <= 8192
 *   max_blocks_per_seq >= 1 (row stride of block_tables)
 *   num_blocks         >= 1, num_blocks*n_kv_heads*block_size < 2^31
 *   n_q_heads, n_kv_heads  >= 1, n_q_heads % n_kv_heads == 0, G <= 16
 *   head_dim           64 or 128
 *   block_size         8, 16 or 32
 *   scale              softmax scale (e.g. 1/sqrt(head_dim))
 *   partition_tokens   0 = balanced split, else the partition length (see
 *                      pa_decode_partition_tokens)
 *   max_seq_len        host-side upper bound of seq_lens (sizes the
 *                      workspace); longer sequences are clamped and flagged
 *   workspace          >= pa_decode_workspace_bytes(...) bytes, 256-B
 *                      aligned, zeroed before first use (see above)
 *   err_word           nullable device int32, see PA_DEV_ERR_*
 */
pa_status pa_decode(void* out, const void* q, const void* k_pool, const void* v_pool,
                    const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                    int max_blocks_per_seq, int num_blocks, int n_q_heads, int n_kv_heads,
                    int head_dim, int block_size, float scale, int partition_tokens,
                    int max_seq_len, void* workspace, size_t workspace_bytes,
                    int32_t* err_word, pa_stream_t stream);

/*
 * pa_prefill — chunked-prefill attention over the paged cache.
 * Defined by "Serving: vLLM and PagedAttention", section 2.4 (chunked
 * prefill: a long prompt is processed in chunks that share steps with
 * decodes) together with the paged gather of "03 · PagedAttention", "The
 * part the analogy hides: the kernel". The chunk's own K/V are written to
 * the pool first (pa_reshape_and_cache with one slot per chunk token).
 *
 * Sequence s contributes c_s = cu_q[s+1] - cu_q[s] query tokens, rows
 * cu_q[s] .. cu_q[s+1]-1 of q and out, which are its LAST c_s tokens:
 * seq_lens[s] counts every cached token, the chunk included. Query token i
 * of s is at position p = seq_lens[s] - c_s + i and, for query head h with
 * kv head g = h / G,
 *   out[cu_q[s]+i][h][:] = sum_{j <= p} softmax_j(scale * q . K_j) V_j
 * with K_j = k_pool[block_tables[s][j / block_size]][g][j % block_size][:].
 * c_s = 1 for every s is decode; cu_q[s] = 0 history (seq_lens = c_s) is a
 * whole-prompt prefill.
 *
 *   out            bf16 [total_q][n_q_heads][head_dim], 16-B aligned
 *   q              bf16 [total_q][n_q_heads][head_dim], 16-B aligned
 *   cu_q           int32 [num_seqs + 1], non-decreasing, cu_q[0] = 0 (device)
 *   total_q        rows (tokens) of q and out, >= cu_q[num_seqs]; a chunk
 *                  reaching past it is flagged PA_DEV_ERR_SEQ_LEN and its
 *                  rows past total_q are neither read nor written
 *   max_q_len      host bound of max_s c_s (sizes the grid); rows of a
 *                  longer chunk are not written and PA_DEV_ERR_SEQ_LEN is set
 *   n_q_heads / n_kv_heads  <= 64
 *   scale          finite and > 0 (else PA_ERR_INVALID_ARG)
 *   others         as pa_decode (head_dim 64/128, block_size 8/16/32)
 * seq_lens[s] > max_blocks_per_seq * block_size is clamped and flagged
 * PA_DEV_ERR_SEQ_LEN; c_s > seq_lens[s] is flagged and that sequence's rows
 * are not written. Bad block ids are skipped (their tokens weigh zero) and
 * flagged PA_DEV_ERR_BLOCK_ID. No workspace. Launched as a programmatic
 * dependent of the preceding kernel; it waits for it before reading.
 */
pa_status pa_prefill(void* out, const void* q, const void* k_pool, const void* v_pool,
                     const int32_t* block_tables, const int32_t* seq_lens, const int32_t* cu_q,
                     int num_seqs, int total_q, int max_blocks_per_seq, int num_blocks,
                     int n_q_heads, int n_kv_heads, int head_dim, int block_size, float scale,
                     int max_q_len, int32_t* err_word, pa_stream_t stream);

/*
 * pa_reshape_and_cache — write new tokens' K/V into their pool slots.
 * Defined by the "A DECODE STEP" diagram of "PagedAttention"
 * (mlapandio.dev): the step writes the new K and V into the sequence's
 * current block; "03 · PagedAttention", "Blocks and block tables": that
 * block was taken when the previous one filled.
 *
 * For token t with slot = slot_mapping[t] >= 0, every kv head h:
 *   k_pool[slot / block_size][h][slot % block_size][:] = k[t][h][:]
 *   v_pool[slot / block_size][h][slot % block_size][:] = v[t][h][:]
 * (bit copy). The kernel signals programmatic completion as soon as it
 * starts, so a following pa_decode may begin its set-up meanwhile (it waits
 * for this kernel before reading the pools). slot < 0 is padding and is
 * skipped silently; slot >=
 * num_blocks*block_size is skipped and flagged PA_DEV_ERR_SLOT. Two tokens
 * naming the same slot race (the caller must not do that).
 *
 *   k, v          bf16 [num_tokens][n_kv_heads][head_dim], 16-B aligned
 *   k_pool, v_pool as in pa_decode
 *   slot_mapping  int32 [num_tokens]
 *   num_tokens    >= 0 (0: nothing is launched)
 */
pa_status pa_reshape_and_cache(const void* k, const void* v, void* k_pool, void* v_pool,
                               const int32_t* slot_mapping, int num_tokens, int num_blocks,
                               int n_kv_heads, int head_dim, int block_size,
                               int32_t* err_word, pa_stream_t stream);

/*
 * pa_copy_blocks — copy-on-write block duplication.
 * Defined by "03 · PagedAttention", "Sharing: copy-on-write, straight from
 * fork()" (a writer into a block with refcount > 1 gets a copy and its
 * table is repointed) and the "COPY-ON-WRITE ON A SHARED PREFIX" diagram of
 * "PagedAttention" (mlapandio.dev: the runtime copies the shared block,
 * then writes). The refcount bookkeeping and the table update are the
 * caller's (host) business; this call moves the bytes.
 *
 * For each pair p: block pairs[p][1] of k_pool and of v_pool (all kv heads)
 * becomes a bit copy of block pairs[p][0]. A pair with an id outside
 * [0, num_blocks) is skipped and flagged PA_DEV_ERR_PAIR. Precondition: no
 * destination id is also a source id or appears twice (else the result
 * depends on scheduling).
 *
 *   pairs    int32 [n_pairs][2] (src, dst), device memory
 *   n_pairs  >= 0 (0: nothing is launched)
 */
pa_status pa_copy_blocks(void* k_pool, void* v_pool, const int32_t* pairs, int n_pairs,
                         int n_kv_heads, int head_dim, int block_size, int num_blocks,
                         int32_t* err_word, pa_stream_t stream);

/*
 * FP8 KV cache. "PagedAttention" (mlapandio.dev), "Cons and honest limits",
 * and "Serving: vLLM and PagedAttention", section 3.1, name an fp8 KV cache
 * as the way to halve the cache (and with it the bytes every decode step
 * reads). The pages fix no format; these calls use OCP FP8 E4M3 (bias 7, no
 * infinities, codes 0x7F/0xFF are NaN, largest finite value 448) with one
 * fp32 scale per tensor: a stored code c stands for e4m3(c) * scale.
 * Pools are uint8 [num_blocks][n_kv_heads][block_size][head_dim], one byte
 * per element, otherwise laid out like the bf16 pools.
 */

/*
 * pa_reshape_and_cache_fp8 — pa_reshape_and_cache into fp8 pools.
 * For token t with slot >= 0 and every kv head h and column d:
 *   k_pool[slot / bs][h][slot % bs][d] = E4M3(fp32(k[t][h][d]) / k_scale)
 * (the division rounded to nearest in fp32; the conversion rounded to
 * nearest even and saturated to +-448; NaN gives a NaN code), likewise v
 * with v_scale. Padding, range checks, flags and the early completion
 * signal are those of pa_reshape_and_cache.
 *
 *   k, v              bf16 [num_tokens][n_kv_heads][head_dim], 16-B aligned
 *   k_pool, v_pool    uint8 pools, 16-B aligned
 *   head_dim          64 or 128; block_size 8, 16 or 32
 *   k_scale, v_scale  finite, > 0 (else PA_ERR_INVALID_ARG)
 */
pa_status pa_reshape_and_cache_fp8(const void* k, const void* v, void* k_pool, void* v_pool,
                                   const int32_t* slot_mapping, int num_tokens, int num_blocks,
                                   int n_kv_heads, int head_dim, int block_size, float k_scale,
                                   float v_scale, int32_t* err_word, pa_stream_t stream);

/*
 * pa_copy_blocks_fp8 — pa_copy_blocks on uint8 (fp8) pools: block
 * pairs[p][1] becomes a bit copy of block pairs[p][0] in both pools.
 * Arguments, checks and flags as pa_copy_blocks.
 */
pa_status pa_copy_blocks_fp8(void* k_pool, void* v_pool, const int32_t* pairs, int n_pairs,
                             int n_kv_heads, int head_dim, int block_size, int num_blocks,
                             int32_t* err_word, pa_stream_t stream);

/*
 * pa_decode_fp8 — pa_decode over fp8 pools. For each (sequence, query head)
 * the result is attention with
 *   K_i = e4m3(k code) * k_scale,  V_i = e4m3(v code) * v_scale
 * and the softmax scale `scale`, exactly as pa_decode defines it otherwise.
 * Always the balanced split (no partition argument); the workspace is that
 * of pa_decode_workspace_bytes(num_seqs, n_q_heads, n_kv_heads, 128,
 * block_size, max_seq_len, 0), with the same zeroing rule.
 *
 * Arithmetic: codes are exact in f16; q is rounded from bf16 to f16 (exact
 * for |q| in [2^-14, 65504]; smaller values lose low bits, larger ones are
 * out of range) and the scores and the weighted sum of V are f16 tensor-core
 * products with fp32 accumulation; softmax in fp32.
 *
 *   k_pool, v_pool    uint8 pools, 16-B aligned
 *   head_dim          128 only (else PA_ERR_UNSUPPORTED)
 *   k_scale, v_scale  finite, > 0 (else PA_ERR_INVALID_ARG)
 *   everything else   as pa_decode
 */
pa_status pa_decode_fp8(void* out, const void* q, const void* k_pool, const void* v_pool,
                        const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                        int max_blocks_per_seq, int num_blocks, int n_q_heads, int n_kv_heads,
                        int head_dim, int block_size, float scale, float k_scale, float v_scale,
                        int max_seq_len, void* workspace, size_t workspace_bytes,
                        int32_t* err_word, pa_stream_t stream);

/*
 * pa_swap_blocks — copy whole blocks between two pools, one of which is
 * normally in host memory: preemption by swapping. "03 · PagedAttention",
 * "Memory management, in brief": when memory runs out a sequence can be
 * preempted by swapping its blocks to CPU memory and back later; "Serving:
 * vLLM and PagedAttention" names the same swap. Swap-out copies device
 * blocks to host blocks, swap-in copies them back, possibly under other
 * ids; the allocator's bookkeeping (which ids, the tables) is the caller's.
 *
 * For each pair p: block pairs[p][1] of (dst_k, dst_v) becomes a byte copy
 * of block pairs[p][0] of (src_k, src_v). A block is block_bytes bytes
 * (n_kv_heads * block_size * head_dim * element size; a multiple of 16), so
 * the call serves bf16 and fp8 pools alike. A pair with an id outside
 * [0, src_num_blocks) or [0, dst_num_blocks) is skipped and flagged
 * PA_DEV_ERR_PAIR. Destination ids must be distinct.
 *
 * Every pointer (the four pools, pairs and err_word) must be memory this
 * device can address: its own device memory, managed memory, or page-locked
 * host memory (cudaHostAlloc / cudaMallocHost / registered), which the
 * kernel reads or writes directly through its mapped address. Anything else
 * (pageable host memory, another device's memory) returns
 * PA_ERR_INVALID_ARG before anything is launched. The kernel is ordered on
 * `stream` like the other calls; host memory it writes is complete once the
 * stream has reached the call.
 */
pa_status pa_swap_blocks(void* dst_k, void* dst_v, const void* src_k, const void* src_v,
                         const int32_t* pairs, int n_pairs, size_t block_bytes,
                         int src_num_blocks, int dst_num_blocks, int32_t* err_word,
                         pa_stream_t stream);

/*
 * pa_check_bounded_wait — a check that the library's waits give up. The pages
 * have no counterpart: it tests the failure behaviour of the kernels here.
 *
 * Every wait inside the library's kernels (on a copy landing, on tensor-core
 * work, on another role's progress) is bounded: after a time limit (2 s in the
 * kernels) it gives up, sets PA_DEV_ERR_TIMEOUT in the error word and lets the
 * kernel finish, so a lost arrival cannot hang the GPU. This entry point runs
 * the same bounded wait on a barrier that nothing arrives on, with the given
 * limit (1 ns .. 2 s), in one thread on `stream`: afterwards *err_word has
 * PA_DEV_ERR_TIMEOUT set and the context is usable.
 *
 * err_word: device int32 (required). Returns PA_ERR_INVALID_ARG for a null
 * err_word or a limit outside (0, 2e9] ns; PA_ERR_CUDA on a launch failure.
 */
pa_status pa_check_bounded_wait(int32_t* err_word, int64_t limit_ns, pa_stream_t stream);

/*
 * pa_copy_host — a byte copy between device memory of the current device and
 * page-locked host memory (either side may be either), done by the SMs as a
 * kernel on `stream`. The pages have no counterpart: it serves the
 * end-to-end step, whose small inputs (the new tokens' q/k/v, tables,
 * lengths, slots) and output cross the chip-to-chip link each step; as a
 * kernel the copy joins the stream of the step's own kernels without a
 * copy-engine hand-off between them.
 *
 * dst, src: 16-byte aligned, caller-owned, not overlapping; page-locked host
 * memory must be mapped for the device (cudaHostAlloc / cudaHostRegister
 * default flags on a unified-address system). nbytes: a multiple of 16
 * (0 does nothing). Returns PA_ERR_INVALID_ARG for null or misaligned
 * pointers, a size not a multiple of 16, or memory the device cannot address
 * (pageable host memory, another device's memory); PA_ERR_CUDA on a launch
 * failure. Asynchronous on `stream`, ordered after the work before it.
 */
pa_status pa_copy_host(void* dst, const void* src, size_t nbytes, pa_stream_t stream);

/*
 * pa_decode_noalloc — pa_decode for callers that cannot allocate device
 * memory. The paper has no counterpart; this is a library convenience.
 *
 * Some callers cannot obtain device memory at the point where they decode:
 * a serving engine that hands all free HBM to its KV pool at start-up and
 * allows no allocation afterwards, a plugin running inside a framework whose
 * allocator owns the device, or latency-critical code that cannot afford an
 * allocation call that may synchronise the device. They still own their
 * inputs and outputs, but cannot provide pa_decode's workspace.
 *
 * This entry point computes exactly what pa_decode computes, with the same
 * arguments minus the workspace. Its scratch is a fixed array of
 * PA_NOALLOC_SCRATCH_BYTES (64 MiB) inside the library's device image: every
 * GPU that loads the library holds those 64 MiB until the process exits. It
 * calls no allocator (no cudaMalloc, cudaFree or allocating library routine).
 *
 *  - The first call from a CUDA context (normally the device's primary
 *    context) looks the array's device address up: one cudaGetSymbolAddress
 *    with that context current, cached under the context's id. A context
 *    made after a device reset, or one the caller created, gets its own
 *    lookup. Make the first call on each device before any stream capture.
 *  - Each call checks every argument first; a refused call launches
 *    nothing. Then it clears the scratch's counters on `stream` (an
 *    asynchronous memset) and runs the decode on `stream`.
 *  - All calls in the process share the one array. Calls that may overlap on
 *    the GPU (different streams without ordering, or several host threads)
 *    race on it and give wrong results; order them on one stream.
 *  - If the call would need more scratch than PA_NOALLOC_SCRATCH_BYTES
 *    (compare pa_decode_workspace_bytes with it beforehand), it returns
 *    PA_ERR_INVALID_ARG without launching anything. Everything else returns
 *    what pa_decode returns for the same arguments.
 */
#define PA_NOALLOC_SCRATCH_BYTES (64u << 20)

pa_status pa_decode_noalloc(void* out, const void* q, const void* k_pool, const void* v_pool,
                            const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                            int max_blocks_per_seq, int num_blocks, int n_q_heads,
                            int n_kv_heads, int head_dim, int block_size, float scale,
                            int partition_tokens, int max_seq_len, int32_t* err_word,
                            pa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
