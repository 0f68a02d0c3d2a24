/*
 * pkv.h -- C ABI of libpkv.so: attention for one continuous-batching engine
 * step over a paged KV cache, on one GB300 (sm_103a), plus the host-side block
 * pool and iteration-level scheduler that build the step's metadata.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Plain C types only.  Device pointers are owned by the caller (this
 *   library never allocates or frees device memory on these paths); host
 *   pointers are owned by whoever the function says.
 * - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   Every device entry point only enqueues work on that stream and returns;
 *   results are ready when the stream reaches that point.
 * - Kernels are launched with programmatic dependent launch: one may start
 *   while the kernel before it on the stream is still running, and waits for
 *   that kernel to finish before it touches anything the kernel may write.
 *   The one exception is context_lens in the decode entry points (see
 *   pkv_paged_decode_attention).
 * - Return value: PKV_OK (0) or a negative PKV_ERR_* code.  Arguments are
 *   validated on the host before any launch; on an error nothing is enqueued.
 *   PKV_ERR_CUDA means a CUDA call failed; pkv_last_cuda_error() names it.
 * - Contents of index arrays (block ids, context lengths, slots) are the
 *   caller's contract.  The kernels still never read or write outside the
 *   buffers whose sizes they are given: an out-of-range block id reads zeros
 *   and sets PKV_DEV_BAD_BLOCK_ID in *dev_status, a context length beyond the
 *   table is clamped and sets PKV_DEV_BAD_CONTEXT, an out-of-range slot is
 *   skipped and sets PKV_DEV_BAD_SLOT.  dev_status (device int, may be NULL)
 *   is OR-ed, never cleared, by the library.  Nothing traps.
 * - Dtypes: PKV_DTYPE_F16 or PKV_DTYPE_BF16 for Q/K/V; outputs may also be
 *   PKV_DTYPE_F32.  Accumulation and softmax are fp32; a 16-bit output is
 *   rounded once, to nearest even, at the final store.
 *
 * Cache layout (both k_cache and v_cache): [num_blocks][num_kv_heads]
 * [block_size][head_dim], row-major, 16-byte aligned.  One (block, KV head)
 * tile is a contiguous block_size x head_dim run.  Physical block b of a
 * sequence holds its logical tokens 16*j .. 16*j+15 where block_tables row
 * entry j == b ("Project 17: Production Serving: Continuous Batching and
 * PagedAttention", section "PagedAttention, the thing you build for memory":
 * fixed-size pages, a per-sequence page table from logical to physical page).
 * Entries past ceil(context_len / block_size) are never read and may hold -1
 * (tiny-vllm part 7, "Termination and returning blocks": -1 = unassigned).
 *
 * Supported instantiations: head_dim 64 or 128, block_size 16, grouped-query
 * ratio num_q_heads / num_kv_heads between 1 and 16.  Query head h reads KV
 * head h / (num_q_heads / num_kv_heads).
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes --------------------------------------------------------- */
#define PKV_OK 0
#define PKV_ERR_INVALID_ARG (-1)   /* null/misaligned pointer, inconsistent sizes */
#define PKV_ERR_UNSUPPORTED (-2)   /* dtype, head_dim, block_size or group size not built */
#define PKV_ERR_WORKSPACE (-3)     /* workspace too small or misaligned */
#define PKV_ERR_CUDA (-4)          /* a CUDA runtime/driver call failed */
#define PKV_ERR_OUT_OF_BLOCKS (-5) /* block pool exhausted (host allocator) */
#define PKV_ERR_NO_DEVICE (-6)     /* no CUDA device is current / visible */
#define PKV_ERR_NO_MEMORY (-7)     /* a host allocation inside the library failed */

/* ---- dtypes ---------------------------------------------------------------- */
#define PKV_DTYPE_F16 0
#define PKV_DTYPE_BF16 1
#define PKV_DTYPE_F32 2

/* ---- device status bits (OR-ed into *dev_status) ---------------------------- */
#define PKV_DEV_BAD_BLOCK_ID 1  /* a block-table entry in use was outside [0, num_blocks) */
#define PKV_DEV_BAD_CONTEXT 2   /* a context length < 0 or > max_blocks_per_seq*block_size */
#define PKV_DEV_WAIT_TIMEOUT 4  /* a bounded wait for a tile gave up; outputs are invalid */
#define PKV_DEV_BAD_SLOT 8      /* a slot_mapping entry pointed outside the pool */
#define PKV_DEV_BAD_CHUNK 16    /* a prefill chunk had q_len > context_len or q_len < 0 */
#define PKV_DEV_SPLIT 32        /* decode's own bookkeeping failed a self-check: the pieces of a
                                   split range did not tile it exactly, or the blocks streamed
                                   differ from the planned total; the affected outputs are wrong.
                                   Never expected; a library bug if seen. */

/* Human-readable name of a status code (static string, never NULL). */
const char *pkv_status_string(int status);

/* Name of the last CUDA error seen by this thread inside the library, or the
 * reason for the last size-limit rejection ("no error" if none).
 * Static/thread-local string, never NULL. */
const char *pkv_last_cuda_error(void);

/* Library version string, e.g. "pkv 0.1 sm_103a". */
const char *pkv_version(void);

/*
 * pkv_kv_append -- write this step's new keys and values into the paged cache.
 *
 * Defined by "Project 17", Step 4 "Implement the paged KV cache" (append
 * stores a token's K and V at (page, slot in page)), with the slot of each new
 * token given by slot_mapping, part of the per-step metadata of "Continuous
 * Batching" (infra.pidoku.co.in) §6 "Under the hood"; it runs before
 * attention (tiny-vllm part 7, "Uploading the active arrays to the GPU").
 *
 *   k, v           device, [num_tokens][num_kv_heads][head_dim], dtype, 16-B aligned
 *   slot_mapping   device int64 [num_tokens]; slot = block * block_size + offset;
 *                  a negative slot means "padding, write nothing"
 *   k_cache, v_cache  device caches (layout above), modified in place
 * For every token t with slot_mapping[t] >= 0 and every KV head h, the bytes
 * of k[t][h][:] and v[t][h][:] are copied unchanged to
 * cache[slot / block_size][h][slot % block_size][:].  Bit-exact.  Slots must be
 * unique within one call (duplicates leave one of the writers' rows).
 * num_tokens == 0 is a no-op.
 */
int pkv_kv_append(const void *k, const void *v, const int64_t *slot_mapping, int num_tokens,
                  void *k_cache, void *v_cache, int num_blocks, int block_size, int num_kv_heads,
                  int head_dim, int dtype, int *dev_status, void *stream);

/*
 * pkv_copy_blocks -- copy whole cache blocks by index pairs, for preemption by
 * swap ("Continuous Batching" §5 "Preemption": copy the victim's KV blocks to
 * CPU memory, later copy them back).  For every i < num_pairs, the
 * block_bytes bytes of block pairs[2i] of src go to block pairs[2i+1] of dst.
 *   dst, src   [dst_blocks] / [src_blocks] blocks of block_bytes each, 16-B
 *              aligned; device memory or pinned host memory (the GPU reads
 *              and writes the latter directly); one call per cache array
 *              (a K or a V cache of one layer)
 *   pairs      device-accessible int32 [num_pairs][2] (source, destination)
 *   block_bytes  multiple of 16 (Hkv * block_size * head_dim * element size)
 * An index out of range skips that pair and sets PKV_DEV_BAD_BLOCK_ID.
 * Destinations must be distinct within a call (else one writer wins).
 */
int pkv_copy_blocks(void *dst, int64_t dst_blocks, const void *src, int64_t src_blocks, const int32_t *pairs,
                    int num_pairs, int64_t block_bytes, int *dev_status, void *stream);

/*
 * Bytes of device workspace pkv_paged_decode_attention should be given on the
 * current device for these head counts and head_dim (independent of the
 * contexts).  The call also accepts less, down to two partial records per
 * warp of its grid and four piece slots per (sequence, KV head) range (it
 * then rebalances work between SMs less, and a step of at most 1024 ranges
 * finds a range's pieces past the fourth through a list instead of 32 slots);
 * below that it returns PKV_ERR_WORKSPACE.  Returns 0 if no device is current.
 */
size_t pkv_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim);

/*
 * pkv_paged_decode_attention -- one query token per sequence attends its whole
 * paged context.
 *
 * Defined by "Project 17", Step 6 "Implement attention over paged storage":
 * walk the page table, score each stored key against the query scaled by
 * 1/sqrt(head_dim), softmax over the sequence, weighted sum of the stored
 * values -- taken per query head, with grouped KV heads.  For sequence s and
 * query head h (g = h / (Hq/Hkv)):
 *     out[s][h][:] = sum_{t < ctx_s} softmax_t(scale * q[s][h] . K_t) V_t,
 *     K_t, V_t = cache[block_tables[s][t / 16]][g][t % 16][:]
 * where ctx_s = context_lens[s] counts the token(s) appended this step
 * (tiny-vllm part 7: K/V are written first, then attention reads length + 1).
 * ctx_s == 0 gives an all-zero row.
 *
 *   out            device, [num_seqs][num_q_heads][head_dim], out_dtype (dtype or F32)
 *   q              device, [num_seqs][num_q_heads][head_dim], dtype, 4-B aligned
 *   k_cache, v_cache  device caches, 16-B aligned, num_blocks blocks
 *   block_tables   device int32 [num_seqs][max_blocks_per_seq]
 *   context_lens   device int32 [num_seqs]
 *   scale          score scale (pass 1/sqrt(head_dim) for the standard one)
 *   workspace      device, >= pkv_decode_workspace_size(...) bytes, 16-B aligned;
 *                  scratch for split-context partial results, contents on entry
 *                  ignored: the call first enqueues a small kernel that zeroes
 *                  the workspace's control region (its first few KB: counters
 *                  and list heads, about 16 bytes per (sequence, KV head)),
 *                  and everything else it reads there it wrote earlier in the
 *                  same call.  Owned by the caller; must not be used by another
 *                  call that may run concurrently.
 *   dev_status     device int or NULL (see conventions)
 * When num_seqs <= 256 the decode kernel reads context_lens to plan its work
 * before it waits for the work enqueued ahead of the call.  By then that work
 * has ended, or has signalled its dependents through programmatic dependent
 * launch.  So context_lens must not be written by a kernel just before the
 * call that signals its dependents before that write (the library's own
 * kernels never write it).  Everything else is read and written only after
 * the wait.
 * One persistent kernel: every warp starts on an equal share of the
 * (sequence, KV head, block) list, and warps that finish early take over the
 * far half of busier warps' unclaimed blocks.  A (sequence, KV head) range
 * processed in several pieces is combined by a log-sum-exp merge, done by the
 * warp that finishes the range's last block, pieces taken in block order.
 * Which blocks are taken over depends on timing, so the last bits of the
 * output may differ from call to call; with the environment variable
 * PKV_DETERMINISTIC=1 (read at every call) nothing is taken over and equal
 * inputs give equal bits.  With head_dim 64, groups of at most 4 query heads
 * and an even num_kv_heads, a unit of work can be a block of two adjacent KV
 * heads (one 4 KB run of K and one of V in the cache), with ranges per
 * (sequence, KV-head pair).  The call takes that form for steps of at least
 * 256 such ranges (512 when max_blocks_per_seq > 128) whose layout fits the
 * workspace; pkv_decode_workspace_size covers both forms.
 */
int pkv_paged_decode_attention(void *out, const void *q, const void *k_cache, const void *v_cache,
                               const int32_t *block_tables, int max_blocks_per_seq,
                               const int32_t *context_lens, int num_seqs, int num_blocks,
                               int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                               float scale, int dtype, int out_dtype, void *workspace,
                               size_t workspace_bytes, int *dev_status, void *stream);

/*
 * pkv_paged_decode_append_attention -- the decode step's append and its
 * attention in one launch: the same result as pkv_kv_append of k_new / v_new
 * followed by pkv_paged_decode_attention ("tiny-vllm part 7": the new token's
 * K/V are written into its block first, then attention runs over the whole
 * context including it), with the slot of sequence s's new token taken from
 * its block table: position context_lens[s] - 1, i.e. slot
 * block_tables[s][(ctx-1)/16] * 16 + (ctx-1) % 16.
 *   k_new, v_new  [num_seqs][num_kv_heads][head_dim], 16-B aligned
 *   k_cache, v_cache  written at those slots (and read, as in decode)
 * The warp that streams the last block of (s, KV head) loads the new rows
 * with that block, uses them in place of the block's stale row and stores
 * them to the cache, so the cache holds after the call exactly what the
 * separate append would have written.  A sequence with context 0 appends
 * nothing; a block id out of range skips the store and sets
 * PKV_DEV_BAD_BLOCK_ID.  Everything else as pkv_paged_decode_attention.
 */
int pkv_paged_decode_append_attention(void *out, const void *q, const void *k_new, const void *v_new,
                                      void *k_cache, void *v_cache, const int32_t *block_tables,
                                      int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                                      int num_blocks, int num_q_heads, int num_kv_heads, int head_dim,
                                      int block_size, float scale, int dtype, int out_dtype, void *workspace,
                                      size_t workspace_bytes, int *dev_status, void *stream);

/*
 * pkv_paged_prefill_attention -- chunked prefill: a chunk of new query tokens
 * per sequence attends the sequence's prior context plus the chunk, causally.
 *
 * Defined by "Continuous Batching" §5 "Mixed batching (prefill + decode in one
 * step)": prompts are split into chunks that ride with the decode step, and
 * variable-length kernels take the ragged shape through cu_seqlens (§6).  For
 * chunk c with q_len = cu_seqlens[c+1] - cu_seqlens[c] and ctx = context_lens[c]
 * (which counts the chunk), query row i sits at position p = ctx - q_len + i and
 *     out[cu[c]+i][h][:] = sum_{t <= p} softmax_t(scale * q[cu[c]+i][h] . K_t) V_t
 * with K_t, V_t gathered through block_tables[c] as in decode.
 *
 *   out, q         device, [total_q][num_q_heads][head_dim]
 *   cu_seqlens     device int32 [num_seqs + 1], cu[0] = 0, non-decreasing
 *   max_q_len      host int, >= every chunk's q_len (sizes the grid)
 *   total_q        host int, == cu_seqlens[num_seqs]
 *   other arguments as in decode.  No workspace is needed.
 * A chunk with q_len > ctx is skipped and sets PKV_DEV_BAD_CHUNK.
 */
int pkv_paged_prefill_attention(void *out, const void *q, const int32_t *cu_seqlens, int num_seqs,
                                int max_q_len, int total_q, const void *k_cache,
                                const void *v_cache, const int32_t *block_tables,
                                int max_blocks_per_seq, const int32_t *context_lens,
                                int num_blocks, int num_q_heads, int num_kv_heads, int head_dim,
                                int block_size, float scale, int dtype, int out_dtype,
                                int *dev_status, void *stream);

/*
 * pkv_paged_mixed_attention -- the attention of one mixed engine step, prefill
 * chunks and decodes in one batch ("Continuous Batching" §5 "Mixed batching
 * (prefill + decode in one step)"), with the two kernels side by side.
 *
 * Layout as the scheduler emits it: the first num_prefill sequences are
 * prefill chunks (rows [0, prefill_tokens) of q/out, cu_seqlens with
 * num_prefill + 1 entries, prefill_tokens = cu_seqlens[num_prefill]), the
 * next num_decode sequences are decodes (one row each, rows prefill_tokens
 * onward); block_tables and context_lens hold num_prefill + num_decode rows.
 * Results equal pkv_paged_prefill_attention on the first part and
 * pkv_paged_decode_attention on the second (workspace as for decode, sized
 * for num_decode sequences).
 *
 * The decode kernel runs on decode_sms SMs and the prefill kernel on the
 * others, on a library-owned side stream forked from and joined back into
 * `stream` with events (one per device, created on first use; the fork and
 * join of concurrent calls are serialised).  decode_sms <= 0 picks the split:
 * from pkv_mixed_split when cu_seqlens_host and context_lens_host (host
 * copies of the same arrays, num_prefill + 1 and num_prefill + num_decode
 * entries) are given, else 3/5 of the SMs.  The pages describe no such
 * overlap; it exists because prefill is bound by the tensor cores and decode
 * by HBM.
 */
int pkv_paged_mixed_attention(void *out, const void *q, const int32_t *cu_seqlens, int num_prefill,
                              int prefill_tokens, int max_q_len, int num_decode, const void *k_cache,
                              const void *v_cache, const int32_t *block_tables, int max_blocks_per_seq,
                              const int32_t *context_lens, int num_blocks, int num_q_heads, int num_kv_heads,
                              int head_dim, int block_size, float scale, int dtype, int out_dtype, void *workspace,
                              size_t workspace_bytes, const int32_t *cu_seqlens_host,
                              const int32_t *context_lens_host, int decode_sms, int *dev_status, void *stream);

/*
 * pkv_paged_mixed_append_attention -- one whole mixed step in one call: the
 * append of the step's new tokens ("tiny-vllm part 7": each new token's K/V
 * is written into its block before attention) and then the attention of
 * pkv_paged_mixed_attention.
 *   k_new, v_new   [prefill_tokens + num_decode][num_kv_heads][head_dim],
 *                  rows in the order of q; 16-B aligned
 *   slot_mapping   int64 [prefill_tokens]: slots of the prefill chunks' rows
 *                  (as pkv_kv_append; < 0 skips).  A decode row s goes to
 *                  position context_lens[s] - 1 through its block table, as
 *                  in pkv_paged_decode_append_attention.
 * The prefill rows are appended just before the prefill kernel (on the side
 * stream, where both kinds of work are present) and the decode rows inside the
 * decode kernel, so the append no longer delays the decode kernel's start.
 * Results (outputs and caches) equal pkv_kv_append of all rows followed by
 * pkv_paged_mixed_attention.  Prefill chunks and decodes must not write the
 * same block (true of scheduler output: a shared prefix page is never
 * written).
 */
int pkv_paged_mixed_append_attention(void *out, const void *q, const void *k_new, const void *v_new,
                                     const int64_t *slot_mapping, const int32_t *cu_seqlens, int num_prefill,
                                     int prefill_tokens, int max_q_len, int num_decode, void *k_cache, void *v_cache,
                                     const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
                                     int num_blocks, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                     float scale, int dtype, int out_dtype, void *workspace, size_t workspace_bytes,
                                     const int32_t *cu_seqlens_host, const int32_t *context_lens_host, int decode_sms,
                                     int *dev_status, void *stream);

/*
 * The SMs pkv_paged_mixed_attention gives the decode kernel for a step (host
 * arrays as above): the split that balances the two kernels' times under a
 * model of their per-SM rates on GB300 -- prefill ~7 TFLOP/s of algorithmic
 * work per SM, decode ~55 GB/s per SM up to 6.2 TB/s in total.  num_sms when
 * there is no prefill, 0 when there is no decode.  Pure host code.
 */
int pkv_mixed_split(int num_sms, const int32_t *cu_seqlens, int num_prefill, const int32_t *context_lens,
                    int num_decode, int num_q_heads, int num_kv_heads, int head_dim, int elem_bytes);

/*
 * pkv_paged_decode_attention_static -- the same decode attention, for callers
 * that cannot allocate device memory.  The pages describe no counterpart:
 * this entry point exists only for the memory model of some callers.
 *
 * pkv_paged_decode_attention needs a caller-provided workspace.  Some callers
 * cannot allocate one: a serving engine that hands all free HBM to its KV
 * pool at start-up and allows no allocation afterwards, a plugin whose host
 * framework owns every device allocation, or a latency-critical loop that must
 * not call cudaMalloc because it can synchronise the device.  This entry point
 * takes the same arguments minus the workspace and uses one scratch array of
 * PKV_STATIC_SCRATCH_BYTES that the library keeps in device global memory
 * (a file-scope __device__ array: every GPU that loads the library holds it
 * until the process exits).  It calls no cudaMalloc/cudaFree and no
 * allocating library routine.
 *
 * - Limits: num_seqs <= PKV_STATIC_MAX_SEQS, and the smallest workspace the
 *   shape accepts must fit in PKV_STATIC_SCRATCH_BYTES.  On a GB300 (152
 *   SMs, 1216 warps) that smallest workspace is about
 *       44 * num_seqs * U + 8 * num_seqs + 10 KB
 *       + 2432 * 4 * (2G + G * head_dim + 8)  bytes,  G = num_q_heads / U,
 *   with U = num_kv_heads; when head_dim is 64, the group has at most 4
 *   query heads and num_kv_heads is even, also with U = num_kv_heads / 2
 *   (two adjacent KV heads as one unit), whichever is less.
 *   So with num_seqs = 16384 the largest num_kv_heads that fits is 27 for
 *   head_dim 128 and G = 4 (452,000 (sequence, KV head) pairs), 20 for G = 8,
 *   and 6 for G = 16 (whose records alone take 20.3 MB); with 256 sequences
 *   every group size fits with several hundred KV heads.  Anything larger
 *   returns PKV_ERR_WORKSPACE before anything is enqueued, and
 *   pkv_last_cuda_error() names the limit.  The rest of the array is room for
 *   rebalancing work between SMs.
 * - The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture.
 * - All calls on a device share the one array, and it keeps the last call's
 *   contents.  Each call first zeroes the array's small control region (as
 *   pkv_paged_decode_attention does with its workspace), and everything else
 *   it reads there it wrote earlier in the same call, so what an earlier call
 *   left behind does not matter; but calls that overlap on the GPU (different
 *   streams, or different host threads, without ordering between them) race
 *   on the array and give wrong results.  Serialise them.
 * Results equal pkv_paged_decode_attention's for the same inputs.
 */
#define PKV_STATIC_SCRATCH_BYTES (24u << 20)
#define PKV_STATIC_MAX_SEQS 16384
int pkv_paged_decode_attention_static(void *out, const void *q, const void *k_cache, const void *v_cache,
                                      const int32_t *block_tables, int max_blocks_per_seq,
                                      const int32_t *context_lens, int num_seqs, int num_blocks,
                                      int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                      float scale, int dtype, int out_dtype, int *dev_status, void *stream);

/* ---- host block pool ----------------------------------------------------------
 * A preallocated set of physical block ids with a free list used as a stack
 * ("Project 17", Step 4: BlockPool.alloc pops from the end of the free list,
 * free appends; "Build a pure-Python continuous batching LLM serving engine",
 * Step 2: the free list is a stack).  Pure host code, no GPU needed.
 */
typedef struct pkv_pool pkv_pool;

/* initial_order: NULL for [0, 1, ..., num_blocks-1] (so block num_blocks-1 is
 * popped first), or a permutation of [0, num_blocks) to start from (copied).
 * Returns NULL on invalid arguments or allocation failure. */
pkv_pool *pkv_pool_create(int num_blocks, const int32_t *initial_order);
void pkv_pool_destroy(pkv_pool *pool);
/* All-or-nothing: pops n ids into out_ids (host array of >= n) in pop order,
 * or returns PKV_ERR_OUT_OF_BLOCKS and changes nothing ("Project 17" Step 4
 * raises OutOfPagesError; "Continuous Batching" §4 returns an error). */
int pkv_pool_alloc(pkv_pool *pool, int n, int32_t *out_ids);
/* Pushes ids back in the given order.  PKV_ERR_INVALID_ARG if an id is out of
 * range or already free (nothing is changed then). */
int pkv_pool_free(pkv_pool *pool, const int32_t *ids, int n);
int pkv_pool_free_count(const pkv_pool *pool);
/* Copies the free list (bottom to top) into out (host, >= free_count ints). */
int pkv_pool_free_list(const pkv_pool *pool, int32_t *out);
/* Fault injection for tests: the nth alloc call from now (1 = the next one)
 * fails with PKV_ERR_OUT_OF_BLOCKS; 0 disarms. */
int pkv_pool_inject_failure(pkv_pool *pool, int64_t nth);

/* ---- host iteration-level scheduler --------------------------------------------
 * Builds each step's metadata for the kernels above and nothing else:
 * retire -> run the running requests -> admit, once per engine step
 * ("Project 17" Step 2, "Continuous Batching" §4 Engine.Step):
 *   - running requests are scheduled first, in admission order: a decode gets
 *     1 token, a request still prefilling gets min(remaining, chunk) tokens,
 *     all within max_num_batched_tokens per step (§5 "Mixed batching");
 *   - before a request runs, it gets blocks for all tokens it will hold after
 *     this step; if the pool is empty, the most recently admitted running
 *     request is preempted (blocks freed, moved to the FRONT of the waiting
 *     queue, recomputed later from prompt + generated tokens), repeatedly; if
 *     that is the request itself it is preempted (§4 preempt, §5 Preemption,
 *     "Victim selection": LIFO);
 *   - waiting requests are admitted first-come-first-served while the batch
 *     has room, the budget is not spent and blocks for all their known tokens
 *     can be allocated; admission stops at the first that does not fit (§4);
 *   - after the iteration, a request whose cache caught up emits one token;
 *     it retires on its pre-drawn EOS step, on max_tokens or when its length
 *     reaches max_model_len, and its blocks are freed at once (§1 lifecycle,
 *     tiny-vllm part 7 "Termination and returning blocks").
 * Emitted sequences: prefill chunks (q_len > 1) first, then decodes
 * (q_len == 1), each group in scheduling order.  Pure host code.
 */
typedef struct pkv_sched pkv_sched;

typedef struct pkv_sched_config {
    int num_blocks;             /* physical blocks in the pool */
    int block_size;             /* tokens per block (16) */
    int max_batch;              /* max running requests */
    int max_num_batched_tokens; /* token budget per step */
    int chunk;                  /* max prefill tokens per request per step */
    int max_model_len;          /* max prompt + generated tokens */
    const int32_t *initial_order; /* NULL or a permutation of [0, num_blocks) (copied) */
    int policy;                 /* PKV_SCHED_CONTINUOUS (0) or PKV_SCHED_STATIC (1) */
    int prefix_caching;         /* 1: share full prompt pages between requests added with tokens */
    int preemption;             /* PKV_PREEMPT_RECOMPUTE (0) or PKV_PREEMPT_SWAP (1) */
    int swap_blocks;            /* host slots for swapped-out blocks (PKV_PREEMPT_SWAP) */
} pkv_sched_config;

/* Preemption ("Continuous Batching" §5 "Preemption").  Recompute: the
 * victim's blocks are freed and it is re-prefilled later.  Swap: the blocks
 * holding its computed tokens are copied to host slots, the device blocks are
 * freed, and when it is admitted again (it waits at the front of the queue)
 * fresh device blocks are allocated, the host slots copied back and its
 * computed length restored -- nothing is recomputed.  A victim whose blocks
 * do not fit in the free host slots is recomputed instead.  The copies are
 * the caller's: each step lists them (pkv_step_meta swap_out / swap_in) and
 * they must run before the step's kernels, all swap-outs before the
 * swap-ins (a block freed by a swap-out may be refilled by a swap-in of the
 * same step).  A host slot freed by a swap-in is reused from the next step
 * on. */
#define PKV_PREEMPT_RECOMPUTE 0
#define PKV_PREEMPT_SWAP 1

/* Admission policies.  Continuous: the rules above, every step ("Continuous
 * Batching" §4-5).  Static: the baseline that page's opening section
 * describes -- a batch of up to max_batch waiting requests is admitted only
 * when nothing runs, and runs until its last request retires; its prefill
 * chunks still take the token budget step by step.  Everything else (block
 * accounting, growth, preemption, retirement) is the same. */
#define PKV_SCHED_CONTINUOUS 0
#define PKV_SCHED_STATIC 1

/* Arrays are owned by the scheduler and valid until the next pkv_sched_step
 * or pkv_sched_destroy on the same scheduler. */
typedef struct pkv_step_meta {
    int num_seqs;       /* sequences scheduled this step */
    int num_prefill;    /* the first num_prefill sequences are prefill chunks */
    int num_tokens;     /* new tokens this step (sum of q_lens) */
    int max_blocks;     /* row length of block_tables = ceil(max_model_len / block_size) */
    const int64_t *seq_rids;      /* [num_seqs] request ids */
    const int32_t *q_lens;        /* [num_seqs] new tokens per sequence */
    const int32_t *context_lens;  /* [num_seqs] tokens attended, including the new ones */
    const int32_t *cu_seqlens;    /* [num_seqs + 1] prefix sums of q_lens */
    const int32_t *block_tables;  /* [num_seqs][max_blocks], -1 padded */
    const int64_t *slot_mapping;  /* [num_tokens] cache slot of every new token */
    const int64_t *token_rids;    /* [num_tokens] request id of every new token */
    const int32_t *token_pos;     /* [num_tokens] position of every new token in its request */
    int num_finished;             /* requests retired at the end of this step */
    const int64_t *finished_rids; /* [num_finished] their ids, in scheduling order */
    int num_swap_out;             /* blocks to copy device -> host before this step's kernels */
    const int32_t *swap_out;      /* [num_swap_out][2]: device block, host slot */
    int num_swap_in;              /* blocks to copy host -> device, after the swap-outs */
    const int32_t *swap_in;       /* [num_swap_in][2]: host slot, device block */
} pkv_step_meta;

typedef struct pkv_sched_stats {
    int64_t steps;          /* pkv_sched_step calls */
    int64_t preemptions;    /* preemption events */
    int64_t admitted;       /* admissions (a recomputed request counts again) */
    int64_t finished;       /* retired requests */
    int64_t sum_running;    /* sum over steps of running requests (average batch) */
    int64_t tokens;         /* scheduled tokens, all steps */
    int64_t prefill_tokens; /* of which in prefill chunks */
    int running;
    int waiting;
    int free_blocks;
    double host_ms;         /* wall time spent inside pkv_sched_step */
    int64_t prefix_hit_blocks; /* blocks taken from the prefix cache at admissions */
    int cached_blocks;      /* pages registered in the prefix cache now */
    int64_t swapped_out_blocks; /* blocks copied to host slots */
    int64_t swapped_in_blocks;  /* blocks copied back */
    int free_swap_slots;    /* host slots free now (including those usable from the next step) */
} pkv_sched_stats;

/* Prefix caching ("Project 17" Step 8 "Prefix caching"; "Continuous Batching"
 * §7 names the gain).  For requests added with their prompt tokens
 * (pkv_sched_add_tokens) and prefix_caching = 1:
 *   - a full page (block_size tokens) of a prompt is registered once its K/V
 *     are computed, keyed by the block holding the preceding page and its own
 *     tokens (which identifies the whole page-aligned prefix, as the page's
 *     tuple key does); it is registered only if that preceding page is;
 *   - at admission the longest chain of registered pages matching the prompt
 *     is taken, covering at most prompt_len - 1 tokens (at least one prompt
 *     token is always computed, so a request never writes into a page it
 *     shares); those blocks join the request's block table with their
 *     reference counts raised, and its computed length starts past them;
 *   - a block returns to the free list when its last holder retires or is
 *     preempted, and its cache entry goes with it.
 * Block tables then carry shared block ids; the kernels need no change. */
pkv_sched *pkv_sched_create(const pkv_sched_config *config);
void pkv_sched_destroy(pkv_sched *sched);
/* Queue a request.  eos_after >= 1 is the output length at which it emits
 * EOS.  PKV_ERR_INVALID_ARG for prompt_len < 1, prompt_len >= max_model_len,
 * max_tokens < 1, eos_after < 1 or a duplicate rid.  A request needing more
 * blocks than the pool holds is accepted but never admitted. */
int pkv_sched_add(pkv_sched *sched, int64_t rid, int prompt_len, int max_tokens, int eos_after);
/* As pkv_sched_add, with the prompt's token ids (copied; prompt_len of them)
 * so that the request can share prompt pages through the prefix cache. */
int pkv_sched_add_tokens(pkv_sched *sched, int64_t rid, const int32_t *tokens, int prompt_len, int max_tokens,
                         int eos_after);
/* One engine step.  Returns the number of scheduled sequences (0 = nothing to
 * run; *out then has num_seqs = 0), or a negative status. */
int pkv_sched_step(pkv_sched *sched, pkv_step_meta *out);
int pkv_sched_get_stats(const pkv_sched *sched, pkv_sched_stats *out);
/* Fault injection for tests: forwarded to the scheduler's pool. */
int pkv_sched_inject_alloc_failure(pkv_sched *sched, int64_t nth);
/* Request state: 0 waiting, 1 running, 2 finished, -1 unknown rid.
 * generated (may be NULL) receives its output-token count. */
int pkv_sched_request_state(const pkv_sched *sched, int64_t rid, int *generated);
/* Drops a finished request's record (its blocks, prompt tokens and swap
 * slots were already released when it finished; what remains are a few
 * counters), so that a long-running scheduler's memory stays bounded; its rid
 * may then be added again.  PKV_ERR_INVALID_ARG for an unknown rid or a
 * request that has not finished. */
int pkv_sched_forget(pkv_sched *sched, int64_t rid);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
