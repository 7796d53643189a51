/*
 * pa.h -- C ABI of the paged-KV attention library (GB300, sm_103a).
 *
 * The operations follow the pages on vLLM's PagedAttention:
 *   "vLLM PagedAttention chuyen sau: Phan manh bo nho KV Cache, Prefill theo
 *   khoi & Prefix Caching" (locionic.com) -- sections "Tuong tu phan trang bo
 *   nho ao" (logical blocks, physical blocks, block table, dynamic growth),
 *   "Co che PagedAttention" (look up, gather, attend), "Chunked Prefill"
 *   (mechanism, KV accumulation) and "Co che APC" step 3 (copy-on-write);
 *   "vLLM" (tellworld.net), section "PagedAttention" (fixed-size blocks
 *   located through a table; sharing).
 *
 * Conventions for every entry point
 * ---------------------------------
 * Pointers.  Every data pointer is a DEVICE pointer owned by the caller; the
 *   library allocates nothing and keeps no pointer after a call returns.
 *   16-bit tensors must be 16-byte aligned.  The only host arguments are the
 *   scalars.
 * Streams.  `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *   stream).  Every call only enqueues work on it and returns; results are
 *   ready when the stream is synchronised.
 * Cache layout.  k_cache and v_cache are each
 *   [num_blocks][num_kv_heads][block_size][head_dim], row-major, elements of
 *   `dtype`.  Token slot t of the pool is block t / block_size, offset
 *   t % block_size.  One (block, kv head) tile is block_size*head_dim
 *   contiguous elements.
 * Head grouping.  Query head h reads KV head h / (num_heads / num_kv_heads).
 * Argument errors (null pointers, bad sizes, unsupported shapes, misaligned
 *   pointers, a too-small workspace) are found on the host before anything
 *   is launched: the call returns a negative pa_status and enqueues nothing.
 * Data errors (a slot or table entry outside the pool, a context length past
 *   the table, a conflicting copy pair, a pipeline wait that gave up) are
 *   found on the device: the offending unit is skipped and a PA_DEVERR_* bit
 *   is OR-ed into *d_err (d_err may be NULL to ignore them).  No kernel traps;
 *   the context stays usable.  Read *d_err after the stream synchronises.
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { PA_F16 = 0, PA_BF16 = 1 } pa_dtype;

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = -1,   /* null pointer, non-positive size, bad enum */
    PA_ERR_UNSUPPORTED = -2,   /* a shape this build has no kernel for */
    PA_ERR_OUT_OF_RANGE = -3,  /* a host scalar outside its allowed range */
    PA_ERR_CUDA = -4,          /* a CUDA runtime call failed (launch, attribute) */
    PA_ERR_WORKSPACE = -5,     /* workspace missing or smaller than required */
    PA_ERR_ALIGNMENT = -6,     /* a pointer is not 16-byte aligned */
    PA_ERR_SCRATCH_LIMIT = -7, /* pa_decode_noalloc: partials exceed its fixed scratch array */
    PA_ERR_NO_BLOCKS = -8      /* block manager: no free block and nothing evictable */
} pa_status;

/* Size of the device array pa_decode_noalloc keeps its split-K partials in. */
#define PA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

/* Bits OR-ed into *d_err by the kernels. */
#define PA_DEVERR_SLOT_RANGE 0x1    /* slot_mapping entry >= num_blocks*block_size */
#define PA_DEVERR_BLOCK_RANGE 0x2   /* block-table entry outside [0, num_blocks) */
#define PA_DEVERR_CONTEXT_RANGE 0x4 /* context length < 0, > max_context_len or > table */
#define PA_DEVERR_COPY_PAIR 0x8     /* copy pair out of pool, src==dst, or dst conflict */
#define PA_DEVERR_TIMEOUT 0x10      /* a bounded pipeline wait gave up */
#define PA_DEVERR_PREFIX 0x20       /* pa_decode_shared_prefix: a group's prefix table rows differ */

/* Human-readable name of a pa_status value. */
PA_API const char *pa_status_string(int status);

/*
 * pa_reshape_and_cache -- write new tokens' K and V rows into their slots.
 * ("vLLM PagedAttention chuyen sau" (locionic.com), section "Tuong tu phan
 * trang bo nho ao": a growing sequence gets each new token a slot in one of
 * its physical blocks; section "Chunked Prefill", mechanism step 3: a
 * chunk's KV accumulates in the cache the same way.)
 *
 *   key, value     [num_tokens][num_kv_heads][head_dim] dtype, contiguous
 *   k_cache,v_cache pool as above, written in place
 *   slot_mapping   int64 [num_tokens]; slot < 0 = padding, nothing written;
 *                  slot >= num_blocks*block_size sets PA_DEVERR_SLOT_RANGE
 * Requires head_dim % 8 == 0.  num_tokens == 0 is a no-op.  Two tokens with
 * the same slot race (one of them wins); the caller must not do that.
 * The copy is bit-exact.
 */
PA_API int pa_reshape_and_cache(const void *key, const void *value, void *k_cache, void *v_cache,
                         const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                         int head_dim, int block_size, int num_blocks, pa_dtype dtype,
                         int *d_err, void *stream);

/*
 * pa_decode_partition_tokens -- the split-K partition length pa_decode uses
 * for these arguments: partition_tokens itself when > 0, otherwise the
 * automatic choice (a power of two in [256, 4096] that grows with
 * num_seqs * max_context_len * num_kv_heads, so units stay few and long when
 * the batch alone fills the GPU and get shorter when it does not).  Returns 0
 * when the arguments are invalid.
 */
PA_API int pa_decode_partition_tokens(int num_seqs, int num_heads, int num_kv_heads, int block_size,
                                      int max_context_len, int partition_tokens);

/*
 * pa_decode_workspace_bytes -- device workspace pa_decode needs for split-K
 * partials with these arguments (0 when every sequence fits one partition).
 * Layout (internal): fp32 partial accumulators and (max, sum) pairs per
 * (sequence, query head, partition).
 */
PA_API size_t pa_decode_workspace_bytes(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                        int block_size, int max_context_len, int partition_tokens);

/*
 * pa_decode -- single-query paged attention (one decode step).
 * For each sequence s and query head h, with L = context_lens[s] and
 * kvh = h / (num_heads/num_kv_heads):
 *   1. look up physical block block_tables[s][j / block_size] for j < L,
 *   2. gather K and V rows from those blocks,
 *   3. out[s][h] = sum_j softmax_j(scale * q[s][h] . K_j) V_j,
 * accumulated in fp32 and rounded once to dtype (round to nearest even).
 * Groups of 8 at head_dim 128 run on the tensor cores: the products
 * accumulate in fp32, and each softmax weight enters the weighted sum as
 * two dtype values (its rounding and the rounded residual), which keeps it
 * to about twice dtype's precision (smaller groups, and head_dim 64, keep
 * the weights in fp32).
 *
 *   out            [num_seqs][num_heads][head_dim] dtype (written)
 *   query          [num_seqs][num_heads][head_dim] dtype
 *   block_tables   int32 [num_seqs][max_blocks_per_seq]; entries past
 *                  ceil(L/block_size) are never read
 *   context_lens   int32 [num_seqs], includes the newest token; 0 gives zeros
 *   max_context_len  host upper bound on every context_lens[s]
 *   partition_tokens 0 = automatic; otherwise a positive multiple of
 *                  block_size: each sequence is split into partitions of this
 *                  many tokens, attended independently, then merged by a
 *                  log-sum-exp reduction (a second kernel on the same stream)
 *   workspace      device buffer of >= pa_decode_workspace_bytes(...) bytes
 *                  (may be NULL when that is 0); its contents are scratch
 * Supported: head_dim in {64, 128}; block_size in {8, 16, 32, 64, 128};
 *   num_heads / num_kv_heads in {1, 2, 4, 8}; dtype f16 or bf16.
 * Invalid lengths are clamped to [0, min(max_context_len,
 * max_blocks_per_seq*block_size)] and flagged; invalid table entries are
 * flagged and the keys they would supply are left out of the softmax (on
 * the CUDA-core path at block_size 8, the whole 16-key tile holding such a
 * block).
 */
PA_API int pa_decode(void *out, const void *query, const void *k_cache, const void *v_cache,
              const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
              int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
              int num_blocks, int max_context_len, float scale, int partition_tokens,
              pa_dtype dtype, void *workspace, size_t workspace_bytes, int *d_err,
              void *stream);

/*
 * pa_decode_shared_prefix -- pa_decode for batches in which consecutive
 * groups of sequences share the physical blocks of a common prefix (several
 * samples of one prompt; the pages' parallel sampling / shared-prefix case:
 * "vLLM PagedAttention chuyen sau" (locionic.com), "Co che APC", and "vLLM"
 * (tellworld.net), "PagedAttention").  Each shared block is read from memory
 * once per group instead of once per sequence.
 *
 * Same arguments, layout, results and errors as pa_decode, plus:
 *   group_size     sequences g*group_size .. g*group_size+group_size-1 form
 *                  group g; num_seqs % group_size == 0, and group_size times
 *                  num_heads/num_kv_heads must be 1, 2, 4 or 8
 *   prefix_blocks  >= 1: the first prefix_blocks entries of every block-table
 *                  row of a group are the same physical blocks, and every
 *                  sequence's context covers them (context_lens[s] >=
 *                  prefix_blocks*block_size).  A group whose rows differ there
 *                  sets PA_DEVERR_PREFIX (its outputs are then undefined); a
 *                  context shorter than the prefix sets PA_DEVERR_CONTEXT_RANGE.
 *   workspace      always required: pa_decode_shared_prefix_workspace_bytes().
 * The output equals pa_decode's within the attention tolerance (the same
 * softmax, merged from partials of the prefix and of each sequence's own
 * tokens; not bit-identical to pa_decode).  Internally: one pass attends each
 * group's queries over its shared blocks as one head group, one pass attends
 * each sequence over its own tokens, and a log-sum-exp merge combines them.
 */
PA_API size_t pa_decode_shared_prefix_workspace_bytes(int num_seqs, int num_heads, int num_kv_heads,
                                                      int head_dim, int block_size, int max_context_len,
                                                      int prefix_blocks, int partition_tokens);
PA_API int pa_decode_shared_prefix(void *out, const void *query, const void *k_cache,
                                   const void *v_cache, const int32_t *block_tables,
                                   int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                                   int group_size, int prefix_blocks, int num_heads, int num_kv_heads,
                                   int head_dim, int block_size, int num_blocks, int max_context_len,
                                   float scale, int partition_tokens, pa_dtype dtype, void *workspace,
                                   size_t workspace_bytes, int *d_err, void *stream);

/*
 * pa_decode_noalloc -- pa_decode for callers that must not allocate device
 * memory.  The pages have no counterpart; this exists for hosts that cannot
 * call cudaMalloc on this path: an inference engine that has already handed
 * nearly all HBM to its KV-cache pool (there is nothing left to allocate from,
 * and a failed allocation mid-step is fatal), or a latency-critical loop that
 * cannot afford the device-wide synchronisation cudaMalloc/cudaFree imply.
 *
 * Same arguments, results and errors as pa_decode, minus the workspace: the
 * split-K partials go to one array of PA_NOALLOC_SCRATCH_BYTES (64 MiB) that
 * the library declares as a static device variable.  Every GPU that loads the
 * library holds that array until the process exits, whether or not this entry
 * point is ever called.
 *   - Sizes whose partials would not fit (pa_decode_workspace_bytes(...) >
 *     PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_SCRATCH_LIMIT and launch
 *     nothing; use pa_decode with a caller-owned workspace, or a longer
 *     partition_tokens, for those.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - All calls on a device share the one array.  Calls whose kernels can
 *     overlap on the GPU (different streams, no ordering between them) race
 *     on it and corrupt each other's results; serialise them.  The array
 *     needs no clearing: every partial is written before it is read.
 * Nothing here calls cudaMalloc, cudaFree or any allocating routine.
 */
PA_API int pa_decode_noalloc(void *out, const void *query, const void *k_cache, const void *v_cache,
                             const int32_t *block_tables, int max_blocks_per_seq,
                             const int32_t *context_lens, int num_seqs, int num_heads,
                             int num_kv_heads, int head_dim, int block_size, int num_blocks,
                             int max_context_len, float scale, int partition_tokens,
                             pa_dtype dtype, int *d_err, void *stream);

/*
 * pa_decode_step_host -- one whole decode step whose inputs sit in host
 * memory, as a scheduler holds them (the step the pages' engine runs per
 * generated token: copy-on-write of shared blocks, the new tokens' K/V into
 * their slots, then attention; "vLLM PagedAttention chuyen sau"
 * (locionic.com), sections "Co che PagedAttention" and "Co che APC").
 * In order on `stream`: the host inputs are brought into `staging` -- those
 * in page-locked host memory the device can address by one gather kernel
 * that reads them all, any other with its own cudaMemcpyAsync -- then
 * pa_copy_blocks (when num_pairs > 0),
 * pa_reshape_and_cache (when num_new_tokens > 0), pa_decode -- or
 * pa_decode_shared_prefix when group_size > 1 -- and the output lands in
 * out_host: written there by the kernels when out_host is page-locked host
 * memory the device can address (16-byte aligned), else written into staging
 * and copied with cudaMemcpyAsync.  All of it is asynchronous: the host buffers
 * must stay valid and unchanged until the stream has finished the step, and
 * out_host holds the result only after the caller synchronises.  Host
 * buffers should be page-locked (pinned) for the copies to be asynchronous.
 *   out_host           [num_seqs][num_heads][head_dim] dtype (written)
 *   query_host         [num_seqs][num_heads][head_dim] dtype
 *   new_key_host, new_value_host  [num_new_tokens][num_kv_heads][head_dim] dtype
 *   slot_mapping_host  int64 [num_new_tokens] (as for pa_reshape_and_cache)
 *   pairs_host         int64 [num_pairs][2] (as for pa_copy_blocks; NULL if 0)
 *   block_tables_host  int32 [num_seqs][max_blocks_per_seq]
 *   context_lens_host  int32 [num_seqs]
 *   k_cache, v_cache   the device pool, as for pa_decode
 *   group_size, prefix_blocks  0 and 0 for plain decode; otherwise as for
 *                      pa_decode_shared_prefix
 *   staging            device buffer of >= pa_decode_step_host_staging_bytes
 *                      (same shape arguments) bytes, 256-byte aligned; its
 *                      contents are scratch (it also holds the decode workspace)
 * Returns the first failing call's status (argument checks happen before any
 * copy is queued); PA_ERR_WORKSPACE if staging is missing or too small.
 */
PA_API size_t pa_decode_step_host_staging_bytes(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                                int block_size, int max_blocks_per_seq, int max_context_len,
                                                int num_new_tokens, int num_pairs, int group_size,
                                                int prefix_blocks, int partition_tokens);
PA_API int pa_decode_step_host(void *out_host, const void *query_host, const void *new_key_host,
                               const void *new_value_host, const int64_t *slot_mapping_host, int num_new_tokens,
                               const int64_t *pairs_host, int num_pairs, const int32_t *block_tables_host,
                               int max_blocks_per_seq, const int32_t *context_lens_host, int num_seqs,
                               int group_size, int prefix_blocks, int num_heads, int num_kv_heads, int head_dim,
                               int block_size, int num_blocks, void *k_cache, void *v_cache,
                               int max_context_len, float scale, int partition_tokens, pa_dtype dtype,
                               void *staging, size_t staging_bytes, int *d_err, void *stream);

/*
 * pa_mixed_step -- one continuous-batching step over one pool: the prompt
 * chunks of num_prefill sequences (as pa_prefill_batch) and one decode token
 * for each of num_decode other sequences (as pa_decode), together.  The
 * pages' chunked prefill, whose point is to batch prompt chunks with decodes
 * ("vLLM PagedAttention chuyen sau" (locionic.com), "Chunked Prefill",
 * mechanism steps 2 and 4).  Both halves read the pool as it is when the call
 * is reached on `stream`: write the step's new K/V first (pa_reshape_and_cache).
 * Arguments as for pa_prefill_batch (prefill_*, prefix_lens, chunk_lens on
 * the host) and pa_decode (decode_*, context_lens on the device), with the
 * pool and the model shape shared.
 *
 * One launch: with head_dim 128, 2, 4 or 8 query heads per kv head, block_size 16 to
 * 128, max_context_len <= 16384, at most 64 non-empty chunks, and a
 * workspace of at least pa_mixed_step_workspace_bytes(...) bytes, 256-byte
 * aligned and ZERO-FILLED before its first use, the step is one kernel of one
 * CTA per SM: some CTAs run the chunks (the stream-K prefill over those
 * CTAs), the others decode (sequence, kv head) units drawn from a queue the
 * whole grid shares (one partition each, so no reduce), and the chunks' CTAs
 * join the queue when their share of the chunks is done; the split of the
 * SMs follows the chunks' key tiles and the decodes' estimated K/V bytes, so
 * the tensor cores and HBM work at the same time.  The calls leave the
 * workspace's counters at zero, so one workspace serves every later step
 * whose sizes it covers; two steps must not run on one workspace at the same
 * time.  Results equal the separate calls' up to rounding.
 * Two launches otherwise (or when the workspace is smaller, e.g. only
 * pa_decode's): the chunks' kernel first on a high-priority stream the library
 * forks from `stream` and joins back into it, the decode on `stream` over the
 * SMs the chunks leave free; the workspace is then pa_decode's.  The fork
 * stream and its two events are created on the first such call on a device
 * and kept; calls from several host threads are serialised around the fork.
 * A half with no sequences is skipped.  Returns the first failing half's
 * status (the other half may have been queued).
 */
PA_API size_t pa_mixed_step_workspace_bytes(int num_prefill, int total_chunk_len, int num_decode, int num_heads,
                                            int num_kv_heads, int head_dim, int block_size, int max_context_len,
                                            int partition_tokens);
PA_API int pa_mixed_step(void *prefill_out, const void *prefill_query, const int32_t *prefill_block_tables,
                         int prefill_max_blocks, const int *prefix_lens, const int *chunk_lens, int num_prefill,
                         void *decode_out, const void *decode_query, const int32_t *decode_block_tables,
                         int decode_max_blocks, const int32_t *context_lens, int num_decode, int max_context_len,
                         int partition_tokens, void *workspace, size_t workspace_bytes, const void *k_cache,
                         const void *v_cache, int num_heads, int num_kv_heads, int head_dim, int block_size,
                         int num_blocks, float scale, pa_dtype dtype, int *d_err, void *stream);

/*
 * Failure detection.  Every wait inside the kernels (on TMA copies, MMA
 * completions, other warps) is bounded: after pa_bounded_wait_polls() polls
 * it gives up, ORs PA_DEVERR_TIMEOUT into *d_err and lets the kernel finish,
 * so a stuck pipeline is reported and the context stays usable.
 * pa_selftest_bounded_wait runs that same wait, with max_polls polls, on a
 * barrier nothing ever arrives on: it must set PA_DEVERR_TIMEOUT in *d_err
 * (device int) and, if d_cycles is not NULL, write the SM clock cycles the
 * wait took to *d_cycles (device long long).  Asynchronous on `stream`.
 */
PA_API int pa_bounded_wait_polls(void);
PA_API int pa_selftest_bounded_wait(int max_polls, int *d_err, long long *d_cycles, void *stream);

/*
 * pa_copy_blocks -- copy-on-write of shared blocks ("vLLM PagedAttention
 * chuyen sau" (locionic.com), section "Co che APC", step 3: a block that
 * several sequences share is copied before one of them writes into it).
 * For each pair (src, dst) of `pairs` (int64 [num_pairs][2], device), copy
 * the whole K block and V block (all kv heads) of src to dst, bit-exact.  A
 * pair is skipped and PA_DEVERR_COPY_PAIR set when an id is outside the
 * pool, src == dst, its dst appears as another pair's dst, or its dst is any
 * pair's src -- so the result never depends on the order in which pairs run.
 *
 *   workspace  device scratch of at least
 *              pa_copy_blocks_workspace_bytes(num_pairs) bytes, 16-byte
 *              aligned, owned by the caller (NULL allowed when num_pairs is
 *              0).  The call counts, in one pass over the pairs, how often
 *              each block id appears as a dst and as a src (a hash table in
 *              the workspace); each pair's copy then reads its dst's counts
 *              once, so validation costs O(num_pairs) in total.  Its content
 *              on entry is ignored; it must not be shared with work that
 *              overlaps the call on the device.
 * num_pairs above PA_COPY_MAX_PAIRS returns PA_ERR_OUT_OF_RANGE; a missing
 * or too small workspace returns PA_ERR_WORKSPACE.  Three launches (clear
 * the table, count, copy).
 */
#define PA_COPY_MAX_PAIRS (1 << 26)
PA_API size_t pa_copy_blocks_workspace_bytes(int num_pairs);
PA_API int pa_copy_blocks(void *k_cache, void *v_cache, const int64_t *pairs, int num_pairs,
                   int num_kv_heads, int head_dim, int block_size, int num_blocks,
                   pa_dtype dtype, void *workspace, size_t workspace_bytes, int *d_err, void *stream);

/*
 * pa_prefill_chunk -- attention of one prompt chunk over its sequence's paged
 * KV ("vLLM PagedAttention chuyen sau" (locionic.com), section "Chunked
 * Prefill", mechanism: a long prompt is processed chunk by chunk, each chunk
 * attending to the KV its sequence has accumulated so far), causal: row i
 * (absolute position prefix_len + i) attends to keys 0 .. prefix_len + i.  The chunk's own K/V must already be in the cache
 * (pa_reshape_and_cache).  QK^T and PV run on the 5th-generation tensor cores
 * (tcgen05.mma, accumulators in TMEM) with fp32 accumulation; P is rounded
 * to dtype for the PV product;
 * the output is rounded once to dtype.
 *
 *   out    [chunk_len][num_heads][head_dim] dtype (written)
 *   query  [chunk_len][num_heads][head_dim] dtype
 *   block_table int32 [>= ceil((prefix_len+chunk_len)/block_size)]
 * scale must be finite and > 0.
 * Supported: head_dim 128, block_size in {16, 32, 64, 128}, group size in {1,2,4,8},
 * dtype f16 or bf16.
 *
 *   workspace  NULL, or device scratch of at least
 *              pa_prefill_workspace_bytes(1, chunk_len, ...) bytes, 256-byte
 *              aligned, owned by the caller, ZERO-FILLED before its first use.
 *              The work is cut into units of 256 query rows (chunk positions
 *              x the heads of one kv head).  With a workspace the kernel runs
 *              one CTA per SM, each over an equal share of the units' key
 *              tiles; a unit shared by several CTAs is finished by merging
 *              their log-sum-exp partials, which live in the workspace with a
 *              counter per unit.  Every call that completes leaves the
 *              counters at zero again, so no call needs to clear anything;
 *              after a call that set PA_DEVERR_TIMEOUT, zero-fill the
 *              workspace again.  It must not be shared with work that overlaps
 *              the call on the device.  Without a workspace each CTA computes
 *              one whole unit: the same result up to rounding, slower when the
 *              units do not fill the GPU.  A non-NULL workspace that is too
 *              small returns PA_ERR_WORKSPACE; one not 256-byte aligned,
 *              PA_ERR_ALIGNMENT.
 */
PA_API int pa_prefill_chunk(void *out, const void *query, const void *k_cache, const void *v_cache,
                     const int32_t *block_table, int prefix_len, int chunk_len, int num_heads,
                     int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
                     pa_dtype dtype, void *workspace, size_t workspace_bytes, int *d_err, void *stream);

/*
 * pa_prefill_batch -- pa_prefill_chunk for several sequences in one launch
 * (continuous batching of prompt chunks: "vLLM PagedAttention chuyen sau"
 * (locionic.com), section "Chunked Prefill").  Sequence i's chunk is rows
 * row_i .. row_i + chunk_lens[i] - 1 of query and out, where row_i is the sum
 * of the earlier chunk lengths; its row r (absolute position prefix_lens[i] +
 * r) attends to keys 0 .. prefix_lens[i] + r of its own block-table row.
 *
 *   out, query    [sum(chunk_lens)][num_heads][head_dim] dtype (device)
 *   block_tables  int32 [num_seqs][max_blocks_per_seq] (device)
 *   prefix_lens, chunk_lens  int [num_seqs], HOST memory (scheduling
 *                 metadata the caller knows when it builds the batch); a
 *                 chunk length of 0 skips the sequence; prefix + chunk must
 *                 fit in max_blocks_per_seq * block_size
 * Same numerics, shapes, workspace and errors as pa_prefill_chunk; one
 * launch per 64 sequences with a non-empty chunk.  Without a workspace a
 * sequence's rows are bit-identical to a pa_prefill_chunk call on it alone
 * without one (every unit is computed whole, in the same order); with one,
 * where the key tiles are cut depends on the whole batch.
 */
PA_API int pa_prefill_batch(void *out, const void *query, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, int max_blocks_per_seq, const int *prefix_lens,
                            const int *chunk_lens, int num_seqs, int num_heads, int num_kv_heads,
                            int head_dim, int block_size, int num_blocks, float scale, pa_dtype dtype,
                            void *workspace, size_t workspace_bytes, int *d_err, void *stream);

/*
 * pa_prefill_workspace_bytes -- workspace for pa_prefill_chunk (num_seqs 1)
 * or pa_prefill_batch: enough for any num_seqs chunks whose lengths add up
 * to at most total_chunk_len, on the current device.  0 for invalid arguments.
 */
PA_API size_t pa_prefill_workspace_bytes(int num_seqs, int total_chunk_len, int num_heads, int num_kv_heads,
                                         int head_dim);

/*
 * Block manager -- host bookkeeping of the paged pool: which physical blocks
 * each sequence's block table holds, reference counts of shared blocks,
 * copy-on-write, and automatic prefix caching ("vLLM PagedAttention chuyen
 * sau" (locionic.com), "Tuong tu phan trang bo nho ao" and "Co che APC").
 * It produces exactly what the kernels consume: block-table rows, slot
 * mappings for pa_reshape_and_cache and (src, dst) pairs for pa_copy_blocks.
 * Pure host code; no GPU needed.  Not thread-safe: one owner per manager.
 *
 *   pa_bm_create(num_blocks, block_size, enable_prefix_cache)
 *       -> manager, or NULL on bad sizes.  Free blocks go out in id order.
 *   pa_bm_add_sequence(m, seq_id, tokens, n, slots, num_cached)
 *       registers a new sequence with its n prompt token ids.  With prefix
 *       caching, the longest run of whole blocks whose token ids match blocks
 *       already cached (a path in the prefix tree) is linked into the table
 *       and counted as hits; those tokens get slot -1.  Every other token
 *       gets the slot its K/V must be written to.  Each block that fills up
 *       joins the prefix tree.  PA_ERR_INVALID_ARG for a known seq_id,
 *       PA_ERR_NO_BLOCKS (nothing changed) when the pool runs out.
 *   pa_bm_fork(m, parent, child)
 *       child starts with all of parent's blocks, shared (parallel sampling).
 *   pa_bm_append_token(m, seq_id, token, slot, copy_src, copy_dst)
 *       one more token (decode step): its slot; a new block when the last
 *       one is full; if the last block is partially filled and shared, a
 *       private copy first (copy-on-write) whose (src, dst) is returned, else
 *       src = dst = -1.  The caller copies the block before writing the slot.
 *   pa_bm_free_sequence(m, seq_id)
 *       drops the sequence's references.  Unreferenced blocks in the prefix
 *       tree stay cached (reusable) until evicted; the others are free.
 *       Allocation evicts the least recently released cached leaf block when
 *       no free block is left.
 *   pa_bm_block_table(m, seq_id, out, max_blocks) -> number of blocks, or
 *       PA_ERR_OUT_OF_RANGE if max_blocks is too small.
 *   pa_bm_seq_len, pa_bm_block_refcount, pa_bm_stats: introspection.  The
 *       prefix-cache hit rate is hit_tokens / query_tokens.
 */
typedef struct pa_block_manager pa_block_manager;
typedef struct {
    int num_blocks, free_blocks, cached_free_blocks, used_blocks, num_sequences;
    long long query_tokens, hit_tokens, evictions, cow_copies;
} pa_bm_counters;
PA_API pa_block_manager *pa_bm_create(int num_blocks, int block_size, int enable_prefix_cache);
PA_API void pa_bm_destroy(pa_block_manager *m);
PA_API int pa_bm_add_sequence(pa_block_manager *m, int64_t seq_id, const int32_t *tokens, int num_tokens,
                              int64_t *slots, int *num_cached_tokens);
PA_API int pa_bm_fork(pa_block_manager *m, int64_t parent_id, int64_t child_id);
PA_API int pa_bm_append_token(pa_block_manager *m, int64_t seq_id, int32_t token, int64_t *slot,
                              int64_t *copy_src, int64_t *copy_dst);
PA_API int pa_bm_free_sequence(pa_block_manager *m, int64_t seq_id);
PA_API int pa_bm_block_table(const pa_block_manager *m, int64_t seq_id, int32_t *out, int max_blocks);
PA_API int64_t pa_bm_seq_len(const pa_block_manager *m, int64_t seq_id);
PA_API int pa_bm_block_refcount(const pa_block_manager *m, int block);
PA_API int pa_bm_stats(const pa_block_manager *m, pa_bm_counters *out);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
