// Host-side declarations shared by the C-ABI layer and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

#include "../../include/pa.h"

namespace pa {

// Streaming multiprocessors of the current device, queried once per device
// (152 on a GB300; also the answer when no device is present).
inline int sm_count() {
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
    int n = cached[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 152;
    cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

// Raise a kernel's dynamic shared-memory limit once per device (the attribute
// is per device; `done` is the caller's per-kernel record of devices set).
template <typename Kernel>
int ensure_smem_attr(Kernel kern, int bytes, std::atomic<uint64_t> &done) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PA_ERR_CUDA;
    const uint64_t bit = 1ull << dev;
    if (done.load(std::memory_order_acquire) & bit) return PA_OK;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return PA_ERR_CUDA;
    done.fetch_or(bit, std::memory_order_release);
    return PA_OK;
}

// Everything a decode launch needs; passed by value to the kernels.
struct DecodeParams {
    void *out;                   // [B][Hq][D] dtype
    const void *query;           // [B][Hq][D] dtype
    const void *k_cache;         // [NB][Hkv][bs][D]
    const void *v_cache;
    const int32_t *block_tables; // [B][MB]
    const int32_t *context_lens; // [B]
    float *ws_acc;               // [B][Hq][max_partitions][D] unnormalised partial sums
    float2 *ws_ml;               // [B][Hq][max_partitions] (running max in log2 units, sum)
    int *d_err;
    int num_seqs, num_heads, num_kv_heads, max_blocks_per_seq, num_blocks, max_context_len;
    int block_size, partition_tokens, max_partitions;
    float scale_log2;            // scale * log2(e)
    // Kernel sequence s and its head (kvh, h < G) stand for the real row
    // ((s*grp_size + h / grp_inner) * num_heads + kvh*grp_inner + h % grp_inner) of
    // query/out; ordinary decode has grp_size 1 and grp_inner G.  The
    // shared-prefix pass sets grp_size to the sequences sharing a prefix.
    int grp_size, grp_inner;
    int table_stride;            // block-table entries between kernel sequences
    int len_fixed;               // > 0: every kernel sequence has this many tokens
    int len_offset;              // tokens before this position are skipped (multiple of block_size)
    int part_base;               // partials go to partition slot part_base + part ...
    int slots;                   // ... of `slots` per (row); the reduce merges slots
    int force_partials;          // write partials even for one-partition units; no reduce
    int red_fixed_slots;         // reduce: slots before the per-sequence ones
};

// One sequence's chunk in a prefill launch.  Its work units are (kv head,
// row tile of 256 query rows); their key tiles are laid end to end after the
// previous sequences' (the launcher fills in the schedule fields).
struct PrefillSeq {
    const int32_t *block_table;  // [>= ceil((prefix_len+chunk_len)/bs)]
    int prefix_len, chunk_len;
    int row_start;               // first row of the chunk in query/out
    int row_tiles;               // row tiles of the chunk (ceil(chunk_len * group / 256))
    int tiles_per_head;          // key tiles of all its row tiles for one kv head
    int tile_start;              // global index of its first key tile
    int unit_start;              // global index of its first unit
};

constexpr int kPrefillMaxSeqs = 64;  // sequences per launch (kernel-parameter table)

struct PrefillParams {
    void *out;                   // [rows][Hq][D], the chunks one after another
    const void *query;           // [rows][Hq][D]
    const void *k_cache;
    const void *v_cache;
    int *d_err;
    int num_heads, num_kv_heads, num_blocks;
    float scale_log2;
    int num_seqs;                // entries of seqs in use (1 .. kPrefillMaxSeqs)
    int query_rows;              // rows of query/out (all chunks of the call, across launches)
    int total_tiles;             // key tiles of all units
    int split;                   // 1: stream-K ranges over gridDim.x CTAs, with merging; 0: one unit per CTA
    float *part_o;               // split: [2 * CTAs][2 Q tiles][128 rows][128] unnormalised O of partial units
    float2 *part_ml;             // split: [2 * CTAs][2 Q tiles][128 rows] (running max, sum)
    unsigned *counters;          // split: [units][2 Q tiles] segments counted so far; zero on entry, and
                                 // the merging segment resets its unit's to zero before the call ends
    PrefillSeq seqs[kPrefillMaxSeqs];
};

// One launch of a continuous-batching step: CTAs 0 .. prefill_ctas-1 run the
// prompt chunks (the stream-K prefill over those CTAs), the others the decodes
// as a persistent role (one partition per sequence, so no reduce).
struct MixedParams {
    PrefillParams pp;
    DecodeParams dp;
    int prefill_ctas;
    int decode_units;            // sequences x kv heads
    unsigned *decode_next;       // the decode CTAs' shared unit queue (0 between launches)
};

// Split-K partition length for the automatic setting.
int auto_partition_tokens(int num_seqs, int num_heads, int num_kv_heads, int block_size, int max_context_len);

// Kernel launchers.  Each returns PA_OK, PA_ERR_UNSUPPORTED (no instance for
// the shape) or PA_ERR_CUDA (launch / attribute failure).
int launch_decode(pa_dtype dt, int head_dim, int block_size, int group, const DecodeParams &p,
                  cudaStream_t stream);
// Groups whose decode runs on the tensor cores at head_dim 128: only groups
// of 8, where every K/V byte feeds 8 dot products and 8 weighted sums and the
// CUDA-core kernel runs out of issue slots well below the HBM bound.  Groups
// of 1, 2 and 4 are HBM-bound on the CUDA cores and stay there.
inline bool decode_tc_group(int group) { return group == 8; }
// Decode on the tensor cores (the decode kernel only; the caller launches the
// reduce).  PA_ERR_UNSUPPORTED for any other shape, or when the driver
// refuses the kernel's tensor maps.
int launch_decode_tc(pa_dtype dt, int head_dim, int block_size, int group, const DecodeParams &p,
                     cudaStream_t stream);
// Log-sum-exp merge of the partials in p's workspace into p.out.
int launch_decode_reduce(pa_dtype dt, int head_dim, const DecodeParams &p, cudaStream_t stream);
int launch_reshape_and_cache(const void *key, const void *value, void *k_cache, void *v_cache,
                             const int64_t *slots, int num_tokens, int num_kv_heads, int head_dim,
                             int block_size, int num_blocks, int *d_err, cudaStream_t stream);
// Copies of up to kGatherMax buffers in one launch, each from memory the
// device can address (pinned host memory through its device view included)
// to device memory: 16-byte vectors where both ends and the size allow,
// bytes otherwise.
constexpr int kGatherMax = 8;
struct GatherList {
    const void *src[kGatherMax];
    void *dst[kGatherMax];
    unsigned long long bytes[kGatherMax];
    int n;
};
int launch_gather(const GatherList &list, cudaStream_t stream);
size_t copy_blocks_workspace_bytes(int num_pairs);
int launch_copy_blocks(void *k_cache, void *v_cache, const int64_t *pairs, int num_pairs,
                       int num_kv_heads, int head_dim, int block_size, int num_blocks, void *workspace,
                       int *d_err, cudaStream_t stream);
// Workspace for the stream-K prefill schedule (an upper bound for any batch of
// num_seqs chunks totalling total_chunk_len rows).
size_t prefill_workspace_bytes(int num_seqs, long long total_chunk_len, int group, int num_kv_heads);
// workspace may be NULL (or too small): each CTA then computes one whole unit.
int launch_prefill(pa_dtype dt, int head_dim, int block_size, int group, const PrefillParams &p,
                   void *workspace, size_t workspace_bytes, cudaStream_t stream);
// Whether launch_mixed has a kernel for these (head_dim 128, a tensor-core
// decode group, block_size 16..128).
bool mixed_supported(int head_dim, int block_size, int group);
// The one-launch step's kernel instances, one translation unit per dtype.
int launch_mixed_bf16(int block_size, int group, const MixedParams &mp, unsigned grid, cudaStream_t stream);
int launch_mixed_f16(int block_size, int group, const MixedParams &mp, unsigned grid, cudaStream_t stream);
// The fused step: pp as for launch_prefill (at most kPrefillMaxSeqs chunks),
// dp as for launch_decode with one partition per sequence; prefill_ws as for
// launch_prefill (required); decode_bytes: the decodes' K/V bytes, estimated,
// to split the SMs between the two halves.
int launch_mixed(pa_dtype dt, int block_size, int group, const PrefillParams &pp, const DecodeParams &dp,
                 void *workspace, size_t workspace_bytes, double decode_bytes, cudaStream_t stream);

}  // namespace pa
