// C-ABI entry points: host-side argument validation, then kernel dispatch.
// Nothing here allocates device memory or synchronises the stream.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "../../include/pa.h"
#include "pa_internal.h"

namespace pa {
int launch_decode_bf16(int head_dim, int block_size, int group, const DecodeParams &p,
                       cudaStream_t stream);
int launch_decode_f16(int head_dim, int block_size, int group, const DecodeParams &p,
                      cudaStream_t stream);

int launch_decode_reduce_bf16(int head_dim, const DecodeParams &p, cudaStream_t stream);
int launch_decode_reduce_f16(int head_dim, const DecodeParams &p, cudaStream_t stream);

// Head groups of 8 at head_dim 128 run on the tensor cores; every other shape
// (and that one, should its tensor maps be refused) on the CUDA cores.
int launch_decode(pa_dtype dt, int head_dim, int block_size, int group, const DecodeParams &p,
                  cudaStream_t stream) {
    const int rc = launch_decode_tc(dt, head_dim, block_size, group, p, stream);
    if (rc == PA_ERR_UNSUPPORTED)
        return dt == PA_BF16 ? launch_decode_bf16(head_dim, block_size, group, p, stream)
                             : launch_decode_f16(head_dim, block_size, group, p, stream);
    if (rc != PA_OK) return rc;
    if (p.max_partitions > 1 && !p.force_partials) return launch_decode_reduce(dt, head_dim, p, stream);
    return PA_OK;
}

int launch_decode_reduce(pa_dtype dt, int head_dim, const DecodeParams &p, cudaStream_t stream) {
    return dt == PA_BF16 ? launch_decode_reduce_bf16(head_dim, p, stream)
                         : launch_decode_reduce_f16(head_dim, p, stream);
}

// Automatic split-K partition length: about an eighth of one CTA slot's
// share of the step's work per partition, so units are long enough to
// amortise their set-up and the merge, and short enough to balance.  The work
// is estimated from the host-side arguments only (every sequence's length is
// on the device): num_seqs * max_context_len / 2 tokens per kv head, spread
// over the GPU's SMs (152) x the resident CTAs of the kernel that runs (3 for
// the CUDA-core kernel at groups up to 4; 2 for groups of 8, which run on the
// tensor cores at head_dim 128 and hold 2 CTAs per SM on the CUDA cores).
// The result is the power of two nearest that estimate within [256, 4096] (a
// multiple of block_size).  Measured on the decode workloads: LLaMA GQA picks
// 1024 (98.8% of HBM peak against 96.5% at 512), long context 2048, OPT MHA
// 512, the shared-prefix batch 2048 (1.84x against 1.55x logical).
int auto_partition_tokens(int num_seqs, int num_heads, int num_kv_heads, int block_size, int max_context_len) {
    const int group = num_heads / num_kv_heads;
    const double slots = (double)pa::sm_count() * (group <= 4 ? 3 : 2);
    const double per_part = (double)num_seqs * max_context_len * 0.5 * num_kv_heads / slots / 8.0;
    int pt = 256;
    while (pt < 4096 && per_part > pt * 1.41421356) pt *= 2;
    if (pt % block_size) pt = (pt + block_size - 1) / block_size * block_size;
    return pt;
}
}  // namespace pa

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool good_dtype(pa_dtype d) { return d == PA_F16 || d == PA_BF16; }

bool decode_shape_supported(int head_dim, int block_size, int group) {
    return (head_dim == 64 || head_dim == 128) &&
           (block_size == 8 || block_size == 16 || block_size == 32 || block_size == 64 || block_size == 128) &&
           (group == 1 || group == 2 || group == 4 || group == 8);
}

int resolve_partition(int num_seqs, int num_heads, int num_kv_heads, int block_size, int max_context_len,
                      int partition_tokens) {
    if (partition_tokens < 0) return -1;
    if (partition_tokens == 0)
        return pa::auto_partition_tokens(num_seqs, num_heads, num_kv_heads, block_size, max_context_len);
    if (partition_tokens % block_size) return -1;
    return partition_tokens;
}

int max_parts(int max_context_len, int pt) {
    return max_context_len > 0 ? (max_context_len + pt - 1) / pt : 1;
}

}  // namespace

extern "C" {

const char *pa_status_string(int status) {
    switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG: null pointer, bad size or bad enum";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED: no kernel for this shape";
    case PA_ERR_OUT_OF_RANGE: return "PA_ERR_OUT_OF_RANGE: scalar argument out of range";
    case PA_ERR_CUDA: return "PA_ERR_CUDA: CUDA runtime call failed";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE: workspace missing or too small";
    case PA_ERR_ALIGNMENT: return "PA_ERR_ALIGNMENT: pointer not 16-byte aligned";
    case PA_ERR_SCRATCH_LIMIT:
        return "PA_ERR_SCRATCH_LIMIT: split-K partials exceed the fixed scratch of pa_decode_noalloc";
    case PA_ERR_NO_BLOCKS: return "PA_ERR_NO_BLOCKS: block pool exhausted and nothing evictable";
    default: return "unknown pa_status";
    }
}

int pa_reshape_and_cache(const void *key, const void *value, void *k_cache, void *v_cache,
                         const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                         int head_dim, int block_size, int num_blocks, pa_dtype dtype, int *d_err,
                         void *stream) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0 ||
        !good_dtype(dtype))
        return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!key || !value || !k_cache || !v_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
    if (head_dim % 8) return PA_ERR_UNSUPPORTED;
    if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_ALIGNMENT;
    return pa::launch_reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, num_tokens,
                                        num_kv_heads, head_dim, block_size, num_blocks, d_err,
                                        static_cast<cudaStream_t>(stream));
}

int pa_decode_partition_tokens(int num_seqs, int num_heads, int num_kv_heads, int block_size,
                               int max_context_len, int partition_tokens) {
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads || block_size <= 0 ||
        max_context_len < 0)
        return 0;
    const int pt = resolve_partition(num_seqs, num_heads, num_kv_heads, block_size, max_context_len,
                                     partition_tokens);
    return pt > 0 ? pt : 0;
}

size_t pa_decode_workspace_bytes(int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                                 int max_context_len, int partition_tokens) {
    if (num_seqs <= 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads || head_dim <= 0 ||
        block_size <= 0 || max_context_len < 0)
        return 0;
    const int pt = resolve_partition(num_seqs, num_heads, num_kv_heads, block_size, max_context_len,
                                     partition_tokens);
    if (pt <= 0) return 0;
    const int mp = max_parts(max_context_len, pt);
    if (mp <= 1) return 0;
    const size_t n = (size_t)num_seqs * num_heads * mp;
    const size_t acc = (n * head_dim * sizeof(float) + 255) / 256 * 256;
    return acc + n * 2 * sizeof(float);
}

int pa_decode(void *out, const void *query, const void *k_cache, const void *v_cache,
              const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
              int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
              int num_blocks, int max_context_len, float scale, int partition_tokens,
              pa_dtype dtype, void *workspace, size_t workspace_bytes, int *d_err, void *stream) {
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        num_blocks <= 0 || max_blocks_per_seq <= 0 || max_context_len < 0 || !good_dtype(dtype))
        return PA_ERR_INVALID_ARG;
    if (num_heads % num_kv_heads) return PA_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return PA_ERR_OUT_OF_RANGE;
    if (num_seqs == 0) return PA_OK;
    if (!out || !query || !k_cache || !v_cache || !block_tables || !context_lens)
        return PA_ERR_INVALID_ARG;
    const int group = num_heads / num_kv_heads;
    if (!decode_shape_supported(head_dim, block_size, group)) return PA_ERR_UNSUPPORTED;
    if (!aligned16(out) || !aligned16(query) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_ALIGNMENT;
    const int pt = resolve_partition(num_seqs, num_heads, num_kv_heads, block_size, max_context_len,
                                     partition_tokens);
    if (pt <= 0) return PA_ERR_OUT_OF_RANGE;
    const int mp = max_parts(max_context_len, pt);
    pa::DecodeParams p{};
    p.out = out;
    p.query = query;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.d_err = d_err;
    p.num_seqs = num_seqs;
    p.num_heads = num_heads;
    p.num_kv_heads = num_kv_heads;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.num_blocks = num_blocks;
    p.max_context_len = max_context_len;
    p.block_size = block_size;
    p.partition_tokens = pt;
    p.max_partitions = mp;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.grp_size = 1;
    p.grp_inner = group;
    p.table_stride = max_blocks_per_seq;
    p.slots = mp;
    if (mp > 1) {
        const size_t need = pa_decode_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                                      max_context_len, pt);
        if (!workspace || workspace_bytes < need) return PA_ERR_WORKSPACE;
        if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PA_ERR_ALIGNMENT;
        const size_t n = (size_t)num_seqs * num_heads * mp;
        const size_t acc = (n * head_dim * sizeof(float) + 255) / 256 * 256;
        p.ws_acc = static_cast<float *>(workspace);
        p.ws_ml = reinterpret_cast<float2 *>(static_cast<char *>(workspace) + acc);
    }
    return pa::launch_decode(dtype, head_dim, block_size, group, p,
                             static_cast<cudaStream_t>(stream));
}

size_t pa_decode_shared_prefix_workspace_bytes(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                                int block_size, int max_context_len, int prefix_blocks,
                                                int partition_tokens) {
    if (num_seqs <= 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads || head_dim <= 0 ||
        block_size <= 0 || max_context_len < 0 || prefix_blocks <= 0)
        return 0;
    const int pt = resolve_partition(num_seqs, num_heads, num_kv_heads, block_size, max_context_len,
                                     partition_tokens);
    if (pt <= 0) return 0;
    const int prefix_tokens = prefix_blocks * block_size;
    const int slots = max_parts(prefix_tokens, pt) + max_parts(std::max(max_context_len - prefix_tokens, 0), pt);
    const size_t n = (size_t)num_seqs * num_heads * slots;
    const size_t acc = (n * head_dim * sizeof(float) + 255) / 256 * 256;
    return acc + n * 2 * sizeof(float);
}

int pa_decode_shared_prefix(void *out, const void *query, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
                            int num_seqs, int group_size, int prefix_blocks, int num_heads, int num_kv_heads,
                            int head_dim, int block_size, int num_blocks, int max_context_len, float scale,
                            int partition_tokens, pa_dtype dtype, void *workspace, size_t workspace_bytes,
                            int *d_err, void *stream) {
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        num_blocks <= 0 || max_blocks_per_seq <= 0 || max_context_len < 0 || !good_dtype(dtype) ||
        group_size <= 0 || prefix_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    if (num_heads % num_kv_heads || num_seqs % group_size) return PA_ERR_INVALID_ARG;
    if (prefix_blocks > max_blocks_per_seq || (long long)prefix_blocks * block_size > max_context_len)
        return PA_ERR_OUT_OF_RANGE;
    if (!std::isfinite(scale)) return PA_ERR_OUT_OF_RANGE;
    if (num_seqs == 0) return PA_OK;
    if (!out || !query || !k_cache || !v_cache || !block_tables || !context_lens) return PA_ERR_INVALID_ARG;
    const int group = num_heads / num_kv_heads;
    const long long vgroup = (long long)group * group_size;  // heads per kv head in the prefix pass
    if (!decode_shape_supported(head_dim, block_size, group) || vgroup > 8 ||
        !decode_shape_supported(head_dim, block_size, (int)vgroup))
        return PA_ERR_UNSUPPORTED;
    if (!aligned16(out) || !aligned16(query) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_ALIGNMENT;
    const int pt = resolve_partition(num_seqs, num_heads, num_kv_heads, block_size, max_context_len,
                                     partition_tokens);
    if (pt <= 0) return PA_ERR_OUT_OF_RANGE;
    const int prefix_tokens = prefix_blocks * block_size;
    const int p_pre = max_parts(prefix_tokens, pt);
    const int p_tail = max_parts(std::max(max_context_len - prefix_tokens, 0), pt);
    const size_t need = pa_decode_shared_prefix_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim,
                                                                block_size, max_context_len, prefix_blocks, pt);
    if (!workspace || workspace_bytes < need) return PA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PA_ERR_ALIGNMENT;
    const size_t n = (size_t)num_seqs * num_heads * (p_pre + p_tail);
    const size_t acc = (n * head_dim * sizeof(float) + 255) / 256 * 256;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    pa::DecodeParams p{};
    p.out = out;
    p.query = query;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.d_err = d_err;
    p.num_heads = num_heads;
    p.num_kv_heads = num_kv_heads;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.num_blocks = num_blocks;
    p.max_context_len = max_context_len;
    p.block_size = block_size;
    p.partition_tokens = pt;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.ws_acc = static_cast<float *>(workspace);
    p.ws_ml = reinterpret_cast<float2 *>(static_cast<char *>(workspace) + acc);
    p.slots = p_pre + p_tail;
    p.force_partials = 1;

    // pass 1: each group's queries over its shared blocks, one head group per kv head
    pa::DecodeParams pre = p;
    pre.num_seqs = num_seqs / group_size;
    pre.grp_size = group_size;
    pre.grp_inner = group;
    pre.table_stride = group_size * max_blocks_per_seq;
    pre.len_fixed = prefix_tokens;
    pre.max_partitions = p_pre;
    int rc = pa::launch_decode(dtype, head_dim, block_size, (int)vgroup, pre, st);
    if (rc != PA_OK) return rc;

    // pass 2: every sequence over its own tokens after the prefix
    pa::DecodeParams tail = p;
    tail.num_seqs = num_seqs;
    tail.grp_size = 1;
    tail.grp_inner = group;
    tail.table_stride = max_blocks_per_seq;
    tail.len_offset = prefix_tokens;
    tail.part_base = p_pre;
    tail.max_partitions = p_tail;
    rc = pa::launch_decode(dtype, head_dim, block_size, group, tail, st);
    if (rc != PA_OK) return rc;

    // merge: p_pre prefix slots plus one per partition of the sequence's own tokens
    pa::DecodeParams red = tail;
    red.red_fixed_slots = p_pre;
    return pa::launch_decode_reduce(dtype, head_dim, red, st);
}

size_t pa_copy_blocks_workspace_bytes(int num_pairs) {
    if (num_pairs < 0 || num_pairs > PA_COPY_MAX_PAIRS) return 0;
    return pa::copy_blocks_workspace_bytes(num_pairs);
}

int pa_copy_blocks(void *k_cache, void *v_cache, const int64_t *pairs, int num_pairs,
                   int num_kv_heads, int head_dim, int block_size, int num_blocks, pa_dtype dtype,
                   void *workspace, size_t workspace_bytes, int *d_err, void *stream) {
    if (num_pairs < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0 ||
        !good_dtype(dtype))
        return PA_ERR_INVALID_ARG;
    if (num_pairs > PA_COPY_MAX_PAIRS) return PA_ERR_OUT_OF_RANGE;
    if (num_pairs == 0) return PA_OK;
    if (!k_cache || !v_cache || !pairs) return PA_ERR_INVALID_ARG;
    if (((long long)num_kv_heads * block_size * head_dim) % 8) return PA_ERR_UNSUPPORTED;
    if (!aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_ALIGNMENT;
    if (!workspace || workspace_bytes < pa::copy_blocks_workspace_bytes(num_pairs)) return PA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return PA_ERR_ALIGNMENT;
    return pa::launch_copy_blocks(k_cache, v_cache, pairs, num_pairs, num_kv_heads, head_dim,
                                  block_size, num_blocks, workspace, d_err, static_cast<cudaStream_t>(stream));
}

size_t pa_prefill_workspace_bytes(int num_seqs, int total_chunk_len, int num_heads, int num_kv_heads,
                                  int head_dim) {
    if (num_seqs <= 0 || total_chunk_len < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads ||
        head_dim <= 0)
        return 0;
    return pa::prefill_workspace_bytes(num_seqs < pa::kPrefillMaxSeqs ? num_seqs : pa::kPrefillMaxSeqs,
                                       total_chunk_len, num_heads / num_kv_heads, num_kv_heads);
}

int pa_prefill_chunk(void *out, const void *query, const void *k_cache, const void *v_cache,
                     const int32_t *block_table, int prefix_len, int chunk_len, int num_heads,
                     int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
                     pa_dtype dtype, void *workspace, size_t workspace_bytes, int *d_err, void *stream) {
    if (prefix_len < 0 || chunk_len < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        block_size <= 0 || num_blocks <= 0 || !good_dtype(dtype))
        return PA_ERR_INVALID_ARG;
    if (num_heads % num_kv_heads) return PA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return PA_ERR_OUT_OF_RANGE;
    if (chunk_len == 0) return PA_OK;
    if (!out || !query || !k_cache || !v_cache || !block_table) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(query) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_ALIGNMENT;
    pa::PrefillParams p{};
    p.out = out;
    p.query = query;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.d_err = d_err;
    p.num_heads = num_heads;
    p.num_kv_heads = num_kv_heads;
    p.num_blocks = num_blocks;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.num_seqs = 1;
    p.query_rows = chunk_len;
    p.seqs[0].block_table = block_table;
    p.seqs[0].prefix_len = prefix_len;
    p.seqs[0].chunk_len = chunk_len;
    p.seqs[0].row_start = 0;
    return pa::launch_prefill(dtype, head_dim, block_size, num_heads / num_kv_heads, p, workspace, workspace_bytes,
                              static_cast<cudaStream_t>(stream));
}

int pa_prefill_batch(void *out, const void *query, const void *k_cache, const void *v_cache,
                     const int32_t *block_tables, int max_blocks_per_seq, const int *prefix_lens,
                     const int *chunk_lens, int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                     int block_size, int num_blocks, float scale, pa_dtype dtype, void *workspace,
                     size_t workspace_bytes, int *d_err, void *stream) {
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        num_blocks <= 0 || max_blocks_per_seq <= 0 || !good_dtype(dtype))
        return PA_ERR_INVALID_ARG;
    if (num_heads % num_kv_heads) return PA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return PA_ERR_OUT_OF_RANGE;
    if (num_seqs == 0) return PA_OK;
    if (!prefix_lens || !chunk_lens) return PA_ERR_INVALID_ARG;
    long long rows = 0;
    for (int i = 0; i < num_seqs; ++i) {
        if (prefix_lens[i] < 0 || chunk_lens[i] < 0) return PA_ERR_INVALID_ARG;
        if ((long long)prefix_lens[i] + chunk_lens[i] > (long long)max_blocks_per_seq * block_size)
            return PA_ERR_OUT_OF_RANGE;
        rows += chunk_lens[i];
    }
    if (rows == 0) return PA_OK;
    if (rows > 0x7fffffffLL) return PA_ERR_OUT_OF_RANGE;
    if (!out || !query || !k_cache || !v_cache || !block_tables) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(query) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_ALIGNMENT;
    pa::PrefillParams p{};
    p.out = out;
    p.query = query;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.d_err = d_err;
    p.num_heads = num_heads;
    p.num_kv_heads = num_kv_heads;
    p.num_blocks = num_blocks;
    p.scale_log2 = scale * 1.4426950408889634f;
    // sequences with a non-empty chunk, kPrefillMaxSeqs per launch
    p.query_rows = (int)rows;
    int row = 0;
    for (int i = 0; i < num_seqs; ++i) {
        if (chunk_lens[i] > 0) {
            pa::PrefillSeq &q = p.seqs[p.num_seqs++];
            q.block_table = block_tables + (size_t)i * max_blocks_per_seq;
            q.prefix_len = prefix_lens[i];
            q.chunk_len = chunk_lens[i];
            q.row_start = row;
        }
        row += chunk_lens[i];
        if (p.num_seqs == pa::kPrefillMaxSeqs || (i == num_seqs - 1 && p.num_seqs > 0)) {
            const int rc = pa::launch_prefill(dtype, head_dim, block_size, num_heads / num_kv_heads, p, workspace,
                                              workspace_bytes, static_cast<cudaStream_t>(stream));
            if (rc != PA_OK) return rc;
            p.num_seqs = 0;
        }
    }
    return PA_OK;
}

}  // extern "C"

// ---- a whole decode step from host-resident inputs ----------------------------

namespace {

size_t round256(size_t n) { return (n + 255) / 256 * 256; }

// Staging regions of pa_decode_step_host, in order: out, query, new keys, new
// values, slots, copy pairs, block tables, context lengths, decode workspace.
struct StepLayout {
    size_t off[10];
    size_t total;
};

bool step_layout(int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                 int max_blocks_per_seq, int max_context_len, int num_new_tokens, int num_pairs, int group_size,
                 int prefix_blocks, int partition_tokens, StepLayout *lay) {
    if (num_seqs <= 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads || head_dim <= 0 ||
        block_size <= 0 || max_blocks_per_seq <= 0 || max_context_len < 0 || num_new_tokens < 0 || num_pairs < 0 ||
        num_pairs > PA_COPY_MAX_PAIRS)
        return false;
    const size_t qbytes = (size_t)num_seqs * num_heads * head_dim * 2;
    const size_t kvbytes = (size_t)num_new_tokens * num_kv_heads * head_dim * 2;
    size_t ws = 0;
    if (group_size > 1) {
        if (prefix_blocks <= 0) return false;
        ws = pa_decode_shared_prefix_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                                     max_context_len, prefix_blocks, partition_tokens);
    } else {
        ws = pa_decode_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_context_len,
                                       partition_tokens);
    }
    const size_t sizes[10] = {qbytes, qbytes, kvbytes, kvbytes, (size_t)num_new_tokens * 8,
                              (size_t)num_pairs * 16, (size_t)num_seqs * max_blocks_per_seq * 4,
                              (size_t)num_seqs * 4, pa::copy_blocks_workspace_bytes(num_pairs), ws};
    size_t at = 0;
    for (int i = 0; i < 10; ++i) {
        lay->off[i] = at;
        at += round256(sizes[i]);
    }
    lay->total = at;
    return true;
}

}  // namespace

extern "C" {

size_t pa_decode_step_host_staging_bytes(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                         int block_size, int max_blocks_per_seq, int max_context_len,
                                         int num_new_tokens, int num_pairs, int group_size, int prefix_blocks,
                                         int partition_tokens) {
    StepLayout lay;
    if (!step_layout(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                     max_context_len, num_new_tokens, num_pairs, group_size, prefix_blocks, partition_tokens,
                     &lay))
        return 0;
    return lay.total;
}

int pa_decode_step_host(void *out_host, const void *query_host, const void *new_key_host,
                        const void *new_value_host, const int64_t *slot_mapping_host, int num_new_tokens,
                        const int64_t *pairs_host, int num_pairs, const int32_t *block_tables_host,
                        int max_blocks_per_seq, const int32_t *context_lens_host, int num_seqs, int group_size,
                        int prefix_blocks, int num_heads, int num_kv_heads, int head_dim, int block_size,
                        int num_blocks, void *k_cache, void *v_cache, int max_context_len, float scale,
                        int partition_tokens, pa_dtype dtype, void *staging, size_t staging_bytes, int *d_err,
                        void *stream) {
    if (num_seqs <= 0 || num_blocks <= 0 || !good_dtype(dtype)) return PA_ERR_INVALID_ARG;
    StepLayout lay;
    if (!step_layout(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                     max_context_len, num_new_tokens, num_pairs, group_size, prefix_blocks, partition_tokens,
                     &lay))
        return PA_ERR_INVALID_ARG;
    if (!out_host || !query_host || !block_tables_host || !context_lens_host || !k_cache || !v_cache)
        return PA_ERR_INVALID_ARG;
    if (num_new_tokens > 0 && (!new_key_host || !new_value_host || !slot_mapping_host)) return PA_ERR_INVALID_ARG;
    if (num_pairs > 0 && !pairs_host) return PA_ERR_INVALID_ARG;
    if (!staging || staging_bytes < lay.total) return PA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(staging) & 255u) != 0) return PA_ERR_ALIGNMENT;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    char *base = static_cast<char *>(staging);
    void *d_out = base + lay.off[0], *d_q = base + lay.off[1], *d_k = base + lay.off[2], *d_v = base + lay.off[3];
    // An output in page-locked host memory the device can address is written
    // there by the kernels themselves (no copy after the step).
    bool out_direct = false;
    {
        cudaPointerAttributes at{};
        const cudaError_t qa = cudaPointerGetAttributes(&at, out_host);
        if (qa != cudaSuccess) cudaGetLastError();
        if (qa == cudaSuccess && at.type == cudaMemoryTypeHost && at.devicePointer != nullptr &&
            aligned16(at.devicePointer)) {
            d_out = at.devicePointer;
            out_direct = true;
        }
    }
    int64_t *d_slots = reinterpret_cast<int64_t *>(base + lay.off[4]);
    int64_t *d_pairs = reinterpret_cast<int64_t *>(base + lay.off[5]);
    int32_t *d_bt = reinterpret_cast<int32_t *>(base + lay.off[6]);
    int32_t *d_lens = reinterpret_cast<int32_t *>(base + lay.off[7]);
    void *d_cow_ws = base + lay.off[8];
    const size_t cow_ws_bytes = lay.off[9] - lay.off[8];
    void *d_ws = base + lay.off[9];
    const size_t ws_bytes = lay.total - lay.off[9];
    const size_t qbytes = (size_t)num_seqs * num_heads * head_dim * 2;
    const size_t kvbytes = (size_t)num_new_tokens * num_kv_heads * head_dim * 2;
    // Inputs in page-locked host memory the device can address are read by
    // one gather kernel (the copies' fixed costs, paid once); any other input
    // is copied with its own cudaMemcpyAsync.
    pa::GatherList gl{};
    auto h2d = [&](void *dst, const void *src, size_t n) {
        if (n == 0) return true;
        cudaPointerAttributes at{};
        const cudaError_t qa = cudaPointerGetAttributes(&at, src);
        if (qa != cudaSuccess) cudaGetLastError();  // a pointer the runtime does not know: no error kept
        if (qa == cudaSuccess && at.type == cudaMemoryTypeHost && at.devicePointer != nullptr &&
            gl.n < pa::kGatherMax) {
            gl.src[gl.n] = at.devicePointer;
            gl.dst[gl.n] = dst;
            gl.bytes[gl.n] = n;
            ++gl.n;
            return true;
        }
        return cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, st) == cudaSuccess;
    };
    if (!h2d(d_q, query_host, qbytes) || !h2d(d_k, new_key_host, kvbytes) || !h2d(d_v, new_value_host, kvbytes) ||
        !h2d(d_slots, slot_mapping_host, (size_t)num_new_tokens * 8) ||
        !h2d(d_pairs, pairs_host, (size_t)num_pairs * 16) ||
        !h2d(d_bt, block_tables_host, (size_t)num_seqs * max_blocks_per_seq * 4) ||
        !h2d(d_lens, context_lens_host, (size_t)num_seqs * 4))
        return PA_ERR_CUDA;
    if (pa::launch_gather(gl, st) != PA_OK) return PA_ERR_CUDA;
    int rc = pa_copy_blocks(k_cache, v_cache, d_pairs, num_pairs, num_kv_heads, head_dim, block_size, num_blocks,
                            dtype, d_cow_ws, cow_ws_bytes, d_err, stream);
    if (rc != PA_OK) return rc;
    rc = pa_reshape_and_cache(d_k, d_v, k_cache, v_cache, d_slots, num_new_tokens, num_kv_heads, head_dim,
                              block_size, num_blocks, dtype, d_err, stream);
    if (rc != PA_OK) return rc;
    if (group_size > 1)
        rc = pa_decode_shared_prefix(d_out, d_q, k_cache, v_cache, d_bt, max_blocks_per_seq, d_lens, num_seqs,
                                     group_size, prefix_blocks, num_heads, num_kv_heads, head_dim, block_size,
                                     num_blocks, max_context_len, scale, partition_tokens, dtype, d_ws, ws_bytes,
                                     d_err, stream);
    else
        rc = pa_decode(d_out, d_q, k_cache, v_cache, d_bt, max_blocks_per_seq, d_lens, num_seqs, num_heads,
                       num_kv_heads, head_dim, block_size, num_blocks, max_context_len, scale, partition_tokens,
                       dtype, d_ws, ws_bytes, d_err, stream);
    if (rc != PA_OK) return rc;
    if (out_direct) return PA_OK;
    return cudaMemcpyAsync(out_host, d_out, qbytes, cudaMemcpyDeviceToHost, st) == cudaSuccess ? PA_OK
                                                                                                  : PA_ERR_CUDA;
}

}  // extern "C"

// ---- one continuous-batching step: prompt chunks and decodes together ----------

namespace {

// A high-priority stream and two events per device, created on first use and
// kept for the life of the process; the mutex keeps one call's fork, launches
// and join together when several host threads use them.
struct ForkStream {
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
std::mutex g_fork_mutex;
ForkStream g_fork[64];

int fork_stream(ForkStream **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PA_ERR_CUDA;
    ForkStream &f = g_fork[dev];
    if (!f.stream) {
        int least = 0, greatest = 0;
        if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess ||
            cudaEventCreateWithFlags(&f.fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&f.join, cudaEventDisableTiming) != cudaSuccess ||
            cudaStreamCreateWithPriority(&f.stream, cudaStreamNonBlocking, greatest) != cudaSuccess)
            return PA_ERR_CUDA;
    }
    *out = &f;
    return PA_OK;
}

// Longest context the fused step decodes as one partition per sequence.
constexpr int kMixedMaxContext = 16384;

// The fused step's workspace: the decode's split-K region (used when the step
// runs as two launches), then the stream-K prefill region, which must stay
// zero-filled between calls (the decode region never overlaps it).
size_t mixed_decode_region(int num_decode, int num_heads, int num_kv_heads, int head_dim, int block_size,
                           int max_context_len, int partition_tokens) {
    if (num_decode <= 0) return 0;
    const size_t d = pa_decode_workspace_bytes(num_decode, num_heads, num_kv_heads, head_dim, block_size,
                                               max_context_len, partition_tokens);
    return round256(d);
}

}  // namespace

extern "C" {

size_t pa_mixed_step_workspace_bytes(int num_prefill, int total_chunk_len, int num_decode, int num_heads,
                                     int num_kv_heads, int head_dim, int block_size, int max_context_len,
                                     int partition_tokens) {
    if (num_prefill < 0 || total_chunk_len < 0 || num_decode < 0 || num_heads <= 0 || num_kv_heads <= 0 ||
        num_heads % num_kv_heads || head_dim <= 0 || block_size <= 0 || max_context_len < 0)
        return 0;
    const size_t dec = mixed_decode_region(num_decode, num_heads, num_kv_heads, head_dim, block_size,
                                           max_context_len, partition_tokens);
    const size_t pre = num_prefill > 0 ? pa_prefill_workspace_bytes(num_prefill, total_chunk_len, num_heads,
                                                                    num_kv_heads, head_dim)
                                       : 0;
    return dec + pre;
}

}  // extern "C"

namespace {

// The step as one launch (pa::launch_mixed) when the shape allows it; returns
// PA_ERR_UNSUPPORTED (having queued nothing) when it does not.
int mixed_fused(void *prefill_out, const void *prefill_query, const int32_t *prefill_block_tables,
                int prefill_max_blocks, const int *prefix_lens, const int *chunk_lens, int num_prefill,
                void *decode_out, const void *decode_query, const int32_t *decode_block_tables, int decode_max_blocks,
                const int32_t *context_lens, int num_decode, int max_context_len, int partition_tokens,
                void *workspace, size_t workspace_bytes, const void *k_cache, const void *v_cache, int num_heads,
                int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale, pa_dtype dtype,
                int *d_err, void *stream) {
    const int group = num_heads / num_kv_heads;
    if (!pa::mixed_supported(head_dim, block_size, group) || max_context_len > kMixedMaxContext ||
        max_context_len <= 0 || !workspace || !good_dtype(dtype))
        return PA_ERR_UNSUPPORTED;
    if (!std::isfinite(scale) || !(scale > 0.f)) return PA_ERR_UNSUPPORTED;
    if (!prefill_out || !prefill_query || !prefill_block_tables || !prefix_lens || !chunk_lens || !decode_out ||
        !decode_query || !decode_block_tables || !context_lens || !k_cache || !v_cache)
        return PA_ERR_UNSUPPORTED;
    if (!aligned16(prefill_out) || !aligned16(prefill_query) || !aligned16(decode_out) ||
        !aligned16(decode_query) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_UNSUPPORTED;
    if (prefill_max_blocks <= 0 || decode_max_blocks <= 0 || num_blocks <= 0) return PA_ERR_UNSUPPORTED;
    // the prompt chunks, one launch's worth
    pa::PrefillParams pp{};
    pp.out = prefill_out;
    pp.query = prefill_query;
    pp.k_cache = k_cache;
    pp.v_cache = v_cache;
    pp.d_err = d_err;
    pp.num_heads = num_heads;
    pp.num_kv_heads = num_kv_heads;
    pp.num_blocks = num_blocks;
    pp.scale_log2 = scale * 1.4426950408889634f;
    long long rows = 0;
    int row = 0;
    for (int i = 0; i < num_prefill; ++i) {
        if (prefix_lens[i] < 0 || chunk_lens[i] < 0) return PA_ERR_UNSUPPORTED;
        if ((long long)prefix_lens[i] + chunk_lens[i] > (long long)prefill_max_blocks * block_size)
            return PA_ERR_UNSUPPORTED;
        if (chunk_lens[i] > 0) {
            if (pp.num_seqs == pa::kPrefillMaxSeqs) return PA_ERR_UNSUPPORTED;
            pa::PrefillSeq &q = pp.seqs[pp.num_seqs++];
            q.block_table = prefill_block_tables + (size_t)i * prefill_max_blocks;
            q.prefix_len = prefix_lens[i];
            q.chunk_len = chunk_lens[i];
            q.row_start = row;
        }
        row += chunk_lens[i];
        rows += chunk_lens[i];
    }
    if (pp.num_seqs == 0 || rows > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    pp.query_rows = (int)rows;
    // the decodes, one partition per sequence
    pa::DecodeParams dp{};
    dp.out = decode_out;
    dp.query = decode_query;
    dp.k_cache = k_cache;
    dp.v_cache = v_cache;
    dp.block_tables = decode_block_tables;
    dp.context_lens = context_lens;
    dp.d_err = d_err;
    dp.num_seqs = num_decode;
    dp.num_heads = num_heads;
    dp.num_kv_heads = num_kv_heads;
    dp.max_blocks_per_seq = decode_max_blocks;
    dp.num_blocks = num_blocks;
    dp.max_context_len = max_context_len;
    dp.block_size = block_size;
    dp.partition_tokens = (max_context_len + block_size - 1) / block_size * block_size;
    dp.max_partitions = 1;
    dp.scale_log2 = pp.scale_log2;
    dp.grp_size = 1;
    dp.grp_inner = group;
    dp.table_stride = decode_max_blocks;
    dp.slots = 1;
    const size_t dec = mixed_decode_region(num_decode, num_heads, num_kv_heads, head_dim, block_size, max_context_len,
                                           partition_tokens);
    if (workspace_bytes <= dec) return PA_ERR_UNSUPPORTED;
    // the decodes' K/V bytes, estimated from the longest context (lengths are on the device)
    const double decode_bytes = (double)num_decode * num_kv_heads * (0.5 * max_context_len) * head_dim * 2 * 2;
    const int rc = pa::launch_mixed(dtype, block_size, group, pp, dp, static_cast<char *>(workspace) + dec,
                                    workspace_bytes - dec, decode_bytes, static_cast<cudaStream_t>(stream));
    return rc == PA_ERR_WORKSPACE || rc == PA_ERR_ALIGNMENT ? PA_ERR_UNSUPPORTED : rc;
}

}  // namespace

extern "C" {

int pa_mixed_step(void *prefill_out, const void *prefill_query, const int32_t *prefill_block_tables,
                  int prefill_max_blocks, const int *prefix_lens, const int *chunk_lens, int num_prefill,
                  void *decode_out, const void *decode_query, const int32_t *decode_block_tables,
                  int decode_max_blocks, const int32_t *context_lens, int num_decode, int max_context_len,
                  int partition_tokens, void *workspace, size_t workspace_bytes, const void *k_cache,
                  const void *v_cache, int num_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks,
                  float scale, pa_dtype dtype, int *d_err, void *stream) {
    if (num_prefill < 0 || num_decode < 0) return PA_ERR_INVALID_ARG;
    if (num_prefill == 0 || num_decode == 0) {
        // one half only: no fork
        int rc = pa_prefill_batch(prefill_out, prefill_query, k_cache, v_cache, prefill_block_tables,
                                  num_prefill ? prefill_max_blocks : 1, prefix_lens, chunk_lens, num_prefill,
                                  num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, dtype, nullptr, 0,
                                  d_err, stream);
        if (rc != PA_OK) return rc;
        return pa_decode(decode_out, decode_query, k_cache, v_cache, decode_block_tables,
                         num_decode ? decode_max_blocks : 1, context_lens, num_decode, num_heads, num_kv_heads,
                         head_dim, block_size, num_blocks, max_context_len, scale, partition_tokens, dtype,
                         workspace, workspace_bytes, d_err, stream);
    }
    {
        // one launch when the shape and the workspace allow it
        const int rc = mixed_fused(prefill_out, prefill_query, prefill_block_tables, prefill_max_blocks, prefix_lens,
                                   chunk_lens, num_prefill, decode_out, decode_query, decode_block_tables,
                                   decode_max_blocks, context_lens, num_decode, max_context_len, partition_tokens,
                                   workspace, workspace_bytes, k_cache, v_cache, num_heads, num_kv_heads, head_dim,
                                   block_size, num_blocks, scale, dtype, d_err, stream);
        if (rc != PA_ERR_UNSUPPORTED) return rc;
    }
    std::lock_guard<std::mutex> guard(g_fork_mutex);
    ForkStream *f = nullptr;
    int rc = fork_stream(&f);
    if (rc != PA_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the prompt chunks go first, on the high-priority stream, so their CTAs
    // are placed before the decode's; the decode streams KV on the SMs the
    // chunks leave free, then on all of them
    if (cudaEventRecord(f->fork, st) != cudaSuccess || cudaStreamWaitEvent(f->stream, f->fork, 0) != cudaSuccess)
        return PA_ERR_CUDA;
    const int rc_pf = pa_prefill_batch(prefill_out, prefill_query, k_cache, v_cache, prefill_block_tables,
                                       prefill_max_blocks, prefix_lens, chunk_lens, num_prefill, num_heads,
                                       num_kv_heads, head_dim, block_size, num_blocks, scale, dtype, nullptr, 0, d_err,
                                       f->stream);
    const int rc_dec = pa_decode(decode_out, decode_query, k_cache, v_cache, decode_block_tables, decode_max_blocks,
                                 context_lens, num_decode, num_heads, num_kv_heads, head_dim, block_size,
                                 num_blocks, max_context_len, scale, partition_tokens, dtype, workspace,
                                 workspace_bytes, d_err, stream);
    // join even when a half failed, so the caller's stream never runs ahead of queued work
    if (cudaEventRecord(f->join, f->stream) != cudaSuccess || cudaStreamWaitEvent(st, f->join, 0) != cudaSuccess)
        return PA_ERR_CUDA;
    return rc_pf != PA_OK ? rc_pf : rc_dec;
}

}  // extern "C"
