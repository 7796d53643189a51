// The chunked-prefill kernel and its launcher: one CTA per unit, or the
// persistent stream-K schedule over one CTA per SM (device code and the
// schedule in pa_prefill.cuh).
#include "pa_prefill.cuh"

namespace pa {
namespace {
using namespace pf;

template <typename T, int BS, int G>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ PrefillParams p, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmq) {
    pdl_wait();  // the kernel before this one on the stream (the chunk's cache write) has finished
    prefill_cta<T, BS, G>(p, tmk, tmv, tmq, (int)blockIdx.x, (int)gridDim.x);
}

template <typename T, int BS, int G>
int launch_tc_t(const PrefillParams &p, unsigned grid, cudaStream_t stream) {
    auto kern = prefill_tc_kernel<T, BS, G>;
    static std::atomic<uint64_t> attr_done{0};
    if (ensure_smem_attr(kern, kSmemAlloc, attr_done) != PA_OK) return PA_ERR_CUDA;
    const bool bf16 = std::is_same<T, __nv_bfloat16>::value;
    CUtensorMap tmk, tmv, tmq;
    if (!make_pool_map(&tmk, p.k_cache, p, BS, bf16) || !make_pool_map(&tmv, p.v_cache, p, BS, bf16) ||
        !make_query_map(&tmq, p, G, bf16))
        return PA_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemAlloc;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    // programmatic dependent launch: scheduled while the cache write drains
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p, tmk, tmv, tmq) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

template <typename T>
int launch_tc_dtype(int block_size, int group, const PrefillParams &p, unsigned grid, cudaStream_t stream) {
#define PA_TC_CASE(BB, GG) \
    if (block_size == BB && group == GG) return launch_tc_t<T, BB, GG>(p, grid, stream);
#define PA_TC_GROUPS(BB) PA_TC_CASE(BB, 1) PA_TC_CASE(BB, 2) PA_TC_CASE(BB, 4) PA_TC_CASE(BB, 8)
    PA_TC_GROUPS(16)
    PA_TC_GROUPS(32)
    PA_TC_GROUPS(64)
    PA_TC_GROUPS(128)
#undef PA_TC_GROUPS
#undef PA_TC_CASE
    return PA_ERR_UNSUPPORTED;
}
}  // namespace

size_t prefill_workspace_bytes(int num_seqs, long long total_chunk_len, int group, int num_kv_heads) {
    // units <= kv heads x (sum of ceil(chunk * group / rows per unit)) <= kv heads x (total rows / 256 + seqs)
    const long long units = (long long)num_kv_heads * ((total_chunk_len * group + kUnitRows - 1) / kUnitRows + num_seqs);
    return prefill_ws(sm_count(), units).total();
}

int launch_prefill(pa_dtype dt, int head_dim, int block_size, int group, const PrefillParams &p_in,
                   void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (head_dim != kD) return PA_ERR_UNSUPPORTED;
    // TMA row coordinates are 32-bit
    if ((long long)p_in.num_blocks * p_in.num_kv_heads * block_size >= (1LL << 31)) return PA_ERR_UNSUPPORTED;
    if (p_in.num_seqs < 1 || p_in.num_seqs > kPrefillMaxSeqs) return PA_ERR_INVALID_ARG;
    if (group < 1 || kM % group) return PA_ERR_UNSUPPORTED;
    PrefillParams p = p_in;
    long long units = 0;
    const int rc = prefill_schedule(p, group, &units);
    if (rc != PA_OK) return rc;
    if (units == 0) return PA_OK;
    const long long tiles = p.total_tiles;
    const long long ctas = std::min<long long>(sm_count(), tiles);
    // The layout depends on the device only (partial regions for one CTA per
    // SM, counters after them), never on the call: the counters must stay put
    // from one call to the next, since each call relies on the previous ones
    // having left them at zero.
    const PrefillWs ws = prefill_ws(sm_count(), units);
    // Stream-K pays when the units do not fill the GPU a couple of times over;
    // with more, one CTA per unit keeps the concurrently running units on the
    // same kv heads (whose K/V they share through L2) and the hardware
    // balances the tail.
    if (workspace) {
        if (workspace_bytes < ws.total()) return PA_ERR_WORKSPACE;
        if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PA_ERR_ALIGNMENT;
    }
    unsigned grid;
    if (workspace && units < 2LL * sm_count()) {
        char *base = static_cast<char *>(workspace);
        p.split = 1;
        p.part_o = reinterpret_cast<float *>(base);
        p.part_ml = reinterpret_cast<float2 *>(base + ws.o_bytes);
        // zero on entry: the caller zero-fills the workspace once, and the
        // segment that merges a unit resets its counter before the call ends
        p.counters = reinterpret_cast<unsigned *>(base + ws.cnt_off());
        grid = (unsigned)ctas;
    } else {
        p.split = 0;
        grid = (unsigned)units;
    }
    return dt == PA_BF16 ? launch_tc_dtype<__nv_bfloat16>(block_size, group, p, grid, stream)
                         : launch_tc_dtype<__half>(block_size, group, p, grid, stream);
}
}  // namespace pa
