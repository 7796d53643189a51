// The one-launch continuous-batching step's kernel and its launch templates:
// prompt-chunk CTAs (the stream-K prefill of pa_prefill.cuh) and decode
// instances (the tensor-core decode pipeline of pa_decode_tc.cuh) in one grid
// of one CTA per SM.  Instantiated per dtype in pa_mixed_bf16.cu and
// pa_mixed_f16.cu (compiled side by side); the host side is in pa_mixed.cu.
#pragma once

#include "pa_decode_tc.cuh"
#include "pa_prefill.cuh"

namespace pa {
namespace mx {
using namespace pf;

// ---- one launch of a continuous-batching step --------------------------------
//
// Every CTA runs two decode instances of six warps each, every instance the
// tensor-core decode's pipeline (its own three-slot ring, TMEM columns and
// softmax barrier) over units (sequence, kv head) drawn one after another from
// a queue the grid shares; CTAs 0 .. prefill_ctas-1 first run the prompt
// chunks exactly as the prefill kernel (stream-K over those CTAs; the two
// extra warps wait at its final barrier) and join the queue when their range
// is done.  Two instances keep as many K/V bytes in flight on an SM as two
// standalone decode CTAs, and the shared queue spreads long and short
// contexts, and the SMs the prompt chunks free, over the decodes as they go.
// The prefill CTAs keep the tensor cores busy while the decode CTAs stream
// K/V from HBM, in one grid of one CTA per SM, so neither half waits for the
// other to release SMs.
constexpr int kMixedThreads = kThreads + 32;  // twelve warps: two decode instances
constexpr int kDecodeSlotsMixed = tcd::kSlotsStandalone;
constexpr uint32_t kDecodeInst1 = (tcd::TcLayout<kDecodeSlotsMixed>::kSmemUsed + 1023u) & ~1023u;
constexpr uint32_t kMixedHolder = kOffBar + 248;  // TMEM base of a decode-only CTA (past the prefill's barriers)
static_assert(kMixedThreads == 2 * tcd::kThreads, "two decode instances");
static_assert(kDecodeInst1 + tcd::TcLayout<kDecodeSlotsMixed>::kSmemUsed <= (uint32_t)kOffBar,
              "both decode instances fit below the prefill's barriers");
static_assert((2 * kSlots + 2 + 2 * kQT) * 8 + 4 + 4 * kQT <= 248, "the holder is past the prefill's barriers");
static_assert(2 * tcd::kTmemCols <= kTmemCols, "both instances' columns in the prefill's allocation");

template <typename T, int BS, int G>
__global__ void __launch_bounds__(kMixedThreads, 1)
    mixed_tc_kernel(const __grid_constant__ MixedParams mp, const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmq) {
    const bool prefill = (int)blockIdx.x < mp.prefill_ctas;
    const int warp = threadIdx.x >> 5, inst = (int)threadIdx.x / tcd::kThreads;
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    volatile uint32_t *holder =
        reinterpret_cast<volatile uint32_t *>(smem_raw + (((raw + 1023u) & ~1023u) - raw) + kMixedHolder);
    uint32_t tmem = 0;
    if (prefill)  // ends with a CTA barrier: every warp is past the prefill's use of shared memory and TMEM
        tmem = prefill_cta<T, BS, G, true>(mp.pp, tmk, tmv, tmq, (int)blockIdx.x, mp.prefill_ctas);
    tcd::TcRun r;
    tcd::tc_init<kDecodeSlotsMixed>(r, inst * kDecodeInst1, inst * 6, kBarL + 1 + inst);
    if (!prefill && warp == 1) tcd::tc_alloc(holder, 2 * tcd::kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (!prefill) tmem = *holder;
    r.tmem = tmem + inst * tcd::kTmemCols;
    tcd::tc_queue_loop<T, BS, G, kDecodeSlotsMixed>(mp.dp, &tmk, &tmv, r, mp.decode_next, mp.decode_units,
                                                    2 * (int)gridDim.x);
    tcd::tc_drain<kDecodeSlotsMixed>(r);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tcd::tc_dealloc(tmem, prefill ? (uint32_t)kTmemCols : 2 * tcd::kTmemCols);
}

template <typename T, int BS, int G>
int launch_mixed_t(const MixedParams &mp, unsigned grid, cudaStream_t stream) {
    auto kern = mixed_tc_kernel<T, BS, G>;
    static std::atomic<uint64_t> attr_done{0};
    if (ensure_smem_attr(kern, kSmemAlloc, attr_done) != PA_OK) return PA_ERR_CUDA;
    const bool bf16 = std::is_same<T, __nv_bfloat16>::value;
    CUtensorMap tmk, tmv, tmq;
    if (!make_pool_map(&tmk, mp.pp.k_cache, mp.pp, BS, bf16) || !make_pool_map(&tmv, mp.pp.v_cache, mp.pp, BS, bf16) ||
        !make_query_map(&tmq, mp.pp, G, bf16))
        return PA_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kMixedThreads);
    cfg.dynamicSmemBytes = kSmemAlloc;
    cfg.stream = stream;
    // launched in plain stream order: launched early behind the cache write
    // (which lets dependents start at once), the step measured about 0.17 ms
    // slower, its CTAs starting that much later
    return cudaLaunchKernelEx(&cfg, kern, mp, tmk, tmv, tmq) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

template <typename T, int G>
int launch_mixed_group(int block_size, const MixedParams &mp, unsigned grid, cudaStream_t stream) {
    switch (block_size) {
        case 16: return launch_mixed_t<T, 16, G>(mp, grid, stream);
        case 32: return launch_mixed_t<T, 32, G>(mp, grid, stream);
        case 64: return launch_mixed_t<T, 64, G>(mp, grid, stream);
        case 128: return launch_mixed_t<T, 128, G>(mp, grid, stream);
        default: return PA_ERR_UNSUPPORTED;
    }
}

// Head groups of 2, 4 and 8 query heads per kv head: the decode instances
// run the tensor-core decode for any group up to 8 (the heads fill the first
// G of the MMA's 16 N rows), the chunks the prefill's G.
template <typename T>
int launch_mixed_dtype(int block_size, int group, const MixedParams &mp, unsigned grid, cudaStream_t stream) {
    switch (group) {
        case 2: return launch_mixed_group<T, 2>(block_size, mp, grid, stream);
        case 4: return launch_mixed_group<T, 4>(block_size, mp, grid, stream);
        case 8: return launch_mixed_group<T, 8>(block_size, mp, grid, stream);
        default: return PA_ERR_UNSUPPORTED;
    }
}

}  // namespace mx
}  // namespace pa
