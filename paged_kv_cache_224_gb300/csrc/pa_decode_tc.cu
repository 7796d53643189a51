// Paged decode attention for head groups of 8 on the tensor cores (tcgen05).
//
// Same operation and work units as the CUDA-core decode kernel (the three
// steps of the page "vLLM PagedAttention chuyen sau" (locionic.com), section
// "Co che PagedAttention": look up each logical block in the block table,
// gather its K/V rows, attend), for the shape where the CUDA cores run out of
// issue slots well below the HBM bound: with 8 query heads per kv head every
// K/V byte feeds 8 dot products and 8 weighted sums, and the group's scores
// and weighted sums are dense contractions.  (Smaller groups are HBM-bound on
// the CUDA cores and stay there; the kernel is written for any G up to 8.)
// Keys are the MMA's M dimension, so nothing is padded along the long axis:
//   S^T[128 keys][16] = K[128 keys][128 dims] . Q^T    (Q: the G heads, zero rows up to N = 16)
//   O^T[128 dims][16] += V^T[128 dims][128 keys] . P^T (V read in place, MN-major)
// fp32 accumulators in tensor memory.  P enters the MMA as two 16-bit rows
// per head, its rounding and the rounding residual, in the N padding (rows 8-15),
// so the PV product keeps P to about twice the input type's precision.
//
// One CTA = one unit (sequence, kv head, partition), 128-key tiles:
//   warp 0    TMA producer: one 4-D tensor copy per (block, K or V) from the
//             paged pool into a 128-byte-swizzled layout in which a tile's
//             8-key groups sit 2 KB apart with the two 64-dim halves 1 KB
//             apart inside each group -- uniform strides across the tile's
//             blocks, so one descriptor covers a whole tile.  A ring of three
//             32 KB slots holds K and V tiles in the order the MMAs consume
//             them: K(0), then K(j), V(j-1), ...;
//   warp 1    MMA issuer (one thread): QK^T of tile j into one of two S
//             buffers, then O += P V of tile j-1;
//   warps 2-5 softmax, one thread per key of the tile (= TMEM lane): read the
//             key's scores for 8 head slots (the G heads, then zero rows), mask keys past the unit, find each head's tile
//             maximum (warp reduce-scatter, then an exchange across the four
//             warps), rescale O in TMEM only when a head's maximum grows by
//             more than 2^8, write P^T for the PV MMA.  At the end each thread
//             owns one dimension (= TMEM lane of O^T) and writes it for the G
//             heads: the normalised output when the unit is a whole sequence,
//             else the unnormalised partial (acc, running max, sum) that the
//             log-sum-exp reduce merges.
// All waits are bounded; a wait that gives up flags PA_DEVERR_TIMEOUT.
#include "pa_decode_tc.cuh"

namespace pa {
namespace {

using namespace tcd;

template <typename T, int BS, int G>
__global__ void __launch_bounds__(kThreads, 2)
    decode_tc_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv) {
    pdl_wait();     // the kernel before this one on the stream (e.g. the cache write) has finished
    pdl_trigger();  // the reduce may be scheduled once every CTA of this grid has started
    const TcUnit u = tc_unit_of<BS>(p, (int)blockIdx.x, (int)threadIdx.x);
    if (u.skip) return;
    if (u.ntiles == 0) {
        tc_empty_unit<T, G>(p, u, (int)threadIdx.x);
        return;
    }
    TcRun r;
    tc_init<kSlotsStandalone>(r, 0, 0, 1);
    if (threadIdx.x >> 5 == 1) tc_alloc(r.tmem_holder, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    r.tmem = *r.tmem_holder;
    tc_unit<T, BS, G, kSlotsStandalone>(p, &tmk, &tmv, u, r);
    tc_drain<kSlotsStandalone>(r);
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x >> 5 == 1) tc_dealloc(r.tmem, kTmemCols);
}

// ---- host side -------------------------------------------------------------

// The pool as a 4-D tensor {64 dims, 8 rows, 2 dim halves, 8-row groups}
// (strides 2, 256, 128 and 2048 bytes): a block of block_size rows is one box
// of block_size/8 groups, which lands as [group][half][8 rows][128 bytes],
// 128-byte swizzled.
bool make_pool_map4(CUtensorMap *map, const void *pool, const DecodeParams &p, int bs, bool bf16) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {64, 8, 2, (cuuint64_t)p.num_blocks * p.num_kv_heads * (bs / 8)};
    const cuuint64_t strides[3] = {(cuuint64_t)kTD * 2, 128, (cuuint64_t)8 * kTD * 2};
    const cuuint32_t box[4] = {64, 8, 2, (cuuint32_t)(bs / 8)};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
              const_cast<void *>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T, int BS, int G>
int launch_tc_t(const DecodeParams &p, cudaStream_t stream) {
    auto kern = decode_tc_kernel<T, BS, G>;
    static std::atomic<uint64_t> attr_done{0};
    if (ensure_smem_attr(kern, TcLayout<kSlotsStandalone>::kSmemAlloc, attr_done) != PA_OK) return PA_ERR_CUDA;
    const bool bf16 = std::is_same<T, __nv_bfloat16>::value;
    CUtensorMap tmk, tmv;
    if (!make_pool_map4(&tmk, p.k_cache, p, BS, bf16) || !make_pool_map4(&tmv, p.v_cache, p, BS, bf16))
        return PA_ERR_UNSUPPORTED;  // the CUDA-core kernel takes over
    const long long units = (long long)p.max_partitions * p.num_seqs * p.num_kv_heads;
    if (units <= 0) return PA_OK;
    if (units > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    return launch_pdl(kern, dim3((unsigned)units), dim3(kThreads), TcLayout<kSlotsStandalone>::kSmemAlloc, stream, p,
                      tmk, tmv) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

template <typename T, int G>
int launch_tc_group(int block_size, const DecodeParams &p, cudaStream_t stream) {
    switch (block_size) {
        case 8: return launch_tc_t<T, 8, G>(p, stream);
        case 16: return launch_tc_t<T, 16, G>(p, stream);
        case 32: return launch_tc_t<T, 32, G>(p, stream);
        case 64: return launch_tc_t<T, 64, G>(p, stream);
        case 128: return launch_tc_t<T, 128, G>(p, stream);
        default: return PA_ERR_UNSUPPORTED;
    }
}

template <typename T>
int launch_tc_dtype(int block_size, int group, const DecodeParams &p, cudaStream_t stream) {
    switch (group) {
        case 8: return launch_tc_group<T, 8>(block_size, p, stream);
        default: return PA_ERR_UNSUPPORTED;
    }
}

}  // namespace

int launch_decode_tc(pa_dtype dt, int head_dim, int block_size, int group, const DecodeParams &p,
                     cudaStream_t stream) {
    if (head_dim != kTD || !decode_tc_group(group)) return PA_ERR_UNSUPPORTED;
    // TMA coordinates are 32-bit
    if ((long long)p.num_blocks * p.num_kv_heads * (block_size / 8) >= (1LL << 31)) return PA_ERR_UNSUPPORTED;
    return dt == PA_BF16 ? launch_tc_dtype<__nv_bfloat16>(block_size, group, p, stream)
                         : launch_tc_dtype<__half>(block_size, group, p, stream);
}

}  // namespace pa
