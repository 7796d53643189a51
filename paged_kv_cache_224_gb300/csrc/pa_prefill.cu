// Chunked-prefill attention on the 5th-generation tensor cores (tcgen05).
//
// Follows the page "vLLM PagedAttention chuyen sau" (locionic.com), section
// "Chunked Prefill": each chunk of a long prompt attends to the sequence's
// paged cache built so far.  Query row i of the chunk sits at position
// prefix_len + i and sees keys 0 .. prefix_len + i, gathered through the
// block table.
//
// One CTA computes 128 query rows -- 128/G chunk positions times the G query
// heads of one kv head -- against 64-key tiles:
//   warp 0    TMA producer: for each key tile, one 2-D tensor copy per
//             (block, 64-dim half) of K and of V, straight from the paged pool
//             into a 128-byte-swizzled shared layout (four stages in flight);
//   warp 1    MMA issuer (one thread): S = Q K^T into TMEM (two buffers), then
//             O += P V into TMEM, tcgen05.mma kind::f16, fp32 accumulation;
//   warps 2-5 softmax: each thread owns one query row = one TMEM lane; reads
//             its S row, applies the causal mask, updates the running max
//             (rescaling O in TMEM only when the max grows by more than 2^8),
//             writes P (rounded to the input type) into one of two TMEM
//             buffers, the A operand of the PV MMA, and finally normalises O and stores the
//             row.  With two P buffers the softmax of tile j overlaps PV of
//             tile j-1; it waits for that PV only when O must be rescaled.
//             On the last tile it zeroes the V rows past the CTA's last key,
//             so garbage (even NaN) in unused slots never reaches O.
// All waits are bounded; a wait that gives up flags PA_DEVERR_TIMEOUT.
#include <cuda.h>

#include <type_traits>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kD = 128;                        // head_dim
constexpr int kM = 128;                        // query rows per CTA
constexpr int kNK = 64;                        // keys per tile
constexpr int kStages = 4;                     // K/V tiles in flight
constexpr int kQHalf = kM * 128;               // one 64-dim half of Q: 128 rows x 128 bytes
constexpr int kKVHalf = kNK * 128;             // one 64-dim half of a K or V tile
constexpr int kKVTile = 2 * kKVHalf;           // 16 KB
constexpr int kStageBytes = 2 * kKVTile;       // K tile + V tile
constexpr int kOffQ = 0;
constexpr int kOffKV = kOffQ + 2 * kQHalf;                 // 32 KB
constexpr int kOffBar = kOffKV + kStages * kStageBytes;    // 160 KB
constexpr int kSmemUsed = kOffBar + 256;
constexpr int kSmemAlloc = kSmemUsed + 1024;               // room to align the base to 1 KB
constexpr int kThreads = 192;
// TMEM columns: S0, S1 (64 fp32 each), P0, P1 (64 keys as 32 packed pairs each), O (128 fp32)
constexpr uint32_t kColS = 0, kColP = 128, kColO = 256;
constexpr uint32_t kTmemCols = 512;

// ---- tcgen05 / TMA wrappers (inline PTX) ---------------------------------

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: start, leading / stride byte offsets,
// descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, A and B both fp16 or
// both bf16, A K-major, B K-major or MN-major, M = 128, N given.
__host__ __device__ constexpr uint32_t instr_desc(bool bf16, bool b_mn_major, int n) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
           ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"((uint32_t)accumulate)
        : "memory");
}

// Same, with A read from tensor memory (row i in lane i, K pairs packed per column).
__device__ __forceinline__ void mma_f16_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc,
                                           bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
        "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"((uint32_t)accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32u(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void mbar_arrive1(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void wait_or_flag(uint64_t *bar, uint32_t parity, int *d_err) {
    if (!mbar_wait(bar, parity)) flag_error(d_err, PA_DEVERR_TIMEOUT);
}

// ---- the kernel ------------------------------------------------------------

template <typename T, int BS, int G>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv) {
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr int kBlocksPerTile = kNK / BS;
    static_assert(kNK % BS == 0 && kBlocksPerTile <= 32, "block_size");
    static_assert(kM % G == 0, "group");

    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t sb = (raw + 1023u) & ~1023u;  // 1 KB aligned: swizzle atoms start on 1 KB
    unsigned char *gb = smem_raw + (sb - raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(gb + kOffBar);
    uint64_t *kv_full = bars + 0;   // [kStages] TMA -> MMA
    uint64_t *kv_empty = bars + 4;  // [kStages] MMA -> TMA
    uint64_t *q_full = bars + 8;    // softmax threads -> MMA (Q tile written)
    uint64_t *s_full = bars + 9;    // [2] MMA -> softmax (S ready)
    uint64_t *s_free = bars + 11;   // [2] softmax -> MMA (S read)
    uint64_t *p_full = bars + 13;   // [2] softmax -> MMA (P buffer written, O rescaled)
    uint64_t *pv_done = bars + 15;  // [2] MMA -> softmax (PV of that P buffer finished)
    volatile uint32_t *tmem_holder = reinterpret_cast<volatile uint32_t *>(bars + 17);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kvh = blockIdx.y;
    const int row0 = blockIdx.x * kM;
    const int nrows = p.chunk_len * G;
    const int i_last = min(p.chunk_len - 1, (row0 + kM - 1) / G);
    const int kend = p.prefix_len + i_last;  // last key any row of this CTA sees
    const int ntiles = kend / kNK + 1;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&kv_full[i], 1);
            mbar_init(&kv_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_free[i], 128);
            mbar_init(&p_full[i], 128);
            mbar_init(&pv_done[i], 1);
        }
        mbar_init(q_full, 128);
        fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(const_cast<uint32_t *>(tmem_holder))),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const uint32_t tS0 = tmem + kColS, tP0 = tmem + kColP, tO = tmem + kColO;

    if (warp == 0) {
        // ============================================================ producer
        const int32_t *table = p.block_table;
        const int oob_row = p.num_blocks * p.num_kv_heads * BS;  // first row past the pool: zero fill
        // lane b < kBlocksPerTile handles block b of each tile; entries load one tile ahead
        auto entry = [&](int jt) {
            const int key0 = jt * kNK + lane * BS;
            return (lane < kBlocksPerTile && key0 <= kend) ? table[key0 / BS] : -1;
        };
        int blk_next = entry(0);
        for (int j = 0; j < ntiles; ++j) {
            const int st = j % kStages;
            const int blk = blk_next;
            if (j + 1 < ntiles) blk_next = entry(j + 1);
            int y = oob_row;
            if (lane < kBlocksPerTile && j * kNK + lane * BS <= kend) {
                if (blk >= 0 && blk < p.num_blocks) y = (blk * p.num_kv_heads + kvh) * BS;
                else flag_error(p.d_err, PA_DEVERR_BLOCK_RANGE);
            }
            if (lane == 0) {
                if (j >= kStages) wait_or_flag(&kv_empty[st], (uint32_t)(j / kStages - 1) & 1u, p.d_err);
                mbar_arrive_expect_tx(&kv_full[st], 2u * kKVTile);
            }
            __syncwarp();
            if (lane < kBlocksPerTile) {
                const uint32_t k_dst = sb + kOffKV + st * kStageBytes + lane * BS * 128;
                const uint32_t v_dst = k_dst + kKVTile;
                tma_2d(k_dst, &tmk, 0, y, &kv_full[st]);
                tma_2d(k_dst + kKVHalf, &tmk, 64, y, &kv_full[st]);
                tma_2d(v_dst, &tmv, 0, y, &kv_full[st]);
                tma_2d(v_dst + kKVHalf, &tmv, 64, y, &kv_full[st]);
            }
        }
    } else if (warp == 1) {
        // ============================================================ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = instr_desc(kBf16, false, kNK);
            constexpr uint32_t idesc_pv = instr_desc(kBf16, true, kD);
            const uint32_t q_s = sb + kOffQ;
            auto issue_pv = [&](int jj) {
                const int pb = jj & 1;
                const int stage = jj % kStages;
                wait_or_flag(&p_full[pb], (uint32_t)(jj >> 1) & 1u, p.d_err);
                tc_fence_after();
                const uint32_t v_s = sb + kOffKV + stage * kStageBytes + kKVTile;
#pragma unroll
                for (int kk = 0; kk < kNK / 16; ++kk) {
                    const uint64_t b = smem_desc(v_s + kk * 2048, kKVHalf, 1024);
                    mma_f16_ts(tO, tP0 + pb * (kNK / 2) + kk * 8, b, idesc_pv, jj > 0 || kk > 0);
                }
                mma_commit(&pv_done[pb]);
                mma_commit(&kv_empty[stage]);
            };
            wait_or_flag(q_full, 0, p.d_err);
            tc_fence_after();
            for (int j = 0; j < ntiles; ++j) {
                const int st = j % kStages;
                const int sbuf = j & 1;
                wait_or_flag(&kv_full[st], (uint32_t)(j / kStages) & 1u, p.d_err);
                if (j >= 2) wait_or_flag(&s_free[sbuf], (uint32_t)((j - 2) >> 1) & 1u, p.d_err);
                tc_fence_after();
                const uint32_t k_s = sb + kOffKV + st * kStageBytes;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    mma_f16(tS0 + sbuf * kNK, smem_desc(q_s + (kk >> 2) * kQHalf + (kk & 3) * 32, 16, 1024),
                            smem_desc(k_s + (kk >> 2) * kKVHalf + (kk & 3) * 32, 16, 1024), idesc_qk, kk > 0);
                }
                mma_commit(&s_full[sbuf]);
                if (j >= 1) issue_pv(j - 1);
            }
            issue_pv(ntiles - 1);
        }
    } else {
        // ============================================================ softmax
        const int quarter = warp & 3;
        const int t = quarter * 32 + lane;  // query row of this thread = TMEM lane
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const int gr = row0 + t;
        const bool valid = gr < nrows;
        const int ipos = valid ? gr / G : 0, head = valid ? gr % G : 0;
        const int plim = p.prefix_len + min(gr / G, p.chunk_len - 1);
        const int plim_cta = p.prefix_len + row0 / G;  // smallest limit of any row in the CTA
        const float csc = p.scale_log2;                 // > 0 (checked on the host)

        // Q row t into the swizzled K-major tile
        {
            const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const T *>(p.query) +
                                                               ((size_t)ipos * p.num_heads + kvh * G + head) * kD);
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const uint4 v = valid ? src[c] : make_uint4(0, 0, 0, 0);
                const uint32_t dst = sb + kOffQ + (c >> 3) * kQHalf + t * 128 + (((c & 7) ^ (t & 7)) << 4);
                asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(v.x), "r"(v.y), "r"(v.z),
                             "r"(v.w)
                             : "memory");
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive1(q_full);
        }

        float m_run = -INFINITY;  // running max in scaled log2 units
        float l8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) l8[e] = 0.f;
        for (int j = 0; j < ntiles; ++j) {
            const int st = j & 1;
            wait_or_flag(&s_full[st], (uint32_t)(j >> 1) & 1u, p.d_err);
            tc_fence_after();
            float s[kNK];
#pragma unroll
            for (int c = 0; c < kNK / 32; ++c) {
                float v[32];
                tmem_ld32(tS0 + st * kNK + lane_off + c * 32, v);
#pragma unroll
                for (int e = 0; e < 32; ++e) s[c * 32 + e] = v[e];
            }
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive1(&s_free[st]);

            // causal mask only on tiles that reach past some row's limit
            const int kb = j * kNK;
            if (kb + kNK - 1 > plim_cta) {
#pragma unroll
                for (int c = 0; c < kNK; ++c) s[c] = (kb + c <= plim) ? s[c] : -INFINITY;
            }
            float mx8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) mx8[e] = s[e];
#pragma unroll
            for (int c = 8; c < kNK; ++c) mx8[c & 7] = fmaxf(mx8[c & 7], s[c]);
            float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
            mx *= csc;

            // the P buffer of this tile was last read by PV of tile j-2
            const int pb = j & 1;
            if (j >= 2) {
                wait_or_flag(&pv_done[pb], (uint32_t)((j - 2) >> 1) & 1u, p.d_err);
                tc_fence_after();
            }
            if (mx > m_run + 8.0f) {
                if (j >= 1 && m_run != -INFINITY) {
                    // O must hold every PV so far before it is rescaled
                    wait_or_flag(&pv_done[(j - 1) & 1], (uint32_t)((j - 1) >> 1) & 1u, p.d_err);
                    tc_fence_after();
                    const float alpha = fast_exp2(m_run - mx);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float v[32];
                        tmem_ld32(tO + lane_off + c * 32, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] *= alpha;
                        tmem_st32(tO + lane_off + c * 32, v);
                    }
                    tmem_wait_st();
#pragma unroll
                    for (int e = 0; e < 8; ++e) l8[e] *= alpha;
                }
                m_run = mx;
            }
            // P row t = 2^(s*scale - max), rounded to the input type, into TMEM lane t
            const float neg_m = -m_run;
            uint32_t pk[kNK / 2];
#pragma unroll
            for (int c = 0; c < kNK / 8; ++c) {
                float pr[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    pr[e] = fast_exp2(fmaf(s[c * 8 + e], csc, neg_m));
                    l8[e] += pr[e];
                }
                const uint4 u = pack8<T>(pr);
                pk[c * 4 + 0] = u.x;
                pk[c * 4 + 1] = u.y;
                pk[c * 4 + 2] = u.z;
                pk[c * 4 + 3] = u.w;
            }
            tmem_st32u(tP0 + pb * (kNK / 2) + lane_off, pk);
            if (j == ntiles - 1 && kb + kNK - 1 > kend) {
                // V rows past the last key any row sees hold whatever the pool
                // has there (possibly NaN, and 0 * NaN poisons O): zero them
                const int st_kv = j % kStages;
                wait_or_flag(&kv_full[st_kv], (uint32_t)(j / kStages) & 1u, p.d_err);
                const int z0 = kend + 1 - kb;
                const uint32_t v_s = sb + kOffKV + st_kv * kStageBytes + kKVTile;
                for (int idx = t; idx < (kNK - z0) * 16; idx += 128) {
                    const int r = z0 + (idx >> 4), h = (idx >> 3) & 1, c = idx & 7;
                    asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(v_s + h * kKVHalf + r * 128 + c * 16),
                                 "r"(0u)
                                 : "memory");
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive1(&p_full[pb]);
        }

        // epilogue: O row / l, rounded once, stored
        wait_or_flag(&pv_done[(ntiles - 1) & 1], (uint32_t)((ntiles - 1) >> 1) & 1u, p.d_err);
        tc_fence_after();
        const float l_run = ((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7]));
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        T *orow = static_cast<T *>(p.out) + ((size_t)ipos * p.num_heads + kvh * G + head) * kD;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float v[32];
            tmem_ld32(tO + lane_off + c * 32, v);
            tmem_wait_ld();
            if (valid) {
#pragma unroll
                for (int q8 = 0; q8 < 4; ++q8) {
                    float o8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) o8[e] = v[q8 * 8 + e] * inv;
                    *reinterpret_cast<uint4 *>(orow + c * 32 + q8 * 8) = pack8<T>(o8);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
    }
}

// ---- host side -------------------------------------------------------------

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

// The pool as a 2-D tensor [num_blocks*num_kv_heads*block_size rows][128]; a
// box is 64 elements (128 bytes) by block_size rows, 128-byte swizzled.
bool make_pool_map(CUtensorMap *map, const void *pool, const PrefillParams &p, int bs, bool bf16) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)p.num_blocks * p.num_kv_heads * bs};
    const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)bs};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
              const_cast<void *>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T, int BS, int G>
int launch_tc_t(const PrefillParams &p, cudaStream_t stream) {
    auto kern = prefill_tc_kernel<T, BS, G>;
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc) != cudaSuccess)
            return PA_ERR_CUDA;
        attr_set = true;
    }
    const bool bf16 = std::is_same<T, __nv_bfloat16>::value;
    CUtensorMap tmk, tmv;
    if (!make_pool_map(&tmk, p.k_cache, p, BS, bf16) || !make_pool_map(&tmv, p.v_cache, p, BS, bf16))
        return PA_ERR_CUDA;
    dim3 grid((p.chunk_len * G + kM - 1) / kM, p.num_kv_heads);
    kern<<<grid, kThreads, kSmemAlloc, stream>>>(p, tmk, tmv);
    return cudaPeekAtLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

template <typename T>
int launch_tc_dtype(int block_size, int group, const PrefillParams &p, cudaStream_t stream) {
#define PA_TC_CASE(BB, GG) \
    if (block_size == BB && group == GG) return launch_tc_t<T, BB, GG>(p, stream);
#define PA_TC_GROUPS(BB) PA_TC_CASE(BB, 1) PA_TC_CASE(BB, 2) PA_TC_CASE(BB, 4) PA_TC_CASE(BB, 8)
    PA_TC_GROUPS(16)
    PA_TC_GROUPS(32)
#undef PA_TC_GROUPS
#undef PA_TC_CASE
    return PA_ERR_UNSUPPORTED;
}

}  // namespace

int launch_prefill(pa_dtype dt, int head_dim, int block_size, int group, const PrefillParams &p,
                   cudaStream_t stream) {
    if (head_dim != kD) return PA_ERR_UNSUPPORTED;
    // TMA row coordinates are 32-bit
    if ((long long)p.num_blocks * p.num_kv_heads * block_size >= (1LL << 31)) return PA_ERR_UNSUPPORTED;
    return dt == PA_BF16 ? launch_tc_dtype<__nv_bfloat16>(block_size, group, p, stream)
                         : launch_tc_dtype<__half>(block_size, group, p, stream);
}

}  // namespace pa
