// Chunked-prefill attention on the 5th-generation tensor cores (tcgen05).
//
// Follows the page "vLLM PagedAttention chuyen sau" (locionic.com), section
// "Chunked Prefill": each chunk of a long prompt attends to the sequence's
// paged cache built so far.  Query row i of the chunk sits at position
// prefix_len + i and sees keys 0 .. prefix_len + i, gathered through the
// block table.
//
// One CTA computes two tiles of 128 query rows -- 256/G chunk positions times
// the G query heads of one kv head -- against 128-key tiles that both Q tiles
// share (each K/V byte brought into shared memory serves 256 rows).
//   warp 0    TMA producer: for each key tile, one 4-D tensor copy per block
//             of K and of V, straight from the paged pool into a
//             128-byte-swizzled shared layout in which the tile's 8-key groups
//             sit 2 KB apart and the two 64-dim halves 1 KB apart inside each
//             group (uniform strides across the tile's blocks, so one
//             descriptor covers the tile, and one copy per block instead of
//             one per (block, half): the copy engine's cost is per copy).  K
//             and V have rings of their own (two stages each): K(j) is free
//             once the QKs of tile j ran, a whole MMA round before V(j), so
//             K(j+2) streams in while V(j) is still in use.  Block-table
//             entries are read 32 at a time, a chunk ahead;
//   warp 1    MMA issuer (one thread): per key tile j and Q tile g, first
//             O_g += P_g(j-1) V(j-1), then S_g = Q_g K(j)^T, tcgen05.mma
//             kind::f16 with fp32 accumulation in TMEM.  P_g is written over
//             the first half of S_g's TMEM columns and read from there as the
//             A operand; the tensor pipe runs one thread's MMAs in order, so
//             the PV of tile j-1 has read P before the QK of tile j writes S,
//             and S_g(j) being complete means O_g holds every PV up to j-1;
//   warps 2-5 softmax of Q tile 0, warps 6-9 of Q tile 1: each thread owns one
//             query row = one TMEM lane; it reads its S row, applies the causal
//             mask, updates the running max (rescaling O in TMEM only when the
//             max grows by more than 2^8), writes P (rounded to the input
//             type) into TMEM, and finally normalises O and stores the row.
//             The two groups interleave, so the tensor pipe works on one Q
//             tile's MMAs while the other's softmax runs.  On the last key tile
//             each group zeroes the V rows past the CTA's last key, so garbage
//             (even NaN) in unused slots never reaches O.
// All waits are bounded; a wait that gives up flags PA_DEVERR_TIMEOUT.
#include <cuda.h>

#include <type_traits>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_tcgen05.cuh"

namespace pa {
namespace {

constexpr int kD = 128;                        // head_dim
constexpr int kM = 128;                        // query rows per Q tile (one per TMEM lane)
constexpr int kQT = 2;                         // Q tiles per CTA
constexpr int kNK = 128;                       // keys per tile
constexpr int kStages = 2;                     // K/V tiles in flight
constexpr int kQHalf = kM * 128;               // one 64-dim half of a Q tile: 128 rows x 128 bytes
constexpr int kQTile = 2 * kQHalf;             // 32 KB
constexpr int kKVTile = kNK * kD * 2;          // 32 KB: [16 key groups][2 dim halves][8 keys][128 B]
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQT * kQTile;                // 64 KB: K ring
constexpr int kOffV = kOffK + kStages * kKVTile;           // 128 KB: V ring
constexpr int kOffBar = kOffV + kStages * kKVTile;         // 192 KB
constexpr int kSmemUsed = kOffBar + 256;
constexpr int kSmemAlloc = kSmemUsed + 1024;               // room to align the base to 1 KB
constexpr int kThreads = 64 + kQT * 128;
// TMEM columns: S of each Q tile (128 fp32; P overwrites its first 64 columns
// as 128 packed pairs), O of each Q tile (128 fp32)
constexpr uint32_t kColS = 0, kColO = 256;
constexpr uint32_t kTmemCols = 512;

// ---- the kernel ------------------------------------------------------------

template <typename T, int BS, int G>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv) {
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr int kBlocksPerTile = kNK / BS;
    static_assert(kNK % BS == 0 && BS % 8 == 0 && 32 % kBlocksPerTile == 0, "block_size");
    static_assert(kM % G == 0, "group");

    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t sb = (raw + 1023u) & ~1023u;  // 1 KB aligned: swizzle atoms start on 1 KB
    unsigned char *gb = smem_raw + (sb - raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(gb + kOffBar);
    uint64_t *k_full = bars + 0;                // [kStages] TMA -> MMA
    uint64_t *k_empty = bars + kStages;         // [kStages] MMA -> TMA
    uint64_t *v_full = bars + 2 * kStages;      // [kStages] TMA -> MMA
    uint64_t *v_empty = bars + 3 * kStages;     // [kStages] MMA -> TMA
    uint64_t *q_full = bars + 4 * kStages;      // softmax threads -> MMA (both Q tiles written)
    uint64_t *s_full = q_full + 1;              // [kQT] MMA -> softmax (S ready, O holds all PVs before it)
    uint64_t *p_full = s_full + kQT;            // [kQT] softmax -> MMA (S read, P written, O rescaled)
    uint64_t *o_done = p_full + kQT;            // [kQT] MMA -> softmax (last PV finished)
    volatile uint32_t *tmem_holder = reinterpret_cast<volatile uint32_t *>(o_done + kQT);
    static_assert((4 * kStages + 1 + 3 * kQT + 1) * 8 <= kSmemUsed - kOffBar, "barrier area");

    pdl_wait();  // the kernel before this one on the stream (the chunk's cache write) has finished
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kvh = blockIdx.y;
    // the sequence of this CTA: the last one whose first CTA is at or before it
    int si = 0;
    for (int i = 1; i < p.num_seqs; ++i)
        if (p.seqs[i].cta_start <= (int)blockIdx.x) si = i;
    const PrefillSeq &sq = p.seqs[si];
    const int prefix_len = sq.prefix_len, chunk_len = sq.chunk_len;
    const int cta = (int)blockIdx.x - sq.cta_start;  // CTA index within the sequence
    const int row0 = cta * (kQT * kM);
    const int nrows = chunk_len * G;
    // key tiles up to the last key any row of this CTA sees
    const int i_last = max(0, min(chunk_len - 1, (row0 + kQT * kM - 1) / G));
    const int kend = prefix_len + i_last;
    const int ntiles = kend / kNK + 1;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
        }
        mbar_init(q_full, kQT * 128);
        for (int g = 0; g < kQT; ++g) {
            mbar_init(&s_full[g], 1);
            mbar_init(&p_full[g], 128);
            mbar_init(&o_done[g], 1);
        }
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

    if (warp == 0) {
        // ============================================================ producer
        const int32_t *table = sq.block_table;
        const int oob = p.num_blocks * p.num_kv_heads * (BS / 8);  // first 8-row group past the pool: zero fill
        const uint64_t pol = policy_evict_last();  // every row tile of this kv head reads the same K/V
        // Table entries come 32 at a time, one per lane, a whole chunk ahead of
        // use (a chunk covers 32 / kBlocksPerTile tiles), so the producer never
        // waits on a table load; lane b < kBlocksPerTile handles block b of a tile.
        const int nent = kend / BS + 1;
        auto chunk = [&](int c) { return c * 32 + lane < nent ? table[c * 32 + lane] : -1; };
        int ent_cur = chunk(0), ent_nxt = chunk(1);
        constexpr int kTilesPerChunk = 32 / kBlocksPerTile;
        // first 8-row group of block `lane` of tile j in the pool (zero fill when past kend)
        auto tile_y = [&](int j, int blk) {
            int y = oob;
            if (lane < kBlocksPerTile && j * kNK + lane * BS <= kend) {
                if (blk >= 0 && blk < p.num_blocks) y = (blk * p.num_kv_heads + kvh) * (BS / 8);
                else flag_error(p.d_err, PA_DEVERR_BLOCK_RANGE);
            }
            return y;
        };
        auto load = [&](const CUtensorMap *map, uint64_t *full, uint64_t *empty, uint32_t ring, int j, int y) {
            const int st = j % kStages;
            if (lane == 0) {
                if (j >= kStages) wait_or_flag(&empty[st], (uint32_t)(j / kStages - 1) & 1u, p.d_err);
                mbar_arrive_expect_tx(&full[st], (uint32_t)kKVTile);
            }
            __syncwarp();
            // block `lane`: both 64-dim halves of its BS rows, BS * 256 bytes
            if (lane < kBlocksPerTile) tma_4d(ring + st * kKVTile + lane * (BS * 256), map, y, &full[st], pol);
        };
        // order: K(0), then K(j) before V(j-1) -- both are first needed by the
        // same MMA round, and K(j)'s slot frees up earlier
        int y_prev = oob;
        for (int j = 0; j < ntiles; ++j) {
            if (j > 0 && j % kTilesPerChunk == 0) {
                ent_cur = ent_nxt;
                ent_nxt = chunk(j / kTilesPerChunk + 1);
            }
            const int blk = __shfl_sync(0xffffffffu, ent_cur, (j % kTilesPerChunk) * kBlocksPerTile + (lane % kBlocksPerTile));
            const int y = tile_y(j, blk);
            load(&tmk, k_full, k_empty, sb + kOffK, j, y);
            if (j >= 1) load(&tmv, v_full, v_empty, sb + kOffV, j - 1, y_prev);
            y_prev = y;
        }
        load(&tmv, v_full, v_empty, sb + kOffV, ntiles - 1, y_prev);
        // every copy has normally been consumed by now; after a timeout, let
        // the ones in flight land before the CTA can exit
        if (lane == 0) {
            for (int j = max(0, ntiles - kStages); j < ntiles; ++j) {
                mbar_wait(&k_full[j % kStages], (uint32_t)(j / kStages) & 1u);
                mbar_wait(&v_full[j % kStages], (uint32_t)(j / kStages) & 1u);
            }
        }
    } else if (warp == 1) {
        // ============================================================ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = instr_desc(kBf16, false, false, kM, kNK);
            constexpr uint32_t idesc_pv = instr_desc(kBf16, false, true, kM, kD);
            constexpr uint32_t hi_q = desc_hi(1024);   // Q: 8-row groups 1 KB apart
            constexpr uint32_t hi_kv = desc_hi(2048);  // K, V: 8-key groups 2 KB apart
            // descriptor low words of Q tile 0 and of stage 0's K and V; the
            // rest are fixed offsets from these
            const uint32_t q_lo0 = desc_lo(sb + kOffQ, 16);
            const uint32_t k_lo0 = desc_lo(sb + kOffK, 16);     // K-major: leading offset unused
            const uint32_t v_lo0 = desc_lo(sb + kOffV, 1024);   // MN-major: second 64-dim half 1 KB on
            wait_or_flag(q_full, 0, p.d_err);
            tc_fence_after();
            for (int j = 0; j <= ntiles; ++j) {
                const int st = j % kStages, stp = (j + kStages - 1) % kStages;
                if (j >= 1) wait_or_flag(&v_full[stp], (uint32_t)((j - 1) / kStages) & 1u, p.d_err);
#pragma unroll
                for (int g = 0; g < kQT; ++g) {
                    const uint32_t tS = tmem + kColS + g * kNK;
                    if (j >= 1) {
                        // O_g += P_g(j-1) V(j-1); P sits in S_g's first 64 columns
                        wait_or_flag(&p_full[g], (uint32_t)(j - 1) & 1u, p.d_err);
                        tc_fence_after();
                        const uint32_t v_lo = v_lo0 + stp * (kKVTile >> 4);
#pragma unroll
                        for (int kk = 0; kk < kNK / 16; ++kk)
                            mma_f16_ts(tmem + kColO + g * kD, tS + kk * 8, desc_of(v_lo + kk * (4096 >> 4), hi_kv),
                                       idesc_pv, j > 1 || kk > 0);
                        if (j == ntiles) mma_commit(&o_done[g]);
                        // release V(j-1)'s slot only if the producer will wait for it
                        if (g == kQT - 1 && j - 1 + kStages < ntiles) mma_commit(&v_empty[stp]);
                    }
                    if (j < ntiles) {
                        if (g == 0) {
                            wait_or_flag(&k_full[st], (uint32_t)(j / kStages) & 1u, p.d_err);
                            tc_fence_after();
                        }
                        // S_g = Q_g K(j)^T
                        const uint32_t q_lo = q_lo0 + g * (kQTile >> 4);
                        const uint32_t k_lo = k_lo0 + st * (kKVTile >> 4);
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint32_t qo = ((kk >> 2) * kQHalf + (kk & 3) * 32) >> 4;
                            const uint32_t ko = ((kk >> 2) * 1024 + (kk & 3) * 32) >> 4;
                            mma_f16(tS, desc_of(q_lo + qo, hi_q), desc_of(k_lo + ko, hi_kv), idesc_qk, kk > 0);
                        }
                        mma_commit(&s_full[g]);
                        if (g == kQT - 1 && j + kStages < ntiles) mma_commit(&k_empty[st]);
                    }
                }
            }
        }
    } else {
        // ============================================================ softmax
        const int g = (warp - 2) >> 2;         // Q tile of this warp group
        const int quarter = warp & 3;          // TMEM lanes 32*quarter .. +31 (fixed by the warp id)
        const int t = quarter * 32 + lane;     // query row of this thread within its Q tile = TMEM lane
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const int gr = row0 + g * kM + t;
        const bool valid = gr < nrows;
        const int ipos = valid ? gr / G : 0, head = valid ? gr % G : 0;
        const int plim = prefix_len + min(gr / G, chunk_len - 1);
        const int plim_min = prefix_len + min((row0 + g * kM) / G, chunk_len - 1);  // smallest limit in the tile
        const float csc = p.scale_log2;                   // > 0 (checked on the host)
        const uint32_t tS = tmem + kColS + g * kNK + lane_off;
        const uint32_t tO = tmem + kColO + g * kD + lane_off;

        // Q row t into the swizzled K-major tile of this group
        {
            const uint4 *src = reinterpret_cast<const uint4 *>(
                static_cast<const T *>(p.query) + ((size_t)(sq.row_start + ipos) * p.num_heads + kvh * G + head) * kD);
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const uint4 v = valid ? src[c] : make_uint4(0, 0, 0, 0);
                const uint32_t dst =
                    sb + kOffQ + g * kQTile + (c >> 3) * kQHalf + t * 128 + (((c & 7) ^ (t & 7)) << 4);
                asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(v.x), "r"(v.y), "r"(v.z),
                             "r"(v.w)
                             : "memory");
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive1(q_full);
        }

        float m_run = -INFINITY;  // running max in scaled log2 units
        float2 l2[4];             // row sum as four pairs of partial sums
#pragma unroll
        for (int e = 0; e < 4; ++e) l2[e] = make_float2(0.f, 0.f);
        for (int j = 0; j < ntiles; ++j) {
            wait_or_flag(&s_full[g], (uint32_t)j & 1u, p.d_err);
            tc_fence_after();
            // causal mask only on tiles that reach past some row's limit
            const int kb = j * kNK;
            const bool need_mask = kb + kNK - 1 > plim_min;
            // pass 1: row max, 64 columns at a time (128 live values would spill)
            float mx8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) mx8[e] = -INFINITY;
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                float s0[32], s1[32];
                tmem_ld32(tS + h * 64, s0);
                tmem_ld32(tS + h * 64 + 32, s1);
                tmem_wait_ld();
                float s[64];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    s[e] = s0[e];
                    s[32 + e] = s1[e];
                }
                if (need_mask) {
#pragma unroll
                    for (int c = 0; c < 64; ++c) s[c] = (kb + h * 64 + c <= plim) ? s[c] : -INFINITY;
                }
#pragma unroll
                for (int c = 0; c < 64; ++c) mx8[c & 7] = fmaxf(mx8[c & 7], s[c]);
            }
            float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
            mx *= csc;

            // Lazy rescale.  The TMEM loads and stores are warp-collective, so
            // the warp decides together: lanes whose maximum did not grow past
            // the threshold scale by 1.
            const bool up = mx > m_run + 8.0f;
            if (__any_sync(kFull, up)) {
                const float m_new = up ? mx : m_run;
                if (j >= 1) {
                    // S(j) complete means O holds every PV before it: rescale in place
                    const float alpha = !up ? 1.f : (m_run == -INFINITY ? 0.f : fast_exp2(m_run - m_new));
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float v[32];
                        tmem_ld32(tO + c * 32, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] *= alpha;
                        tmem_st32(tO + c * 32, v);
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) l2[e] = __fmul2_rn(l2[e], make_float2(alpha, alpha));
                }
                m_run = m_new;
            }
            // pass 2: P row t = 2^(s*scale - max), rounded to the input type,
            // packed over S's first 64 columns (half h goes to columns 32h..32h+31,
            // which pass 2 of half h-1 has already read)
            const float2 csc2 = make_float2(csc, csc), negm2 = make_float2(-m_run, -m_run);
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                float s0[32], s1[32];
                tmem_ld32(tS + h * 64, s0);
                tmem_ld32(tS + h * 64 + 32, s1);
                tmem_wait_ld();
                float s[64];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    s[e] = s0[e];
                    s[32 + e] = s1[e];
                }
                if (need_mask) {
#pragma unroll
                    for (int c = 0; c < 64; ++c) s[c] = (kb + h * 64 + c <= plim) ? s[c] : -INFINITY;
                }
                // exponent arguments and row sums in packed fp32x2 arithmetic
                uint32_t pk[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const float2 a = __ffma2_rn(make_float2(s[2 * c], s[2 * c + 1]), csc2, negm2);
                    const float2 q = make_float2(fast_exp2(a.x), fast_exp2(a.y));
                    l2[c & 3] = __fadd2_rn(l2[c & 3], q);
                    pk[c] = Elem<T>::pack2(q.x, q.y);
                }
                tmem_st32u(tS + h * 32, pk);
            }
            if (j == ntiles - 1 && kb + kNK - 1 > kend) {
                // V rows past the last key any row sees hold whatever the pool
                // has there (possibly NaN, and 0 * NaN poisons O): zero them
                const int st_kv = j % kStages;
                wait_or_flag(&v_full[st_kv], (uint32_t)(j / kStages) & 1u, p.d_err);
                const int z0 = kend + 1 - kb;
                const uint32_t v_s = sb + kOffV + st_kv * kKVTile;
                for (int idx = t; idx < (kNK - z0) * 16; idx += 128) {
                    const int r = z0 + (idx >> 4), h = (idx >> 3) & 1, c = idx & 7;
                    asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(
                                     v_s + (r >> 3) * 2048 + h * 1024 + (r & 7) * 128 + c * 16),
                                 "r"(0u)
                                 : "memory");
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive1(&p_full[g]);
        }

        // epilogue: O row / l, rounded once, stored
        wait_or_flag(&o_done[g], 0, p.d_err);
        tc_fence_after();
        const float l_run = ((l2[0].x + l2[0].y) + (l2[1].x + l2[1].y)) + ((l2[2].x + l2[2].y) + (l2[3].x + l2[3].y));
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        T *orow = static_cast<T *>(p.out) + ((size_t)(sq.row_start + ipos) * p.num_heads + kvh * G + head) * kD;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float v[32];
            tmem_ld32(tO + c * 32, v);
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

// The pool as a 4-D tensor {64 dims, 8 rows, 2 dim halves, 8-row groups}
// with strides {2, 256, 128, 2048} bytes; a box is one block (block_size / 8
// groups), landing as [group][half][8 rows][128 B], 128-byte swizzled.
bool make_pool_map(CUtensorMap *map, const void *pool, const PrefillParams &p, int bs, bool bf16) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {64, 8, 2, (cuuint64_t)p.num_blocks * p.num_kv_heads * (bs / 8)};
    const cuuint64_t strides[3] = {(cuuint64_t)kD * 2, 128, (cuuint64_t)8 * kD * 2};
    const cuuint32_t box[4] = {64, 8, 2, (cuuint32_t)(bs / 8)};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
              const_cast<void *>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T, int BS, int G>
int launch_tc_t(const PrefillParams &p, cudaStream_t stream) {
    auto kern = prefill_tc_kernel<T, BS, G>;
    static std::atomic<uint64_t> attr_done{0};
    if (ensure_smem_attr(kern, kSmemAlloc, attr_done) != PA_OK) return PA_ERR_CUDA;
    const bool bf16 = std::is_same<T, __nv_bfloat16>::value;
    CUtensorMap tmk, tmv;
    if (!make_pool_map(&tmk, p.k_cache, p, BS, bf16) || !make_pool_map(&tmv, p.v_cache, p, BS, bf16))
        return PA_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.num_ctas, p.num_kv_heads);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemAlloc;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    // programmatic dependent launch: scheduled while the cache write drains
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p, tmk, tmv) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

template <typename T>
int launch_tc_dtype(int block_size, int group, const PrefillParams &p, cudaStream_t stream) {
#define PA_TC_CASE(BB, GG) \
    if (block_size == BB && group == GG) return launch_tc_t<T, BB, GG>(p, stream);
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

int launch_prefill(pa_dtype dt, int head_dim, int block_size, int group, const PrefillParams &p_in,
                   cudaStream_t stream) {
    if (head_dim != kD) return PA_ERR_UNSUPPORTED;
    // TMA row coordinates are 32-bit
    if ((long long)p_in.num_blocks * p_in.num_kv_heads * block_size >= (1LL << 31)) return PA_ERR_UNSUPPORTED;
    if (p_in.num_seqs < 1 || p_in.num_seqs > kPrefillMaxSeqs) return PA_ERR_INVALID_ARG;
    // each sequence's CTAs: its rows (chunk positions x group) in tiles of kQT*kM
    PrefillParams p = p_in;
    long long ctas = 0;
    for (int i = 0; i < p.num_seqs; ++i) {
        p.seqs[i].cta_start = (int)ctas;
        const long long rows = (long long)p.seqs[i].chunk_len * group;
        const long long tiles = (rows + kQT * kM - 1) / (kQT * kM);
        ctas += tiles;
    }
    if (ctas == 0) return PA_OK;
    if (ctas > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    p.num_ctas = (int)ctas;
    return dt == PA_BF16 ? launch_tc_dtype<__nv_bfloat16>(block_size, group, p, stream)
                         : launch_tc_dtype<__half>(block_size, group, p, stream);
}

}  // namespace pa
