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
#include <cuda.h>

#include <type_traits>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_tcgen05.cuh"

namespace pa {
namespace {

constexpr int kTG = 8;                    // head slots: the group's G query heads, then zero rows
constexpr int kTN = 16;                   // MMA N: the slots padded to the smallest N allowed with M = 128
constexpr int kTD = 128;                  // head_dim
constexpr int kTK = 128;                  // keys per tile (M of the QK^T MMA)
constexpr int kSlot = kTK * kTD * 2;      // 32 KB: one K or V tile
constexpr int kSlots = 3;                 // ring slots
constexpr int kOffQ = kSlots * kSlot;     // Q^T: [2 dim halves][16 rows][128 B]
constexpr int kOffP = kOffQ + 4096;       // P^T: 2 buffers x [2 key halves][16 rows][128 B]
constexpr int kOffBar = kOffP + 2 * 4096;
constexpr int kOffXch = kOffBar + 256;    // [2][4 warps][8] tile maxima, then [4 warps][8] row sums
constexpr int kSmemUsed = kOffXch + (2 * 4 * kTG + 4 * kTG) * 4;
constexpr int kSmemAlloc = kSmemUsed + 1024;  // room to align the base to 1 KB
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 64;        // S^T x 2 buffers (16 columns each), O^T (16)
constexpr uint32_t kColS = 0, kColO = 32;
constexpr float kTcRescale = 8.0f;        // log2 units

// Reduce 8 per-lane values across the warp (max or sum); lane l ends with the
// result for value l >> 2.  Halving exchanges: each lane keeps the half of
// its values that its lane-index bit selects and sends the other half.
template <bool kMax>
__device__ __forceinline__ float warp_scatter8(const float (&v)[8], int lane) {
    auto op = [](float a, float b) { return kMax ? fmaxf(a, b) : a + b; };
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
    float a[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float keep = b4 ? v[k + 4] : v[k], send = b4 ? v[k] : v[k + 4];
        a[k] = op(keep, __shfl_xor_sync(kFull, send, 16));
    }
    float c[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const float keep = b3 ? a[k + 2] : a[k], send = b3 ? a[k] : a[k + 2];
        c[k] = op(keep, __shfl_xor_sync(kFull, send, 8));
    }
    float e = op(b2 ? c[1] : c[0], __shfl_xor_sync(kFull, b2 ? c[0] : c[1], 4));
    e = op(e, __shfl_xor_sync(kFull, e, 2));
    e = op(e, __shfl_xor_sync(kFull, e, 1));
    return e;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void sts16(uint32_t addr, uint16_t v) {
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

template <typename T, int BS, int G>
__global__ void __launch_bounds__(kThreads, 2)
    decode_tc_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv) {
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr int kBPT = kTK / BS;  // blocks per tile
    static_assert(kTK % BS == 0 && BS % 8 == 0 && 32 % kBPT == 0, "block_size");
    static_assert(G >= 1 && G <= kTG, "group");

    pdl_wait();     // the kernel before this one on the stream (e.g. the cache write) has finished
    pdl_trigger();  // the reduce may be scheduled once every CTA of this grid has started

    // ---- unit = (partition, sequence, kv head); partition-major order
    const int per_part = p.num_seqs * p.num_kv_heads;
    const int part = blockIdx.x / per_part;
    const int rem = blockIdx.x - part * per_part;
    const int s = rem / p.num_kv_heads;
    const int kvh = rem - s * p.num_kv_heads;

    int L;
    if (p.len_fixed > 0) {
        L = p.len_fixed;
    } else {
        L = p.context_lens[s] - p.len_offset;
        const int Lcap = min(p.max_context_len, p.max_blocks_per_seq * BS) - p.len_offset;
        if (L < 0 || L > Lcap) {
            if (threadIdx.x == 0 && part == 0 && kvh == 0) flag_error(p.d_err, PA_DEVERR_CONTEXT_RANGE);
            L = L < 0 ? 0 : Lcap;
        }
    }
    if (p.grp_size > 1 && part == 0 && kvh == 0 && threadIdx.x < 32) {
        // shared-prefix pass: every member's table must start with the leader's blocks
        const int32_t *lead = p.block_tables + (size_t)s * p.table_stride;
        bool same = true;
        for (int m = 1; m < p.grp_size; ++m) {
            const int32_t *row = lead + (size_t)m * p.max_blocks_per_seq;
            for (int j = threadIdx.x; j < L / BS; j += 32) same = same && row[j] == lead[j];
        }
        if (!same) flag_error(p.d_err, PA_DEVERR_PREFIX);
    }
    const int PT = p.partition_tokens;
    const int nparts = L > 0 ? (L + PT - 1) / PT : 1;
    if (part >= nparts) return;
    const int tok0 = part * PT;
    const int ntok = max(0, min(L, tok0 + PT) - tok0);
    const int ntiles = (ntok + kTK - 1) / kTK;
    const bool direct = nparts == 1 && !p.force_partials;
    // real query/out row of head h of this unit
    auto row_of = [&](int h) -> size_t {
        return (size_t)(s * p.grp_size + h / p.grp_inner) * p.num_heads + (size_t)kvh * p.grp_inner +
               h % p.grp_inner;
    };

    if (ntiles == 0) {
        // no keys: zeros, or an empty partial (max -inf, sum 0)
        if (threadIdx.x < G * 16) {
            const int h = threadIdx.x >> 4, c = threadIdx.x & 15;
            const size_t row = row_of(h);
            if (direct) {
                *reinterpret_cast<uint4 *>(static_cast<T *>(p.out) + row * kTD + c * 8) = make_uint4(0, 0, 0, 0);
            } else {
                const size_t slot = row * p.slots + p.part_base + part;
                float4 *dst = reinterpret_cast<float4 *>(p.ws_acc + slot * kTD + c * 8);
                dst[0] = make_float4(0.f, 0.f, 0.f, 0.f);
                dst[1] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (c == 0) p.ws_ml[slot] = make_float2(-INFINITY, 0.f);
            }
        }
        return;
    }

    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t sb = (raw + 1023u) & ~1023u;  // 1 KB aligned: swizzle atoms start on 1 KB
    unsigned char *gb = smem_raw + (sb - raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(gb + kOffBar);
    uint64_t *full = bars;                  // [kSlots] TMA -> MMA
    uint64_t *empty = bars + kSlots;        // [kSlots] MMA -> TMA
    uint64_t *q_full = bars + 2 * kSlots;   // softmax threads -> MMA (Q^T written)
    uint64_t *s_full = q_full + 1;          // [2] MMA -> softmax (S^T of a tile ready)
    uint64_t *p_full = s_full + 2;          // [2] softmax -> MMA (S read, P^T written, O rescaled)
    uint64_t *pv_done = p_full + 2;         // [2] MMA -> softmax (PV of a tile complete)
    volatile uint32_t *tmem_holder = reinterpret_cast<volatile uint32_t *>(pv_done + 2);
    static_assert((2 * kSlots + 7) * 8 + 4 <= kOffXch - kOffBar, "barrier area");
    float *xmax = reinterpret_cast<float *>(gb + kOffXch);  // [2][4][8]
    float *xsum = xmax + 2 * 4 * kTG;                       // [4][8]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(q_full, 128);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&p_full[b], 128);
            mbar_init(&pv_done[b], 1);
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

    // ring items in consumption order: K(0), then K(j), V(j-1) for j >= 1, then V(last)
    auto item_k = [](int j) { return j == 0 ? 0 : 2 * j - 1; };
    auto item_v = [ntiles](int j) { return j + 1 < ntiles ? 2 * j + 2 : 2 * j + 1; };

    if (warp == 0) {
        // ============================================================ producer
        const int32_t *table = p.block_tables + (size_t)s * p.table_stride + p.len_offset / BS + tok0 / BS;
        const int nblk = (ntok + BS - 1) / BS;
        const int oob = p.num_blocks * p.num_kv_heads * (BS / 8);  // first 8-row group past the pool: zero fill
        const uint64_t pol = policy_evict_first();
        // table entries 32 at a time, one per lane, a chunk ahead of use
        constexpr int kTilesPerChunk = 32 / kBPT;
        auto chunk = [&](int c) { return c * 32 + lane < nblk ? table[c * 32 + lane] : -1; };
        int ent_cur = chunk(0), ent_nxt = chunk(1);
        int item = 0;
        auto load = [&](const CUtensorMap *map, int y) {
            const int sl = item % kSlots;
            if (lane == 0) {
                if (item >= kSlots) wait_or_flag(&empty[sl], (uint32_t)(item / kSlots - 1) & 1u, p.d_err);
                mbar_arrive_expect_tx(&full[sl], (uint32_t)kSlot);
            }
            __syncwarp();
            if (lane < kBPT) tma_4d(sb + sl * kSlot + lane * (BS * 256), map, y, &full[sl], pol);
            ++item;
        };
        int y_prev = oob;
        for (int j = 0; j < ntiles; ++j) {
            if (j > 0 && j % kTilesPerChunk == 0) {
                ent_cur = ent_nxt;
                ent_nxt = chunk(j / kTilesPerChunk + 1);
            }
            const int e = __shfl_sync(kFull, ent_cur, (j % kTilesPerChunk) * kBPT + (lane % kBPT));
            int y = oob;
            if (lane < kBPT && j * kBPT + lane < nblk) {
                if (e >= 0 && e < p.num_blocks) y = (e * p.num_kv_heads + kvh) * (BS / 8);
                else flag_error(p.d_err, PA_DEVERR_BLOCK_RANGE);
            }
            load(&tmk, y);
            if (j >= 1) load(&tmv, y_prev);
            y_prev = y;
        }
        load(&tmv, y_prev);
        // every copy has normally been consumed by now; after a timeout, let
        // the ones in flight land before the CTA can exit
        if (lane == 0)
            for (int i = max(0, item - kSlots); i < item; ++i) mbar_wait(&full[i % kSlots], (uint32_t)(i / kSlots) & 1u);
    } else if (warp == 1) {
        // ============================================================ MMA issuer
        if (lane == 0) {
            constexpr uint32_t id_qk = instr_desc(kBf16, false, false, kTK, kTN);
            constexpr uint32_t id_pv = instr_desc(kBf16, true, false, kTD, kTN);
            constexpr uint32_t hi_kv = desc_hi(2048);  // K, V: 8-key groups 2 KB apart
            constexpr uint32_t hi_qp = desc_hi(1024);  // Q^T, P^T: 8-row groups 1 KB apart
            const uint32_t k_lo0 = desc_lo(sb, 16);     // K-major: leading offset unused
            const uint32_t v_lo0 = desc_lo(sb, 1024);   // MN-major: second 64-dim half 1 KB on
            const uint32_t q_lo = desc_lo(sb + kOffQ, 16);
            const uint32_t p_lo0 = desc_lo(sb + kOffP, 16);
            wait_or_flag(q_full, 0, p.d_err);
            tc_fence_after();
            for (int j = 0; j <= ntiles; ++j) {
                if (j < ntiles) {
                    // S^T(j) = K(j) Q^T into buffer j & 1 (its previous tile's
                    // softmax finished before the PV issued last iteration)
                    const int it = item_k(j), sl = it % kSlots;
                    wait_or_flag(&full[sl], (uint32_t)(it / kSlots) & 1u, p.d_err);
                    tc_fence_after();
                    const uint32_t tS = tmem + kColS + (j & 1) * kTN;
                    const uint32_t k_lo = k_lo0 + ((uint32_t)(sl * kSlot) >> 4);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t ko = (uint32_t)((kk >> 2) * 1024 + (kk & 3) * 32) >> 4;
                        const uint32_t qo = (uint32_t)((kk >> 2) * 2048 + (kk & 3) * 32) >> 4;
                        mma_f16(tS, desc_of(k_lo + ko, hi_kv), desc_of(q_lo + qo, hi_qp), id_qk, kk > 0);
                    }
                    mma_commit(&s_full[j & 1]);
                    mma_commit(&empty[sl]);
                }
                if (j >= 1) {
                    // O^T += V^T(j-1) P^T(j-1)
                    const int jj = j - 1;
                    wait_or_flag(&p_full[jj & 1], (uint32_t)(jj >> 1) & 1u, p.d_err);
                    const int it = item_v(jj), sl = it % kSlots;
                    wait_or_flag(&full[sl], (uint32_t)(it / kSlots) & 1u, p.d_err);
                    tc_fence_after();
                    const uint32_t v_lo = v_lo0 + ((uint32_t)(sl * kSlot) >> 4);
                    const uint32_t p_lo = p_lo0 + ((uint32_t)((jj & 1) * 4096) >> 4);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t vo = (uint32_t)(kk * 4096) >> 4;
                        const uint32_t po = (uint32_t)((kk >> 2) * 2048 + (kk & 3) * 32) >> 4;
                        mma_f16(tmem + kColO, desc_of(v_lo + vo, hi_kv), desc_of(p_lo + po, hi_qp), id_pv,
                                jj > 0 || kk > 0);
                    }
                    mma_commit(&pv_done[jj & 1]);
                    mma_commit(&empty[sl]);
                }
            }
        }
    } else {
        // ============================================================ softmax
        const int quarter = warp & 3;         // TMEM lanes 32*quarter .. +31 (fixed by the warp id)
        const int t = quarter * 32 + lane;    // key of the tile (S^T row) and dimension (O^T row)
        const int sw = warp - 2;              // index among the softmax warps
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const float csc = p.scale_log2;
        {
            // Q^T rows 0..G-1 = the group's query heads, the rest zero
            const uint4 z = make_uint4(0, 0, 0, 0);
            const int h = t >> 4, c = t & 15;
            const uint4 q = h < G ? *reinterpret_cast<const uint4 *>(static_cast<const T *>(p.query) +
                                                                     row_of(h) * kTD + c * 8)
                                  : z;
            sts128(sb + kOffQ + (c >> 3) * 2048 + h * 128 + (((c & 7) ^ h) << 4), q);
            sts128(sb + kOffQ + (c >> 3) * 2048 + (8 + h) * 128 + (((c & 7) ^ h) << 4), z);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive1(q_full);
        }

        float m_run[kTG], l_part[kTG];
#pragma unroll
        for (int h = 0; h < kTG; ++h) {
            m_run[h] = -INFINITY;
            l_part[h] = 0.f;
        }
        const int32_t *table = p.block_tables + (size_t)s * p.table_stride + p.len_offset / BS + tok0 / BS;
        for (int j = 0; j < ntiles; ++j) {
            const int b = j & 1;
            // this key's block must be in the pool (the producer flags a bad
            // entry and fetches zeros; the key is left out here); the load is
            // issued before the wait so its latency hides behind it
            const int key = j * kTK + t;
            const int ent = key < ntok ? table[key / BS] : -1;
            wait_or_flag(&s_full[b], (uint32_t)(j >> 1) & 1u, p.d_err);
            tc_fence_after();
            float sc[kTG];
            tmem_ld8(tmem + lane_off + kColS + b * kTN, sc);
            tmem_wait_ld();
            const bool valid = key < ntok && ent >= 0 && ent < p.num_blocks;
#pragma unroll
            for (int h = 0; h < kTG; ++h) sc[h] = valid ? sc[h] * csc : -INFINITY;
            // each head's maximum over the tile's 128 keys
            const float wmax = warp_scatter8<true>(sc, lane);
            if ((lane & 3) == 0) xmax[(b * 4 + sw) * kTG + (lane >> 2)] = wmax;
            named_bar_sync(1, 128);
            float tmax[kTG];
            {
                const float4 *x = reinterpret_cast<const float4 *>(xmax + b * 4 * kTG);
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const float4 lo = x[2 * w], hi = x[2 * w + 1];
                    const float v[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
                    for (int h = 0; h < kTG; ++h) tmax[h] = w == 0 ? v[h] : fmaxf(tmax[h], v[h]);
                }
            }
            // lazy rescale (the same decision in every thread)
            bool grow = false;
            float alpha[kTG];
#pragma unroll
            for (int h = 0; h < kTG; ++h) {
                const float nm = tmax[h] > m_run[h] + kTcRescale ? tmax[h] : m_run[h];
                alpha[h] = m_run[h] == -INFINITY ? 0.f : fast_exp2(m_run[h] - nm);
                grow |= nm != m_run[h];
                m_run[h] = nm;
            }
            if (grow && j > 0) {
                // O must hold the PV of tile j-1 before it is scaled
                wait_or_flag(&pv_done[(j - 1) & 1], (uint32_t)((j - 1) >> 1) & 1u, p.d_err);
                tc_fence_after();
                float o[2 * kTG];  // the P_hi and P_lo columns of each head
                tmem_ld16(tmem + lane_off + kColO, o);
                tmem_wait_ld();
#pragma unroll
                for (int h = 0; h < kTG; ++h) {
                    o[h] *= alpha[h];
                    o[kTG + h] *= alpha[h];
                    l_part[h] *= alpha[h];
                }
                tmem_st16(tmem + lane_off + kColO, o);
            }
            float pr[kTG];
#pragma unroll
            for (int h = 0; h < kTG; ++h) {
                pr[h] = valid ? fast_exp2(sc[h] - m_run[h]) : 0.f;  // no NaN while every key so far is masked
                l_part[h] += pr[h];
            }
            // P^T buffer b is free once the PV of tile j-2 completed
            if (j >= 2) wait_or_flag(&pv_done[b], (uint32_t)((j - 2) >> 1) & 1u, p.d_err);
            {
                // P of head h is stored twice: rounded to the input type in
                // row h, and the rounding residual (rounded again) in row 8 + h,
                // the MMA's padding rows.  The PV MMA then yields V.P_hi in
                // column h and V.P_lo in column 8 + h of O^T, and their fp32
                // sum carries P to about twice the input type's precision at
                // no extra MMA (a 16-bit P alone would add up to 2^-9 |v|
                // per weight to bf16 outputs)
                const uint32_t pb = sb + kOffP + b * 4096 + (t >> 6) * 2048 + (t & 7) * 2;
                const int ch = (t & 63) >> 3;
#pragma unroll
                for (int h = 0; h < kTG; h += 2) {
                    const uint32_t w2 = Elem<T>::pack2(pr[h], pr[h + 1]);
                    float h0, h1;
                    Elem<T>::unpack2(w2, h0, h1);
                    const uint32_t r2 = Elem<T>::pack2(pr[h] - h0, pr[h + 1] - h1);
                    sts16(pb + h * 128 + ((ch ^ h) << 4), (uint16_t)(w2 & 0xffffu));
                    sts16(pb + (h + 1) * 128 + ((ch ^ (h + 1)) << 4), (uint16_t)(w2 >> 16));
                    sts16(pb + (kTG + h) * 128 + ((ch ^ h) << 4), (uint16_t)(r2 & 0xffffu));
                    sts16(pb + (kTG + h + 1) * 128 + ((ch ^ (h + 1)) << 4), (uint16_t)(r2 >> 16));
                }
            }
            if (j == ntiles - 1 && key >= ntok) {
                // this key's V row holds whatever the pool has past the
                // context (possibly NaN, and 0 * NaN poisons O): zero it
                const int it = item_v(j), sl = it % kSlots;
                wait_or_flag(&full[sl], (uint32_t)(it / kSlots) & 1u, p.d_err);
                const uint32_t vr = sb + sl * kSlot + (t >> 3) * 2048 + (t & 7) * 128;
                const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    sts128(vr + c * 16, z);
                    sts128(vr + 1024 + c * 16, z);
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive1(&p_full[b]);
        }

        // row sums over the 128 key lanes, then the four warps
        const float wsum = warp_scatter8<false>(l_part, lane);
        if ((lane & 3) == 0) xsum[sw * kTG + (lane >> 2)] = wsum;
        named_bar_sync(1, 128);
        float lsum[kTG];
#pragma unroll
        for (int h = 0; h < kTG; ++h)
            lsum[h] = (xsum[h] + xsum[kTG + h]) + (xsum[2 * kTG + h] + xsum[3 * kTG + h]);

        wait_or_flag(&pv_done[(ntiles - 1) & 1], (uint32_t)((ntiles - 1) >> 1) & 1u, p.d_err);
        tc_fence_after();
        float o[kTG];
        {
            float o2[2 * kTG];
            tmem_ld16(tmem + lane_off + kColO, o2);
            tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < kTG; ++h) o[h] = o2[h] + o2[kTG + h];  // V.P_hi + V.P_lo
        }
        const int d = t;  // O^T row = dimension
        if (direct) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float inv = lsum[h] > 0.f ? 1.f / lsum[h] : 0.f;
                const uint32_t w2 = Elem<T>::pack2(o[h] * inv, 0.f);
                *reinterpret_cast<uint16_t *>(static_cast<T *>(p.out) + row_of(h) * kTD + d) = (uint16_t)(w2 & 0xffffu);
            }
        } else {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const size_t slot = row_of(h) * p.slots + p.part_base + part;
                p.ws_acc[slot * kTD + d] = o[h];
                if (d == h) p.ws_ml[slot] = make_float2(m_run[h], lsum[h]);
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
    if (ensure_smem_attr(kern, kSmemAlloc, attr_done) != PA_OK) return PA_ERR_CUDA;
    const bool bf16 = std::is_same<T, __nv_bfloat16>::value;
    CUtensorMap tmk, tmv;
    if (!make_pool_map4(&tmk, p.k_cache, p, BS, bf16) || !make_pool_map4(&tmv, p.v_cache, p, BS, bf16))
        return PA_ERR_UNSUPPORTED;  // the CUDA-core kernel takes over
    const long long units = (long long)p.max_partitions * p.num_seqs * p.num_kv_heads;
    if (units <= 0) return PA_OK;
    if (units > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    return launch_pdl(kern, dim3((unsigned)units), dim3(kThreads), kSmemAlloc, stream, p, tmk, tmv) == cudaSuccess
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
