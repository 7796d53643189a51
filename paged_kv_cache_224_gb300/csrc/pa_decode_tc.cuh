// Device code of the tensor-core decode (head groups up to 8 at head_dim 128),
// shared by the decode kernel (one unit per CTA, two CTAs per SM) and the
// one-launch mixed prefill + decode kernel (two six-warp decode instances per
// CTA, each drawing units from a queue the grid shares).  An instance is a
// producer warp, an MMA warp and four softmax warps with their own three-slot
// ring, barriers and 64 TMEM columns; its ring, barrier phases and TMEM run on
// from one unit to the next.  See pa_decode_tc.cu for the design.
#pragma once

#include <cuda.h>

#include <type_traits>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_tcgen05.cuh"

namespace pa {
namespace tcd {


constexpr int kTG = 8;                    // head slots: the group's G query heads, then zero rows
constexpr int kTN = 16;                   // MMA N: the slots padded to the smallest N allowed with M = 128
constexpr int kTD = 128;                  // head_dim
constexpr int kTK = 128;                  // keys per tile (M of the QK^T MMA)
constexpr int kSlot = kTK * kTD * 2;      // 32 KB: one K or V tile
// Shared memory of a CTA with a ring of S slots: the ring, then Q^T: [2 dim
// halves][16 rows][128 B], P^T: 2 buffers x [2 key halves][16 rows][128 B],
// the barriers, and [2][4 warps][8] tile maxima then [4 warps][8] row sums.
template <int S>
struct TcLayout {
    static constexpr int kSlots = S;
    static constexpr int kOffQ = S * kSlot;
    static constexpr int kOffP = kOffQ + 4096;
    static constexpr int kOffBar = kOffP + 2 * 4096;
    static constexpr int kOffXch = kOffBar + 256;
    static constexpr int kSmemUsed = kOffXch + (2 * 4 * kTG + 4 * kTG) * 4;
    static constexpr int kSmemAlloc = kSmemUsed + 1024;  // room to align the base to 1 KB
};
constexpr int kSlotsStandalone = 3;       // two CTAs per SM
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

// ---- one unit ----------------------------------------------------------------

// A unit (partition, sequence, kv head) and what its CTA needs to know about it.
struct TcUnit {
    int part, s, kvh;
    int tok0, ntok, ntiles;
    bool skip;    // a partition past the sequence's end: nothing to do
    bool direct;  // the whole sequence: the normalised output, else a partial
};

template <int BS>
__device__ __forceinline__ TcUnit tc_unit_of(const DecodeParams &p, int unit, int tid) {
    // partition-major order
    TcUnit u;
    const int per_part = p.num_seqs * p.num_kv_heads;
    u.part = unit / per_part;
    const int rem = unit - u.part * per_part;
    u.s = rem / p.num_kv_heads;
    u.kvh = rem - u.s * p.num_kv_heads;
    int L;
    if (p.len_fixed > 0) {
        L = p.len_fixed;
    } else {
        L = p.context_lens[u.s] - p.len_offset;
        const int Lcap = min(p.max_context_len, p.max_blocks_per_seq * BS) - p.len_offset;
        if (L < 0 || L > Lcap) {
            if (tid == 0 && u.part == 0 && u.kvh == 0) flag_error(p.d_err, PA_DEVERR_CONTEXT_RANGE);
            L = L < 0 ? 0 : Lcap;
        }
    }
    if (p.grp_size > 1 && u.part == 0 && u.kvh == 0 && tid >= 0 && tid < 32) {
        // shared-prefix pass: every member's table must start with the leader's blocks
        const int32_t *lead = p.block_tables + (size_t)u.s * p.table_stride;
        bool same = true;
        for (int m = 1; m < p.grp_size; ++m) {
            const int32_t *row = lead + (size_t)m * p.max_blocks_per_seq;
            for (int j = tid; j < L / BS; j += 32) same = same && row[j] == lead[j];
        }
        if (!same) flag_error(p.d_err, PA_DEVERR_PREFIX);
    }
    const int PT = p.partition_tokens;
    const int nparts = L > 0 ? (L + PT - 1) / PT : 1;
    u.skip = u.part >= nparts;
    u.tok0 = u.part * PT;
    u.ntok = u.skip ? 0 : max(0, min(L, u.tok0 + PT) - u.tok0);
    u.ntiles = (u.ntok + kTK - 1) / kTK;
    u.direct = nparts == 1 && !p.force_partials;
    return u;
}

// real query/out row of head h of a unit
__device__ __forceinline__ size_t tc_row(const DecodeParams &p, const TcUnit &u, int h) {
    return (size_t)(u.s * p.grp_size + h / p.grp_inner) * p.num_heads + (size_t)u.kvh * p.grp_inner + h % p.grp_inner;
}

// A unit without keys: zeros, or an empty partial (max -inf, sum 0).  The
// threads with tid 0 .. G*16-1 write.
template <typename T, int G>
__device__ __forceinline__ void tc_empty_unit(const DecodeParams &p, const TcUnit &u, int tid) {
    if (tid >= 0 && tid < G * 16) {
        const int h = tid >> 4, c = tid & 15;
        const size_t row = tc_row(p, u, h);
        if (u.direct) {
            *reinterpret_cast<uint4 *>(static_cast<T *>(p.out) + row * kTD + c * 8) = make_uint4(0, 0, 0, 0);
        } else {
            const size_t slot = row * p.slots + p.part_base + u.part;
            float4 *dst = reinterpret_cast<float4 *>(p.ws_acc + slot * kTD + c * 8);
            dst[0] = make_float4(0.f, 0.f, 0.f, 0.f);
            dst[1] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (c == 0) p.ws_ml[slot] = make_float2(-INFINITY, 0.f);
        }
    }
}

// One decode instance: six warps (producer, MMA issuer, four softmax warps
// from warp wb on) with their own shared memory, barriers and TMEM, and the
// counts that give each barrier's phase (ring items, key tiles, units), which
// carry from one unit to the next.  Every thread of the instance keeps the
// same counts.  A CTA holds one instance (the decode kernel) or two (the
// mixed kernel's decode CTAs).
struct TcRun {
    uint32_t sb;  // 1 KB-aligned shared base of the instance
    uint64_t *full, *empty, *q_full, *s_full, *p_full, *pv_done;
    uint64_t *u_full, *u_empty;  // [2] unit queue: producer -> MMA + softmax, and back
    volatile int *u_slot;        // [2]
    float *xmax, *xsum;
    volatile uint32_t *tmem_holder;
    uint32_t tmem;
    int wb;   // first warp (the producer)
    int bar;  // hardware barrier of the four softmax warps
    int items, tiles, units;
};

// Set up an instance whose shared memory starts `offset` bytes into the
// CTA's 1 KB-aligned dynamic shared memory: its barriers, by its first
// thread.  TMEM is the caller's: one allocation per CTA (a CTA gives up its
// right to allocate after the first), and r.tmem is set once the caller has
// synchronised the CTA.
template <int S>
__device__ __forceinline__ void tc_init(TcRun &r, uint32_t offset, int wb, int bar) {
    using Lay = TcLayout<S>;
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // 1 KB aligned: swizzle atoms start on 1 KB
    r.sb = base + offset;
    unsigned char *gb = smem_raw + (r.sb - raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(gb + Lay::kOffBar);
    r.full = bars;                   // [S] TMA -> MMA
    r.empty = bars + S;              // [S] MMA -> TMA
    r.q_full = bars + 2 * S;         // softmax threads -> MMA (Q^T written)
    r.s_full = r.q_full + 1;         // [2] MMA -> softmax (S^T of a tile ready)
    r.p_full = r.s_full + 2;         // [2] softmax -> MMA (S read, P^T written, O rescaled)
    r.pv_done = r.p_full + 2;        // [2] MMA -> softmax (PV of a tile complete)
    r.u_full = r.pv_done + 2;        // [2]
    r.u_empty = r.u_full + 2;        // [2]
    r.tmem_holder = reinterpret_cast<volatile uint32_t *>(r.u_empty + 2);
    r.u_slot = reinterpret_cast<volatile int *>(r.tmem_holder + 2);
    static_assert((2 * S + 11) * 8 + 16 <= Lay::kOffXch - Lay::kOffBar, "barrier area");
    r.xmax = reinterpret_cast<float *>(gb + Lay::kOffXch);  // [2][4][8]
    r.xsum = r.xmax + 2 * 4 * kTG;                          // [4][8]
    r.wb = wb;
    r.bar = bar;
    r.tmem = 0;
    r.items = r.tiles = r.units = 0;
    if ((int)threadIdx.x == wb * 32) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&r.full[i], 1);
            mbar_init(&r.empty[i], 1);
        }
        mbar_init(r.q_full, 128);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&r.s_full[b], 1);
            mbar_init(&r.p_full[b], 128);
            mbar_init(&r.pv_done[b], 1);
            mbar_init(&r.u_full[b], 1);
            mbar_init(&r.u_empty[b], 1 + 128);  // the MMA thread and the softmax threads
        }
        fence_barrier_init();
    }
}

// TMEM for a CTA, by one whole warp: `cols` columns (a power of two, >= 32),
// base address written to *holder; the CTA makes no further allocation.
__device__ __forceinline__ void tc_alloc(volatile uint32_t *holder, uint32_t cols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(const_cast<uint32_t *>(holder))),
                 "r"(cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

// Free a CTA's TMEM, by one whole warp, after the CTA's final barrier.
__device__ __forceinline__ void tc_dealloc(uint32_t tmem, uint32_t cols) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(cols) : "memory");
}

// After the instance's last unit, before the CTA's final barrier: let copies
// still in flight (only after a timeout) land.
template <int S>
__device__ __forceinline__ void tc_drain(const TcRun &r) {
    if ((int)threadIdx.x == r.wb * 32)
        for (int i = max(0, r.items - S); i < r.items; ++i) mbar_wait(&r.full[i % S], (uint32_t)(i / S) & 1u);
}

// One unit with keys, by the instance's six warps; the ring, the barrier
// phases and TMEM continue from the previous unit (r's counts advance).
template <typename T, int BS, int G, int S>
__device__ __forceinline__ void tc_unit(const DecodeParams &p, const CUtensorMap *tmk, const CUtensorMap *tmv,
                                        const TcUnit &u, TcRun &r) {
    using Lay = TcLayout<S>;
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr int kBPT = kTK / BS;  // blocks per tile
    static_assert(kTK % BS == 0 && BS % 8 == 0 && 32 % kBPT == 0, "block_size");
    static_assert(G >= 1 && G <= kTG, "group");
    const int warp = (int)(threadIdx.x >> 5) - r.wb, lane = threadIdx.x & 31;  // warp within the instance
    const int ntiles = u.ntiles, ntok = u.ntok, kvh = u.kvh;
    const uint32_t sb = r.sb, tmem = r.tmem;
    // ring items of this unit in consumption order: K(0), then K(j), V(j-1) for
    // j >= 1, then V(last); item i of the CTA sits in slot i % S
    const int ib = r.items;
    auto item_k = [ib](int j) { return ib + (j == 0 ? 0 : 2 * j - 1); };
    auto item_v = [ib, ntiles](int j) { return ib + (j + 1 < ntiles ? 2 * j + 2 : 2 * j + 1); };
    const int tb = r.tiles;  // key tiles of earlier units: tile j's buffers and phases follow tb + j

    if (warp == 0) {
        // ============================================================ producer
        const int32_t *table = p.block_tables + (size_t)u.s * p.table_stride + p.len_offset / BS + u.tok0 / BS;
        const int nblk = (ntok + BS - 1) / BS;
        const int oob = p.num_blocks * p.num_kv_heads * (BS / 8);  // first 8-row group past the pool: zero fill
        const uint64_t pol = policy_evict_first();
        // table entries 32 at a time, one per lane, a chunk ahead of use
        constexpr int kTilesPerChunk = 32 / kBPT;
        auto chunk = [&](int c) { return c * 32 + lane < nblk ? table[c * 32 + lane] : -1; };
        int ent_cur = chunk(0), ent_nxt = chunk(1);
        int item = ib;
        auto load = [&](const CUtensorMap *map, int y) {
            const int sl = item % S;
            if (lane == 0) {
                if (item >= S) wait_or_flag(&r.empty[sl], (uint32_t)(item / S - 1) & 1u, p.d_err);
                mbar_arrive_expect_tx(&r.full[sl], (uint32_t)kSlot);
            }
            __syncwarp();
            if (lane < kBPT) tma_4d(sb + sl * kSlot + lane * (BS * 256), map, y, &r.full[sl], pol);
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
            load(tmk, y);
            if (j >= 1) load(tmv, y_prev);
            y_prev = y;
        }
        load(tmv, y_prev);
    } else if (warp == 1) {
        // ============================================================ MMA issuer
        if (lane == 0) {
            constexpr uint32_t id_qk = instr_desc(kBf16, false, false, kTK, kTN);
            constexpr uint32_t id_pv = instr_desc(kBf16, true, false, kTD, kTN);
            constexpr uint32_t hi_kv = desc_hi(2048);  // K, V: 8-key groups 2 KB apart
            constexpr uint32_t hi_qp = desc_hi(1024);  // Q^T, P^T: 8-row groups 1 KB apart
            const uint32_t k_lo0 = desc_lo(sb, 16);     // K-major: leading offset unused
            const uint32_t v_lo0 = desc_lo(sb, 1024);   // MN-major: second 64-dim half 1 KB on
            const uint32_t q_lo = desc_lo(sb + Lay::kOffQ, 16);
            const uint32_t p_lo0 = desc_lo(sb + Lay::kOffP, 16);
            wait_or_flag(r.q_full, (uint32_t)r.units & 1u, p.d_err);
            tc_fence_after();
            for (int j = 0; j <= ntiles; ++j) {
                if (j < ntiles) {
                    // S^T(j) = K(j) Q^T into buffer (tb+j) & 1 (its previous
                    // tile's softmax finished before the PV issued last iteration)
                    const int it = item_k(j), sl = it % S, g = tb + j;
                    wait_or_flag(&r.full[sl], (uint32_t)(it / S) & 1u, p.d_err);
                    tc_fence_after();
                    const uint32_t tS = tmem + kColS + (g & 1) * kTN;
                    const uint32_t k_lo = k_lo0 + ((uint32_t)(sl * kSlot) >> 4);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t ko = (uint32_t)((kk >> 2) * 1024 + (kk & 3) * 32) >> 4;
                        const uint32_t qo = (uint32_t)((kk >> 2) * 2048 + (kk & 3) * 32) >> 4;
                        mma_f16(tS, desc_of(k_lo + ko, hi_kv), desc_of(q_lo + qo, hi_qp), id_qk, kk > 0);
                    }
                    mma_commit(&r.s_full[g & 1]);
                    mma_commit(&r.empty[sl]);
                }
                if (j >= 1) {
                    // O^T += V^T(j-1) P^T(j-1)
                    const int jj = j - 1, g = tb + jj;
                    wait_or_flag(&r.p_full[g & 1], (uint32_t)(g >> 1) & 1u, p.d_err);
                    const int it = item_v(jj), sl = it % S;
                    wait_or_flag(&r.full[sl], (uint32_t)(it / S) & 1u, p.d_err);
                    tc_fence_after();
                    const uint32_t v_lo = v_lo0 + ((uint32_t)(sl * kSlot) >> 4);
                    const uint32_t p_lo = p_lo0 + ((uint32_t)((g & 1) * 4096) >> 4);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t vo = (uint32_t)(kk * 4096) >> 4;
                        const uint32_t po = (uint32_t)((kk >> 2) * 2048 + (kk & 3) * 32) >> 4;
                        mma_f16(tmem + kColO, desc_of(v_lo + vo, hi_kv), desc_of(p_lo + po, hi_qp), id_pv,
                                jj > 0 || kk > 0);
                    }
                    mma_commit(&r.pv_done[g & 1]);
                    mma_commit(&r.empty[sl]);
                }
            }
        }
    } else if (warp >= 2 && warp < 6) {
        // ============================================================ softmax
        const int quarter = (threadIdx.x >> 5) & 3;  // TMEM lanes 32*quarter .. +31 (fixed by the CTA warp id)
        const int t = quarter * 32 + lane;    // key of the tile (S^T row) and dimension (O^T row)
        const int sw = warp - 2;              // index among the softmax warps
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const float csc = p.scale_log2;
        {
            // Q^T rows 0..G-1 = the group's query heads, the rest zero (the
            // previous unit's QKs have all completed: its last S was read)
            const uint4 z = make_uint4(0, 0, 0, 0);
            const int h = t >> 4, c = t & 15;
            const uint4 q = h < G ? *reinterpret_cast<const uint4 *>(static_cast<const T *>(p.query) +
                                                                     tc_row(p, u, h) * kTD + c * 8)
                                  : z;
            sts128(sb + Lay::kOffQ + (c >> 3) * 2048 + h * 128 + (((c & 7) ^ h) << 4), q);
            sts128(sb + Lay::kOffQ + (c >> 3) * 2048 + (8 + h) * 128 + (((c & 7) ^ h) << 4), z);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive1(r.q_full);
        }

        float m_run[kTG], l_part[kTG];
#pragma unroll
        for (int h = 0; h < kTG; ++h) {
            m_run[h] = -INFINITY;
            l_part[h] = 0.f;
        }
        const int32_t *table = p.block_tables + (size_t)u.s * p.table_stride + p.len_offset / BS + u.tok0 / BS;
        for (int j = 0; j < ntiles; ++j) {
            const int g = tb + j, b = g & 1;
            // this key's block must be in the pool (the producer flags a bad
            // entry and fetches zeros; the key is left out here); the load is
            // issued before the wait so its latency hides behind it
            const int key = j * kTK + t;
            const int ent = key < ntok ? table[key / BS] : -1;
            wait_or_flag(&r.s_full[b], (uint32_t)(g >> 1) & 1u, p.d_err);
            tc_fence_after();
            float sc[kTG];
            tmem_ld8(tmem + lane_off + kColS + b * kTN, sc);
            tmem_wait_ld();
            const bool valid = key < ntok && ent >= 0 && ent < p.num_blocks;
#pragma unroll
            for (int h = 0; h < kTG; ++h) sc[h] = valid ? sc[h] * csc : -INFINITY;
            // each head's maximum over the tile's 128 keys
            const float wmax = warp_scatter8<true>(sc, lane);
            if ((lane & 3) == 0) r.xmax[(b * 4 + sw) * kTG + (lane >> 2)] = wmax;
            named_bar_sync(r.bar, 128);
            float tmax[kTG];
            {
                const float4 *x = reinterpret_cast<const float4 *>(r.xmax + b * 4 * kTG);
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
                wait_or_flag(&r.pv_done[(g - 1) & 1], (uint32_t)((g - 1) >> 1) & 1u, p.d_err);
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
            // P^T buffer b is free once the PV of tile g-2 completed (the last
            // tile of the previous unit's PV completed before its output)
            if (j >= 2) wait_or_flag(&r.pv_done[b], (uint32_t)((g - 2) >> 1) & 1u, p.d_err);
            {
                // P of head h is stored twice: rounded to the input type in
                // row h, and the rounding residual (rounded again) in row 8 + h,
                // the MMA's padding rows.  The PV MMA then yields V.P_hi in
                // column h and V.P_lo in column 8 + h of O^T, and their fp32
                // sum carries P to about twice the input type's precision at
                // no extra MMA (a 16-bit P alone would add up to 2^-9 |v|
                // per weight to bf16 outputs)
                const uint32_t pb = sb + Lay::kOffP + b * 4096 + (t >> 6) * 2048 + (t & 7) * 2;
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
                const int it = item_v(j), sl = it % S;
                wait_or_flag(&r.full[sl], (uint32_t)(it / S) & 1u, p.d_err);
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
            mbar_arrive1(&r.p_full[b]);
        }

        // row sums over the 128 key lanes, then the four warps
        const float wsum = warp_scatter8<false>(l_part, lane);
        if ((lane & 3) == 0) r.xsum[sw * kTG + (lane >> 2)] = wsum;
        named_bar_sync(r.bar, 128);
        float lsum[kTG];
#pragma unroll
        for (int h = 0; h < kTG; ++h)
            lsum[h] = (r.xsum[h] + r.xsum[kTG + h]) + (r.xsum[2 * kTG + h] + r.xsum[3 * kTG + h]);

        const int gl = tb + ntiles - 1;
        wait_or_flag(&r.pv_done[gl & 1], (uint32_t)(gl >> 1) & 1u, p.d_err);
        tc_fence_after();
        float o[kTG];
        {
            float o2[2 * kTG];
            tmem_ld16(tmem + lane_off + kColO, o2);
            tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < kTG; ++h) o[h] = o2[h] + o2[kTG + h];  // V.P_hi + V.P_lo
        }
        // the next unit's row sums land in xsum only after every warp read
        // this unit's (its first tile has a barrier first)
        const int d = t;  // O^T row = dimension
        if (u.direct) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float inv = lsum[h] > 0.f ? 1.f / lsum[h] : 0.f;
                const uint32_t w2 = Elem<T>::pack2(o[h] * inv, 0.f);
                *reinterpret_cast<uint16_t *>(static_cast<T *>(p.out) + tc_row(p, u, h) * kTD + d) =
                    (uint16_t)(w2 & 0xffffu);
            }
        } else {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const size_t slot = tc_row(p, u, h) * p.slots + p.part_base + u.part;
                p.ws_acc[slot * kTD + d] = o[h];
                if (d == h) p.ws_ml[slot] = make_float2(m_run[h], lsum[h]);
            }
        }
    }
    r.items += 2 * ntiles;
    r.tiles += ntiles;
    r.units += 1;
}

// Units from a queue that every instance of the grid shares: the producer's
// lane 0 takes the next unit number from *next (an atomic counter) and hands
// it to the MMA thread and the softmax threads through a two-entry queue in
// shared memory, so an instance that drew short units takes more of them.  A
// number >= nunits ends the instance; each of the ninst instances draws one,
// and the draw that returns the last number handed out (nunits + ninst - 1)
// puts the counter back to 0 for the next launch.
template <typename T, int BS, int G, int S>
__device__ __forceinline__ void tc_queue_loop(const DecodeParams &p, const CUtensorMap *tmk, const CUtensorMap *tmv,
                                              TcRun &r, unsigned *next, int nunits, int ninst) {
    const int rel = (int)threadIdx.x - r.wb * 32;  // thread within the instance
    const int warp = rel >> 5, lane = rel & 31;
    for (int k = 0;; ++k) {
        const int q = k & 1;
        const uint32_t ph = (uint32_t)(k >> 1) & 1u;
        int unit = 0;
        if (warp == 0) {
            if (lane == 0) {
                unit = (int)atomicAdd(next, 1u);
                if (unit == nunits + ninst - 1) atomicExch(next, 0u);
                if (k >= 2) wait_or_flag(&r.u_empty[q], ph ^ 1u, p.d_err);
                r.u_slot[q] = unit;
                mbar_arrive1(&r.u_full[q]);
            }
        } else if (warp >= 2 || lane == 0) {
            wait_or_flag(&r.u_full[q], ph, p.d_err);
            unit = r.u_slot[q];
            mbar_arrive1(&r.u_empty[q]);
        }
        if (warp < 2) unit = __shfl_sync(kFull, unit, 0);
        if (unit >= nunits) break;
        const TcUnit u = tc_unit_of<BS>(p, unit, rel);
        if (u.skip) continue;
        if (u.ntiles == 0) {
            tc_empty_unit<T, G>(p, u, rel - 64);  // by the softmax threads
            continue;
        }
        tc_unit<T, BS, G, S>(p, tmk, tmv, u, r);
    }
}

}  // namespace tcd
}  // namespace pa
