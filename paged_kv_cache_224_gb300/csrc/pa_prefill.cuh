// Chunked-prefill attention on the 5th-generation tensor cores (tcgen05):
// the CTA-level device code and host helpers, shared by the prefill kernel
// (pa_prefill.cu) and the one-launch continuous-batching step (pa_mixed.cu).
//
// Follows the page "vLLM PagedAttention chuyen sau" (locionic.com), section
// "Chunked Prefill": each chunk of a long prompt attends to the sequence's
// paged cache built so far.  Query row i of the chunk sits at position
// prefix_len + i and sees keys 0 .. prefix_len + i, gathered through the
// block table.
//
// Work unit = (sequence, kv head, row tile): 256 query rows -- 256/G chunk
// positions times the G query heads of one kv head -- against the unit's
// 128-key tiles, computed as two Q tiles of 128 rows that share every K/V
// tile (each K/V byte brought into shared memory serves 256 rows).
//
// Schedule.  With a workspace the kernel is persistent and stream-K: the
// units' key tiles, laid end to end (sequence, kv head, row tile, key tile),
// are cut into one contiguous range per CTA, one CTA per SM, so every SM gets
// the same number of tiles whatever the number of units (a 512-token chunk of
// a 64/8-head model has 128 units for 152 SMs).  A CTA walks its range unit
// by unit ("segments"); a unit cut by a range boundary is finished by
// log-sum-exp merging: each of its segments writes its unnormalised O, running
// maximum and sum to a per-CTA slot of the workspace and counts itself on the
// unit's counter, and the segment that arrives last merges all of them in
// key order (so the result does not depend on which arrived last) and writes
// the output.  No CTA ever waits for another.  Without a workspace each CTA
// computes one whole unit (grid = units).
//
// Warp roles inside a CTA (the ring, the barrier phases and the tile count
// run on across segments):
//   warp 0    TMA producer: for each key tile, one 4-D tensor copy per block
//             of K and then of V, straight from the paged pool into a
//             128-byte-swizzled shared layout in which the tile's 8-key groups
//             sit 2 KB apart and the two 64-dim halves 1 KB apart inside each
//             group (uniform strides across the tile's blocks, so one
//             descriptor covers the tile; one copy per block, not per (block,
//             half)).  One ring of five 32 KB slots, K(0), V(0), K(1), V(1),
//             ...; block-table entries are read 32 at a time, a chunk ahead;
//   warp 1    MMA issuer (one thread): per key tile j and Q tile g, first
//             O_g += P_g(j-1) V(j-1), then S_g = Q_g K(j)^T, tcgen05.mma
//             kind::f16 with fp32 accumulation in TMEM.  P_g is written over
//             the first half of S_g's TMEM columns and read from there as the
//             A operand; the tensor pipe runs one thread's MMAs in order, so
//             the PV of tile j-1 has read P before the QK of tile j writes S,
//             and S_g(j) being complete means O_g holds every PV up to j-1.
//             Every mbarrier wait or commit costs this thread a few hundred
//             cycles in which it issues nothing, so it commits only S and the
//             last PV, and learns that P is written and that the copies have
//             landed through hardware barriers the other warps arrive on or
//             sync with;
//   warps 2-5 softmax of Q tile 0, warps 6-9 of Q tile 1: each thread owns one
//             query row = one TMEM lane; it reads its whole S row (one TMEM
//             wait), applies the causal mask, updates the running max
//             (rescaling O in TMEM only when the max grows by more than 2^8),
//             writes P (rounded to the input type) into TMEM, and at the end
//             of the segment stores the normalised row or its partial.  The
//             two groups interleave, so the tensor pipe works on one Q tile's
//             MMAs while the other's softmax runs.  Q tile 1's threads hand
//             K(j) and V(j-1)'s ring slots back to the producer once S_1(j) is
//             complete (every MMA before it has finished).  On the unit's last
//             key tile each group zeroes the V rows past the unit's last key,
//             so garbage (even NaN) in unused slots never reaches O;
//   warp 10   load watcher: per key tile j, waits for the V(j) and K(j+1)
//             copies and then syncs with the MMA warp before it issues the PV
//             of tile j and the QK of tile j+1.
// All waits are bounded; a wait that gives up flags PA_DEVERR_TIMEOUT.
#pragma once

#include <cuda.h>

#include <type_traits>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_tcgen05.cuh"

namespace pa {
namespace pf {

constexpr int kD = 128;                        // head_dim
constexpr int kM = 128;                        // query rows per Q tile (one per TMEM lane)
constexpr int kQT = 2;                         // Q tiles per unit
constexpr int kUnitRows = kQT * kM;            // query rows per unit
constexpr int kNK = 128;                       // keys per tile
constexpr int kSlots = 5;                      // K/V tiles in flight (one ring)
constexpr int kQHalf = kM * 128;               // one 64-dim half of a Q tile: 128 rows x 128 bytes
constexpr int kQTile = 2 * kQHalf;             // 32 KB
constexpr int kKVTile = kNK * kD * 2;          // 32 KB: [16 key groups][2 dim halves][8 keys][128 B]
constexpr int kOffQ = 0;
constexpr int kOffKV = kOffQ + kQT * kQTile;               // 64 KB: K/V ring
constexpr int kOffBar = kOffKV + kSlots * kKVTile;         // 224 KB
constexpr int kSmemUsed = kOffBar + 256;
constexpr int kSmemAlloc = kSmemUsed + 1024;               // room to align the base to 1 KB
constexpr int kThreads = 64 + kQT * 128 + 32;
// TMEM columns: S of each Q tile (128 fp32; P overwrites its first 64 columns
// as 128 packed pairs), O of each Q tile (128 fp32)
constexpr uint32_t kColS = 0, kColO = 256;
constexpr uint32_t kTmemCols = 512;
// Hardware barriers: 1 + g over Q tile g's softmax warps (merging), kBarP + g
// over those warps and the MMA warp (P of Q tile g written)
constexpr int kBarP = 3;
constexpr int kBarL = kBarP + kQT;

// Key tiles of row tile r of sequence q: up to the last key its last row sees.
__host__ __device__ __forceinline__ int unit_tiles(int prefix_len, int chunk_len, int G, int r) {
    const int last_row = min(chunk_len * G, (r + 1) * kUnitRows) - 1;
    return (prefix_len + last_row / G) / kNK + 1;
}

// A run of consecutive key tiles of one unit.
struct Seg {
    int si, h, r;  // sequence (entry of p.seqs), kv head, row tile
    int t0, t1;    // key tiles [t0, t1) of the unit's n
    int n;
    int x_unit;    // global index of the unit's first key tile
    int unit;      // global index of the unit
};

// The segment that starts at global tile x and ends at x_end or at the end of its unit.
template <int G>
__device__ __forceinline__ Seg seg_at(const PrefillParams &p, int x, int x_end) {
    int si = 0;
    for (int i = 1; i < p.num_seqs; ++i)
        if (p.seqs[i].tile_start <= x) si = i;
    const PrefillSeq &q = p.seqs[si];
    const int off = x - q.tile_start;
    Seg s;
    s.si = si;
    s.h = off / q.tiles_per_head;
    int rem = off - s.h * q.tiles_per_head;
    int r = 0, n = unit_tiles(q.prefix_len, q.chunk_len, G, 0);
    while (rem >= n) {
        rem -= n;
        ++r;
        n = unit_tiles(q.prefix_len, q.chunk_len, G, r);
    }
    s.r = r;
    s.n = n;
    s.t0 = rem;
    s.t1 = min(n, rem + (x_end - x));
    s.x_unit = x - rem;
    s.unit = q.unit_start + s.h * q.row_tiles + r;
    return s;
}

// Global tile range of unit u (the schedule without a workspace).
template <int G>
__device__ __forceinline__ void unit_range(const PrefillParams &p, int u, int &x0, int &x1) {
    int si = 0;
    for (int i = 1; i < p.num_seqs; ++i)
        if (p.seqs[i].unit_start <= u) si = i;
    const PrefillSeq &q = p.seqs[si];
    const int off = u - q.unit_start;
    const int h = off / q.row_tiles, r = off - h * q.row_tiles;
    int x = q.tile_start + h * q.tiles_per_head;
    for (int rr = 0; rr < r; ++rr) x += unit_tiles(q.prefix_len, q.chunk_len, G, rr);
    x0 = x;
    x1 = x + unit_tiles(q.prefix_len, q.chunk_len, G, r);
}

// CTA whose stream-K range holds global tile x (ranges start at W*c/N).
__device__ __forceinline__ int cta_of(int x, long long W, long long N) { return (int)(((x + 1) * N - 1) / W); }

// ---- the end of a segment that is part of a unit ----------------------------
//
// Out of line, so that its registers do not weigh on the softmax loop.  The
// calling thread owns row t of Q tile g; its unnormalised O is in TMEM at tO,
// its running max and sum are m_run, l_run.  Partials are laid out as
// [slot][Q tile][32 float4 columns][128 rows] (a warp's stores and loads of
// one column are 512 contiguous bytes) and (max, sum) as [slot][Q tile][128
// rows]; the unit's counter counts the segments that have published theirs.
//
// The unit's c_hi - c_lo + 1 segments are merged by the last of them to
// finish, folding every segment's (O, max, sum) in CTA (= key) order with an
// online maximum, so the result does not depend on which segment merges.
//   * The CTA's last segment (no next segment; its S columns are free) first
//     looks whether all the others have published: if so it merges at once,
//     its own O read from TMEM where the fold reaches it and the fold
//     accumulated in the S columns, without publishing its own.  A range's
//     last segment is a unit's first key tiles, whose other parts the next
//     CTAs computed at the start of their ranges, so this is the usual case.
//   * Otherwise it publishes (partial, fence, count); the segment whose count
//     completes the unit merges, everything read from the workspace and the
//     fold accumulated in its O columns.
template <typename T>
__device__ __noinline__ void finish_partial(float4 *part_o, float2 *part_ml, unsigned *counter, T *orow, bool valid,
                                            uint32_t tO, uint32_t tS, bool last_seg, int g, int t, int slot, int my_cta,
                                            int c_lo, int c_hi, int x_unit, long long W, long long N, float m_run,
                                            float l_run, volatile int *merge_flag) {
    auto po = [&](int sl, int c4) { return part_o + ((size_t)(sl * kQT + g) * (kD / 4) + c4) * kM + t; };
    auto pml = [&](int sl) { return part_ml + (size_t)(sl * kQT + g) * kM + t; };
    auto slot_of = [&](int cc) { return 2 * cc + ((int)(W * cc / N) >= x_unit ? 0 : 1); };
    const unsigned others = (unsigned)(c_hi - c_lo);
    bool direct = false;  // merge without publishing: every other segment has published
    if (last_seg) {
        if (t == 0) {
            unsigned v;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
            merge_flag[g] = v == others;
        }
        named_bar_sync(1 + g, 128);
        direct = merge_flag[g];
        named_bar_sync(1 + g, 128);
    }
    if (!direct) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            float v[32];
            tmem_ld32(tO + c * 32, v);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 8; ++e) __stcg(po(slot, c * 8 + e), make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]));
        }
        __stcg(pml(slot), make_float2(m_run, l_run));
        __threadfence();
        named_bar_sync(1 + g, 128);
        if (t == 0) merge_flag[g] = atomicAdd(counter, 1u) == others;
        named_bar_sync(1 + g, 128);
        if (!merge_flag[g]) return;
    }
    __threadfence();
    // the fold; its accumulator: the S columns when merging directly (O holds
    // this segment's own part), else the O columns (every part is in the workspace)
    const uint32_t tA = direct ? tS : tO;
    float m_acc = -INFINITY, lsum = 0.f;
    for (int cc = c_lo; cc <= c_hi; ++cc) {
        const bool own = direct && cc == my_cta;
        const int sl = slot_of(cc);
        const float2 ml = own ? make_float2(m_run, l_run) : __ldcg(pml(sl));
        const float m_new = fmaxf(m_acc, ml.x);
        const float a = m_acc == -INFINITY ? 0.f : fast_exp2(m_acc - m_new);  // rescales what is accumulated
        const float w = ml.x == -INFINITY ? 0.f : fast_exp2(ml.x - m_new);
        lsum = lsum * a + ml.y * w;
        m_acc = m_new;
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {
            float4 ld[16];
            if (own) {
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                    float v[32];
                    tmem_ld32(tO + (hh * 2 + c2) * 32, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 8; ++e) ld[c2 * 8 + e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 16; ++e) ld[e] = __ldcg(po(sl, hh * 16 + e));
            }
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
                const uint32_t col = tA + (hh * 2 + c2) * 32;
                float v[32];
                if (cc == c_lo) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = 0.f;
                } else {
                    tmem_ld32(col, v);
                    tmem_wait_ld();
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float4 o = ld[c2 * 8 + e];
                    v[4 * e] = v[4 * e] * a + w * o.x;
                    v[4 * e + 1] = v[4 * e + 1] * a + w * o.y;
                    v[4 * e + 2] = v[4 * e + 2] * a + w * o.z;
                    v[4 * e + 3] = v[4 * e + 3] * a + w * o.w;
                }
                tmem_st32(col, v);
            }
        }
        tmem_wait_st();
    }
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
        float v[32];
        tmem_ld32(tA + c * 32, v);
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
    if (t == 0) *counter = 0u;  // ready for the next call
}

// ---- the kernel ------------------------------------------------------------

// The prefill work of CTA `cta` of `ncta`: with the stream-K schedule, its
// share of the key tiles; without, unit `cta` (all of the CTA's threads call this).
// Returns the CTA's TMEM base; with kKeepTmem (the one-launch step, whose
// prefill CTAs go on to decode) the allocation is left for the caller to free.
template <typename T, int BS, int G, bool kKeepTmem = false>
__device__ __forceinline__ uint32_t prefill_cta(const PrefillParams &p, const CUtensorMap &tmk,
                                                const CUtensorMap &tmv, const CUtensorMap &tmq, int cta, int ncta) {
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr int kBlocksPerTile = kNK / BS;
    static_assert(kNK % BS == 0 && BS % 8 == 0 && 32 % kBlocksPerTile == 0, "block_size");
    static_assert(kM % G == 0, "group");

    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t sb = (raw + 1023u) & ~1023u;  // 1 KB aligned: swizzle atoms start on 1 KB
    unsigned char *gb = smem_raw + (sb - raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(gb + kOffBar);
    uint64_t *full = bars + 0;                  // [kSlots] TMA -> MMA
    uint64_t *empty = bars + kSlots;            // [kSlots] softmax (Q tile 1) -> TMA
    uint64_t *q_full = bars + 2 * kSlots;       // TMA -> MMA (both Q tiles of a segment landed)
    uint64_t *q_empty = q_full + 1;             // softmax (Q tile 1) -> TMA (the segment's last QKs finished)
    uint64_t *s_full = q_empty + 1;             // [kQT] MMA -> softmax (S ready, O holds all PVs before it)
    uint64_t *o_done = s_full + kQT;            // [kQT] MMA -> softmax (last PV of the segment finished)
    volatile uint32_t *tmem_holder = reinterpret_cast<volatile uint32_t *>(o_done + kQT);
    volatile int *merge_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);  // [kQT]
    static_assert((2 * kSlots + 2 + 2 * kQT) * 8 + 4 + 4 * kQT <= kSmemUsed - kOffBar, "barrier area");

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // this CTA's key tiles [x0, x1) of the global order
    int x0, x1;
    const long long W = p.total_tiles, N = ncta;
    if (p.split) {
        x0 = (int)(W * cta / N);
        x1 = (int)(W * (cta + 1) / N);
    } else {
        unit_range<G>(p, cta, x0, x1);
    }
    const int nitems = 2 * (x1 - x0);  // ring items: K and V of every tile

    if (threadIdx.x == 0) {
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int g = 0; g < kQT; ++g) {
            mbar_init(&s_full[g], 1);
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
        const int oob = p.num_blocks * p.num_kv_heads * (BS / 8);  // first 8-row group past the pool: zero fill
        const uint64_t pol = policy_evict_last();  // every row tile of a kv head reads the same K/V
        constexpr int kTilesPerChunk = 32 / kBlocksPerTile;
        int item = 0;
        auto load = [&](const CUtensorMap *map, int y) {
            const int sl = item % kSlots;
            if (lane == 0) {
                if (item >= kSlots) wait_or_flag(&empty[sl], (uint32_t)(item / kSlots - 1) & 1u, p.d_err);
                mbar_arrive_expect_tx(&full[sl], (uint32_t)kKVTile);
            }
            __syncwarp();
            // block `lane`: both 64-dim halves of its BS rows, BS * 256 bytes
            if (lane < kBlocksPerTile)
                tma_4d(sb + kOffKV + sl * kKVTile + lane * (BS * 256), map, y, &full[sl], pol);
            ++item;
        };
        // The segment's two Q tiles: its unit's 256 query rows are 256/G
        // consecutive chunk positions times the G heads of its kv head, i.e. a
        // box of the query viewed as {128 dims, heads, rows}; per Q tile two
        // boxes of {64 dims, G heads, 128/G positions}, which land as 128 rows
        // of 128 bytes, 128-byte swizzled: the K-major layout the QK MMA reads.
        // (Rows past the chunk read the next chunk's queries or zeros past the
        // tensor; their outputs are never stored.)  Issued once the previous
        // segment's last QKs have finished reading the tiles.
        auto load_q = [&](const Seg &sg, int sc) {
            if (lane == 0) {
                if (sc > 0) wait_or_flag(q_empty, (uint32_t)(sc - 1) & 1u, p.d_err);
                mbar_arrive_expect_tx(q_full, (uint32_t)(kQT * kQTile));
                const PrefillSeq &q = p.seqs[sg.si];
                for (int g = 0; g < kQT; ++g) {
                    const int pos0 = q.row_start + (sg.r * kUnitRows + g * kM) / G;
                    for (int hf = 0; hf < 2; ++hf)
                        tma_3d(sb + kOffQ + g * kQTile + hf * kQHalf, &tmq, hf * 64, sg.h * G, pos0, q_full);
                }
            }
            __syncwarp();
        };
        int sc = 0;
        for (int x = x0; x < x1; ++sc) {
            const Seg sg = seg_at<G>(p, x, x1);
            const PrefillSeq &q = p.seqs[sg.si];
            const int32_t *table = q.block_table;
            const int kend = q.prefix_len + min(q.chunk_len - 1, ((sg.r + 1) * kUnitRows - 1) / G);
            // Table entries come 32 at a time, one per lane, a whole chunk ahead
            // of use (a chunk covers 32 / kBlocksPerTile tiles); lane b <
            // kBlocksPerTile handles block b of a tile.
            const int nent = kend / BS + 1;
            auto chunk = [&](int c) { return c * 32 + lane < nent ? table[c * 32 + lane] : -1; };
            int c_cur = sg.t0 / kTilesPerChunk;
            int ent_cur = chunk(c_cur), ent_nxt = chunk(c_cur + 1);
            for (int j = sg.t0; j < sg.t1; ++j) {
                if (j / kTilesPerChunk != c_cur) {
                    ++c_cur;
                    ent_cur = ent_nxt;
                    ent_nxt = chunk(c_cur + 1);
                }
                const int blk = __shfl_sync(kFull, ent_cur, (j % kTilesPerChunk) * kBlocksPerTile + lane % kBlocksPerTile);
                // first 8-row group of block `lane` in the pool (zero fill past kend)
                int y = oob;
                if (lane < kBlocksPerTile && j * kNK + lane * BS <= kend) {
                    if (blk >= 0 && blk < p.num_blocks) y = (blk * p.num_kv_heads + sg.h) * (BS / 8);
                    else flag_error(p.d_err, PA_DEVERR_BLOCK_RANGE);
                }
                load(&tmk, y);
                load(&tmv, y);
                // the segment's Q after its first K/V tile: for a later
                // segment its slots free up only as the previous one ends
                if (j == sg.t0) load_q(sg, sc);
            }
            x += sg.t1 - sg.t0;
        }
        // every copy has normally been consumed by now; after a timeout, let
        // the ones in flight land before the CTA can exit
        if (lane == 0)
            for (int i = max(0, nitems - kSlots); i < nitems; ++i) mbar_wait(&full[i % kSlots], (uint32_t)(i / kSlots) & 1u);
    } else if (warp == 1) {
        // ============================================================ MMA issuer
        // One thread issues; the whole warp takes the P announcements, which
        // come through hardware barriers (kBarP + g, the four softmax warps of
        // Q tile g arrive, this warp syncs) rather than mbarriers: a wait on an
        // mbarrier costs the issuing thread a few hundred cycles even when the
        // phase is long complete.
        {
            constexpr uint32_t idesc_qk = instr_desc(kBf16, false, false, kM, kNK);
            constexpr uint32_t idesc_pv = instr_desc(kBf16, false, true, kM, kD);
            constexpr uint32_t hi_q = desc_hi(1024);   // Q: 8-row groups 1 KB apart
            constexpr uint32_t hi_kv = desc_hi(2048);  // K, V: 8-key groups 2 KB apart
            // descriptor low words of Q tile 0 and of slot 0's K and V; the
            // rest are fixed offsets from these
            const uint32_t q_lo0 = desc_lo(sb + kOffQ, 16);
            const uint32_t k_lo0 = desc_lo(sb + kOffKV, 16);     // K-major: leading offset unused
            const uint32_t v_lo0 = desc_lo(sb + kOffKV, 1024);   // MN-major: second 64-dim half 1 KB on
            int tc = 0;  // tiles of earlier segments
            for (int x = x0, sc = 0; x < x1; ++sc) {
                const Seg sg = seg_at<G>(p, x, x1);
                const int nt = sg.t1 - sg.t0;
                if (lane == 0) wait_or_flag(q_full, (uint32_t)sc & 1u, p.d_err);
                for (int k = 0; k <= nt; ++k) {
                    const int gt = tc + k;  // this CTA's tile count
                    const int sl_v = (2 * gt - 1) % kSlots, sl_k = (2 * gt) % kSlots;
                    // K of a segment's first tile is the only copy this warp
                    // waits for: Q tile 0's softmax announces P(j) only once
                    // V(j) and K(j+1) have landed
                    if (k == 0 && lane == 0) {
                        wait_or_flag(&full[sl_k], (uint32_t)(2 * gt / kSlots) & 1u, p.d_err);
                        tc_fence_after();
                    }
#pragma unroll
                    for (int g = 0; g < kQT; ++g) {
                        const uint32_t tS = tmem + kColS + g * kNK;
                        if (k >= 1) {
                            // O_g += P_g(k-1) V(k-1); P sits in S_g's first 64 columns
                            __syncwarp();
                            if (g == 0) named_bar_sync(kBarL, 64);
                            named_bar_sync(kBarP + g, 160);
                            if (lane == 0) {
                                tc_fence_after();
                                const uint32_t v_lo = v_lo0 + sl_v * (kKVTile >> 4);
#pragma unroll
                                for (int kk = 0; kk < kNK / 16; ++kk)
                                    mma_f16_ts(tmem + kColO + g * kD, tS + kk * 8,
                                               desc_of(v_lo + kk * (4096 >> 4), hi_kv), idesc_pv, k > 1 || kk > 0);
                                if (k == nt) mma_commit(&o_done[g]);
                            }
                        }
                        if (k < nt && lane == 0) {
                            // S_g = Q_g K(k)^T
                            const uint32_t q_lo = q_lo0 + g * (kQTile >> 4);
                            const uint32_t k_lo = k_lo0 + sl_k * (kKVTile >> 4);
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk) {
                                const uint32_t qo = ((kk >> 2) * kQHalf + (kk & 3) * 32) >> 4;
                                const uint32_t ko = ((kk >> 2) * 1024 + (kk & 3) * 32) >> 4;
                                mma_f16(tS, desc_of(q_lo + qo, hi_q), desc_of(k_lo + ko, hi_kv), idesc_qk, kk > 0);
                            }
                            mma_commit(&s_full[g]);
                        }
                    }
                }
                tc += nt;
                x += nt;
            }
        }
    } else if (warp == 2 + 4 * kQT) {
        // ============================================================ load watcher
        // Tile by tile, V(j) and the segment's K(j+1) have landed before the
        // MMA warp issues the PV of tile j and the QK of tile j+1: this warp
        // waits on their mbarriers and then syncs with the MMA warp on a
        // hardware barrier, so the issuing thread touches no mbarrier in the
        // steady state
        int gt = 0;
        for (int x = x0; x < x1;) {
            const Seg sg = seg_at<G>(p, x, x1);
            const int nt = sg.t1 - sg.t0;
            for (int k = 0; k < nt; ++k, ++gt) {
                if (lane == 0) {
                    const int iv = 2 * gt + 1;
                    wait_or_flag(&full[iv % kSlots], (uint32_t)(iv / kSlots) & 1u, p.d_err);
                    if (k + 1 < nt) {
                        const int ik = 2 * gt + 2;
                        wait_or_flag(&full[ik % kSlots], (uint32_t)(ik / kSlots) & 1u, p.d_err);
                    }
                }
                __syncwarp();
                named_bar_sync(kBarL, 64);
            }
            x += nt;
        }
    } else if (warp < 2 + 4 * kQT) {
        // ============================================================ softmax
        const int g = (warp - 2) >> 2;         // Q tile of this warp group
        const int quarter = warp & 3;          // TMEM lanes 32*quarter .. +31 (fixed by the warp id)
        const int t = quarter * 32 + lane;     // query row of this thread within its Q tile = TMEM lane
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const float csc = p.scale_log2;        // > 0 (checked on the host)
        const uint32_t tS = tmem + kColS + g * kNK + lane_off;
        const uint32_t tO = tmem + kColO + g * kD + lane_off;
        // this thread's row of a segment's unit: query row (chunk position, head) and its last key
        struct Row {
            bool valid;
            int ipos, head, plim;
        };
        auto row_of = [&](const Seg &sg) {
            const PrefillSeq &q = p.seqs[sg.si];
            const int gr = sg.r * kUnitRows + g * kM + t;  // row of the sequence's chunk x heads
            Row rw;
            rw.valid = gr < q.chunk_len * G;
            rw.ipos = rw.valid ? gr / G : 0;
            rw.head = rw.valid ? gr % G : 0;
            rw.plim = q.prefix_len + min(gr / G, q.chunk_len - 1);
            return rw;
        };
        // O (TMEM) times inv, rounded once, into this thread's output row if
        // the row exists.  Every lane runs the TMEM loads: they are
        // warp-collective, and a warp of the last row tile can hold rows on
        // both sides of the chunk's end.
        auto store_out = [&](T *orow, float inv, bool valid) {
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
        };

        // Only what the tile loop needs stays live across it; the segment is
        // computed again for its epilogue (the softmax runs at the register limit).
        int gt = 0;  // this CTA's tile count: ring items and barrier phases
        for (int x = x0, sc = 0; x < x1; ++sc) {
            int nt, j0, jn, plim, plim_min, kend;
            {
                const Seg sg = seg_at<G>(p, x, x1);
                const PrefillSeq &q = p.seqs[sg.si];
                nt = sg.t1 - sg.t0;
                j0 = sg.t0;
                jn = sg.n - 1;  // the unit's last key tile
                plim = row_of(sg).plim;
                // smallest limit in the Q tile, and the unit's last key
                plim_min = q.prefix_len + min((sg.r * kUnitRows + g * kM) / G, q.chunk_len - 1);
                kend = q.prefix_len + min(q.chunk_len - 1, ((sg.r + 1) * kUnitRows - 1) / G);
            }

            float m_run = -INFINITY;  // running max in scaled log2 units
            float2 l2[4];             // row sum as four pairs of partial sums
#pragma unroll
            for (int e = 0; e < 4; ++e) l2[e] = make_float2(0.f, 0.f);
            for (int k = 0; k < nt; ++k, ++gt) {
                const int j = j0 + k;  // key tile of the unit
                wait_or_flag(&s_full[g], (uint32_t)gt & 1u, p.d_err);
                tc_fence_after();
                if (g == kQT - 1 && t == 0) {
                    // S of the last Q tile complete means every MMA issued
                    // before it has finished too (one thread issues them, and a
                    // commit tracks all of its earlier MMAs): K of this tile and
                    // V of the one before are read for good
                    if (2 * gt + kSlots < nitems) mbar_arrive1(&empty[(2 * gt) % kSlots]);
                    if (gt >= 1 && 2 * gt - 1 + kSlots < nitems) mbar_arrive1(&empty[(2 * gt - 1) % kSlots]);
                    // and on the segment's last tile, both QKs of it have read Q
                    if (k == nt - 1) mbar_arrive1(q_empty);
                }
                // causal mask only on tiles that reach past some row's limit
                const int kb = j * kNK;
                const bool need_mask = kb + kNK - 1 > plim_min;
                // the whole S row in registers: four loads, one wait
                float s[kNK];
                tmem_ld32p(tS + 0, s + 0);
                tmem_ld32p(tS + 32, s + 32);
                tmem_ld32p(tS + 64, s + 64);
                tmem_ld32p(tS + 96, s + 96);
                tmem_wait_ld();
                if (need_mask) {
#pragma unroll
                    for (int c = 0; c < kNK; ++c) s[c] = (kb + c <= plim) ? s[c] : -INFINITY;
                }
                // row max with three-input maxima: 8 chains over the 128 columns
                float mx8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) mx8[e] = fmaxf(s[e], s[8 + e]);
                static_assert(kNK % 16 == 0, "columns in steps of 16");
#pragma unroll
                for (int c = 16; c < kNK; c += 16) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) mx8[e] = fmax3(mx8[e], s[c + e], s[c + 8 + e]);
                }
                float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
                mx *= csc;

                // Lazy rescale: the maximum moves only when it grew by more than
                // 2^8.  The TMEM loads and stores of O are warp-collective, so the
                // warp decides together: lanes whose maximum did not grow scale by 1.
                const bool up = mx > m_run + 8.0f;
                const bool any_up = __any_sync(kFull, up);
                float alpha = 1.f;  // factor for what was accumulated against the old maximum
                if (up) {
                    alpha = m_run == -INFINITY ? 0.f : fast_exp2(m_run - mx);
                    m_run = mx;
#pragma unroll
                    for (int e = 0; e < 4; ++e) l2[e] = __fmul2_rn(l2[e], make_float2(alpha, alpha));
                }
                // P row t = 2^(s*scale - max), rounded to the input type, packed
                // two per column over S's first 64 columns, 16 keys at a time (S
                // is already in registers, and each stored piece frees its part
                // of it: 128 scores plus a larger piece would not fit in the 168
                // registers a thread has with ten warps on four sub-partitions).
                // A row whose keys in this segment are all masked (a segment of
                // a unit's last tiles that starts past the row's position) has
                // no maximum yet: its weights are 2^-inf = 0.
                const float m_use = m_run == -INFINITY ? 0.f : m_run;
                const float2 csc2 = make_float2(csc, csc), negm2 = make_float2(-m_use, -m_use);
#pragma unroll
                for (int h = 0; h < kNK / 16; ++h) {
                    uint32_t pk[8];
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const int kk = h * 16 + 2 * c;
                        const float2 a = __ffma2_rn(make_float2(s[kk], s[kk + 1]), csc2, negm2);
                        const float2 e2 = make_float2(fast_exp2(a.x), fast_exp2(a.y));
                        l2[c & 3] = __fadd2_rn(l2[c & 3], e2);
                        pk[c] = Elem<T>::pack2(e2.x, e2.y);
                    }
                    tmem_st8u(tS + h * 8, pk);
                }
                if (any_up && k >= 1) {
                    // S complete means O holds every PV before it: rescale in
                    // place (before P is announced, so the next PV adds to the
                    // scaled O)
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float v[32];
                        tmem_ld32(tO + c * 32, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] *= alpha;
                        tmem_st32(tO + c * 32, v);
                    }
                }
                if (j == jn && kb + kNK - 1 > kend) {
                    // V rows past the unit's last key hold whatever the pool has
                    // there (possibly NaN, and 0 * NaN poisons O): zero them
                    const int iv = 2 * gt + 1, sl = iv % kSlots;
                    wait_or_flag(&full[sl], (uint32_t)(iv / kSlots) & 1u, p.d_err);
                    const int z0 = kend + 1 - kb;
                    const uint32_t v_s = sb + kOffKV + sl * kKVTile;
                    for (int idx = t; idx < (kNK - z0) * 16; idx += 128) {
                        const int rr = z0 + (idx >> 4), hh = (idx >> 3) & 1, cc = idx & 7;
                        asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(
                                         v_s + (rr >> 3) * 2048 + hh * 1024 + (rr & 7) * 128 + cc * 16),
                                     "r"(0u)
                                     : "memory");
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                }
                tmem_wait_st();
                tc_fence_before();
                named_bar_arrive(kBarP + g, 160);
            }

            // ---- end of the segment.  O (unnormalised) is complete in TMEM; it
            // stays there until the next segment's first PV, which comes only
            // after this thread announces that segment's first P, while the
            // tensor pipe already works on the next segment's first S.
            wait_or_flag(&o_done[g], (uint32_t)sc & 1u, p.d_err);
            tc_fence_after();
            const int x_next = x + nt;
            const float l_run =
                ((l2[0].x + l2[0].y) + (l2[1].x + l2[1].y)) + ((l2[2].x + l2[2].y) + (l2[3].x + l2[3].y));
            {
                const Seg sg = seg_at<G>(p, x, x1);
                const PrefillSeq &q = p.seqs[sg.si];
                const Row rw = row_of(sg);
                T *orow = static_cast<T *>(p.out) +
                          ((size_t)(q.row_start + rw.ipos) * p.num_heads + sg.h * G + rw.head) * kD;
                if (sg.t0 == 0 && sg.t1 == sg.n) {
                    // the whole unit: normalise, round once, store
                    store_out(orow, l_run > 0.f ? 1.f / l_run : 0.f, rw.valid);
                } else {
                    // part of a unit: write the partial to this CTA's slot (0 for
                    // the first segment of its range, 1 for the last), count it,
                    // and if it is the unit's last to arrive, merge all of them
                    const long long Wt = p.total_tiles, Nc = ncta;
                    finish_partial<T>(reinterpret_cast<float4 *>(p.part_o), p.part_ml, &p.counters[sg.unit * kQT + g],
                                      orow, rw.valid, tO, tS, x_next >= x1, g, t, 2 * cta + (sc == 0 ? 0 : 1),
                                      cta, cta_of(sg.x_unit, Wt, Nc), cta_of(sg.x_unit + sg.n - 1, Wt, Nc),
                                      sg.x_unit, Wt, Nc, m_run, l_run, merge_flag);
                }
            }
            x = x_next;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (!kKeepTmem && warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
    }
    return tmem;
}

// The pool as a 4-D tensor {64 dims, 8 rows, 2 dim halves, 8-row groups}
// with strides {2, 256, 128, 2048} bytes; a box is one block (block_size / 8
// groups), landing as [group][half][8 rows][128 B], 128-byte swizzled.
inline bool make_pool_map(CUtensorMap *map, const void *pool, const PrefillParams &p, int bs, bool bf16) {
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

// The query [rows][heads][128] as a 3-D tensor {128 dims, heads, rows}; a box
// is {64 dims, G heads, 128/G rows} (128 rows of 128 bytes), 128-byte swizzled.
inline bool make_query_map(CUtensorMap *map, const PrefillParams &p, int G, bool bf16) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)p.num_heads, (cuuint64_t)p.query_rows};
    const cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)p.num_heads * kD * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)(kM / G)};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
              const_cast<void *>(p.query), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline size_t round256(size_t n) { return (n + 255) / 256 * 256; }

// Workspace regions for `ctas` stream-K CTAs and `units` merge counters.
// [ctas][2 slots][kQT][128 rows][128] partial outputs, [ctas][2][kQT][128]
// (max, sum) pairs, 256 bytes holding the one-launch step's decode queue
// counter, then a counter per (unit, Q tile).  Only the counters' length
// depends on the call, so every counter sits at the same place from call to
// call and stays zero between calls.
struct PrefillWs {
    size_t o_bytes, ml_bytes, q_bytes, cnt_bytes;
    size_t queue_off() const { return o_bytes + ml_bytes; }
    size_t cnt_off() const { return o_bytes + ml_bytes + q_bytes; }
    size_t total() const { return o_bytes + ml_bytes + q_bytes + cnt_bytes; }
};
inline PrefillWs prefill_ws(long long ctas, long long units) {
    PrefillWs w;
    w.o_bytes = round256((size_t)ctas * 2 * kQT * kM * kD * sizeof(float));
    w.ml_bytes = round256((size_t)ctas * 2 * kQT * kM * sizeof(float2));
    w.q_bytes = 256;
    w.cnt_bytes = round256((size_t)units * kQT * sizeof(unsigned));
    return w;
}

// Units in (sequence, kv head, row tile) order and their key tiles laid end to
// end: fills the schedule fields of p.  Returns PA_OK, or an error.
inline int prefill_schedule(PrefillParams &p, int group, long long *units_out) {
    long long tiles = 0, units = 0;
    for (int i = 0; i < p.num_seqs; ++i) {
        PrefillSeq &q = p.seqs[i];
        const long long rows = (long long)q.chunk_len * group;
        const int row_tiles = (int)((rows + kUnitRows - 1) / kUnitRows);
        long long per_head = 0;
        for (int r = 0; r < row_tiles; ++r) per_head += unit_tiles(q.prefix_len, q.chunk_len, group, r);
        if (per_head > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
        q.row_tiles = row_tiles;
        q.tiles_per_head = (int)per_head;
        q.tile_start = (int)tiles;
        q.unit_start = (int)units;
        tiles += per_head * p.num_kv_heads;
        units += (long long)row_tiles * p.num_kv_heads;
        if (tiles > 0x3fffffffLL || units > 0x3fffffffLL) return PA_ERR_UNSUPPORTED;
    }
    p.total_tiles = (int)tiles;
    *units_out = units;
    return PA_OK;
}

}  // namespace pf
}  // namespace pa
