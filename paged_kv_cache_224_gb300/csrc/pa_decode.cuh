// Paged single-query decode attention for sm_103a.
//
// Follows the three steps of the PagedAttention kernel described on the page
// "vLLM PagedAttention chuyen sau" (locionic.com), section "Co che
// PagedAttention": (1) look up each logical block's physical block in the
// sequence's block table, (2) gather the K and V rows from those
// non-contiguous blocks, (3) attend.
//
// Work decomposition.  One CTA owns one unit = (sequence, kv head, partition
// of partition_tokens tokens).  The unit's tokens are cut into tiles of TR
// rows (4 KB of K and 4 KB of V: 16 rows at head_dim 128, 32 at 64); a tile
// is gathered from several whole blocks when block_size < TR, or is TR rows
// of one block otherwise.  The CTA's NW warps take the tiles round robin and
// each streams its tiles into a private S-stage shared-memory ring with 1-D
// bulk (TMA) copies completed on mbarriers, so no warp waits on a global load
// in its compute loop.  All G = Hq/Hkv query heads of the group are processed
// against each tile, so every K/V byte is read from HBM once per kv head.
//
// Per tile (see attend_tile): QK partial dots use packed fp32x2 FMAs and are
// combined by a shuffle reduce-scatter across the lanes that share a K row,
// which leaves every score on exactly one lane (no redundant exp).  Softmax is
// online in fp32, in log2 units, with a warp vote that rescales only when a
// score exceeds the running max by more than 2^8 (exact in real arithmetic;
// fp32 keeps its relative precision).  P goes through a small shared buffer,
// stored twice per value so the packed PV FMAs can use it directly, and PV
// accumulates in fp32 registers.  The warps of the CTA merge through shared
// memory; a unit that is a whole sequence writes the rounded output,
// otherwise it writes unnormalised partials (acc, max, sum) for the
// log-sum-exp reduce kernel.
#pragma once

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D, int BS, int G, int NW, int S>
struct DecodeCfg {
    static constexpr int TILE_BYTES = 4096;           // K (or V) bytes of one tile
    static constexpr int ROWB = D * 2;                // bytes per K/V row
    static constexpr int TR = TILE_BYTES / ROWB;      // rows per tile: 16 at D=128, 32 at D=64
    static constexpr bool MULTI = BS < TR;            // a tile spans several blocks
    static constexpr int BPT = MULTI ? TR / BS : 1;   // blocks per tile
    static constexpr int PART_BYTES = MULTI ? BS * ROWB : TILE_BYTES;  // bytes per copy
    // PV layout: LPT lanes per V row, one 16-byte chunk (8 dims) each
    static constexpr int LPT = D / 8;
    static constexpr int TPI = 32 / LPT;              // V rows per warp-wide 512-byte load
    // QK layout: QL lanes per K row, CPL chunks each; fewer lanes per row means
    // a shorter shuffle reduction at the price of more query registers
    static constexpr int CPL = (D == 128 && G <= 4) ? 2 : 1;
    static constexpr int QL = D / 8 / CPL;
    static constexpr int QRP = 32 / QL;               // K rows per pass of the warp
    static constexpr int NQ = TR / QRP;               // K rows per lane per tile
    static constexpr int NQS_CAP = (32 / G) < 8 ? (32 / G) : 8;
    static constexpr int NQS = NQ < NQS_CAP ? NQ : NQS_CAP;  // K rows per lane per softmax step
    static constexpr int STEPS = NQ / NQS;
    static constexpr int STEP_ROWS = NQS * QRP;       // tokens per softmax step
    static constexpr int N = NQS * G;                 // partial scores per lane per step
    static constexpr int R = N >= QL ? N / QL : 1;    // scores a lane owns after reduce-scatter
    static constexpr int DUP = N >= QL ? 1 : QL / N;  // lanes sharing one score when N < QL
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    static constexpr int RING_BYTES = S * STAGE_BYTES;
    static constexpr int PBUF_FLOATS = TR * G * 2;    // P[token][head], stored twice
    static constexpr int OFF_PBUF = NW * RING_BYTES;
    static constexpr int OFF_FLAG = OFF_PBUF + NW * PBUF_FLOATS * 4;
    static constexpr int OFF_BAR = (OFF_FLAG + NW * S * 4 + 7) / 8 * 8;
    static constexpr int SMEM = OFF_BAR + NW * S * 8;
    static constexpr int HDR = (2 * G + 3) / 4 * 4;   // (max, sum) header of a warp's merge area
    static_assert(D % 64 == 0 && TR * ROWB == TILE_BYTES, "head_dim");
    static_assert(MULTI ? (TR % BS == 0 && BPT <= 4) : (BS % TR == 0), "block_size");
    static_assert(TR % QRP == 0 && NQ % NQS == 0 && STEP_ROWS % TPI == 0, "tile rows");
    static_assert(G <= QL, "group larger than lanes per row");
    static_assert((G & (G - 1)) == 0 && (NQS & (NQS - 1)) == 0 && (QL & (QL - 1)) == 0,
                  "the reduce-scatter relabelling XORs indices");
    static_assert((HDR + G * D) * 4 <= RING_BYTES, "merge area must fit in one warp's ring");
    static_assert(NW * 32 >= G * (D / 8), "merge needs one thread per (head, 8 dims)");
    static_assert(OFF_PBUF % 16 == 0, "alignment");
};

// Shuffle reduce-scatter across the lanes of a row group (xor masks M, M/2,
// .., 1).  Each halving step keeps the low half of the array and adds the
// partner's high half; when one value is left the remaining steps are a plain
// all-reduce.  For that to add like to like, every lane lays its partial dots
// out under its own relabelling: array slot k holds the dot for (head, row)
// index k XOR base, where base is the index the lane ends up owning -- R*c
// for lane c of the group if N >= group size, else c / (group size / N) --
// so partners, which differ in one bit of base, send exactly what the other
// keeps.  Afterwards lane c holds indices base + f (f < R).
template <int N, int M>
struct ReduceScatter {
    static __device__ __forceinline__ void run(float *v, int lane) {
        if constexpr (M == 0) {
            return;
        } else if constexpr (N > 1) {
#pragma unroll
            for (int k = 0; k < N / 2; ++k) v[k] += __shfl_xor_sync(kFull, v[k + N / 2], M);
            ReduceScatter<N / 2, M / 2>::run(v, lane);
        } else {
            v[0] += __shfl_xor_sync(kFull, v[0], M);
            ReduceScatter<1, M / 2>::run(v, lane);
        }
    }
};

template <typename T>
__device__ __forceinline__ void unpack8x2(const uint4 &u, float2 (&f)[4]) {
    Elem<T>::unpack2(u.x, f[0].x, f[0].y);
    Elem<T>::unpack2(u.y, f[1].x, f[1].y);
    Elem<T>::unpack2(u.z, f[2].x, f[2].y);
    Elem<T>::unpack2(u.w, f[3].x, f[3].y);
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Per-lane online-softmax state of one warp.
template <int G>
struct WarpState {
    float2 acc[G][4];  // acc[h][j] = (out[h][8c+2j], out[h][8c+2j+1]), unnormalised
    float m_run[G];    // running max per head (log2 units), uniform across the warp
    float m_mine;      // m_run of the head this lane owns scores of
    float l_mine;      // sum of this lane's owned probabilities
};

// One K/V tile: QK, online softmax update, PV.
//   QK layout: lane = (qr, qc): K row step*STEP_ROWS + i*QRP + qr, chunks qc + cc*QL.
//   PV layout: lane = (grp, c): V row step*STEP_ROWS + i*TPI + grp, chunk c.
template <typename T, class C, int G>
__device__ __forceinline__ void attend_tile(const unsigned char *Ks, const unsigned char *Vs, int nvalid,
                                            const float2 (&q2)[G][C::CPL][4], WarpState<G> &st,
                                            float *pbuf, int lane, int idx0, int h_lane, bool owner) {
    const int qr = lane / C::QL, qc = lane % C::QL;
    const int grp = lane / C::LPT, c = lane % C::LPT;
    const bool full = nvalid == C::TR;
#pragma unroll
    for (int step = 0; step < C::STEPS; ++step) {
        if (step * C::STEP_ROWS >= nvalid) break;  // nothing valid left in the tile
        float v[C::N];
        // QK partial dots over this lane's CPL*8 dims, head-major v[h*NQS + i]
#pragma unroll
        for (int i = 0; i < C::NQS; ++i) {
            const int row = step * C::STEP_ROWS + (i ^ (idx0 % C::NQS)) * C::QRP + qr;  // relabelled row
            float2 a[G];
#pragma unroll
            for (int cc = 0; cc < C::CPL; ++cc) {
                float2 k2[4];
                unpack8x2<T>(lds128(Ks + row * C::ROWB + (qc + cc * C::QL) * 16), k2);
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    a[h] = cc == 0 ? __fmul2_rn(q2[h][cc][0], k2[0]) : __ffma2_rn(q2[h][cc][0], k2[0], a[h]);
                    a[h] = __ffma2_rn(q2[h][cc][1], k2[1], a[h]);
                    a[h] = __ffma2_rn(q2[h][cc][2], k2[2], a[h]);
                    a[h] = __ffma2_rn(q2[h][cc][3], k2[3], a[h]);
                }
            }
#pragma unroll
            for (int h = 0; h < G; ++h) v[h * C::NQS + i] = a[h].x + a[h].y;
        }
        ReduceScatter<C::N, C::QL / 2>::run(v, lane);

        // owned scores: index idx0 + f -> K row i = index % NQS of head h_lane
        float sc[C::R];
        bool need = false;
#pragma unroll
        for (int f = 0; f < C::R; ++f) {
            const int i = (idx0 + f) % C::NQS;
            const int tok = step * C::STEP_ROWS + i * C::QRP + qr;
            sc[f] = (full || tok < nvalid) ? v[f] : -INFINITY;
            need |= sc[f] > st.m_mine + kRescaleThreshold;
        }
        if (__any_sync(kFull, need)) {
            float mymax = sc[0];
#pragma unroll
            for (int f = 1; f < C::R; ++f) mymax = fmaxf(mymax, sc[f]);
            float bm[G];
#pragma unroll
            for (int h = 0; h < G; ++h) bm[h] = (h == h_lane) ? mymax : -INFINITY;
#pragma unroll
            for (int m = 16; m >= 1; m >>= 1)
#pragma unroll
                for (int h = 0; h < G; ++h) bm[h] = fmaxf(bm[h], __shfl_xor_sync(kFull, bm[h], m));
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float nm = fmaxf(st.m_run[h], bm[h]);
                const float alpha = st.m_run[h] == -INFINITY ? 0.f : fast_exp2(st.m_run[h] - nm);
                const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                for (int j = 0; j < 4; ++j) st.acc[h][j] = __fmul2_rn(st.acc[h][j], a2);
                if (h == h_lane) {
                    st.l_mine *= alpha;
                    st.m_mine = nm;
                }
                st.m_run[h] = nm;
            }
        }
        if (owner) {
#pragma unroll
            for (int f = 0; f < C::R; ++f) {
                const float pr = fast_exp2(sc[f] - st.m_mine);
                st.l_mine += pr;
                const int i = (idx0 + f) % C::NQS;
                const int tok = step * C::STEP_ROWS + i * C::QRP + qr;
                *reinterpret_cast<float2 *>(pbuf + 2 * (tok * G + h_lane)) = make_float2(pr, pr);
            }
        }
        __syncwarp();
        // PV over this step's tokens and this lane's 8 dims
#pragma unroll
        for (int i = 0; i < C::STEP_ROWS / C::TPI; ++i) {
            const int row = step * C::STEP_ROWS + i * C::TPI + grp;
            float2 v2[4];
            unpack8x2<T>(lds128(Vs + row * C::ROWB + c * 16), v2);
            if (!full && row >= nvalid) {
#pragma unroll
                for (int j = 0; j < 4; ++j) v2[j] = make_float2(0.f, 0.f);  // garbage past the context
            }
            const float *prow = pbuf + 2 * row * G;
            float2 pp[G];
            if constexpr (G >= 2) {
#pragma unroll
                for (int h2 = 0; h2 < G; h2 += 2) {
                    const float4 x = *reinterpret_cast<const float4 *>(prow + 2 * h2);
                    pp[h2] = make_float2(x.x, x.y);
                    pp[h2 + 1] = make_float2(x.z, x.w);
                }
            } else {
                pp[0] = *reinterpret_cast<const float2 *>(prow);
            }
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int j = 0; j < 4; ++j) st.acc[h][j] = __ffma2_rn(pp[h], v2[j], st.acc[h][j]);
        }
        __syncwarp();
    }
}

// Physical block for logical block j of the unit: the first 64 come from two
// lane-distributed registers, later ones (partitions longer than 64 blocks)
// straight from the table.  Every lane of the warp must call this with the
// same j.
__device__ __forceinline__ int unit_block(int j, int e0, int e1, const int32_t *table) {
    if (j < 32) return __shfl_sync(kFull, e0, j);
    if (j < 64) return __shfl_sync(kFull, e1, j - 32);
    return table[j];
}

// Resident CTAs per SM the register budget is sized for: three CTAs of four
// warps for groups up to 4 (<= 170 registers), two for group 8.
template <int G>
constexpr int decode_min_ctas() { return G <= 4 ? 3 : 2; }

template <typename T, int D, int BS, int G, int NW, int S>
__global__ void __launch_bounds__(NW * 32, decode_min_ctas<G>()) decode_kernel(const DecodeParams p) {
    using C = DecodeCfg<D, BS, G, NW, S>;
    extern __shared__ __align__(128) unsigned char smem[];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
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
    const int blk0 = tok0 / BS;
    const int nblk = (ntok + BS - 1) / BS;
    const int ntile_all = (ntok + C::TR - 1) / C::TR;
    const int ntile = ntile_all > warp ? (ntile_all - warp + NW - 1) / NW : 0;  // this warp's tiles

    unsigned char *ring = smem + warp * C::RING_BYTES;
    float *pbuf = reinterpret_cast<float *>(smem + C::OFF_PBUF) + warp * C::PBUF_FLOATS;
    volatile int *sflag = reinterpret_cast<int *>(smem + C::OFF_FLAG) + warp * S;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR) + warp * S;

    if (lane == 0) {
#pragma unroll
        for (int k = 0; k < S; ++k) mbar_init(&bars[k], 1);
        fence_barrier_init();
    }
    __syncwarp();

    // ---- step 1 (look up): the unit's first 64 block-table entries
    const int32_t *table = p.block_tables + (size_t)s * p.table_stride + p.len_offset / BS + blk0;
    const int e0 = lane < nblk ? table[lane] : 0;
    const int e1 = 32 + lane < nblk ? table[32 + lane] : 0;

    const size_t run_elems = (size_t)BS * D;           // one (block, kv head) run
    const size_t blk_elems = run_elems * p.num_kv_heads;
    const T *kbase = static_cast<const T *>(p.k_cache) + (size_t)kvh * run_elems;
    const T *vbase = static_cast<const T *>(p.v_cache) + (size_t)kvh * run_elems;
    const uint64_t pol = policy_evict_first();
    const int num_blocks = p.num_blocks;
    int *const d_err = p.d_err;

    // step 2 (gather): the warp's j-th tile (unit tile warp + j*NW) into stage st
    auto issue = [&](int j, int st) {
        const int t = warp + j * NW;
        int phys[C::BPT];
        int nb = 1;
        bool ok = true;
        size_t roff = 0;
        if constexpr (C::MULTI) {
            nb = min(C::BPT, nblk - t * C::BPT);
#pragma unroll
            for (int b = 0; b < C::BPT; ++b) {
                phys[b] = 0;
                if (b < nb) {
                    phys[b] = unit_block(t * C::BPT + b, e0, e1, table);
                    ok = ok && phys[b] >= 0 && phys[b] < num_blocks;
                }
            }
        } else {
            phys[0] = unit_block((t * C::TR) / BS, e0, e1, table);
            ok = phys[0] >= 0 && phys[0] < num_blocks;
            roff = (size_t)((t * C::TR) % BS) * D;
        }
        if (lane == 0) {
            sflag[st] = ok ? 1 : 0;
            if (ok) {
                unsigned char *dst = ring + st * C::STAGE_BYTES;
                mbar_arrive_expect_tx(&bars[st], 2u * C::PART_BYTES * (uint32_t)nb);
#pragma unroll
                for (int b = 0; b < C::BPT; ++b) {
                    if (b < nb) {
                        const size_t src = (size_t)phys[b] * blk_elems + roff;
                        bulk_g2s(dst + b * C::PART_BYTES, kbase + src, C::PART_BYTES, &bars[st], pol);
                        bulk_g2s(dst + C::TILE_BYTES + b * C::PART_BYTES, vbase + src, C::PART_BYTES,
                                 &bars[st], pol);
                    }
                }
            } else {
                flag_error(d_err, PA_DEVERR_BLOCK_RANGE);
                mbar_arrive(&bars[st]);
            }
        }
    };

#pragma unroll
    for (int k = 0; k < S; ++k)
        if (k < ntile) issue(k, k);

    // ---- query rows of the group in the QK layout, pre-scaled into log2 units
    const int qc = lane % C::QL;
    // real query/out row of head h of this unit (see DecodeParams)
    auto row_of = [&](int h) -> size_t {
        return (size_t)(s * p.grp_size + h / p.grp_inner) * p.num_heads + (size_t)kvh * p.grp_inner +
               h % p.grp_inner;
    };
    // The (head, row) index this lane's scores end with (see ReduceScatter);
    // its slot h of q2 holds head h XOR (idx0 / NQS), its K row i is row i XOR
    // (idx0 % NQS).
    const int idx0 = C::N >= C::QL ? C::R * qc : qc / C::DUP;
    const int h_lane = idx0 / C::NQS;
    const bool owner = C::N >= C::QL || (qc % C::DUP) == 0;
    float2 q2[G][C::CPL][4];
    {
        const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const T *qrow = static_cast<const T *>(p.query) + row_of(h ^ h_lane) * D;
#pragma unroll
            for (int cc = 0; cc < C::CPL; ++cc) {
                const uint4 u = *reinterpret_cast<const uint4 *>(qrow + (qc + cc * C::QL) * 8);
                unpack8x2<T>(u, q2[h][cc]);
#pragma unroll
                for (int j = 0; j < 4; ++j) q2[h][cc][j] = __fmul2_rn(q2[h][cc][j], sc2);
            }
        }
    }


    WarpState<G> st;
#pragma unroll
    for (int h = 0; h < G; ++h) {
        st.m_run[h] = -INFINITY;
#pragma unroll
        for (int j = 0; j < 4; ++j) st.acc[h][j] = make_float2(0.f, 0.f);
    }
    st.m_mine = -INFINITY;
    st.l_mine = 0.f;
    bool timed_out = false;
    int consumed = 0;

    // ---- step 3 (attend) over this warp's tiles
    for (int j = 0; j < ntile; ++j) {
        const int sl = j % S;
        if (!mbar_wait(&bars[sl], (uint32_t)(j / S) & 1u)) {
            timed_out = true;
            break;
        }
        consumed = j + 1;
        const int t = warp + j * NW;
        const int nvalid = min(C::TR, ntok - t * C::TR);
        if (sflag[sl]) {
            const unsigned char *Ks = ring + sl * C::STAGE_BYTES;
            attend_tile<T, C, G>(Ks, Ks + C::TILE_BYTES, nvalid, q2, st, pbuf, lane, idx0, h_lane, owner);
        }
        __syncwarp();
        if (j + S < ntile) issue(j + S, sl);
    }

    if (timed_out) {
        flag_error(d_err, PA_DEVERR_TIMEOUT);
        // let copies already in flight land before the CTA's smem goes away
        const int issued = min(ntile, consumed + S);
        for (int j = consumed; j < issued; ++j) mbar_wait(&bars[j % S], (uint32_t)(j / S) & 1u);
        // contribute nothing from this warp
#pragma unroll
        for (int h = 0; h < G; ++h) {
            st.m_run[h] = -INFINITY;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) st.acc[h][jj] = make_float2(0.f, 0.f);
        }
        st.l_mine = 0.f;
    }

    // ---- merge the row groups of this warp, then the warps of the CTA
    const int grp = lane / C::LPT;
    const int c = lane % C::LPT;
#pragma unroll
    for (int m = C::LPT; m < 32; m <<= 1)
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                st.acc[h][jj].x += __shfl_xor_sync(kFull, st.acc[h][jj].x, m);
                st.acc[h][jj].y += __shfl_xor_sync(kFull, st.acc[h][jj].y, m);
            }
    float lh[G];
#pragma unroll
    for (int h = 0; h < G; ++h) lh[h] = (h == h_lane && owner) ? st.l_mine : 0.f;
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1)
#pragma unroll
        for (int h = 0; h < G; ++h) lh[h] += __shfl_xor_sync(kFull, lh[h], m);

    // merge area in this warp's (now idle) ring: [G] max, [G] sum (padded), [G][D] acc
    float *cm = reinterpret_cast<float *>(ring);
    if (lane == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            cm[h] = st.m_run[h];
            cm[G + h] = lh[h];
        }
    }
    if (grp == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float4 *dst = reinterpret_cast<float4 *>(cm + C::HDR + h * D + c * 8);
            dst[0] = make_float4(st.acc[h][0].x, st.acc[h][0].y, st.acc[h][1].x, st.acc[h][1].y);
            dst[1] = make_float4(st.acc[h][2].x, st.acc[h][2].y, st.acc[h][3].x, st.acc[h][3].y);
        }
    }
    __syncthreads();

    const int tid = threadIdx.x;
    if (tid < G * (D / 8)) {
        const int h = tid / (D / 8);
        const int ch = tid % (D / 8);
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, reinterpret_cast<const float *>(smem + w * C::RING_BYTES)[h]);
        float lsum = 0.f;
        float o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const float *wm = reinterpret_cast<const float *>(smem + w * C::RING_BYTES);
                const float mw = wm[h];
                const float sc = mw == -INFINITY ? 0.f : fast_exp2(mw - M);
                lsum = fmaf(sc, wm[G + h], lsum);
                const float4 a = *reinterpret_cast<const float4 *>(wm + C::HDR + h * D + ch * 8);
                const float4 b = *reinterpret_cast<const float4 *>(wm + C::HDR + h * D + ch * 8 + 4);
                o[0] = fmaf(sc, a.x, o[0]); o[1] = fmaf(sc, a.y, o[1]);
                o[2] = fmaf(sc, a.z, o[2]); o[3] = fmaf(sc, a.w, o[3]);
                o[4] = fmaf(sc, b.x, o[4]); o[5] = fmaf(sc, b.y, o[5]);
                o[6] = fmaf(sc, b.z, o[6]); o[7] = fmaf(sc, b.w, o[7]);
            }
        }
        const size_t row = row_of(h);
        if (nparts == 1 && !p.force_partials) {
            const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) o[e] *= inv;
            T *orow = static_cast<T *>(p.out) + row * D + ch * 8;
            *reinterpret_cast<uint4 *>(orow) = pack8<T>(o);
        } else {
            const size_t slot = row * p.slots + p.part_base + part;
            float4 *dst = reinterpret_cast<float4 *>(p.ws_acc + slot * D + ch * 8);
            dst[0] = make_float4(o[0], o[1], o[2], o[3]);
            dst[1] = make_float4(o[4], o[5], o[6], o[7]);
            if (ch == 0) p.ws_ml[slot] = make_float2(M, lsum);
        }
    }
}

// Log-sum-exp merge of split-K partials: one warp per (sequence, query head).
//   M = max_p m_p,  w_p = 2^(m_p - M),  out = sum_p w_p acc_p / sum_p w_p l_p.
template <typename T, int D>
__global__ void __launch_bounds__(128) decode_reduce_kernel(const DecodeParams p) {
    constexpr int VPL = D / 32;  // values per lane
    pdl_wait();                  // the decode kernel's partials are complete and visible
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pair = blockIdx.x * 4 + warp;
    if (pair >= p.num_seqs * p.num_heads) return;
    const int s = pair / p.num_heads;
    // same clamping as the decode kernel; slots = the fixed ones plus one per
    // partition of the sequence's own tokens
    int L = p.context_lens[s] - p.len_offset;
    const int Lcap = min(p.max_context_len, p.max_blocks_per_seq * p.block_size) - p.len_offset;
    L = L < 0 ? 0 : (L > Lcap ? Lcap : L);
    const int own = L > 0 ? (L + p.partition_tokens - 1) / p.partition_tokens : (p.red_fixed_slots > 0 ? 0 : 1);
    const int nparts = p.red_fixed_slots + own;
    if (nparts <= 1 && !p.force_partials) return;
    const size_t base = (size_t)pair * p.slots;
    float M = -INFINITY;
    for (int i = lane; i < nparts; i += 32) M = fmaxf(M, p.ws_ml[base + i].x);
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, m));
    float lsum = 0.f;
    float o[VPL];
#pragma unroll
    for (int d = 0; d < VPL; ++d) o[d] = 0.f;
#pragma unroll 4
    for (int i = 0; i < nparts; ++i) {
        const float2 ml = p.ws_ml[base + i];
        const float w = fast_exp2(ml.x - M);
        lsum = fmaf(w, ml.y, lsum);
        const float *a = p.ws_acc + (base + i) * D + lane * VPL;
        if constexpr (VPL == 4) {
            const float4 x = *reinterpret_cast<const float4 *>(a);
            o[0] = fmaf(w, x.x, o[0]); o[1] = fmaf(w, x.y, o[1]);
            o[2] = fmaf(w, x.z, o[2]); o[3] = fmaf(w, x.w, o[3]);
        } else {
            const float2 x = *reinterpret_cast<const float2 *>(a);
            o[0] = fmaf(w, x.x, o[0]); o[1] = fmaf(w, x.y, o[1]);
        }
    }
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    T *orow = static_cast<T *>(p.out) + (size_t)pair * D + lane * VPL;
    if constexpr (VPL == 4) {
        uint2 u;
        u.x = Elem<T>::pack2(o[0] * inv, o[1] * inv);
        u.y = Elem<T>::pack2(o[2] * inv, o[3] * inv);
        *reinterpret_cast<uint2 *>(orow) = u;
    } else {
        *reinterpret_cast<uint32_t *>(orow) = Elem<T>::pack2(o[0] * inv, o[1] * inv);
    }
}

constexpr int kDecodeWarps = 4;
constexpr int kDecodeStages = 2;

template <typename T, int D, int BS, int G>
int launch_decode_t(const DecodeParams &p, cudaStream_t stream) {
    constexpr int NW = kDecodeWarps;
    constexpr int S = kDecodeStages;
    using C = DecodeCfg<D, BS, G, NW, S>;
    auto kern = decode_kernel<T, D, BS, G, NW, S>;
    static std::atomic<uint64_t> attr_done{0};
    if (ensure_smem_attr(kern, C::SMEM, attr_done) != PA_OK) return PA_ERR_CUDA;
    const long long units = (long long)p.max_partitions * p.num_seqs * p.num_kv_heads;
    if (units <= 0) return PA_OK;
    if (units > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    if (launch_pdl(kern, dim3((unsigned)units), dim3(NW * 32), C::SMEM, stream, p) != cudaSuccess) return PA_ERR_CUDA;
    if (p.max_partitions > 1 && !p.force_partials) {
        const int pairs = p.num_seqs * p.num_heads;
        if (launch_pdl(decode_reduce_kernel<T, D>, dim3((pairs + 3) / 4), dim3(128), 0, stream, p) != cudaSuccess)
            return PA_ERR_CUDA;
    }
    return PA_OK;
}

template <typename T>
int launch_reduce_dtype(int head_dim, const DecodeParams &p, cudaStream_t stream) {
    const int pairs = p.num_seqs * p.num_heads;
    if (pairs <= 0) return PA_OK;
    cudaError_t e;
    if (head_dim == 128) e = launch_pdl(decode_reduce_kernel<T, 128>, dim3((pairs + 3) / 4), dim3(128), 0, stream, p);
    else if (head_dim == 64) e = launch_pdl(decode_reduce_kernel<T, 64>, dim3((pairs + 3) / 4), dim3(128), 0, stream, p);
    else return PA_ERR_UNSUPPORTED;
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

template <typename T>
int launch_decode_dtype(int head_dim, int block_size, int group, const DecodeParams &p,
                        cudaStream_t stream) {
#define PA_DECODE_CASE(DD, BB, GG)                                           \
    if (head_dim == DD && block_size == BB && group == GG)                   \
        return launch_decode_t<T, DD, BB, GG>(p, stream);
#define PA_DECODE_GROUPS(DD, BB) \
    PA_DECODE_CASE(DD, BB, 1) PA_DECODE_CASE(DD, BB, 2) PA_DECODE_CASE(DD, BB, 4) PA_DECODE_CASE(DD, BB, 8)
    PA_DECODE_GROUPS(128, 16)
    PA_DECODE_GROUPS(128, 32)
    PA_DECODE_GROUPS(128, 8)
    PA_DECODE_GROUPS(128, 64)
    PA_DECODE_GROUPS(128, 128)
    PA_DECODE_GROUPS(64, 16)
    PA_DECODE_GROUPS(64, 32)
    PA_DECODE_GROUPS(64, 8)
    PA_DECODE_GROUPS(64, 64)
    PA_DECODE_GROUPS(64, 128)
#undef PA_DECODE_GROUPS
#undef PA_DECODE_CASE
    return PA_ERR_UNSUPPORTED;
}

}  // namespace pa
