// Paged single-query decode attention for sm_103a.
//
// Follows the three steps of the PagedAttention kernel described on the page
// "vLLM PagedAttention chuyen sau" (locionic.com), section "Co che
// PagedAttention": (1) look up each logical block's physical block in the
// sequence's block table, (2) gather the K and V rows from those
// non-contiguous blocks, (3) attend.
//
// Work decomposition.  One CTA owns one unit = (sequence, kv head, partition
// of partition_tokens tokens).  Its NW warps take the partition's blocks
// round robin; each warp streams its (block, kv head) tiles -- one contiguous
// block_size*head_dim run of K and one of V -- into a private S-stage
// shared-memory ring with 1-D bulk (TMA) copies completed on mbarriers, so a
// warp never waits on global loads in its compute loop.  All G = Hq/Hkv query
// heads of the group are processed against each tile, so every K/V byte is
// read from HBM once per kv head.
//
// Per tile, lane l holds the 16-byte chunk c = l % LPT (dims 8c..8c+7) of rows
// i*TPI + l/LPT.  QK partial dots over 8 dims are combined by a shuffle
// reduce-scatter across the LPT lanes of a row, which leaves every score on
// one lane (no redundant exp).  Softmax is online in fp32, in log2 units, with
// a warp vote that rescales only when a score exceeds the running max by more
// than 2^8 (exact in real arithmetic; fp32 keeps its relative precision).
// P is broadcast through a small shared buffer and PV accumulates in fp32
// registers (acc[G][8] per lane).  Warps merge through shared memory; a unit
// that is a whole sequence writes the rounded output, otherwise it writes
// unnormalised partials (acc, max, sum) for the log-sum-exp reduce kernel.
#pragma once

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D, int BS, int G, int NW, int S>
struct DecodeCfg {
    static constexpr int LPT = D / 8;                 // lanes per K/V row (16-byte chunks)
    static constexpr int TPI = 32 / LPT;              // rows covered by one warp-wide 512-B load
    static constexpr int NT = BS / TPI;               // rows per lane per tile
    static constexpr int NTS_CAP = (32 / G) < 8 ? (32 / G) : 8;
    static constexpr int NTS = NT < NTS_CAP ? NT : NTS_CAP;  // rows per lane per softmax step
    static constexpr int STEPS = NT / NTS;
    static constexpr int N = NTS * G;                 // partial scores per lane per step
    static constexpr int R = N >= LPT ? N / LPT : 1;  // scores a lane owns after reduce-scatter
    static constexpr int DUP = N >= LPT ? 1 : LPT / N;  // lanes sharing one score when N < LPT
    static constexpr int TILE_BYTES = BS * D * 2;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    static constexpr int RING_BYTES = S * STAGE_BYTES;
    static constexpr int PBUF_FLOATS = TPI * N;
    static constexpr int OFF_PBUF = NW * RING_BYTES;
    static constexpr int OFF_FLAG = OFF_PBUF + NW * PBUF_FLOATS * 4;
    static constexpr int OFF_BAR = (OFF_FLAG + NW * S * 4 + 7) / 8 * 8;
    static constexpr int SMEM = OFF_BAR + NW * S * 8;
    static_assert(D % 8 == 0 && 32 % LPT == 0, "head_dim");
    static_assert(BS % TPI == 0 && NT % NTS == 0, "block_size");
    static_assert(G <= LPT, "group larger than lanes per row");
    static_assert(G * (D + 2) * 4 <= RING_BYTES, "combine area must fit in one warp's ring");
    static_assert(NW * 32 >= G * (D / 8), "combine needs one thread per (head, 8 dims)");
    static_assert(TILE_BYTES % 16 == 0, "bulk copy size");
};

// Shuffle reduce-scatter across the LPT lanes of a row group (xor masks M,
// M/2, .., 1).  Each halving step keeps one half of the array and adds the
// partner's copy of it; when one value is left the remaining steps are a
// plain all-reduce.  Afterwards lane c of the group holds original index
// f + R*c (f < R) if N >= LPT, else index c / (LPT/N).
template <int N, int M>
struct ReduceScatter {
    static __device__ __forceinline__ void run(float *v, int lane) {
        if constexpr (M == 0) {
            return;
        } else if constexpr (N > 1) {
            const bool upper = (lane & M) != 0;
#pragma unroll
            for (int k = 0; k < N / 2; ++k) {
                const float a = v[k], b = v[k + N / 2];
                const float send = upper ? a : b;
                const float keep = upper ? b : a;
                v[k] = keep + __shfl_xor_sync(kFull, send, M);
            }
            ReduceScatter<N / 2, M / 2>::run(v, lane);
        } else {
            v[0] += __shfl_xor_sync(kFull, v[0], M);
            ReduceScatter<1, M / 2>::run(v, lane);
        }
    }
};

template <typename T, int D, int BS, int G, int NW, int S>
__global__ void __launch_bounds__(NW * 32) decode_kernel(const DecodeParams p) {
    using C = DecodeCfg<D, BS, G, NW, S>;
    extern __shared__ __align__(128) unsigned char smem[];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int grp = lane / C::LPT;  // which row of a 512-B warp load
    const int c = lane % C::LPT;    // which 16-byte chunk of the row

    // ---- unit = (partition, sequence, kv head); partition-major order
    const int per_part = p.num_seqs * p.num_kv_heads;
    const int part = blockIdx.x / per_part;
    const int rem = blockIdx.x - part * per_part;
    const int s = rem / p.num_kv_heads;
    const int kvh = rem - s * p.num_kv_heads;

    int L = p.context_lens[s];
    const int Lcap = min(p.max_context_len, p.max_blocks_per_seq * BS);
    if (L < 0 || L > Lcap) {
        if (threadIdx.x == 0 && part == 0 && kvh == 0) flag_error(p.d_err, PA_DEVERR_CONTEXT_RANGE);
        L = L < 0 ? 0 : Lcap;
    }
    const int PT = p.partition_tokens;
    const int nparts = L > 0 ? (L + PT - 1) / PT : 1;
    if (part >= nparts) return;
    const int tok0 = part * PT;
    const int tok1 = min(L, tok0 + PT);
    const int blk0 = tok0 / BS;
    const int nblk = tok1 > tok0 ? (tok1 - tok0 + BS - 1) / BS : 0;
    const int ntile = nblk > warp ? (nblk - warp + NW - 1) / NW : 0;

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

    // ---- step 1 (look up): this warp's block-table entries, 32 at a time
    const int32_t *table = p.block_tables + (size_t)s * p.max_blocks_per_seq + blk0 + warp;
    int bt_base = 0;
    int bt_reg = lane < ntile ? table[lane * NW] : 0;

    const size_t tile_elems = (size_t)BS * D;
    const size_t blk_elems = tile_elems * p.num_kv_heads;
    const T *kbase = static_cast<const T *>(p.k_cache) + (size_t)kvh * tile_elems;
    const T *vbase = static_cast<const T *>(p.v_cache) + (size_t)kvh * tile_elems;
    const uint64_t pol = policy_evict_first();

    // step 2 (gather): lane 0 starts the bulk copies of tile tn into stage st
    auto issue = [&](int tn, int st) {
        if (tn - bt_base >= 32) {
            bt_base += 32;
            const int i = bt_base + lane;
            bt_reg = i < ntile ? table[(size_t)i * NW] : 0;
        }
        const int phys = __shfl_sync(kFull, bt_reg, tn - bt_base);
        if (lane == 0) {
            const bool ok = phys >= 0 && phys < p.num_blocks;
            sflag[st] = ok ? 1 : 0;
            if (ok) {
                mbar_arrive_expect_tx(&bars[st], C::STAGE_BYTES);
                bulk_g2s(ring + st * C::STAGE_BYTES, kbase + (size_t)phys * blk_elems, C::TILE_BYTES,
                         &bars[st], pol);
                bulk_g2s(ring + st * C::STAGE_BYTES + C::TILE_BYTES, vbase + (size_t)phys * blk_elems,
                         C::TILE_BYTES, &bars[st], pol);
            } else {
                flag_error(p.d_err, PA_DEVERR_BLOCK_RANGE);
                asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&bars[st]))
                             : "memory");
            }
        }
    };

#pragma unroll
    for (int k = 0; k < S; ++k)
        if (k < ntile) issue(k, k);

    // ---- query rows of the group, pre-scaled into log2 units
    float q[G][8];
    {
        const T *qrow = static_cast<const T *>(p.query) +
                        ((size_t)s * p.num_heads + (size_t)kvh * G) * D + c * 8;
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const uint4 u = *reinterpret_cast<const uint4 *>(qrow + (size_t)h * D);
            unpack8<T>(u, q[h]);
#pragma unroll
            for (int d = 0; d < 8; ++d) q[h][d] *= p.scale_log2;
        }
    }

    // The one head this lane's owned scores belong to (see ReduceScatter).
    const int idx0 = C::N >= C::LPT ? C::R * c : c / C::DUP;
    const int h_lane = idx0 / C::NTS;
    const bool owner = C::N >= C::LPT || (c % C::DUP) == 0;

    float acc[G][8];
    float m_run[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        m_run[h] = -INFINITY;
#pragma unroll
        for (int d = 0; d < 8; ++d) acc[h][d] = 0.f;
    }
    float m_mine = -INFINITY;
    float l_mine = 0.f;
    bool timed_out = false;
    int consumed = 0;

    // ---- step 3 (attend) over this warp's tiles
    for (int t = 0; t < ntile; ++t) {
        const int st = t % S;
        const uint32_t par = (uint32_t)(t / S) & 1u;
        if (!mbar_wait(&bars[st], par)) {
            timed_out = true;
            break;
        }
        consumed = t + 1;
        const int jt = blk0 + warp + t * NW;  // logical block of this tile
        const int nvalid = min(BS, L - jt * BS);
        if (sflag[st]) {
            const unsigned char *Ks = ring + st * C::STAGE_BYTES;
            const unsigned char *Vs = Ks + C::TILE_BYTES;
            const bool full = nvalid == BS;
#pragma unroll
            for (int step = 0; step < C::STEPS; ++step) {
                if (step * C::NTS * C::TPI >= nvalid) break;  // nothing valid left in the tile
                float v[C::N];
                // QK partial dots over this lane's 8 dims, head-major v[h*NTS + i]
#pragma unroll
                for (int i = 0; i < C::NTS; ++i) {
                    const int row = step * C::NTS + i;
                    float k[8];
                    unpack8<T>(lds128(Ks + (row * 32 + lane) * 16), k);
#pragma unroll
                    for (int h = 0; h < G; ++h) {
                        float a = q[h][0] * k[0];
#pragma unroll
                        for (int d = 1; d < 8; ++d) a = fmaf(q[h][d], k[d], a);
                        v[h * C::NTS + i] = a;
                    }
                }
                ReduceScatter<C::N, C::LPT / 2>::run(v, lane);

                // owned scores: index f + idx0 -> token i = index % NTS of head h_lane
                float sc[C::R];
                bool need = false;
#pragma unroll
                for (int f = 0; f < C::R; ++f) {
                    const int i = (idx0 + f) % C::NTS;
                    const int tok = (step * C::NTS + i) * C::TPI + grp;
                    sc[f] = (full || tok < nvalid) ? v[f] : -INFINITY;
                    need |= sc[f] > m_mine + kRescaleThreshold;
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
                        const float nm = fmaxf(m_run[h], bm[h]);
                        const float alpha = m_run[h] == -INFINITY ? 0.f : fast_exp2(m_run[h] - nm);
#pragma unroll
                        for (int d = 0; d < 8; ++d) acc[h][d] *= alpha;
                        if (h == h_lane) {
                            l_mine *= alpha;
                            m_mine = nm;
                        }
                        m_run[h] = nm;
                    }
                }
                float pr[C::R];
#pragma unroll
                for (int f = 0; f < C::R; ++f) {
                    pr[f] = fast_exp2(sc[f] - m_mine);
                    if (owner) l_mine += pr[f];
                }
                if (owner) {
#pragma unroll
                    for (int f = 0; f < C::R; ++f) {
                        const int i = (idx0 + f) % C::NTS;
                        pbuf[grp * C::N + i * G + h_lane] = pr[f];
                    }
                }
                __syncwarp();
                // PV over this lane's rows and dims
#pragma unroll
                for (int i = 0; i < C::NTS; ++i) {
                    const int row = step * C::NTS + i;
                    float vv[8];
                    unpack8<T>(lds128(Vs + (row * 32 + lane) * 16), vv);
                    if (!full && row * C::TPI + grp >= nvalid) {
#pragma unroll
                        for (int d = 0; d < 8; ++d) vv[d] = 0.f;  // garbage past the context
                    }
                    float pp[G];
                    const float *prow = pbuf + grp * C::N + i * G;
                    if constexpr (G % 4 == 0) {
#pragma unroll
                        for (int h4 = 0; h4 < G; h4 += 4) {
                            const float4 x = *reinterpret_cast<const float4 *>(prow + h4);
                            pp[h4] = x.x; pp[h4 + 1] = x.y; pp[h4 + 2] = x.z; pp[h4 + 3] = x.w;
                        }
                    } else if constexpr (G == 2) {
                        const float2 x = *reinterpret_cast<const float2 *>(prow);
                        pp[0] = x.x; pp[1] = x.y;
                    } else {
                        pp[0] = prow[0];
                    }
#pragma unroll
                    for (int h = 0; h < G; ++h)
#pragma unroll
                        for (int d = 0; d < 8; ++d) acc[h][d] = fmaf(pp[h], vv[d], acc[h][d]);
                }
                __syncwarp();
            }
        }
        __syncwarp();
        if (t + S < ntile) issue(t + S, st);
    }

    if (timed_out) {
        flag_error(p.d_err, PA_DEVERR_TIMEOUT);
        // let copies already in flight land before the CTA's smem goes away
        const int issued = min(ntile, consumed + S);
        for (int t = consumed; t < issued; ++t) mbar_wait(&bars[t % S], (uint32_t)(t / S) & 1u);
        // contribute nothing from this warp
#pragma unroll
        for (int h = 0; h < G; ++h) {
            m_run[h] = -INFINITY;
#pragma unroll
            for (int d = 0; d < 8; ++d) acc[h][d] = 0.f;
        }
        l_mine = 0.f;
    }

    // ---- merge the row groups of this warp, then the warps of the CTA
#pragma unroll
    for (int m = C::LPT; m < 32; m <<= 1)
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int d = 0; d < 8; ++d) acc[h][d] += __shfl_xor_sync(kFull, acc[h][d], m);
    float lh[G];
#pragma unroll
    for (int h = 0; h < G; ++h) lh[h] = (h == h_lane && owner) ? l_mine : 0.f;
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1)
#pragma unroll
        for (int h = 0; h < G; ++h) lh[h] += __shfl_xor_sync(kFull, lh[h], m);

    // combine area in this warp's (now idle) ring: [G] max, [G] sum, [G][D] acc
    float *cm = reinterpret_cast<float *>(ring);
    float *cl = cm + G;
    float *ca = cl + G;
    if (lane == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            cm[h] = m_run[h];
            cl[h] = lh[h];
        }
    }
    if (grp == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int d = 0; d < 8; ++d) ca[h * D + c * 8 + d] = acc[h][d];
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
        for (int d = 0; d < 8; ++d) o[d] = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const float *wm = reinterpret_cast<const float *>(smem + w * C::RING_BYTES);
                const float mw = wm[h];
                const float sc = mw == -INFINITY ? 0.f : fast_exp2(mw - M);
                lsum = fmaf(sc, wm[G + h], lsum);
                const float *wa = wm + 2 * G + h * D + ch * 8;
#pragma unroll
                for (int d = 0; d < 8; ++d) o[d] = fmaf(sc, wa[d], o[d]);
            }
        }
        const int hq = kvh * G + h;
        if (nparts == 1) {
            const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
#pragma unroll
            for (int d = 0; d < 8; ++d) o[d] *= inv;
            T *orow = static_cast<T *>(p.out) + ((size_t)s * p.num_heads + hq) * D + ch * 8;
            *reinterpret_cast<uint4 *>(orow) = pack8<T>(o);
        } else {
            const size_t slot = ((size_t)s * p.num_heads + hq) * p.max_partitions + part;
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
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pair = blockIdx.x * 4 + warp;
    if (pair >= p.num_seqs * p.num_heads) return;
    const int s = pair / p.num_heads;
    // same clamping as the decode kernel
    int L = p.context_lens[s];
    const int Lcap = min(p.max_context_len, p.max_blocks_per_seq * p.block_size);
    L = L < 0 ? 0 : (L > Lcap ? Lcap : L);
    const int nparts = L > 0 ? (L + p.partition_tokens - 1) / p.partition_tokens : 1;
    if (nparts <= 1) return;
    const size_t base = (size_t)pair * p.max_partitions;
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
    const float inv = 1.f / lsum;
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

// Stage count per warp: about 24 KB of ring per warp, between 2 and 8 stages.
template <int D, int BS>
constexpr int decode_stages() {
    constexpr int stage = 2 * BS * D * 2;
    constexpr int s = 24576 / stage;
    return s < 2 ? 2 : (s > 8 ? 8 : s);
}

template <typename T, int D, int BS, int G>
int launch_decode_t(const DecodeParams &p, cudaStream_t stream) {
    constexpr int NW = 4;
    constexpr int S = decode_stages<D, BS>();
    using C = DecodeCfg<D, BS, G, NW, S>;
    auto kern = decode_kernel<T, D, BS, G, NW, S>;
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
            return PA_ERR_CUDA;
        attr_set = true;
    }
    const long long units = (long long)p.max_partitions * p.num_seqs * p.num_kv_heads;
    if (units <= 0) return PA_OK;
    if (units > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    kern<<<(unsigned)units, NW * 32, C::SMEM, stream>>>(p);
    if (cudaPeekAtLastError() != cudaSuccess) return PA_ERR_CUDA;
    if (p.max_partitions > 1) {
        const int pairs = p.num_seqs * p.num_heads;
        decode_reduce_kernel<T, D><<<(pairs + 3) / 4, 128, 0, stream>>>(p);
        if (cudaPeekAtLastError() != cudaSuccess) return PA_ERR_CUDA;
    }
    return PA_OK;
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
    PA_DECODE_GROUPS(64, 16)
    PA_DECODE_GROUPS(64, 32)
    PA_DECODE_GROUPS(64, 8)
#undef PA_DECODE_GROUPS
#undef PA_DECODE_CASE
    return PA_ERR_UNSUPPORTED;
}

}  // namespace pa
