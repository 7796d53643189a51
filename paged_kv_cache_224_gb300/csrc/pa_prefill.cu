// Chunked-prefill attention over a paged KV cache (tensor cores).
//
// Follows the page "vLLM PagedAttention chuyen sau" (locionic.com), section
// "Chunked Prefill": a long prompt is processed chunk by chunk, each chunk's
// KV accumulates in the sequence's blocks, and each chunk attends to the
// cache built so far.  Query row i of the chunk sits at absolute position
// prefix_len + i and attends causally to keys 0 .. prefix_len + i, gathered
// through the block table exactly as in decode.
//
// Unlike decode, a chunk against its keys is a dense contraction (C query
// rows x G heads against every key), so QK^T and PV run on the tensor cores:
// m16n8k16 MMAs with fp32 accumulation.  A CTA takes 64 (position, head)
// rows of one kv head -- 64/G chunk positions times the G heads that share
// the kv head -- so every K/V tile staged in shared memory serves all G heads.
// Each of its 4 warps owns 16 rows; the Q fragments stay in registers for the
// whole key loop.  K/V tiles of 64 keys are gathered row by row through the
// block table with 16-byte cp.async copies into an XOR-swizzled layout
// (conflict-free ldmatrix), double-buffered.  Softmax is online in fp32 (log2
// units); P is rounded to the MMA input type for PV, as in any tensor-core
// attention.  Keys past the causal limit of a row are masked; rows past the
// chunk are not stored.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kD = 128;         // head_dim supported by this kernel
constexpr int kRows = 64;       // (position, head) rows per CTA
constexpr int kKeys = 64;       // keys per K/V tile
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kRowBytes = kD * 2;                   // 256 bytes per row
constexpr int kTileBytes = kKeys * kRowBytes;       // 16 KB per K or V tile
constexpr int kQBytes = kRows * kRowBytes;          // 16 KB
constexpr int kSmem = kQBytes + 2 * 2 * kTileBytes; // Q + double-buffered K and V = 80 KB

// Byte offset of 16-byte chunk `ch` (0..15) of row `r` in a swizzled tile:
// the low three bits of the chunk index are XOR-ed with the row, so the 8
// rows an ldmatrix reads at one logical chunk hit 8 different bank groups.
__device__ __forceinline__ int swz(int r, int ch) { return r * kRowBytes + ((ch ^ (r & 7)) << 4); }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
    const int n = valid ? 16 : 0;  // 0 source bytes -> 16 zero bytes
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

template <typename T> struct Mma;
template <> struct Mma<__nv_bfloat16> {
    static __device__ __forceinline__ void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
};
template <> struct Mma<__half> {
    static __device__ __forceinline__ void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
};

// Stage keys [k0, k0 + kKeys) of kv head kvh into a swizzled K tile and V tile.
// Rows past `kend` (the last key any row of this CTA may see) are zero-filled
// and never read from the cache; table entries outside the pool are flagged
// and their rows zero-filled.
template <int BS>
__device__ __forceinline__ void load_kv_tile(const PrefillParams &p, uint32_t ks, uint32_t vs, int k0,
                                             int kend, int kvh, const int32_t *__restrict__ table) {
    const unsigned char *kc = static_cast<const unsigned char *>(p.k_cache);
    const unsigned char *vc = static_cast<const unsigned char *>(p.v_cache);
    // 64 rows x 16 chunks = 1024 chunks for K (and V); 8 per thread
#pragma unroll
    for (int it = 0; it < kKeys * 16 / kThreads; ++it) {
        const int idx = it * kThreads + threadIdx.x;
        const int r = idx >> 4, ch = idx & 15;
        const int key = k0 + r;
        bool valid = key <= kend;
        size_t off = 0;
        if (valid) {
            const int blk = table[key / BS];
            if (blk < 0 || blk >= p.num_blocks) {
                if (ch == 0) flag_error(p.d_err, PA_DEVERR_BLOCK_RANGE);
                valid = false;
            } else {
                off = ((((size_t)blk * p.num_kv_heads + kvh) * BS + (key % BS)) * kD) * 2 + ch * 16;
            }
        }
        const int so = swz(r, ch);
        cp_async16(ks + so, kc + off, valid);
        cp_async16(vs + so, vc + off, valid);
    }
}

template <typename T, int BS, int G>
__global__ void __launch_bounds__(kThreads) prefill_kernel(const PrefillParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kvh = blockIdx.y;
    const int row0 = blockIdx.x * kRows;  // first (position, head) row of this CTA
    const int nrows = p.chunk_len * G;
    const int i_last = min(p.chunk_len - 1, (row0 + kRows - 1) / G);
    const int kend = p.prefix_len + i_last;  // last key any row of this CTA sees
    const int ntiles = kend / kKeys + 1;
    const int32_t *table = p.block_table;

    const uint32_t sq = smem_addr(smem);
    const uint32_t skv = sq + kQBytes;  // buffer b: K at skv + b*2*tile, V right after

    // ---- Q tile: row r = (position i0 + r/G, head kvh*G + r%G), swizzled
    {
        const unsigned char *qg = static_cast<const unsigned char *>(p.query);
#pragma unroll
        for (int it = 0; it < kRows * 16 / kThreads; ++it) {
            const int idx = it * kThreads + threadIdx.x;
            const int r = idx >> 4, ch = idx & 15;
            const int gr = row0 + r;
            const bool valid = gr < nrows;
            const int i = gr / G, h = gr % G;
            const size_t off = valid ? ((((size_t)i * p.num_heads + kvh * G + h) * kD) * 2 + ch * 16) : 0;
            cp_async16(sq + swz(r, ch), qg + off, valid);
        }
    }
    load_kv_tile<BS>(p, skv, skv + kTileBytes, 0, kend, kvh, table);
    cp_async_commit();

    // per-thread rows: g and g+8 of the warp's 16
    const int g = lane >> 2, t4 = lane & 3;
    const int wrow = warp * 16;
    int pos_lim[2];  // last key each of the thread's two rows may see
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        const int gr = row0 + wrow + g + 8 * hr;
        pos_lim[hr] = p.prefix_len + min(gr / G, p.chunk_len - 1);
    }

    float o[16][4];  // O[16 rows][128 dims]: 16 n-tiles of 8 dims
#pragma unroll
    for (int n = 0; n < 16; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[n][e] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY};
    float l_run[2] = {0.f, 0.f};
    uint32_t qa[8][4];  // Q fragments for the 8 k-steps of 16 dims

    for (int tile = 0; tile < ntiles; ++tile) {
        const int buf = tile & 1;
        const uint32_t ks = skv + buf * 2 * kTileBytes;
        const uint32_t vs = ks + kTileBytes;
        if (tile + 1 < ntiles) {
            const uint32_t nks = skv + (buf ^ 1) * 2 * kTileBytes;
            load_kv_tile<BS>(p, nks, nks + kTileBytes, (tile + 1) * kKeys, kend, kvh, table);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        if (tile == 0) {
            // Q fragments: lane l supplies row l%16, column block 8*(l/16) of each 16x16 block
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                ldsm_x4(sq + swz(wrow + (lane & 15), kk * 2 + (lane >> 4)), qa[kk]);
        }

        // ---- S = Q K^T for 64 keys: 8 n-tiles of 8 keys
        float s[8][4];
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[n][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
            for (int n2 = 0; n2 < 4; ++n2) {  // two n-tiles (16 keys) per ldmatrix.x4
                uint32_t b[4];
                const int key = n2 * 16 + (lane & 7) + ((lane >> 4) << 3);
                const int ch = kk * 2 + ((lane >> 3) & 1);
                ldsm_x4(ks + swz(key, ch), b);
                Mma<T>::run(s[2 * n2], qa[kk], b[0], b[1]);
                Mma<T>::run(s[2 * n2 + 1], qa[kk], b[2], b[3]);
            }
        }

        // ---- causal mask, online softmax (log2 units)
        const int kbase = tile * kKeys;
        float mt[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int hr = e >> 1;
                const int key = kbase + n * 8 + 2 * t4 + (e & 1);
                float v = s[n][e] * p.scale_log2;
                v = key <= pos_lim[hr] ? v : -INFINITY;
                s[n][e] = v;
                mt[hr] = fmaxf(mt[hr], v);
            }
        float alpha[2];
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            mt[hr] = fmaxf(mt[hr], __shfl_xor_sync(kFull, mt[hr], 1));
            mt[hr] = fmaxf(mt[hr], __shfl_xor_sync(kFull, mt[hr], 2));
            const float mn = fmaxf(m_run[hr], mt[hr]);
            alpha[hr] = m_run[hr] == -INFINITY ? 0.f : fast_exp2(m_run[hr] - mn);
            m_run[hr] = mn;
            l_run[hr] *= alpha[hr];
        }
#pragma unroll
        for (int n = 0; n < 16; ++n) {
            o[n][0] *= alpha[0];
            o[n][1] *= alpha[0];
            o[n][2] *= alpha[1];
            o[n][3] *= alpha[1];
        }
        uint32_t pa_[4][4];  // P as A fragments for the 4 k-steps of 16 keys
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            const float p0 = m_run[0] == -INFINITY ? 0.f : fast_exp2(s[n][0] - m_run[0]);
            const float p1 = m_run[0] == -INFINITY ? 0.f : fast_exp2(s[n][1] - m_run[0]);
            const float p2 = m_run[1] == -INFINITY ? 0.f : fast_exp2(s[n][2] - m_run[1]);
            const float p3 = m_run[1] == -INFINITY ? 0.f : fast_exp2(s[n][3] - m_run[1]);
            l_run[0] += p0 + p1;
            l_run[1] += p2 + p3;
            const int kk = n >> 1, hi = n & 1;
            pa_[kk][2 * hi] = Elem<T>::pack2(p0, p1);
            pa_[kk][2 * hi + 1] = Elem<T>::pack2(p2, p3);
        }

        // ---- O += P V: 4 k-steps of 16 keys, 16 n-tiles of 8 dims
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
            for (int n2 = 0; n2 < 8; ++n2) {  // two dim n-tiles per ldmatrix.x4.trans
                uint32_t b[4];
                const int key = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
                const int ch = n2 * 2 + (lane >> 4);
                ldsm_x4_t(vs + swz(key, ch), b);
                Mma<T>::run(o[2 * n2], pa_[kk], b[0], b[1]);
                Mma<T>::run(o[2 * n2 + 1], pa_[kk], b[2], b[3]);
            }
        }
        __syncthreads();  // this buffer is refilled in the next iteration
    }

    // ---- normalise and store rows (position, head)
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        float l = l_run[hr];
        l += __shfl_xor_sync(kFull, l, 1);
        l += __shfl_xor_sync(kFull, l, 2);
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const int gr = row0 + wrow + g + 8 * hr;
        if (gr < nrows) {
            const int i = gr / G, h = gr % G;
            T *orow = static_cast<T *>(p.out) + ((size_t)i * p.num_heads + kvh * G + h) * kD;
#pragma unroll
            for (int n = 0; n < 16; ++n) {
                const uint32_t v = Elem<T>::pack2(o[n][2 * hr] * inv, o[n][2 * hr + 1] * inv);
                *reinterpret_cast<uint32_t *>(orow + n * 8 + 2 * t4) = v;
            }
        }
    }
}

template <typename T, int BS, int G>
int launch_prefill_t(const PrefillParams &p, cudaStream_t stream) {
    auto kern = prefill_kernel<T, BS, G>;
    static bool attr_set = false;
    if (!attr_set) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess)
            return PA_ERR_CUDA;
        attr_set = true;
    }
    const int rows = p.chunk_len * G;
    dim3 grid((rows + kRows - 1) / kRows, p.num_kv_heads);
    kern<<<grid, kThreads, kSmem, stream>>>(p);
    return cudaPeekAtLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

template <typename T>
int launch_prefill_dtype(int block_size, int group, const PrefillParams &p, cudaStream_t stream) {
#define PA_PREFILL_CASE(BB, GG) \
    if (block_size == BB && group == GG) return launch_prefill_t<T, BB, GG>(p, stream);
#define PA_PREFILL_GROUPS(BB) \
    PA_PREFILL_CASE(BB, 1) PA_PREFILL_CASE(BB, 2) PA_PREFILL_CASE(BB, 4) PA_PREFILL_CASE(BB, 8)
    PA_PREFILL_GROUPS(16)
    PA_PREFILL_GROUPS(32)
#undef PA_PREFILL_GROUPS
#undef PA_PREFILL_CASE
    return PA_ERR_UNSUPPORTED;
}

}  // namespace

int launch_prefill(pa_dtype dt, int head_dim, int block_size, int group, const PrefillParams &p,
                   cudaStream_t stream) {
    if (head_dim != kD) return PA_ERR_UNSUPPORTED;
    return dt == PA_BF16 ? launch_prefill_dtype<__nv_bfloat16>(block_size, group, p, stream)
                         : launch_prefill_dtype<__half>(block_size, group, p, stream);
}

}  // namespace pa
