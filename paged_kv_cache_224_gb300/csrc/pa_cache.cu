// Cache writes and copy-on-write block copies: pure data movement.
//
// reshape_and_cache follows the page "vLLM PagedAttention chuyen sau"
// (locionic.com), section "Tuong tu phan trang bo nho ao": a growing sequence
// gets new slots in its physical blocks; section "Chunked Prefill", step 3:
// each chunk's KV accumulates in the same blocks.  copy_blocks follows
// section "Co che APC", step 3: a shared block is copied before a sequence
// that diverges writes into it.
//
// Both are HBM-bound streams of 16-byte vectors; every byte is moved once.
#include <algorithm>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

// One thread moves one 16-byte chunk of one (token, kv head) row for both K
// and V.  Reads of key/value are fully coalesced; writes land as contiguous
// head_dim*2-byte rows inside the destination tile.
__global__ void __launch_bounds__(256)
reshape_and_cache_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value,
                         uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                         const int64_t *__restrict__ slots, int num_tokens, int num_kv_heads,
                         int chunks_per_row, int block_size, long long pool_slots, int *d_err) {
    pdl_trigger();  // the decode that follows may be scheduled; it waits for these writes
    const long long per_token = (long long)num_kv_heads * chunks_per_row;
    const long long total = per_token * num_tokens;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long t = i / per_token;
        const long long r = i - t * per_token;  // = h * chunks_per_row + chunk
        const int64_t slot = slots[t];
        if (slot < 0) continue;                 // padding
        if (slot >= pool_slots) {
            if (r == 0) flag_error(d_err, PA_DEVERR_SLOT_RANGE);
            continue;
        }
        const long long blk = slot / block_size;
        const long long off = slot - blk * block_size;
        const long long h = r / chunks_per_row;
        const long long ch = r - h * chunks_per_row;
        const long long dst = ((blk * num_kv_heads + h) * block_size + off) * chunks_per_row + ch;
        k_cache[dst] = key[i];
        v_cache[dst] = value[i];
    }
}

int launch_reshape_and_cache(const void *key, const void *value, void *k_cache, void *v_cache,
                             const int64_t *slots, int num_tokens, int num_kv_heads, int head_dim,
                             int block_size, int num_blocks, int *d_err, cudaStream_t stream) {
    const int cpr = head_dim / 8;
    const long long total = (long long)num_tokens * num_kv_heads * cpr;
    if (total == 0) return PA_OK;
    long long blocks = (total + 255) / 256;
    const long long cap = (long long)sm_count() * 64;  // grid-stride beyond 64 CTAs per SM
    if (blocks > cap) blocks = cap;
    reshape_and_cache_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
        static_cast<const uint4 *>(key), static_cast<const uint4 *>(value),
        static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), slots, num_tokens,
        num_kv_heads, cpr, block_size, (long long)num_blocks * block_size, d_err);
    return cudaPeekAtLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// ---- copy-on-write -----------------------------------------------------------
//
// A pair (src, dst) is copied iff both ids are in the pool, src != dst, no
// other pair has the same dst and no pair (itself included) has dst as its
// src; every other pair is skipped and flagged.  That makes the result
// independent of the order of the pairs.  The verdict needs, for each dst,
// how many pairs name it as dst and as src: one pass over the pairs counts
// both in an open-addressing hash table in the caller's workspace (only ids
// inside the pool are counted; an id outside it cannot equal a valid dst),
// and each copy CTA then looks its dst up once -- O(n) work for n pairs
// instead of every CTA scanning the whole list.

struct CowEntry {
    unsigned int key;   // block id, or kCowEmpty
    unsigned int ndst;  // pairs with this id as dst
    unsigned int nsrc;  // pairs with this id as src
    unsigned int pad;
};
constexpr unsigned int kCowEmpty = 0xffffffffu;

// Slot of a block id: the 32-bit finaliser of MurmurHash3 (so ids with equal
// low bits still spread), masked to the power-of-two table size.
__device__ __forceinline__ unsigned int cow_hash(unsigned int key, unsigned int mask) {
    key ^= key >> 16;
    key *= 0x85ebca6bu;
    key ^= key >> 13;
    key *= 0xc2b2ae35u;
    key ^= key >> 16;
    return key & mask;
}

__global__ void __launch_bounds__(256) cow_clear_kernel(CowEntry *table, unsigned int cap) {
    for (unsigned int i = blockIdx.x * blockDim.x + threadIdx.x; i < cap; i += gridDim.x * blockDim.x)
        table[i] = CowEntry{kCowEmpty, 0u, 0u, 0u};
}

__device__ void cow_count(CowEntry *table, unsigned int mask, unsigned int key, bool as_dst) {
    unsigned int h = cow_hash(key, mask);
    for (unsigned int probe = 0; probe <= mask; ++probe, h = (h + 1) & mask) {
        const unsigned int prev = atomicCAS(&table[h].key, kCowEmpty, key);
        if (prev == kCowEmpty || prev == key) {
            atomicAdd(as_dst ? &table[h].ndst : &table[h].nsrc, 1u);
            return;
        }
    }
}

__global__ void __launch_bounds__(256)
cow_count_kernel(CowEntry *table, unsigned int mask, const int64_t *__restrict__ pairs, int num_pairs,
                 int num_blocks) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < num_pairs; i += gridDim.x * blockDim.x) {
        const int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src >= 0 && src < num_blocks) cow_count(table, mask, (unsigned int)src, false);
        if (dst >= 0 && dst < num_blocks) cow_count(table, mask, (unsigned int)dst, true);
    }
}

// grid = (num_pairs, pieces).  Thread 0 decides whether the pair is valid
// from its dst's counts (every CTA of a pair reaches the same verdict), then
// the CTA copies its piece of the K block and the V block.
__global__ void __launch_bounds__(256)
copy_blocks_kernel(uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                   const int64_t *__restrict__ pairs, const CowEntry *__restrict__ table, unsigned int mask,
                   long long chunks_per_block, long long chunks_per_piece, int num_blocks, int *d_err) {
    __shared__ int s_ok;
    const int i = blockIdx.x;
    const int64_t src = pairs[2 * i];
    const int64_t dst = pairs[2 * i + 1];
    if (threadIdx.x == 0) {
        bool ok = src >= 0 && src < num_blocks && dst >= 0 && dst < num_blocks && src != dst;
        if (ok) {
            // dst was counted by the pass before this kernel, so the probe ends at it
            const unsigned int key = (unsigned int)dst;
            unsigned int h = cow_hash(key, mask);
            ok = false;
            for (unsigned int probe = 0; probe <= mask; ++probe, h = (h + 1) & mask) {
                const unsigned int k = table[h].key;
                if (k == key) {
                    ok = table[h].ndst == 1u && table[h].nsrc == 0u;
                    break;
                }
                if (k == kCowEmpty) break;
            }
        }
        s_ok = ok;
        if (!ok && blockIdx.y == 0) flag_error(d_err, PA_DEVERR_COPY_PAIR);
    }
    __syncthreads();
    if (!s_ok) return;
    const long long begin = (long long)blockIdx.y * chunks_per_piece;
    const long long end = min(begin + chunks_per_piece, chunks_per_block);
    const uint4 *ks = k_cache + src * chunks_per_block;
    const uint4 *vs = v_cache + src * chunks_per_block;
    uint4 *kd = k_cache + dst * chunks_per_block;
    uint4 *vd = v_cache + dst * chunks_per_block;
    for (long long c = begin + threadIdx.x; c < end; c += blockDim.x) {
        const uint4 a = ks[c];
        const uint4 b = vs[c];
        kd[c] = a;
        vd[c] = b;
    }
}

// Entries of the hash table for n pairs: a power of two >= 4n (at most 2n
// distinct ids, so at most half full).
static unsigned long long cow_capacity(int num_pairs) {
    unsigned long long cap = 64;
    while (cap < 4ull * (unsigned long long)num_pairs) cap <<= 1;
    return cap;
}

size_t copy_blocks_workspace_bytes(int num_pairs) {
    if (num_pairs <= 0) return 0;
    return (size_t)cow_capacity(num_pairs) * sizeof(CowEntry);
}

int launch_copy_blocks(void *k_cache, void *v_cache, const int64_t *pairs, int num_pairs,
                       int num_kv_heads, int head_dim, int block_size, int num_blocks, void *workspace,
                       int *d_err, cudaStream_t stream) {
    if (num_pairs == 0) return PA_OK;
    const unsigned long long cap = cow_capacity(num_pairs);
    CowEntry *table = static_cast<CowEntry *>(workspace);
    const int sms = sm_count();
    const unsigned clear_blocks = (unsigned)std::min<unsigned long long>((cap + 255) / 256, (unsigned long long)sms * 8);
    cow_clear_kernel<<<clear_blocks, 256, 0, stream>>>(table, (unsigned int)cap);
    const unsigned count_blocks = (unsigned)std::min<long long>(((long long)num_pairs + 255) / 256, (long long)sms * 8);
    cow_count_kernel<<<count_blocks, 256, 0, stream>>>(table, (unsigned int)(cap - 1), pairs, num_pairs, num_blocks);
    const long long cpb = (long long)num_kv_heads * block_size * head_dim / 8;
    const long long per_piece = 256 * 4;  // 4 vectors per thread per cache
    long long pieces = (cpb + per_piece - 1) / per_piece;
    if (pieces > 65535) pieces = 65535;
    const long long chunks_per_piece = (cpb + pieces - 1) / pieces;
    dim3 grid((unsigned)num_pairs, (unsigned)pieces);
    copy_blocks_kernel<<<grid, 256, 0, stream>>>(static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache),
                                                 pairs, table, (unsigned int)(cap - 1), cpb, chunks_per_piece,
                                                 num_blocks, d_err);
    return cudaPeekAtLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// ---- gather --------------------------------------------------------------------
//
// One launch for a step's small inputs: each CTA strides over the items'
// 16-byte units (or bytes, for an item whose ends or size are not 16-byte
// multiples) so the copies run side by side instead of one after another.
__global__ void __launch_bounds__(256)
gather_kernel(const __grid_constant__ GatherList list) {
    const long long stride = (long long)gridDim.x * blockDim.x;
    const long long t0 = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    for (int it = 0; it < list.n; ++it) {
        const unsigned long long nb = list.bytes[it];
        const bool vec = ((reinterpret_cast<uintptr_t>(list.src[it]) | reinterpret_cast<uintptr_t>(list.dst[it]) |
                           (uintptr_t)nb) & 15u) == 0;
        if (vec) {
            const uint4 *s = static_cast<const uint4 *>(list.src[it]);
            uint4 *d = static_cast<uint4 *>(list.dst[it]);
            for (long long i = t0; i < (long long)(nb / 16); i += stride) d[i] = s[i];
        } else {
            const unsigned char *s = static_cast<const unsigned char *>(list.src[it]);
            unsigned char *d = static_cast<unsigned char *>(list.dst[it]);
            for (long long i = t0; i < (long long)nb; i += stride) d[i] = s[i];
        }
    }
}

int launch_gather(const GatherList &list, cudaStream_t stream) {
    if (list.n <= 0) return PA_OK;
    if (list.n > kGatherMax) return PA_ERR_INVALID_ARG;
    unsigned long long units = 0;
    for (int i = 0; i < list.n; ++i) units += (list.bytes[i] + 15) / 16;
    const long long blocks = std::min<long long>(std::max<long long>(1, (long long)((units + 255) / 256)),
                                                 (long long)sm_count() * 4);
    gather_kernel<<<(unsigned)blocks, 256, 0, stream>>>(list);
    return cudaPeekAtLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa
