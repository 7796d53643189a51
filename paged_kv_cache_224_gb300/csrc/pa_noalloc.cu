// pa_decode_noalloc: the paged decode for callers that cannot allocate device
// memory on this path.  The split-K partials that pa_decode keeps in a
// caller-owned workspace live here in one library-owned device array instead;
// the call then goes through pa_decode unchanged.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/pa.h"

namespace {

// Split-K scratch shared by every pa_decode_noalloc call on a device.  In host
// code this name is only a stand-in for the symbol: its device address comes
// from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_decode_scratch[PA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void *g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current) and cached.
int scratch_address(void **addr) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
    std::lock_guard<std::mutex> guard(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return PA_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return PA_OK;
}

}  // namespace

extern "C" int pa_decode_noalloc(void *out, const void *query, const void *k_cache,
                                 const void *v_cache, const int32_t *block_tables,
                                 int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                                 int num_heads, int num_kv_heads, int head_dim, int block_size,
                                 int num_blocks, int max_context_len, float scale,
                                 int partition_tokens, pa_dtype dtype, int *d_err, void *stream) {
    // Reject sizes the array cannot hold before touching the device.
    const size_t need = pa_decode_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                                  max_context_len, partition_tokens);
    if (need > PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_SCRATCH_LIMIT;
    void *scratch = nullptr;
    const int rc = scratch_address(&scratch);
    if (rc != PA_OK) return rc;
    return pa_decode(out, query, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                     num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                     max_context_len, scale, partition_tokens, dtype, scratch,
                     PA_NOALLOC_SCRATCH_BYTES, d_err, stream);
}
