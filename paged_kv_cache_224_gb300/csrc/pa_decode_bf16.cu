// bf16 instances of the paged decode kernels (one translation unit per dtype
// so the two compile in parallel).
#include "pa_decode.cuh"

namespace pa {
int launch_decode_bf16(int head_dim, int block_size, int group, const DecodeParams &p,
                       cudaStream_t stream) {
    return launch_decode_dtype<__nv_bfloat16>(head_dim, block_size, group, p, stream);
}
int launch_decode_reduce_bf16(int head_dim, const DecodeParams &p, cudaStream_t stream) {
    return launch_reduce_dtype<__nv_bfloat16>(head_dim, p, stream);
}
}  // namespace pa
