// The one-launch step's instances for f16 (see pa_mixed.cuh).
#include "pa_mixed.cuh"

namespace pa {

int launch_mixed_f16(int block_size, int group, const MixedParams &mp, unsigned grid, cudaStream_t stream) {
    return mx::launch_mixed_dtype<__half>(block_size, group, mp, grid, stream);
}

}  // namespace pa
