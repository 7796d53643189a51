// Self-test of the bounded pipeline wait every kernel of the library uses: a
// wait on an mbarrier that nothing ever arrives on must give up after its
// poll limit, flag PA_DEVERR_TIMEOUT and let the kernel return, leaving the
// context usable.  Nothing is copied into the barrier's shared memory, so the
// CTA may exit with the phase incomplete.
#include <cuda_runtime.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

__global__ void __launch_bounds__(32) bounded_wait_selftest_kernel(uint32_t max_polls, int *d_err,
                                                                     long long *d_cycles) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncwarp();
    if (threadIdx.x == 0) {
        const long long t0 = clock64();
        if (!mbar_wait(&bar, 0u, max_polls)) flag_error(d_err, PA_DEVERR_TIMEOUT);
        if (d_cycles) *d_cycles = clock64() - t0;
    }
}

}  // namespace
}  // namespace pa

extern "C" int pa_selftest_bounded_wait(int max_polls, int *d_err, long long *d_cycles, void *stream) {
    if (max_polls <= 0 || !d_err) return PA_ERR_INVALID_ARG;
    pa::bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>((uint32_t)max_polls, d_err,
                                                                                      d_cycles);
    return cudaPeekAtLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

extern "C" int pa_bounded_wait_polls(void) { return (int)pa::kMaxPolls; }
