// Chunked-prefill attention (placeholder until the tensor-core kernel lands).
#include "pa_internal.h"

namespace pa {
int launch_prefill(pa_dtype, int, int, int, const PrefillParams &, cudaStream_t) {
    return PA_ERR_UNSUPPORTED;
}
}  // namespace pa
