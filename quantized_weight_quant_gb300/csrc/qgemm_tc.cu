// Tensor-core prefill path (placeholder until the tcgen05 kernel lands).
#include "qwq_internal.h"

namespace qwq {

cudaError_t launch_prefill_tc(const Tensor &, const Tensor *, const float *, float *, float *, int,
                              cudaStream_t, bool *handled) {
    *handled = false;
    return cudaSuccess;
}

cudaError_t prefill_take_error(unsigned int *code) {
    *code = 0;
    return cudaSuccess;
}

}  // namespace qwq
