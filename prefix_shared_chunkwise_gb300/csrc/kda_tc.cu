// Tensor-core (tcgen05 / TMEM / TMA) kernels for bf16 packed-tree KDA, dk = dv = 128,
// chunk 64.
#include "kda_common.cuh"

namespace harts {

bool tc_supported(bool backward, int dtype, int D, int BC) {
    (void)backward; (void)dtype; (void)D; (void)BC;
    return false;
}

cudaError_t tc_fwd_round(const FwdParams &, const PlanDev &, int32_t, int32_t, int32_t, cudaStream_t) {
    return cudaErrorNotSupported;
}

cudaError_t tc_bwd_round(const BwdParams &, const PlanDev &, int32_t, int32_t, int32_t, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace harts
