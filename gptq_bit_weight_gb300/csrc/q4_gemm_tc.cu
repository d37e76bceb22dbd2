// Tensor-core (tcgen05) GEMM and fused prefill: not built yet.
#include <climits>

#include "q4_internal.cuh"

namespace q4 {
cudaError_t launch_gemm_f16(const uint16_t *, const uint16_t *, const uint16_t *, int, int, int, uint16_t *, int *,
                            cudaStream_t) {
    return cudaErrorNotSupported;
}
cudaError_t launch_prefill(const HandleView &, const uint16_t *, int, uint16_t *, cudaStream_t) {
    return cudaErrorNotSupported;
}
int prefill_default_min_m() { return INT_MAX; }
}  // namespace q4
