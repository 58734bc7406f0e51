// qmm.cu -- tensor-core (tcgen05) quantised matrix-matrix product.  Not built yet.
#include "common.cuh"

namespace lowbit {
uint32_t qmm_timeouts(bool) { return 0; }
cudaError_t launch_qmm(const uint16_t *, const uint8_t *, const uint16_t *, const uint16_t *,
                       const uint16_t *, uint16_t *, int64_t, int64_t, int64_t, int, int,
                       cudaStream_t) {
    return cudaErrorNotSupported;
}
}  // namespace lowbit
