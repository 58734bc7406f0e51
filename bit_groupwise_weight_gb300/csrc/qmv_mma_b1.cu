// qmv_mma_b1.cu -- the warp-level tensor-core decode kernel (qmv_mma.cuh)
// for 1-bit codes; each bit width is its own translation unit so that the
// kernels compile in parallel.
#include "qmv_mma.cuh"

namespace lowbit {
namespace mma {

cudaError_t launch_b1(const uint16_t *x, const uint8_t *w, const uint16_t *s, const uint16_t *z,
                      const uint16_t *bias, uint16_t *y, int64_t M, int K, int N, int group, int F,
                      cudaStream_t stream) {
    return launch_rows<1>(x, w, s, z, bias, y, M, K, N, group, F, stream);
}

uint32_t timeouts_b1(bool reset) { return read_timeouts(reset); }

}  // namespace mma
}  // namespace lowbit
