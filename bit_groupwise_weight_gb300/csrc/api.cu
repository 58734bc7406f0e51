// api.cu -- the C ABI of liblowbit (declared in include/lowbit.h).
//
// Every entry point validates its arguments on the host before it touches
// CUDA, then enqueues the kernel on the caller's stream.  Nothing here
// allocates device memory or synchronises.
#include <atomic>
#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace {

// Self-test of the bounded wait: one thread waits on an mbarrier that nothing
// arrives on, through the same helper every kernel uses.  After the helper's
// limit the wait gives up, counts itself in g_selftest_timeouts and the kernel
// returns; nothing faults and the context stays usable.
__device__ unsigned int g_selftest_timeouts;

__global__ void wait_selftest_kernel(uint32_t *gave_up) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = lowbit::ptx::smem_u32(&bar);
    lowbit::ptx::mbar_init(b, 1);
    lowbit::ptx::fence_mbar_init();
    const bool ok = lowbit::ptx::mbar_wait(b, 0, &g_selftest_timeouts);   // phase 0 never completes
    *gave_up = ok ? 0u : 1u;
}

uint32_t selftest_timeouts(bool reset) {
    unsigned int v = 0;
    cudaMemcpyFromSymbol(&v, g_selftest_timeouts, sizeof(v));
    if (reset) {
        const unsigned int zero = 0;
        cudaMemcpyToSymbol(g_selftest_timeouts, &zero, sizeof(zero));
    }
    return v;
}

bool bits_ok(int bits) { return bits >= 1 && bits <= 7; }
bool group_ok(int g) { return g == 32 || g == 64 || g == 128 || g == 256; }
bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Largest sizes accepted: every index the kernels form stays inside int32 for
// per-row quantities and int64 for whole-buffer offsets.
constexpr int64_t kMaxDim = (int64_t)1 << 30;

// 0 = unknown, 1 = sm_103, 2 = other.  One slot per device ordinal.
std::atomic<int> g_device_ok[64];

lowbit_status check_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LOWBIT_ECUDA;
    if (dev < 0 || dev >= 64) return LOWBIT_EUNSUPPORTED;
    int state = g_device_ok[dev].load(std::memory_order_relaxed);
    if (state == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return LOWBIT_ECUDA;
        state = (major == 10 && minor == 3) ? 1 : 2;
        g_device_ok[dev].store(state, std::memory_order_relaxed);
    }
    return state == 1 ? LOWBIT_OK : LOWBIT_EUNSUPPORTED;
}

lowbit_status from_cuda(cudaError_t e) { return e == cudaSuccess ? LOWBIT_OK : LOWBIT_ECUDA; }

lowbit_status check_pack_args(const void *in, const void *out, int64_t N, int64_t K, int bits,
                              const void *code_buf) {
    if (!bits_ok(bits) || N < 0 || K < 0 || N > kMaxDim || K > kMaxDim || K % 8 != 0)
        return LOWBIT_EINVAL;
    if (N == 0 || K == 0) return LOWBIT_OK;
    if (in == nullptr || out == nullptr || !aligned(code_buf, 8)) return LOWBIT_EINVAL;
    return LOWBIT_OK;
}

lowbit_status check_linear_args(const uint16_t *x, const uint8_t *w, const uint16_t *s,
                                const uint16_t *z, const uint16_t *bias, const uint16_t *y,
                                int64_t M, int64_t K, int64_t N, int bits, int group) {
    if (!bits_ok(bits) || !group_ok(group)) return LOWBIT_EINVAL;
    if (M < 0 || N < 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return LOWBIT_EINVAL;
    if (K % group != 0) return LOWBIT_EINVAL;
    if (M == 0 || N == 0) return LOWBIT_OK;
    if (!x || !w || !s || !z || !y) return LOWBIT_EINVAL;
    if (!aligned(x, 16) || !aligned(w, 16) || !aligned(s, 2) || !aligned(z, 2) || !aligned(y, 2))
        return LOWBIT_EINVAL;
    if (bias != nullptr && !aligned(bias, 2)) return LOWBIT_EINVAL;
    return LOWBIT_OK;
}

// Crossover between the decode kernels and the batched tensor-core kernel
// (qmm), measured on GB300 in-stream at b = 4 for the Llama-3.1-8B shapes and
// the 3B gate+up and down, g = 32 / 64 / 128, M = 2..16.  The tensor-core
// decode kernel reads the weights once per launch of up to 2 (g = 32), 4
// (g = 64) or 8 (g >= 128) rows of x, so its time grows with the launches
// ("passes"); qmm's is nearly flat in M but grows as g shrinks (a K step of
// 128 codes has 128 / g groups to rescale): gate+up takes 47 / 78 / 141 us at
// g = 128 / 64 / 32.  The decode path wins up to 128 / g passes (M <= 8 for
// g <= 128): e.g. g = 32 gate+up at M = 4: 30 against 141 us; g = 64 o at
// M = 8: 11.4 against 15.0 us.  For N >= 24576 (gate+up: qmm runs 232 row
// tiles, a second wave on 80 of the 152 SMs) twice as many passes still win
// (g = 128 at M = 12 / 16: 37.6 / 44.4 against 46.9 / 47.1 us).  With
// K > 8192 the decode kernel splits K over clusters of three or more CTAs and
// loses beyond 4 / 6 / 8 rows at g = 128 / 64 / 32 (down at g = 128, M = 5:
// 26.4 against 24.1 us; g = 64, M = 8: 35.8 against 32.2 us).  Where the
// decode kernel does not take the shape, the CUDA-core kernel reads the
// weights once per two rows of x and wins up to M = 2, or up to M = 6 for
// layers of N >= 9424 outputs.
constexpr int64_t kQmvMaxM = 2;
constexpr int64_t kQmvMaxMWide = 6;
constexpr int64_t kWideN = 9424;          // 76 row tiles of 124: half the SMs
constexpr int64_t kClusterK = 8192;       // above: the decode kernel splits K over >= 3 CTAs
constexpr int64_t kTwoWaveN = 24576;      // qmm needs more than one wave of row tiles at M <= 128

// Decode passes that still beat qmm, and rows of x beyond which a K split over
// clusters loses.  (Group 256 keeps one pass: its qmm rescales once per two K
// steps, and its two-pass crossover was not measured.)
int64_t decode_max_passes(int group, int64_t N) {
    const int64_t p = group >= 128 ? 1 : 128 / group;
    return (N >= kTwoWaveN && group <= 128) ? 2 * p : p;
}
int64_t cluster_max_rows(int group) { return group >= 128 ? 4 : (group == 64 ? 6 : 8); }

}  // namespace

extern "C" {

const char *lowbit_status_string(lowbit_status status) {
    switch (status) {
        case LOWBIT_OK: return "ok";
        case LOWBIT_EINVAL: return "invalid argument";
        case LOWBIT_EUNSUPPORTED: return "unsupported device (needs sm_103 / GB300)";
        case LOWBIT_ECUDA: return "CUDA error";
        default: return "unknown status";
    }
}

size_t lowbit_packed_bytes(int64_t N, int64_t K, int bits) {
    // Range first, so that K * bits cannot overflow.
    if (!bits_ok(bits) || N < 0 || K < 0 || N > kMaxDim || K > kMaxDim) return 0;
    if ((K * bits) % 8 != 0) return 0;
    return (size_t)(N * (K * bits / 8));
}

lowbit_status lowbit_pack_weights(const uint8_t *codes, uint8_t *packed, int64_t N, int64_t K,
                                  int bits, lowbit_stream_t stream) {
    lowbit_status st = check_pack_args(codes, packed, N, K, bits, codes);
    if (st != LOWBIT_OK || N == 0 || K == 0) return st;
    if ((st = check_device()) != LOWBIT_OK) return st;
    return from_cuda(lowbit::launch_pack(codes, packed, N, K, bits, (cudaStream_t)stream));
}

lowbit_status lowbit_unpack_weights(const uint8_t *packed, uint8_t *codes, int64_t N, int64_t K,
                                    int bits, lowbit_stream_t stream) {
    lowbit_status st = check_pack_args(packed, codes, N, K, bits, codes);
    if (st != LOWBIT_OK || N == 0 || K == 0) return st;
    if ((st = check_device()) != LOWBIT_OK) return st;
    return from_cuda(lowbit::launch_unpack(packed, codes, N, K, bits, (cudaStream_t)stream));
}

lowbit_status lowbit_quantize_weights(const void *w, lowbit_dtype dtype, uint8_t *packed,
                                      uint16_t *scales, uint16_t *zeros, int64_t N, int64_t K,
                                      int bits, int group, lowbit_stream_t stream) {
    if (!bits_ok(bits) || !group_ok(group) || N < 0 || K <= 0 || N > kMaxDim || K > kMaxDim ||
        K % group != 0)
        return LOWBIT_EINVAL;
    if (dtype != LOWBIT_DTYPE_F32 && dtype != LOWBIT_DTYPE_BF16 && dtype != LOWBIT_DTYPE_F16)
        return LOWBIT_EINVAL;
    if (N == 0) return LOWBIT_OK;
    if (!w || !packed || !scales || !zeros) return LOWBIT_EINVAL;
    if (!aligned(w, 16) || !aligned(scales, 2) || !aligned(zeros, 2))
        return LOWBIT_EINVAL;
    lowbit_status st = check_device();
    if (st != LOWBIT_OK) return st;
    return from_cuda(lowbit::launch_quantize(w, (int)dtype, packed, scales, zeros, N, K, bits,
                                             group, (cudaStream_t)stream));
}

lowbit_path lowbit_select_path(int64_t M, int64_t K, int64_t N, int bits, int group) {
    if (!bits_ok(bits) || !group_ok(group) || M < 0 || N < 0 || K <= 0 || K % group != 0 ||
        M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return LOWBIT_PATH_AUTO;
    // qmm needs K % 128 == 0; other shapes stay on the decode kernels.
    if (K % 128 != 0) return LOWBIT_PATH_QMV;
    if (lowbit::qmv_mma_shape_ok(K, group)) {
        const int64_t rows = lowbit::qmv_mma_rows(group);
        const int64_t passes = (M + rows - 1) / rows;
        return (passes <= decode_max_passes(group, N) && !(K > kClusterK && M > cluster_max_rows(group)))
                   ? LOWBIT_PATH_QMV : LOWBIT_PATH_QMM;
    }
    return (M <= kQmvMaxM || (M <= kQmvMaxMWide && N >= kWideN)) ? LOWBIT_PATH_QMV : LOWBIT_PATH_QMM;
}

lowbit_status lowbit_linear_ex(const uint16_t *x, const uint8_t *packed_w, const uint16_t *scales,
                               const uint16_t *zeros, const uint16_t *bias, uint16_t *y,
                               int64_t M, int64_t K, int64_t N, int bits, int group,
                               lowbit_path path, lowbit_stream_t stream) {
    if (path != LOWBIT_PATH_AUTO && path != LOWBIT_PATH_QMV && path != LOWBIT_PATH_QMM)
        return LOWBIT_EINVAL;
    lowbit_status st = check_linear_args(x, packed_w, scales, zeros, bias, y, M, K, N, bits, group);
    if (st != LOWBIT_OK || M == 0 || N == 0) return st;
    if ((st = check_device()) != LOWBIT_OK) return st;
    if (path == LOWBIT_PATH_AUTO) path = lowbit_select_path(M, K, N, bits, group);
    cudaStream_t s = (cudaStream_t)stream;
    if (path == LOWBIT_PATH_QMV)
        return from_cuda(lowbit::launch_qmv(x, packed_w, scales, zeros, bias, y, M, K, N, bits, group, s));
    if (!lowbit::qmm_supported(K, x, packed_w)) return LOWBIT_EUNSUPPORTED;
    return from_cuda(lowbit::launch_qmm(x, packed_w, scales, zeros, bias, y, M, K, N, bits, group, s));
}

lowbit_status lowbit_linear(const uint16_t *x, const uint8_t *packed_w, const uint16_t *scales,
                            const uint16_t *zeros, const uint16_t *bias, uint16_t *y, int64_t M,
                            int64_t K, int64_t N, int bits, int group, lowbit_stream_t stream) {
    return lowbit_linear_ex(x, packed_w, scales, zeros, bias, y, M, K, N, bits, group,
                            LOWBIT_PATH_AUTO, stream);
}

lowbit_status lowbit_linear_swiglu(const uint16_t *x, const uint8_t *packed_w, const uint16_t *scales,
                                   const uint16_t *zeros, const uint16_t *bias, uint16_t *y,
                                   int64_t M, int64_t K, int64_t F, int bits, int group,
                                   lowbit_stream_t stream) {
    if (F < 0 || F > kMaxDim / 2) return LOWBIT_EINVAL;
    lowbit_status st = check_linear_args(x, packed_w, scales, zeros, bias, y, M, K, 2 * F, bits, group);
    if (st != LOWBIT_OK || M == 0 || F == 0) return st;
    if ((st = check_device()) != LOWBIT_OK) return st;
    return from_cuda(lowbit::launch_qmv_gated(x, packed_w, scales, zeros, bias, y, M, K, F, bits, group,
                                              (cudaStream_t)stream));
}

lowbit_status lowbit_wait_timeouts(uint32_t *count, int reset) {
    if (count == nullptr) return LOWBIT_EINVAL;
    lowbit_status st = check_device();
    if (st != LOWBIT_OK) return st;
    if (cudaDeviceSynchronize() != cudaSuccess) return LOWBIT_ECUDA;
    *count = lowbit::qmv_timeouts(reset != 0) + lowbit::mma_timeouts(reset != 0) + lowbit::qmm_timeouts(reset != 0) +
             selftest_timeouts(reset != 0);
    return cudaGetLastError() == cudaSuccess ? LOWBIT_OK : LOWBIT_ECUDA;
}

lowbit_status lowbit_selftest_wait_timeout(uint32_t *gave_up, lowbit_stream_t stream) {
    if (gave_up == nullptr || !aligned(gave_up, 4)) return LOWBIT_EINVAL;
    lowbit_status st = check_device();
    if (st != LOWBIT_OK) return st;
    wait_selftest_kernel<<<1, 1, 0, (cudaStream_t)stream>>>(gave_up);
    return from_cuda(cudaGetLastError());
}

}  // extern "C"
