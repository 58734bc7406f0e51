// common.cuh -- device helpers shared by the liblowbit kernels (sm_103a).
#pragma once

#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "lowbit.h"

namespace lowbit {

// Packed layout: code k of a row sits at bits [k*b, k*b+b) of the row's
// little-endian bit stream (ao PR #2167, Summary, bullet 2, read LSB-first).
// 32 consecutive codes therefore fill exactly b 32-bit little-endian words, and
// a row of K codes (K % 32 == 0) is K/32 such "blocks" of 4*b bytes.
constexpr int kBlockCodes = 32;

// Code j (0..31) of a 32-code block held in BITS little-endian words.  All
// indices are compile-time constants, so a code that straddles two words
// becomes one funnel shift and a code inside a word one shift + mask.
template <int BITS, int J>
__device__ __forceinline__ uint32_t block_code(const uint32_t (&w)[BITS]) {
    constexpr int bit = J * BITS;
    constexpr int wi = bit / 32;
    constexpr int off = bit % 32;
    constexpr uint32_t mask = (1u << BITS) - 1u;
    if constexpr (off + BITS <= 32) {
        return (w[wi] >> off) & mask;
    } else {
        return __funnelshift_r(w[wi], w[wi + 1], off) & mask;
    }
}

// Exact small-integer -> fp32: the bit pattern 0x4B000000 | q is 2^23 + q for
// q < 2^23, so one OR and one subtraction replace an int->float conversion.
__device__ __forceinline__ float code_to_float(uint32_t q) {
    return __uint_as_float(0x4B000000u | q) - 8388608.0f;
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ float half_bits_to_float(uint16_t h) {
    return __half2float(__ushort_as_half(h));
}

__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// The gated activation of a gate/up projection pair: silu(a) * u, with
// silu(a) = a / (1 + e^-a), in fp32 (expf from the CUDA math library).
__device__ __forceinline__ float silu_mul(float a, float u) { return a / (1.0f + expf(-a)) * u; }

// 128-bit streaming load that does not allocate in L1 (weights are read once).
__device__ __forceinline__ uint4 ld_stream_v4(const void *p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ uint2 ld_stream_v2(const void *p) {
    uint2 v;
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
                 : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ld_stream_u32(const void *p) {
    uint32_t v;
    asm("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// Load the BITS words of one 32-code block starting at a 4*BITS-byte aligned
// address, with the widest loads that alignment allows.
template <int BITS>
__device__ __forceinline__ void load_block(const uint8_t *p, uint32_t (&w)[BITS]) {
    if constexpr (BITS == 4) {
        uint4 v = ld_stream_v4(p);
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else if constexpr (BITS == 2 || BITS == 6) {
#pragma unroll
        for (int i = 0; i < BITS / 2; ++i) {
            uint2 v = ld_stream_v2(p + 8 * i);
            w[2 * i] = v.x; w[2 * i + 1] = v.y;
        }
    } else {
#pragma unroll
        for (int i = 0; i < BITS; ++i) w[i] = ld_stream_u32(p + 4 * i);
    }
}

// Launch `kernel` with programmatic stream serialisation: the kernel may begin
// while the previous kernel in the stream finishes, and must call
// griddepcontrol.wait before touching global memory (every kernel launched
// this way here does so first thing).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace lowbit

// Launchers implemented in the .cu files (host side, no argument checks: the
// C ABI in api.cu validates everything first).
namespace lowbit {
cudaError_t launch_pack(const uint8_t *codes, uint8_t *packed, int64_t N, int64_t K, int bits,
                        cudaStream_t stream);
cudaError_t launch_unpack(const uint8_t *packed, uint8_t *codes, int64_t N, int64_t K, int bits,
                          cudaStream_t stream);
cudaError_t launch_qmv(const uint16_t *x, const uint8_t *w, const uint16_t *scales,
                       const uint16_t *zeros, const uint16_t *bias, uint16_t *y, int64_t M,
                       int64_t K, int64_t N, int bits, int group, cudaStream_t stream);
// Gated form: packed rows [0, F) are the gate projection and [F, 2F) the up
// projection; y [M, F] = silu(gate) * up (bias, if any, has 2F entries).
cudaError_t launch_qmv_gated(const uint16_t *x, const uint8_t *w, const uint16_t *scales,
                             const uint16_t *zeros, const uint16_t *bias, uint16_t *y, int64_t M,
                             int64_t K, int64_t F, int bits, int group, cudaStream_t stream);
cudaError_t launch_quantize(const void *w, int dtype, uint8_t *packed, uint16_t *scales,
                            uint16_t *zeros, int64_t N, int64_t K, int bits, int group,
                            cudaStream_t stream);
// The decode kernel on the warp-level tensor cores (qmv_mma.cuh), any M in
// launches of up to 8 rows of x; F > 0: the gated form (N = 2F rows).  Returns
// cudaErrorNotSupported, having launched nothing, for shapes it does not take
// (K not a multiple of 256, K > 32768, F not a multiple of 16, x or the
// packed weights not 16-byte aligned).
cudaError_t launch_qmv_mma(const uint16_t *x, const uint8_t *w, const uint16_t *s, const uint16_t *z,
                           const uint16_t *bias, uint16_t *y, int64_t M, int64_t K, int64_t N, int bits, int group,
                           int64_t F, cudaStream_t stream);
// Per-device host state (device.cu), keyed by device ordinal and kernel; a
// failed query returns 0 (or its error) and is not cached.
int current_device();                                                   // -1 on error
int device_sm_count(int dev);
cudaError_t raise_smem_limit(const void *fn, int dev, int bytes);       // once per (device, kernel, bytes)
int blocks_per_sm(const void *fn, int dev, int threads, uint32_t smem);
int clusters_at_once(const void *fn, int dev, int ks, int threads, uint32_t smem);
// A TMA tiled tensor map (element strides 1, no interleave, L2 promotion 256 B,
// out-of-bounds elements read as zero): rank dims (innermost first), rank - 1
// byte strides, the box.  Cached by its arguments.  False when encoding fails.
bool encode_tiled(CUtensorMap *map, CUtensorMapDataType type, uint32_t rank, const void *base,
                  const uint64_t *dims, const uint64_t *strides, const uint32_t *box,
                  CUtensorMapSwizzle swizzle);
// True when the tensor-core decode kernel takes K and group (given 16-byte
// aligned x, weights, scales and zeros), and the rows of x it takes per launch.
bool qmv_mma_shape_ok(int64_t K, int group);
int qmv_mma_rows(int group);
// Bounded waits that gave up, per kernel file (device counters; reading syncs).
uint32_t mma_timeouts(bool reset);
uint32_t qmv_timeouts(bool reset);
uint32_t qmm_timeouts(bool reset);
// True when the tensor-core kernel handles this shape (K a multiple of 128,
// x and packed weights 16-byte aligned).
bool qmm_supported(int64_t K, const void *x, const void *w);
cudaError_t launch_qmm(const uint16_t *x, const uint8_t *w, const uint16_t *scales,
                       const uint16_t *zeros, const uint16_t *bias, uint16_t *y, int64_t M,
                       int64_t K, int64_t N, int bits, int group, cudaStream_t stream);
}  // namespace lowbit
