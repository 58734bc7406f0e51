// pack.cu -- packing and unpacking kernels for the contiguous b-bit layout
// (ao PR #2167 "metal lowbit kernels: qmv_fast optimization", Summary,
// bullet 2: codes stored contiguously, continuing into the next byte when the
// current one is full; bit order read LSB-first).
//
// Eight b-bit codes fill exactly b bytes, so each thread owns one "octet": it
// reads 8 code bytes (one 8-byte load), assembles the 8*b-bit little-endian
// value in a 64-bit register and writes its b bytes.  Rows need no special
// handling: a row of K codes (K % 8 == 0) is K/8 whole octets.
#include "common.cuh"

namespace lowbit {
namespace {

template <int BITS>
__global__ void __launch_bounds__(256) pack_kernel(const uint8_t *__restrict__ codes,
                                                   uint8_t *__restrict__ packed, int64_t octets) {
    constexpr uint64_t mask = (1u << BITS) - 1u;
    for (int64_t o = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; o < octets;
         o += (int64_t)gridDim.x * blockDim.x) {
        const uint2 c = *reinterpret_cast<const uint2 *>(codes + 8 * o);
        uint64_t v = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            v |= ((uint64_t)((c.x >> (8 * j)) & 0xFFu) & mask) << (BITS * j);
            v |= ((uint64_t)((c.y >> (8 * j)) & 0xFFu) & mask) << (BITS * (j + 4));
        }
        uint8_t *dst = packed + BITS * o;
#pragma unroll
        for (int i = 0; i < BITS; ++i) dst[i] = (uint8_t)(v >> (8 * i));
    }
}

template <int BITS>
__global__ void __launch_bounds__(256) unpack_kernel(const uint8_t *__restrict__ packed,
                                                     uint8_t *__restrict__ codes, int64_t octets) {
    constexpr uint64_t mask = (1u << BITS) - 1u;
    for (int64_t o = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; o < octets;
         o += (int64_t)gridDim.x * blockDim.x) {
        const uint8_t *src = packed + BITS * o;
        uint64_t v = 0;
#pragma unroll
        for (int i = 0; i < BITS; ++i) v |= (uint64_t)src[i] << (8 * i);
        uint2 c = make_uint2(0u, 0u);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            c.x |= (uint32_t)((v >> (BITS * j)) & mask) << (8 * j);
            c.y |= (uint32_t)((v >> (BITS * (j + 4))) & mask) << (8 * j);
        }
        *reinterpret_cast<uint2 *>(codes + 8 * o) = c;
    }
}

int grid_for(int64_t octets) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int64_t blocks = (octets + 255) / 256;
    int64_t cap = (int64_t)(sms > 0 ? sms : 148) * 8;
    return (int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

}  // namespace

cudaError_t launch_pack(const uint8_t *codes, uint8_t *packed, int64_t N, int64_t K, int bits,
                        cudaStream_t stream) {
    const int64_t octets = N * (K / 8);
    const int grid = grid_for(octets);
    switch (bits) {
        case 1: pack_kernel<1><<<grid, 256, 0, stream>>>(codes, packed, octets); break;
        case 2: pack_kernel<2><<<grid, 256, 0, stream>>>(codes, packed, octets); break;
        case 3: pack_kernel<3><<<grid, 256, 0, stream>>>(codes, packed, octets); break;
        case 4: pack_kernel<4><<<grid, 256, 0, stream>>>(codes, packed, octets); break;
        case 5: pack_kernel<5><<<grid, 256, 0, stream>>>(codes, packed, octets); break;
        case 6: pack_kernel<6><<<grid, 256, 0, stream>>>(codes, packed, octets); break;
        case 7: pack_kernel<7><<<grid, 256, 0, stream>>>(codes, packed, octets); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_unpack(const uint8_t *packed, uint8_t *codes, int64_t N, int64_t K, int bits,
                          cudaStream_t stream) {
    const int64_t octets = N * (K / 8);
    const int grid = grid_for(octets);
    switch (bits) {
        case 1: unpack_kernel<1><<<grid, 256, 0, stream>>>(packed, codes, octets); break;
        case 2: unpack_kernel<2><<<grid, 256, 0, stream>>>(packed, codes, octets); break;
        case 3: unpack_kernel<3><<<grid, 256, 0, stream>>>(packed, codes, octets); break;
        case 4: unpack_kernel<4><<<grid, 256, 0, stream>>>(packed, codes, octets); break;
        case 5: unpack_kernel<5><<<grid, 256, 0, stream>>>(packed, codes, octets); break;
        case 6: unpack_kernel<6><<<grid, 256, 0, stream>>>(packed, codes, octets); break;
        case 7: unpack_kernel<7><<<grid, 256, 0, stream>>>(packed, codes, octets); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace lowbit
