// pack.cu -- packing and unpacking kernels for the contiguous b-bit layout
// (ao PR #2167 "metal lowbit kernels: qmv_fast optimization", Summary,
// bullet 2: codes stored contiguously, continuing into the next byte when the
// current one is full; bit order read LSB-first).
//
// Eight b-bit codes fill exactly b bytes (an "octet"): a thread reads 8 code
// bytes (one 8-byte load) and assembles the 8*b-bit little-endian value in a
// 64-bit register.  The packing kernel gives each thread U = 16 / gcd(b, 16)
// consecutive octets, whose U*b bytes are a multiple of 16, and writes them
// with 16-byte stores (when the packed matrix is 16-byte aligned; the last
// few octets, and unaligned outputs, take the byte-wise path).  Rows need no
// special handling: a row of K codes (K % 8 == 0) is K/8 whole octets.
#include "common.cuh"

namespace lowbit {
namespace {

// The 8*b-bit value of one octet: code j at bits [b*j, b*j + b).
template <int BITS>
__device__ __forceinline__ uint64_t octet_value(uint2 c) {
    constexpr uint64_t mask = (1u << BITS) - 1u;
    uint64_t v = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        v |= ((uint64_t)((c.x >> (8 * j)) & 0xFFu) & mask) << (BITS * j);
        v |= ((uint64_t)((c.y >> (8 * j)) & 0xFFu) & mask) << (BITS * (j + 4));
    }
    return v;
}

template <int BITS>
constexpr int octets_per_thread() { return BITS % 2 ? 16 : (BITS % 4 ? 8 : 4); }   // 16 / gcd(b, 16)

// Octets [first, octets), one per thread, written byte by byte.
template <int BITS>
__device__ __forceinline__ void pack_bytewise(const uint8_t *__restrict__ codes, uint8_t *__restrict__ packed,
                                              int64_t first, int64_t octets) {
    for (int64_t o = first + blockIdx.x * (int64_t)blockDim.x + threadIdx.x; o < octets;
         o += (int64_t)gridDim.x * blockDim.x) {
        const uint64_t v = octet_value<BITS>(*reinterpret_cast<const uint2 *>(codes + 8 * o));
        uint8_t *dst = packed + BITS * o;
#pragma unroll
        for (int i = 0; i < BITS; ++i) dst[i] = (uint8_t)(v >> (8 * i));
    }
}

template <int BITS, bool WIDE>
__global__ void __launch_bounds__(256) pack_kernel(const uint8_t *__restrict__ codes,
                                                   uint8_t *__restrict__ packed, int64_t octets) {
    if constexpr (!WIDE) {
        pack_bytewise<BITS>(codes, packed, 0, octets);
    } else {
        constexpr int U = octets_per_thread<BITS>();
        constexpr int WORDS = U * BITS / 4;                  // a multiple of 4: whole 16-byte stores
        const int64_t runs = octets / U;
        for (int64_t r = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; r < runs;
             r += (int64_t)gridDim.x * blockDim.x) {
            uint32_t out[WORDS];
#pragma unroll
            for (int i = 0; i < WORDS; ++i) out[i] = 0u;
#pragma unroll
            for (int j = 0; j < U; ++j) {
                const uint64_t v = octet_value<BITS>(*reinterpret_cast<const uint2 *>(codes + 8 * (r * U + j)));
                const int bit = 8 * BITS * j;                    // a multiple of 8
                const int w0 = bit / 32, sh = bit % 32;
                out[w0] |= (uint32_t)(v << sh);
                if (w0 + 1 < WORDS) out[w0 + 1] |= (uint32_t)((v << sh) >> 32);
                if (sh != 0 && w0 + 2 < WORDS) out[w0 + 2] |= (uint32_t)(v >> (64 - sh));
            }
            uint4 *dst = reinterpret_cast<uint4 *>(packed + (int64_t)BITS * U * r);
#pragma unroll
            for (int i = 0; i < WORDS / 4; ++i)
                dst[i] = make_uint4(out[4 * i], out[4 * i + 1], out[4 * i + 2], out[4 * i + 3]);
        }
        pack_bytewise<BITS>(codes, packed, runs * U, octets);
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
    const bool wide = (reinterpret_cast<uintptr_t>(packed) & 15u) == 0;
#define LOWBIT_PACK_CASE(B)                                                                        \
    case B:                                                                                        \
        if (wide) pack_kernel<B, true><<<grid, 256, 0, stream>>>(codes, packed, octets);           \
        else pack_kernel<B, false><<<grid, 256, 0, stream>>>(codes, packed, octets);               \
        break;
    switch (bits) {
        LOWBIT_PACK_CASE(1) LOWBIT_PACK_CASE(2) LOWBIT_PACK_CASE(3) LOWBIT_PACK_CASE(4)
        LOWBIT_PACK_CASE(5) LOWBIT_PACK_CASE(6) LOWBIT_PACK_CASE(7)
        default: return cudaErrorInvalidValue;
    }
#undef LOWBIT_PACK_CASE
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
