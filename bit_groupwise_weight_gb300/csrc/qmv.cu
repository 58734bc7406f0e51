// qmv.cu -- quantised matrix-vector product for decode (small M), on CUDA
// cores with fp32 accumulation.
//
// Method: ao PR #2167 "metal lowbit kernels: qmv_fast optimization" (Summary,
// bullets 1-3) describes a matrix-vector kernel over contiguous b-bit codes
// with N x num_groups scales and zeros; torchchat PR #1415 fixes b = 1..7 and
// g = 32..256.  Per output y[m,n] = sum_k x[m,k] (s q + z) + bias, evaluated per
// 32-code block (one block never straddles a group since g >= 32) as
//     s * (sum_j x_j q_j) + z * (sum_j x_j).
//
// Mapping: a CTA of 128 threads owns RT output rows; thread t walks the
// 32-code blocks t, t+128, ... of K.  For each block it reads the block's
// x values once (bf16 -> fp32, shared by all RT rows) and the b words of each
// row, unpacks the 32 codes with compile-time shifts / funnel shifts and
// accumulates in fp32.  The 128 partial sums per (row, m) are reduced with
// warp shuffles and a small shared-memory step; thread (r, m) adds the bias
// and rounds once to bf16.
#include "common.cuh"

namespace lowbit {
namespace {

constexpr int kQmvThreads = 128;

template <int BITS, int MT, int RT>
__global__ void __launch_bounds__(kQmvThreads)
qmv_kernel(const uint16_t *__restrict__ x, const uint8_t *__restrict__ w,
           const uint16_t *__restrict__ scales, const uint16_t *__restrict__ zeros,
           const uint16_t *__restrict__ bias, uint16_t *__restrict__ y,
           int M, int K, int N, int log2g) {
    const int KB = K >> 5;                       // 32-code blocks per row
    const int G = K >> log2g;                    // groups per row
    const int64_t rb = (int64_t)KB * 4 * BITS;   // packed bytes per row
    const int n0 = blockIdx.x * RT;

    float acc[RT][MT];
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[r][m] = 0.f;

    for (int kb = threadIdx.x; kb < KB; kb += kQmvThreads) {
        // Weights of all RT rows first, so their loads are in flight together.
        uint32_t wv[RT][BITS];
        float sv[RT], zv[RT];
        const int gi = (kb << 5) >> log2g;
#pragma unroll
        for (int r = 0; r < RT; ++r) {
            const int n = min(n0 + r, N - 1);    // clamp: rows past N are computed, not stored
            load_block<BITS>(w + (int64_t)n * rb + (int64_t)kb * 4 * BITS, wv[r]);
            sv[r] = half_bits_to_float(__ldg(scales + (int64_t)n * G + gi));
            zv[r] = half_bits_to_float(__ldg(zeros + (int64_t)n * G + gi));
        }
        // x block: MT rows x 32 values, fp32, plus their sums.
        float xv[MT][32];
        float xs[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            xs[m] = 0.f;
            if (m < M) {
                const uint4 *xp = reinterpret_cast<const uint4 *>(x + (int64_t)m * K + (kb << 5));
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 v = __ldg(xp + q);
                    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        xv[m][8 * q + 2 * i] = bf16_lo(u[i]);
                        xv[m][8 * q + 2 * i + 1] = bf16_hi(u[i]);
                    }
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) xv[m][j] = 0.f;
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) xs[m] += xv[m][j];
        }
#pragma unroll
        for (int r = 0; r < RT; ++r) {
            float d[MT];
#pragma unroll
            for (int m = 0; m < MT; ++m) d[m] = 0.f;
            [&]<int... J>(std::integer_sequence<int, J...>) {
                ((void)[&] {
                    const float q = code_to_float(block_code<BITS, J>(wv[r]));
#pragma unroll
                    for (int m = 0; m < MT; ++m) d[m] = fmaf(xv[m][J], q, d[m]);
                }(), ...);
            }(std::make_integer_sequence<int, 32>{});
#pragma unroll
            for (int m = 0; m < MT; ++m)
                acc[r][m] = fmaf(sv[r], d[m], fmaf(zv[r], xs[m], acc[r][m]));
        }
    }

    // Reduce the 128 partials of every (row, m).
    __shared__ float red[kQmvThreads / 32][RT * MT];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int r = 0; r < RT; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            float v = acc[r][m];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0) red[warp][r * MT + m] = v;
        }
    __syncthreads();
    if (threadIdx.x < RT * MT) {
        const int r = threadIdx.x / MT, m = threadIdx.x % MT;
        const int n = n0 + r;
        if (n < N && m < M) {
            float v = 0.f;
#pragma unroll
            for (int i = 0; i < kQmvThreads / 32; ++i) v += red[i][threadIdx.x];
            if (bias != nullptr) v += half_bits_to_float(bias[n]);
            y[(int64_t)m * N + n] = float_to_bf16_bits(v);
        }
    }
}

template <int BITS, int MT>
cudaError_t launch_mt(const uint16_t *x, const uint8_t *w, const uint16_t *s, const uint16_t *z,
                      const uint16_t *bias, uint16_t *y, int M, int K, int N, int log2g,
                      cudaStream_t stream) {
    constexpr int RT = 4;
    const int grid = (N + RT - 1) / RT;
    qmv_kernel<BITS, MT, RT><<<grid, kQmvThreads, 0, stream>>>(x, w, s, z, bias, y, M, K, N, log2g);
    return cudaGetLastError();
}

template <int BITS>
cudaError_t launch_bits(const uint16_t *x, const uint8_t *w, const uint16_t *s, const uint16_t *z,
                        const uint16_t *bias, uint16_t *y, int64_t M, int K, int N, int log2g,
                        cudaStream_t stream) {
    // Up to 4 rows of x per launch; larger M is processed in chunks of 4.
    for (int64_t m0 = 0; m0 < M; m0 += 4) {
        const int mc = (int)((M - m0) < 4 ? (M - m0) : 4);
        const uint16_t *xc = x + m0 * K;
        uint16_t *yc = y + m0 * N;
        cudaError_t e;
        if (mc == 1) e = launch_mt<BITS, 1>(xc, w, s, z, bias, yc, mc, K, N, log2g, stream);
        else if (mc == 2) e = launch_mt<BITS, 2>(xc, w, s, z, bias, yc, mc, K, N, log2g, stream);
        else e = launch_mt<BITS, 4>(xc, w, s, z, bias, yc, mc, K, N, log2g, stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_qmv(const uint16_t *x, const uint8_t *w, const uint16_t *scales,
                       const uint16_t *zeros, const uint16_t *bias, uint16_t *y, int64_t M,
                       int64_t K, int64_t N, int bits, int group, cudaStream_t stream) {
    const int log2g = __builtin_ctz((unsigned)group);
    const int k = (int)K, n = (int)N;
    switch (bits) {
        case 1: return launch_bits<1>(x, w, scales, zeros, bias, y, M, k, n, log2g, stream);
        case 2: return launch_bits<2>(x, w, scales, zeros, bias, y, M, k, n, log2g, stream);
        case 3: return launch_bits<3>(x, w, scales, zeros, bias, y, M, k, n, log2g, stream);
        case 4: return launch_bits<4>(x, w, scales, zeros, bias, y, M, k, n, log2g, stream);
        case 5: return launch_bits<5>(x, w, scales, zeros, bias, y, M, k, n, log2g, stream);
        case 6: return launch_bits<6>(x, w, scales, zeros, bias, y, M, k, n, log2g, stream);
        case 7: return launch_bits<7>(x, w, scales, zeros, bias, y, M, k, n, log2g, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace lowbit
