// qmv.cu -- quantised matrix-vector product for decode (small M), on CUDA
// cores with fp32 accumulation.  Two kernels:
//   qmv_stream_kernel  -- the decode kernel (M <= 2, K % 1024 == 0): persistent
//                         CTAs stream their rows through a TMA-bulk ring; for
//                         one-bit codes and one row of x it decodes by table
//                         lookup (lut_dot);
//   qmv_generic_kernel -- any shape the library accepts (ragged N, K % 32 == 0,
//                         any M in chunks of 4); used where the stream kernel's
//                         alignment conditions do not hold.
// Both also run the gated form (F > 0): rows [0, F) are a gate projection and
// rows [F, 2F) the matching up projection, and the output is silu(gate) * up.
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
#include <algorithm>
#include <atomic>
#include <numeric>

#include "common.cuh"
#include "ptx.cuh"

namespace lowbit {
namespace {

constexpr int kQmvThreads = 128;

template <int BITS, int MT, int RT>
__global__ void __launch_bounds__(kQmvThreads)
qmv_generic_kernel(const uint16_t *__restrict__ x, const uint8_t *__restrict__ w,
           const uint16_t *__restrict__ scales, const uint16_t *__restrict__ zeros,
           const uint16_t *__restrict__ bias, uint16_t *__restrict__ y,
           int M, int K, int N, int log2g, int F) {
    const int KB = K >> 5;                       // 32-code blocks per row
    const int G = K >> log2g;                    // groups per row
    const int64_t rb = (int64_t)KB * 4 * BITS;   // packed bytes per row
    // Plain: rows n0 .. n0+RT-1.  Gated (F > 0, N = 2F): slots r < RT/2 are the
    // gate rows f0 + r, slots r >= RT/2 the matching up rows F + f0 + r - RT/2.
    static_assert(RT % 2 == 0, "gated CTAs take row pairs");
    const int n0 = blockIdx.x * RT;
    const int f0 = blockIdx.x * (RT / 2);

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
            // Clamp: rows past the end are computed, not stored.
            const int n = F == 0 ? min(n0 + r, N - 1)
                                 : (r < RT / 2 ? 0 : F) + min(f0 + r % (RT / 2), F - 1);
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
    if (F == 0) {
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
    } else if (threadIdx.x < (RT / 2) * MT) {
        const int r = threadIdx.x / MT, m = threadIdx.x % MT;
        const int f = f0 + r;
        if (f < F && m < M) {
            float a = 0.f, u = 0.f;
#pragma unroll
            for (int i = 0; i < kQmvThreads / 32; ++i) {
                a += red[i][r * MT + m];
                u += red[i][(r + RT / 2) * MT + m];
            }
            if (bias != nullptr) {
                a += half_bits_to_float(bias[f]);
                u += half_bits_to_float(bias[F + f]);
            }
            y[(int64_t)m * F + f] = float_to_bf16_bits(silu_mul(a, u));
        }
    }
}

template <int BITS, int MT>
cudaError_t launch_generic_mt(const uint16_t *x, const uint8_t *w, const uint16_t *s,
                              const uint16_t *z, const uint16_t *bias, uint16_t *y, int M, int K,
                              int N, int log2g, int F, cudaStream_t stream) {
    constexpr int RT = 4;
    const int grid = F == 0 ? (N + RT - 1) / RT : (F + RT / 2 - 1) / (RT / 2);
    qmv_generic_kernel<BITS, MT, RT><<<grid, kQmvThreads, 0, stream>>>(x, w, s, z, bias, y, M, K, N,
                                                                      log2g, F);
    return cudaGetLastError();
}

template <int BITS>
cudaError_t launch_generic(const uint16_t *x, const uint8_t *w, const uint16_t *s,
                           const uint16_t *z, const uint16_t *bias, uint16_t *y, int64_t M, int K,
                           int N, int log2g, int F, cudaStream_t stream) {
    // Up to 4 rows of x per launch; larger M is processed in chunks of 4.
    const int64_t ystride = F == 0 ? N : F;
    for (int64_t m0 = 0; m0 < M; m0 += 4) {
        const int mc = (int)((M - m0) < 4 ? (M - m0) : 4);
        const uint16_t *xc = x + m0 * K;
        uint16_t *yc = y + m0 * ystride;
        cudaError_t e;
        if (mc == 1) e = launch_generic_mt<BITS, 1>(xc, w, s, z, bias, yc, mc, K, N, log2g, F, stream);
        else if (mc == 2) e = launch_generic_mt<BITS, 2>(xc, w, s, z, bias, yc, mc, K, N, log2g, F, stream);
        else e = launch_generic_mt<BITS, 4>(xc, w, s, z, bias, yc, mc, K, N, log2g, F, stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// ===========================================================================
// qmv_stream_kernel
//
// Work split.  Output rows are taken R at a time ("passes"); CTA c owns a
// contiguous, balanced run of passes, so the packed weights, scales and zeros
// it needs are three contiguous byte ranges.  A producer warp streams them, SP
// passes per stage, into a ring of shared-memory stages with one-dimensional
// TMA bulk copies (cp.async.bulk), each stage completing on an mbarrier.
//
// Consumers.  T = R*KB threads, KB = K/32 blocks of 32 codes per row: thread t
// always owns block kb = t % KB of row slot rr = t / KB, so its 32 x values
// (per row of x) stay in registers for the whole kernel.  Per pass a thread
// reads its block's b words from shared memory and forms
//     partial = s * (sum_j x_j q_j) + z * (sum_j x_j)
// (the group's scale and zero; a 32-code block never straddles a group).
//
// Code -> float.  Code j is placed by one funnel shift at mantissa bit p_j
// (lo <= p_j <= 23-b) of a shifted copy of the words, and one LOP3 ORs in the
// exponent of 2^(23-p_j): the float is exactly 2^(23-p_j) + q_j.  So
//     sum_j x_j q_j = sum_j x_j f_j - sum_j x_j 2^(23-p_j),
// where the second sum is a per-thread constant computed once.  The products
// run as packed fp32 FMAs (fma.rn.f32x2), two codes per instruction.  lo is
// chosen per bit width so that the constant part stays below about 2^8 times
// the largest code, which costs about 2^-16 relative accuracy per product.
//
// Reduction.  U passes are unrolled; their partials (U*M slots) go through the
// first levels of a transposing butterfly without branches, the rest of a
// batch of 32 slots through a carry chain (one pending value per level).  31
// shuffles per 32 slots leave lane l with the warp's sum for slot l; the KB/32
// warps of a row slot are then summed through shared memory by one thread per
// output, which adds the bias and rounds to bf16.
// ===========================================================================

constexpr int kMaxStages = 8;

__device__ unsigned int g_qmv_timeouts;

// Lowest mantissa bit a code may occupy, per bit width.
template <int BITS>
constexpr int window_lo() { return BITS <= 4 ? 11 : (BITS == 6 ? 9 : 8); }

template <int BITS>
struct Window {
    static constexpr int lo = window_lo<BITS>();
    static constexpr int per_copy = (23 - BITS - lo) / BITS + 1;
    static constexpr int copies = (32 + per_copy - 1) / per_copy;
    static constexpr int first(int c) { return c * per_copy; }
    static constexpr int pos(int j) { return lo + (j % per_copy) * BITS; }
};

// Shifted copy c of the block's words: its first code lands at bit `lo`.
template <int BITS, int C>
__device__ __forceinline__ uint32_t window_copy(const uint32_t (&w)[BITS]) {
    constexpr int lo = Window<BITS>::lo;
    constexpr int P0 = Window<BITS>::first(C) * BITS;
    constexpr int wi = P0 / 32;
    constexpr int o = P0 % 32;
    if constexpr (o >= lo) {
        const uint32_t hi = (wi + 1 < BITS) ? w[wi + 1 < BITS ? wi + 1 : 0] : 0u;
        return __funnelshift_r(w[wi], hi, o - lo);
    } else {
        const uint32_t lw = (wi > 0) ? w[wi > 0 ? wi - 1 : 0] : 0u;
        return __funnelshift_l(lw, w[wi], lo - o);
    }
}

// Code j as the exact float 2^(23-p) + q.
template <int BITS, int J>
__device__ __forceinline__ float window_code(const uint32_t (&cp)[Window<BITS>::copies]) {
    constexpr int c = J / Window<BITS>::per_copy;
    constexpr int p = Window<BITS>::pos(J);
    constexpr uint32_t mask = ((1u << BITS) - 1u) << p;
    constexpr uint32_t expo = (uint32_t)(127 + 23 - p) << 23;
    return __uint_as_float(ptx::and_or_imm<mask>(cp[c], expo));
}

template <int BITS>
__device__ __forceinline__ constexpr float window_const(int j) {
    return (float)(1u << (23 - Window<BITS>::pos(j)));
}

template <int M>
struct XRegs {
    float2 x[M][16];   // x[m][2i], x[m][2i+1] of this thread's block
    float cx[M];       // sum_j x_j 2^(23-p_j)
    float xs[M];       // sum_j x_j
};

// sum_j x_j q_j for each row of x.
template <int BITS, int M>
__device__ __forceinline__ void block_dot(const uint32_t (&w)[BITS], const XRegs<M> &xr,
                                          float (&d)[M]) {
    uint32_t cp[Window<BITS>::copies];
    [&]<int... C>(std::integer_sequence<int, C...>) {
        ((cp[C] = window_copy<BITS, C>(w)), ...);
    }(std::make_integer_sequence<int, Window<BITS>::copies>{});
    float2 acc[M][4];
#pragma unroll
    for (int m = 0; m < M; ++m)
#pragma unroll
        for (int a = 0; a < 4; ++a) acc[m][a] = make_float2(0.f, 0.f);
    [&]<int... I>(std::integer_sequence<int, I...>) {
        ((void)[&] {
            const float2 f = make_float2(window_code<BITS, 2 * I>(cp), window_code<BITS, 2 * I + 1>(cp));
#pragma unroll
            for (int m = 0; m < M; ++m) ptx::ffma2(acc[m][I % 4], f, xr.x[m][I], acc[m][I % 4]);
        }(), ...);
    }(std::make_integer_sequence<int, 16>{});
#pragma unroll
    for (int m = 0; m < M; ++m) {
        const float2 a = ptx::fadd2(ptx::fadd2(acc[m][0], acc[m][1]), ptx::fadd2(acc[m][2], acc[m][3]));
        d[m] = (a.x + a.y) - xr.cx[m];
    }
}

template <int BITS>
__device__ __forceinline__ void lds_block(const uint8_t *p, uint32_t (&w)[BITS]) {
    if constexpr (BITS == 4) {
        const uint4 v = *reinterpret_cast<const uint4 *>(p);
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else if constexpr (BITS == 2 || BITS == 6) {
#pragma unroll
        for (int i = 0; i < BITS / 2; ++i) {
            const uint2 v = *reinterpret_cast<const uint2 *>(p + 8 * i);
            w[2 * i] = v.x; w[2 * i + 1] = v.y;
        }
    } else {
#pragma unroll
        for (int i = 0; i < BITS; ++i) w[i] = reinterpret_cast<const uint32_t *>(p)[i];
    }
}

// Streaming transposing butterfly.  Slot i of a batch of 32 is combined with
// the pending partial sums at every level t whose bit is set in i, using
// shuffle distance 2^t: lanes with bit t clear keep the earlier half, lanes
// with it set the later half.  After slot 31, lane l holds the warp-wide sum of
// slot l.  Levels below L0 are done by static_butterfly on values already in
// registers; this carry chain does levels L0..4 (one pending value each).
template <int L0>
struct CarryReduce {
    float lv[5];
    // Feed the value of slot group `gs`.  Returns true when `val` is complete.
    __device__ __forceinline__ bool feed(float &val, int gs, int lane) {
        bool pending = true;   // val still has to be combined or parked
#pragma unroll
        for (int t = L0; t < 5; ++t) {
            if (pending) {
                if (((gs >> (t - L0)) & 1) == 0) {
                    lv[t] = val;
                    pending = false;
                } else {
                    const bool upper = ((lane >> t) & 1) != 0;
                    const float send = upper ? lv[t] : val;
                    const float keep = upper ? val : lv[t];
                    val = keep + __shfl_xor_sync(0xffffffffu, send, 1 << t);
                }
            }
        }
        return pending;
    }
};

template <int S0>
__device__ __forceinline__ float static_butterfly(float (&v)[S0], int lane) {
#pragma unroll
    for (int t = 0; (1 << t) < S0; ++t) {
        const bool upper = ((lane >> t) & 1) != 0;
#pragma unroll
        for (int i = 0; i < (S0 >> (t + 1)); ++i) {
            const float a = v[2 * i], b = v[2 * i + 1];
            const float send = upper ? a : b;
            const float keep = upper ? b : a;
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 1 << t);
        }
    }
    return v[0];
}

// Passes processed per unrolled group (stage sizes are multiples of it).
template <int BITS>
constexpr int stream_unroll() { return BITS <= 4 ? 8 : 4; }

template <int M>
constexpr int stream_max_consumers() { return M == 1 ? 512 : 256; }

struct StreamParams {
    const uint16_t *x;
    const uint8_t *w;
    const uint16_t *s;
    const uint16_t *z;
    const uint16_t *bias;
    uint16_t *y;
    int N, K, KB, G, log2g, R, T, SP, stages;
    int F;                            // gated: F outputs from rows [0, F) (gate) and [F, 2F) (up); 0: plain
    int chunk;                        // passes per split unit (keeps s/z copies 16-byte sized)
    int chunks, chunks_base, chunks_extra;   // split units in all; per CTA: base (+1 for the first extra)
    int total_passes;                 // ceil(N / R)
    uint32_t row_bytes;               // K*BITS/8
    uint32_t w_stage, sz_stage;       // bytes of a full stage: weights, and scales (= zeros)
    uint32_t stage_bytes;             // w_stage + 2*sz_stage
    uint32_t red_off, ring_off;       // shared-memory offsets
    uint32_t lut_off;                 // b = 1 lookup tables (table decode only)
};

// Table decode (b = 1, one row of x).  Each nibble of a block's word holds
// codes 4j .. 4j+3, so sum_k x_k q_k over the block is the sum over j of
// T_j[nibble j], where T_j[e] = sum of x_{4j+i} over the set bits i of e: 8
// shared-memory lookups and adds per 32 codes instead of a float per code.
// The tables depend only on x, so each CTA builds them once, laid out
// [j][e][kb] (kb fastest): the 32 lanes of a warp hold consecutive blocks kb
// and never share a bank.
__device__ __forceinline__ float lut_dot(uint32_t w, const float *tb, int KB) {
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float t = tb[(j * 16 + (int)((w >> (4 * j)) & 15u)) * KB];
        if (j & 1) s1 += t; else s0 += t;
    }
    return s0 + s1;
}

template <int BITS, int M, bool LUT = false>
__global__ void __launch_bounds__(stream_max_consumers<M>() + 32)
qmv_stream_kernel(const StreamParams p) {
    static_assert(!LUT || (BITS == 1 && M == 1), "table decode: one-bit codes, one row of x");
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int V = 32;              // (pass, m) slots per batch
    constexpr int P = V / M;           // passes per batch
    const int tid = threadIdx.x;
    const int T = p.T;
    const uint32_t sb = ptx::smem_u32(smem);
    const uint32_t full0 = sb, empty0 = sb + 8 * kMaxStages;
    const int S = p.stages;

    // This CTA's passes [pass0, pass0 + npass).
    ptx::pdl_launch_dependents();
    const int c = blockIdx.x;
    const int ch0 = c * p.chunks_base + min(c, p.chunks_extra);
    const int nch = p.chunks_base + (c < p.chunks_extra ? 1 : 0);
    const int pass0 = ch0 * p.chunk;
    const int npass = min(nch * p.chunk, p.total_passes - pass0);
    const int nstage = (npass + p.SP - 1) / p.SP;

    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            ptx::mbar_init(full0 + 8 * i, 1);
            ptx::mbar_init(empty0 + 8 * i, T / 32);
        }
        ptx::fence_mbar_init();
    }
    if (tid == T && nstage > 0) {
        // Ask L2 for the bytes of the first ring's worth of stages while the
        // previous kernel in the stream may still be running (a hint: L2 is
        // coherent, so data still being written is simply fetched again).
        const int pend = pass0 + min(S * p.SP, npass);
        // Plain: one run of rows.  Gated: the gate run and the matching up run.
        const int r0 = p.F == 0 ? pass0 * p.R : (pass0 >> 1) * p.R;
        const int r1 = p.F == 0 ? min(pend * p.R, p.N) : min(((pend + 1) >> 1) * p.R, p.F);
        const uint32_t rows = (uint32_t)(r1 - r0);
        for (int h = 0; h < (p.F == 0 ? 1 : 2); ++h) {
            const int row0 = h * p.F + r0;
            ptx::bulk_prefetch_l2(p.w + (int64_t)row0 * p.row_bytes, (rows * p.row_bytes) & ~15u);
            ptx::bulk_prefetch_l2(p.s + (int64_t)row0 * p.G, (rows * (uint32_t)p.G * 2u) & ~15u);
            ptx::bulk_prefetch_l2(p.z + (int64_t)row0 * p.G, (rows * (uint32_t)p.G * 2u) & ~15u);
        }
    }
    __syncthreads();
    ptx::pdl_wait();            // inputs may come from the previous kernel in the stream

    if (tid >= T) {
        // ---------------- producer warp: one elected lane issues the copies.
        if (tid == T) {
            const uint64_t pol = ptx::policy_evict_first();
            int issued = 0;
            for (int i = 0; i < nstage; ++i, ++issued) {
                const int st = i % S;
                if (i >= S && !ptx::mbar_wait(empty0 + 8 * st, ((i / S) - 1) & 1, &g_qmv_timeouts))
                    break;
                const uint32_t dst = sb + p.ring_off + st * p.stage_bytes;
                const uint32_t bar = full0 + 8 * st;
                if (p.F == 0) {
                    // The stage's passes are one contiguous run of rows.
                    const int row0 = (pass0 + i * p.SP) * p.R;
                    const int row1 = min((pass0 + min((i + 1) * p.SP, npass)) * p.R, p.N);
                    const uint32_t rows = (uint32_t)(row1 - row0);
                    const uint32_t wb = rows * p.row_bytes;
                    const uint32_t szb = rows * (uint32_t)p.G * 2u;
                    ptx::mbar_arrive_expect_tx(bar, wb + 2 * szb);
                    ptx::bulk_g2s(dst, p.w + (int64_t)row0 * p.row_bytes, wb, bar, pol);
                    ptx::bulk_g2s(dst + p.w_stage, p.s + (int64_t)row0 * p.G, szb, bar, pol);
                    ptx::bulk_g2s(dst + p.w_stage + p.sz_stage, p.z + (int64_t)row0 * p.G, szb, bar, pol);
                } else {
                    // Gated: the stage's pass pairs (gate pass 2j, up pass 2j + 1)
                    // cover gate rows [f0, f1) and up rows [F + f0, F + f1).  Each
                    // run is one copy: gate rows fill slots [0, SP/2) of the stage,
                    // up rows slots [SP/2, SP).
                    const int f0 = ((pass0 + i * p.SP) >> 1) * p.R;
                    const int f1 = min(((pass0 + min((i + 1) * p.SP, npass)) >> 1) * p.R, p.F);
                    const uint32_t rows = (uint32_t)(f1 - f0);
                    const uint32_t wb = rows * p.row_bytes;
                    const uint32_t szb = rows * (uint32_t)p.G * 2u;
                    const uint32_t half = (uint32_t)(p.SP / 2);
                    ptx::mbar_arrive_expect_tx(bar, 2u * (wb + 2u * szb));
                    for (int h = 0; h < 2; ++h) {
                        const int64_t row0 = (int64_t)h * p.F + f0;
                        const uint32_t wd = dst + (uint32_t)h * half * (uint32_t)p.R * p.row_bytes;
                        const uint32_t sd = dst + p.w_stage + (uint32_t)h * half * (uint32_t)(p.R * p.G) * 2u;
                        ptx::bulk_g2s(wd, p.w + row0 * p.row_bytes, wb, bar, pol);
                        ptx::bulk_g2s(sd, p.s + row0 * p.G, szb, bar, pol);
                        ptx::bulk_g2s(sd + p.sz_stage, p.z + row0 * p.G, szb, bar, pol);
                    }
                }
            }
            // Do not leave while this thread's last copies may still be landing.
            for (int i = max(0, issued - S); i < issued; ++i)
                if (!ptx::mbar_wait(full0 + 8 * (i % S), (i / S) & 1, &g_qmv_timeouts)) break;
        }
        return;
    }

    // ---------------- consumers.
    const int lane = tid & 31, warp = tid >> 5;
    const int kb = tid % p.KB, rr = tid / p.KB;
    const int gi = (kb << 5) >> p.log2g;
    const int NW = T / 32;
    const int wpr = p.KB / 32;         // warps per row slot

    XRegs<M> xr;
#pragma unroll
    for (int m = 0; m < M; ++m) {
        const uint4 *xp = reinterpret_cast<const uint4 *>(p.x + (int64_t)m * p.K + (kb << 5));
        float s = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 v = __ldg(xp + q);
            const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                xr.x[m][4 * q + i] = make_float2(bf16_lo(u[i]), bf16_hi(u[i]));
                s += bf16_lo(u[i]) + bf16_hi(u[i]);
            }
        }
        xr.xs[m] = s;
        float cx = 0.f;
        [&]<int... I>(std::integer_sequence<int, I...>) {
            ((cx = fmaf(xr.x[m][I].x, window_const<BITS>(2 * I),
                        fmaf(xr.x[m][I].y, window_const<BITS>(2 * I + 1), cx))), ...);
        }(std::make_integer_sequence<int, 16>{});
        xr.cx[m] = cx;
    }
    const float *lut = reinterpret_cast<const float *>(smem + p.lut_off) + kb;
    if constexpr (LUT) {
        // Row slot 0's threads build the tables of their block kb (x is the same
        // for every row slot); everyone waits for them.
        if (rr == 0) {
            float *tw = reinterpret_cast<float *>(smem + p.lut_off) + kb;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float a = xr.x[0][2 * j].x, b = xr.x[0][2 * j].y;
                const float c = xr.x[0][2 * j + 1].x, d = xr.x[0][2 * j + 1].y;
                float t[16];
                t[0] = 0.f; t[1] = a; t[2] = b; t[3] = a + b;
#pragma unroll
                for (int i = 0; i < 4; ++i) t[4 + i] = t[i] + c;
#pragma unroll
                for (int i = 0; i < 8; ++i) t[8 + i] = t[i] + d;
#pragma unroll
                for (int e = 0; e < 16; ++e) tw[(j * 16 + e) * p.KB] = t[e];
            }
        }
        ptx::named_sync(2, T);
    }

    float *red = reinterpret_cast<float *>(smem + p.red_off);
    const uint8_t *ring = smem + p.ring_off;
    const uint32_t wstep = (uint32_t)T * (4 * BITS);         // weights of one pass
    const uint32_t szstep = (uint32_t)p.R * p.G * 2u;       // scales of one pass
    const uint32_t w_own = (uint32_t)tid * (4 * BITS);
    // Offsets from a pass pair's first pass to the next pair and to its second pass.
    const bool gated = p.F != 0;
    const uint32_t w_pair = gated ? wstep : 2u * wstep, sz_pair = gated ? szstep : 2u * szstep;
    const uint32_t w_odd = gated ? (uint32_t)(p.SP / 2) * wstep : wstep;
    const uint32_t sz_odd = gated ? (uint32_t)(p.SP / 2) * szstep : szstep;
    const uint32_t sz_own = (uint32_t)(rr * p.G + gi) * 2u;

    // The output this thread finishes in every batch, if any: pass fj of the
    // batch, row slot fr, row of x fm.
    const bool finisher = tid < P * p.R * M;
    const int fj = tid / (p.R * M), fr = (tid / M) % p.R, fm = tid % M;

    bool ok = true;
    constexpr int U = stream_unroll<BITS>();
    constexpr int S0 = U * M;                        // slots per unrolled group
    constexpr int L0 = S0 == 2 ? 1 : (S0 == 4 ? 2 : (S0 == 8 ? 3 : 4));
    constexpr int GROUPS = 32 / S0;                  // groups per batch of 32 slots
    CarryReduce<L0> cr;
    int gs = 0, batch = 0;

    auto finish_batch = [&](float ws) {
        float *rb = red + (batch & 1) * (NW * V);
        rb[warp * V + lane] = ws;
        ptx::named_sync(1, T);
        if (p.F != 0) {
            // Gated: finisher (pair fj, row slot fr, m) combines passes 2fj and 2fj + 1.
            if (tid < (P / 2) * p.R * M) {
                const int lp = batch * P + 2 * fj;
                const int f = ((pass0 + lp) >> 1) * p.R + fr;
                if (lp < npass && f < p.F) {
                    float a = 0.f, u = 0.f;
                    for (int w2 = fr * wpr; w2 < (fr + 1) * wpr; ++w2) {
                        a += rb[w2 * V + (2 * fj) * M + fm];
                        u += rb[w2 * V + (2 * fj + 1) * M + fm];
                    }
                    if (p.bias != nullptr) {
                        a += half_bits_to_float(p.bias[f]);
                        u += half_bits_to_float(p.bias[p.F + f]);
                    }
                    p.y[(int64_t)fm * p.F + f] = float_to_bf16_bits(silu_mul(a, u));
                }
            }
        } else if (finisher) {
            const int lp = batch * P + fj;
            const int row = (pass0 + lp) * p.R + fr;
            if (lp < npass && row < p.N) {
                float acc = 0.f;
                for (int w2 = fr * wpr; w2 < (fr + 1) * wpr; ++w2) acc += rb[w2 * V + fj * M + fm];
                if (p.bias != nullptr) acc += half_bits_to_float(p.bias[row]);
                p.y[(int64_t)fm * p.N + row] = float_to_bf16_bits(acc);
            }
        }
        ++batch;
    };

    int sp = 0, st = 0;
    uint32_t ph = 0;
    const uint8_t *stage = ring;
#pragma unroll 1
    for (int pass = 0; pass < npass; pass += U) {
        if (sp == 0) {
            if (ok) ok = ptx::mbar_wait(full0 + 8 * st, ph, &g_qmv_timeouts);
            stage = ring + st * p.stage_bytes;
        }
        float v[S0];
        // Slot of the stage's pass sp + u (sp is even): plain sp + u; gated
        // (sp + u) / 2, plus SP/2 for an up pass (u odd).
        const uint8_t *wbase = stage + (gated ? (sp >> 1) : sp) * wstep + w_own;
        const uint8_t *sbase = stage + p.w_stage + (gated ? (sp >> 1) : sp) * szstep + sz_own;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            uint32_t wv[BITS];
            const uint32_t wo = (u >> 1) * w_pair + (u & 1) * w_odd;
            const uint32_t so = (u >> 1) * sz_pair + (u & 1) * sz_odd;
            lds_block<BITS>(wbase + wo, wv);
            const float sv = half_bits_to_float(*reinterpret_cast<const uint16_t *>(sbase + so));
            const float zv = half_bits_to_float(*reinterpret_cast<const uint16_t *>(sbase + p.sz_stage + so));
            float d[M];
            if constexpr (LUT) d[0] = lut_dot(wv[0], lut, p.KB);
            else block_dot<BITS, M>(wv, xr, d);
#pragma unroll
            for (int m = 0; m < M; ++m) v[u * M + m] = fmaf(sv, d[m], zv * xr.xs[m]);
        }
        sp += U;
        if (sp == p.SP || pass + U >= npass) {
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(empty0 + 8 * st);
            sp = 0;
            if (++st == S) { st = 0; ph ^= 1u; }
        }
        float val = static_butterfly<S0>(v, lane);
        if (cr.feed(val, gs, lane)) finish_batch(val);
        gs = (gs + 1) & (GROUPS - 1);
    }
    // Pad the last batch with zeros so that it completes.
    while (gs != 0) {
        float val = 0.f;
        if (cr.feed(val, gs, lane)) finish_batch(val);
        gs = (gs + 1) & (GROUPS - 1);
    }
}

struct StreamPlan {
    bool ok = false;
    StreamParams prm{};
    int grid = 0;
    uint32_t smem = 0;
    int threads = 0;
};

bool aligned16(const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; }

template <int BITS, int M, bool LUT>
const void *stream_kernel_ptr() {
    return reinterpret_cast<const void *>(&qmv_stream_kernel<BITS, M, LUT>);
}

// Resident CTAs per SM of the stream kernel on device dev, for a shared-memory
// size rounded up to the next 8 KB (never optimistic; few distinct queries),
// with the kernel's dynamic shared-memory limit raised first.  0 on error.
template <int BITS, int M, bool LUT>
int stream_occupancy(int dev, int threads, uint32_t smem) {
    const void *fn = stream_kernel_ptr<BITS, M, LUT>();
    if (raise_smem_limit(fn, dev, 200 * 1024) != cudaSuccess) return 0;
    return blocks_per_sm(fn, dev, threads, (smem + 8191u) / 8192u * 8192u);
}

// Shared memory a CTA may fill with ring stages (two CTAs fit on an SM).
constexpr uint32_t kRingBudget = 96u * 1024u;
constexpr uint32_t kStageTarget = 12u * 1024u;
// Table decode: ring stages limited to this so that the tables (16 K bytes
// for K codes per row) and the ring of two CTAs share an SM.
constexpr uint32_t kLutRingBudget = 40u * 1024u;
constexpr int kLutMaxK = 4096;

template <int BITS, int M, bool LUT = false>
StreamPlan plan_stream(const uint16_t *x, const uint8_t *w, const uint16_t *s, const uint16_t *z,
                       const uint16_t *bias, uint16_t *y, int K, int N, int group, int F) {
    StreamPlan pl;
    if (K % 1024 != 0 || K / 32 > stream_max_consumers<M>()) return pl;
    if (LUT && K > kLutMaxK) return pl;
    const int G = K / group;
    if (((int64_t)N * G) % 8 != 0) return pl;
    if (F != 0 && G % 8 != 0) return pl;          // gated passes copy R*G fp16 values each
    if (!aligned16(w) || !aligned16(s) || !aligned16(z) || !aligned16(x)) return pl;
    StreamParams &q = pl.prm;
    q.x = x; q.w = w; q.s = s; q.z = z; q.bias = bias; q.y = y;
    q.N = N; q.K = K; q.KB = K / 32; q.G = G; q.log2g = __builtin_ctz((unsigned)group);
    q.F = F;
    q.R = (M == 1) ? (256 + q.KB - 1) / q.KB : 256 / q.KB;
    q.T = q.R * q.KB;
    const uint32_t w_pass = (uint32_t)q.T * 4u * BITS;
    const uint32_t sz_pass = (uint32_t)q.R * G * 2u;
    // Scale/zero copies must be 16-byte multiples: a split unit of `chunk`
    // passes holds chunk*R*G fp16 values, a multiple of 8.
    // Gated: split units are gate/up pass pairs (each pass is copied on its own).
    q.chunk = F != 0 ? 2 : 8 / std::gcd(8, q.R * G);
    const int U = stream_unroll<BITS>();
    const int step = std::lcm(q.chunk, U);
    int SP = std::max(1, (int)(kStageTarget / (w_pass + 2u * sz_pass)));
    SP = (SP + step - 1) / step * step;
    q.SP = SP;
    q.row_bytes = (uint32_t)K * BITS / 8u;
    q.w_stage = SP * w_pass;
    q.sz_stage = SP * sz_pass;
    q.stage_bytes = q.w_stage + 2u * q.sz_stage;
    const uint32_t budget = LUT ? kLutRingBudget : kRingBudget;
    q.stages = (int)std::min<uint32_t>(kMaxStages, std::max<uint32_t>(2u, budget / q.stage_bytes));
    q.red_off = 16u * kMaxStages;
    const uint32_t red_bytes = 2u * (q.T / 32) * 32u * 4u;
    q.ring_off = (q.red_off + red_bytes + 127u) & ~127u;
    q.lut_off = (q.ring_off + q.stages * q.stage_bytes + 127u) & ~127u;
    pl.smem = q.lut_off + (LUT ? 8u * 16u * (uint32_t)q.KB * 4u : 0u);
    if (pl.smem > 200u * 1024u) return pl;
    pl.threads = q.T + 32;
    q.total_passes = F != 0 ? 2 * ((F + q.R - 1) / q.R) : (N + q.R - 1) / q.R;
    q.chunks = (q.total_passes + q.chunk - 1) / q.chunk;
    const int dev = current_device();
    const int occ = dev < 0 ? 0 : stream_occupancy<BITS, M, LUT>(dev, pl.threads, pl.smem);
    const int sms = dev < 0 ? 0 : device_sm_count(dev);
    if (occ < 1 || sms < 1) return pl;                 // pl.ok stays false: a CUDA error
    pl.grid = std::max(1, std::min(q.chunks, sms * occ));
    q.chunks_base = q.chunks / pl.grid;
    q.chunks_extra = q.chunks % pl.grid;
    pl.ok = true;
    return pl;
}

template <int BITS, int M, bool LUT = false>
cudaError_t launch_stream(const StreamPlan &pl, cudaStream_t stream) {
    cudaError_t e = launch_pdl(qmv_stream_kernel<BITS, M, LUT>, dim3(pl.grid), dim3(pl.threads), pl.smem,
                               stream, pl.prm);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// F == 0: y = x W^T + bias, W with N rows.  F > 0 (N == 2F): the gated form,
// y[m, f] = silu(g) * u with g, u the outputs of rows f and F + f.
template <int BITS>
cudaError_t launch_bits(const uint16_t *x, const uint8_t *w, const uint16_t *s, const uint16_t *z,
                        const uint16_t *bias, uint16_t *y, int64_t M, int K, int N, int group,
                        int F, cudaStream_t stream) {
    // The tensor-core decode kernel takes every shape it supports.
    const cudaError_t em = launch_qmv_mma(x, w, s, z, bias, y, M, K, N, BITS, group, F, stream);
    if (em != cudaErrorNotSupported) return em;
    const int log2g = __builtin_ctz((unsigned)group);
    const int64_t ys = F != 0 ? F : N;           // elements per row of y
    // Rows of x two at a time through the stream kernel when its conditions hold.
    StreamPlan p1 = plan_stream<BITS, 1>(x, w, s, z, bias, y, K, N, group, F);
    if (!p1.ok) return launch_generic<BITS>(x, w, s, z, bias, y, M, K, N, log2g, F, stream);
    for (int64_t m0 = 0; m0 < M; m0 += 2) {
        const int mc = (int)std::min<int64_t>(2, M - m0);
        cudaError_t e;
        if (mc == 1) {
            bool done = false;
            if constexpr (BITS == 1) {             // table decode when its tables fit
                StreamPlan pt = plan_stream<1, 1, true>(x + m0 * K, w, s, z, bias, y + m0 * ys, K, N, group, F);
                if (pt.ok) {
                    e = launch_stream<1, 1, true>(pt, stream);
                    done = true;
                }
            }
            if (!done) {
                StreamPlan pl = plan_stream<BITS, 1>(x + m0 * K, w, s, z, bias, y + m0 * ys, K, N, group, F);
                e = launch_stream<BITS, 1>(pl, stream);
            }
        } else {
            StreamPlan pl = plan_stream<BITS, 2>(x + m0 * K, w, s, z, bias, y + m0 * ys, K, N, group, F);
            if (pl.ok) {
                e = launch_stream<BITS, 2>(pl, stream);
            } else {  // two rows of x that do not fit one CTA's registers: one launch each
                for (int i = 0; i < 2 && (e = cudaSuccess) == cudaSuccess; ++i) {
                    StreamPlan p1r = plan_stream<BITS, 1>(x + (m0 + i) * K, w, s, z, bias,
                                                          y + (m0 + i) * ys, K, N, group, F);
                    e = launch_stream<BITS, 1>(p1r, stream);
                    if (e != cudaSuccess) break;
                }
            }
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

uint32_t qmv_timeouts(bool reset) {
    unsigned int v = 0;
    cudaMemcpyFromSymbol(&v, g_qmv_timeouts, sizeof(v));
    if (reset) {
        const unsigned int zero = 0;
        cudaMemcpyToSymbol(g_qmv_timeouts, &zero, sizeof(zero));
    }
    return v;
}

namespace {
cudaError_t launch_any(const uint16_t *x, const uint8_t *w, const uint16_t *scales,
                       const uint16_t *zeros, const uint16_t *bias, uint16_t *y, int64_t M,
                       int K, int N, int bits, int group, int F, cudaStream_t stream) {
    switch (bits) {
        case 1: return launch_bits<1>(x, w, scales, zeros, bias, y, M, K, N, group, F, stream);
        case 2: return launch_bits<2>(x, w, scales, zeros, bias, y, M, K, N, group, F, stream);
        case 3: return launch_bits<3>(x, w, scales, zeros, bias, y, M, K, N, group, F, stream);
        case 4: return launch_bits<4>(x, w, scales, zeros, bias, y, M, K, N, group, F, stream);
        case 5: return launch_bits<5>(x, w, scales, zeros, bias, y, M, K, N, group, F, stream);
        case 6: return launch_bits<6>(x, w, scales, zeros, bias, y, M, K, N, group, F, stream);
        case 7: return launch_bits<7>(x, w, scales, zeros, bias, y, M, K, N, group, F, stream);
        default: return cudaErrorInvalidValue;
    }
}
}  // namespace

cudaError_t launch_qmv(const uint16_t *x, const uint8_t *w, const uint16_t *scales,
                       const uint16_t *zeros, const uint16_t *bias, uint16_t *y, int64_t M,
                       int64_t K, int64_t N, int bits, int group, cudaStream_t stream) {
    return launch_any(x, w, scales, zeros, bias, y, M, (int)K, (int)N, bits, group, 0, stream);
}

cudaError_t launch_qmv_gated(const uint16_t *x, const uint8_t *w, const uint16_t *scales,
                             const uint16_t *zeros, const uint16_t *bias, uint16_t *y, int64_t M,
                             int64_t K, int64_t F, int bits, int group, cudaStream_t stream) {
    return launch_any(x, w, scales, zeros, bias, y, M, (int)K, (int)(2 * F), bits, group, (int)F, stream);
}

}  // namespace lowbit
