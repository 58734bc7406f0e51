// qmm.cu -- quantised matrix-matrix product on the 5th-generation tensor
// cores (tcgen05, accumulators in tensor memory), for batched inputs.
//
// Method: y = x W^T + bias with W[n,k] = scale[n,k/g] * q[n,k] + zero[n,k/g]
// (torchchat PR #1415 "Add torchao mps ops"; ao PR #2167 "metal lowbit
// kernels: qmv_fast optimization", Summary bullets 1-2, where a reviewer asks
// whether the matrix-vector kernel carries over to gemm; bias per ao issue
// #3446).
//
// Exact-code formulation.  Rounding each dequantised weight to bf16 before
// the product costs 2^-9 of |W| per weight, an error that does not shrink with
// |y| and is too large for near-zero outputs.  Instead the tensor cores
// multiply the integer codes themselves, which bf16 holds exactly (as 128 + q,
// q < 128), and the scale and zero are applied per group in fp32:
//     P_g[n,m] = sum_{k in g} (128 + q[n,k]) x[m,k]       (tensor cores, fp32)
//     X_g[m]   = sum_{k in g} x[m,k]                      (tensor cores, fp32)
//     y[m,n]   = sum_g s[n,g] P_g[n,m] + (z[n,g] - 128 s[n,g]) X_g[m] + bias[n]
// Every product is exact; only fp32 summation rounds.  X_g comes from the
// last row of each 32-row quarter of the A tile (rows 31, 63, 95, 127), which
// hold ones instead of codes, so every warp finds X_g in its own lane 31 and a
// tile covers 124 output rows.
//
// Tiling ("swap AB"): the MMA's 128-row A operand is a tile of weight rows
// (output features n), held in tensor memory; its B operand is a tile of TN
// rows of x (TN <= 128, batch rows m) in shared memory.  K advances 128 codes
// per stage; each group segment (min(g, 128) codes) accumulates into one of
// several TMEM buffers of TN columns.  Keeping A in tensor memory means the
// unpacked codes never travel through shared memory (neither as stores nor as
// MMA operand reads), which leaves shared-memory bandwidth to the x tiles.
//
// Warp roles (480 threads):
//   warp 0       TMA producers: lane 0 streams the 128 x 16b packed-code
//                tiles (one 2D tensor copy per stage) into a deep ring that
//                the unpackers free; lane 1 streams the x tiles (two 2D copies,
//                64-wide, 128-byte swizzle) into a ring that MMA completion
//                frees;
//   warps 1, 2   lane 0 of each issues the MMAs (tcgen05.mma kind::f16, A from
//                tensor memory, bf16 x bf16 -> fp32) of alternate K steps when
//                a segment is one step long (one issuer otherwise) and commits
//                them to mbarriers that free buffers or hand a segment on;
//                warp 1 also allocates and frees tensor memory;
//   warps 3..6   unpack: one thread per tile row (its TMEM lane) turns the
//                row's codes into bf16 pairs and writes them with tcgen05.st;
//   warps 7..14  accumulate: per segment read P_g and X_g from tensor memory,
//                apply scale and zero in fp32, and at the end add the bias and
//                store y (two warps per tensor-memory lane quarter).
// All waits are bounded (about one second) and count a timeout instead of
// hanging; tensor memory is always released before the CTA exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>

#include "common.cuh"
#include "ptx.cuh"

namespace lowbit {
namespace {

constexpr int kBM = 128;             // rows of an A tile (MMA M)
constexpr int kRowsOut = kBM - 4;    // output rows per tile; rows 31, 63, 95, 127 hold ones
constexpr int kBK = 128;             // codes per K stage
constexpr int kMaxPStages = 12;      // packed-code ring (freed by the unpackers)
constexpr int kXStages = 4;          // x ring (freed when the MMAs that read it complete)
constexpr int kAStages = 2;          // code tiles in tensor memory
constexpr int kACols = kBK / 2;      // TMEM columns of one code tile (two bf16 per column)
constexpr int kUnpackWarps = 4;      // one per TMEM lane quarter
constexpr int kAccWarps = 8;
constexpr int kIssuers = 2;          // MMA-issuing threads (warps 1 and 2, lane 0)
constexpr int kFirstUnpackWarp = 1 + kIssuers;                    // 3
constexpr int kFirstAccWarp = kFirstUnpackWarp + kUnpackWarps;    // 7
constexpr int kThreads = (kFirstAccWarp + kAccWarps) * 32;        // 480
constexpr int kMaxTmemBufs = 4;
constexpr uint32_t kBf16Magic = 0x43004300u;                      // bf16 pair (128, 128)

__device__ unsigned int g_qmm_timeouts;

struct QmmParams {
    const uint16_t *s;
    const uint16_t *z;
    const uint16_t *bias;
    uint16_t *y;
    int M, N, K, G, log2g, TN, tmem_cols, nbuf, a_col, ktiles, lseg_log2, nseg;
    int pstages;            // depth of the packed-code ring
    int ksplit;             // CTAs of a cluster that split K (1: no split)
    int kt_unit;            // K tiles per split unit (a group spans whole units)
    uint32_t recv_off;      // split-K: partial sums from the other CTAs (from base)
    uint32_t x_stage;       // TN * kBK * 2 bytes (two swizzle atoms of TN rows)
    uint32_t x_off, p_off;           // offsets from the 1024-aligned base
    uint32_t idesc;         // tcgen05 instruction descriptor
};

// 32 bits of a block's little-endian code stream starting at bit START
// (negative START: zeros shifted in from below).
template <int BITS, int START>
__device__ __forceinline__ uint32_t stream_window(const uint32_t (&w)[BITS]) {
    if constexpr (START < 0) {
        return w[0] << (-START);
    } else {
        constexpr int wi = START / 32, off = START % 32;
        if constexpr (off == 0) {
            return w[wi];
        } else {
            const uint32_t hi = (wi + 1 < BITS) ? w[wi + 1 < BITS ? wi + 1 : 0] : 0u;
            return __funnelshift_r(w[wi], hi, off);
        }
    }
}

// Word I (0..15) of a 32-code block as the bf16 pair (128 + q[2I], 128 + q[2I+1]).
template <int BITS, int I>
__device__ __forceinline__ uint32_t code_pair(const uint32_t (&w)[BITS]) {
    constexpr uint32_t m = (1u << BITS) - 1u;
    if constexpr (BITS == 4) {
        // One byte = the pair; byte * (1 + 2^12) puts its high nibble at bit 16.
        const uint32_t byte = ptx::prmt(w[I / 4], 0u, 0x4440u | (I % 4));
        return ptx::and_or_imm<0x000F000Fu>(byte * 0x1001u, kBf16Magic);
    } else if constexpr (BITS == 2) {
        const uint32_t byte = ptx::prmt(w[I / 8], 0u, 0x4440u | ((I / 2) % 4));
        uint32_t v = byte * (1u + (1u << 14));
        if constexpr (I % 2) v >>= 4;
        return ptx::and_or_imm<0x00030003u>(v, kBf16Magic);
    } else if constexpr (BITS == 1) {
        const uint32_t byte = ptx::prmt(w[I / 16], 0u, 0x4440u | ((I / 4) % 4));
        uint32_t v = byte * (1u + (1u << 15));
        if constexpr (I % 4) v >>= (I % 4) * 2;
        return ptx::and_or_imm<0x00010001u>(v, kBf16Magic);
    } else if constexpr (2 * BITS <= 16 - BITS) {
        // 3 or 5 bits: the pair's 2b bits, spread by one multiply.
        const uint32_t c = stream_window<BITS, 2 * I * BITS>(w) & ((1u << (2 * BITS)) - 1u);
        return ptx::and_or_imm<m | (m << 16)>(c * (1u + (1u << (16 - BITS))), kBf16Magic);
    } else {
        const uint32_t lo = stream_window<BITS, 2 * I * BITS>(w);
        const uint32_t hi = stream_window<BITS, (2 * I + 1) * BITS - 16>(w);
        return ptx::and_or_imm<(m << 16)>(hi, ptx::and_or_imm<m>(lo, kBf16Magic));
    }
}

template <int BITS>
__device__ __forceinline__ void lds_words(const uint8_t *p, uint32_t (&w)[BITS]) {
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

// What an MMA-issuing thread needs (shared addresses of the barriers, tensor
// memory, descriptors).
struct IssueCtx {
    uint32_t tmem, a_tmem;
    uint32_t x_full, a_full, t_full, t_empty, x_empty, a_empty;
    uint64_t xd0;                     // descriptor of x stage 0
    uint32_t xd_stage, xd_atom;       // descriptor address units: next stage, second 64-code half
    uint32_t idesc;
    int nkt, nbuf, TN;
};

// Issues the MMAs of K steps me, me + nis, me + 2 nis, ... of this CTA (SPS
// segments of 128 / SPS codes per step, each into the next accumulator
// buffer).  Returns false after a wait timed out.
//
// One thread issuing every step keeps the tensor core only ~65% busy: any
// instruction between a step's MMAs (barrier waits, buffer bookkeeping) idles
// it, because it holds only a couple of MMAs in its queue.  With two threads
// taking alternate steps, one issues while the other waits, and the MMAs of
// consecutive steps (different buffers, stages and barriers) interleave
// freely.  Two issuers need SPS = 1 and at least two buffers: then every
// barrier phase a thread waits for is at most one behind the one it last saw
// itself, so parity waits cannot alias.
template <int SPS>
__device__ __forceinline__ bool issue_steps(const IssueCtx &c, int me, int nis) {
    constexpr int kPer = (kBK / 16) / SPS;       // MMAs per segment
    int b = (me * SPS) % c.nbuf;                 // buffer of this thread's next segment
    int r = (me * SPS) / c.nbuf;                 // how often that buffer was used before
    for (int kt = me; kt < c.nkt; kt += nis) {
        const int st = kt & (kXStages - 1), as = kt & (kAStages - 1);
        if (!ptx::mbar_wait(c.x_full + 8 * st, (kt / kXStages) & 1, &g_qmm_timeouts) ||
            !ptx::mbar_wait(c.a_full + 8 * as, (kt / kAStages) & 1, &g_qmm_timeouts))
            return false;
        const uint32_t a_st = c.a_tmem + (uint32_t)(as * kACols);
        const uint64_t xd = c.xd0 + (uint64_t)st * c.xd_stage;
#pragma unroll
        for (int j = 0; j < SPS; ++j) {
            if (r > 0 && !ptx::mbar_wait(c.t_empty + 8 * b, (uint32_t)(r - 1) & 1u, &g_qmm_timeouts)) return false;
            ptx::tc_fence_after();
            const uint32_t d = c.tmem + (uint32_t)(b * c.TN);
#pragma unroll
            for (int m = 0; m < kPer; ++m) {
                const int kk = j * kPer + m;
                ptx::mma_f16_tmem_a(d, a_st + (uint32_t)(kk * 8),
                                    xd + (uint64_t)((kk >> 2) * c.xd_atom + (kk & 3) * 2), c.idesc, m != 0);
            }
            ptx::mma_commit(c.t_full + 8 * b);
            if (++b == c.nbuf) {
                b = 0;
                ++r;
            }
        }
        ptx::mma_commit(c.x_empty + 8 * st);
        ptx::mma_commit(c.a_empty + 8 * as);
        for (int i = 0; i < (nis - 1) * SPS; ++i) {      // the other issuers' segments
            if (++b == c.nbuf) {
                b = 0;
                ++r;
            }
        }
    }
    return true;
}

// Final rows of one accumulating thread: y[m, n] = acc + bias for its chunks
// (all of them when ks == 1; with split K only the chunks c with c % ks ==
// rank, summing the partials of CTAs 0..ks-1 in order, its own from `acc`,
// the others from `recv`).
__device__ __forceinline__ void store_rows(const QmmParams &p, const float2 (&acc)[4][8], int h, int nchunk,
                                           int n, int m0, int rank, int ks, const uint8_t *recv = nullptr,
                                           int at = 0) {
    const float bias = p.bias != nullptr ? half_bits_to_float(p.bias[n]) : 0.f;
    const int J = (4 + ks - 1) / ks;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int ch = h + 2 * c;
        if (ch >= nchunk || (ks > 1 && c % ks != rank)) continue;
        float v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = 0.f;
        for (int src = 0; src < ks; ++src) {
            if (src == rank || ks == 1) {
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] += (j & 1) ? acc[c][j / 2].y : acc[c][j / 2].x;
            } else {
                const float4 *r = reinterpret_cast<const float4 *>(recv + ((src * J + c / ks) * 256 + at) * 64);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float4 t = r[j];
                    v[4 * j] += t.x; v[4 * j + 1] += t.y; v[4 * j + 2] += t.z; v[4 * j + 3] += t.w;
                }
            }
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int m = m0 + ch * 16 + j;
            if (m < p.M) p.y[(int64_t)m * p.N + n] = float_to_bf16_bits(v[j] + bias);
        }
    }
}

template <int BITS>
__global__ void __launch_bounds__(kThreads, 1)
qmm_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
           const QmmParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;            // swizzle atoms need 1024-byte alignment
    uint8_t *smem = smem_raw + (base - raw);

    ptx::pdl_launch_dependents();
    ptx::pdl_wait();            // inputs may come from the previous kernel in the stream
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Split K: the ksplit CTAs of a cluster (consecutive blockIdx.x) share a row
    // tile; CTA `rank` takes K tiles [kt0, kt0 + nkt), whole groups each.
    const int ks = p.ksplit;
    const int rank = ks > 1 ? (int)ptx::cluster_ctarank() : 0;
    const int n0 = (blockIdx.x / ks) * kRowsOut;
    const int units = p.ktiles / p.kt_unit;
    const int kt0 = (units * rank / ks) * p.kt_unit;
    const int nkt = (units * (rank + 1) / ks) * p.kt_unit - kt0;
    const int m0 = blockIdx.y * p.TN;
    constexpr uint32_t kPackedStage = kBM * (kBK * BITS / 8);

    // Barriers (8 bytes each), then the TMEM address.
    const uint32_t p_full = base, p_empty = p_full + 8 * kMaxPStages;
    const uint32_t x_full = p_empty + 8 * kMaxPStages, x_empty = x_full + 8 * kXStages;
    const uint32_t a_full = x_empty + 8 * kXStages, a_empty = a_full + 8 * kAStages;
    const uint32_t t_full = a_empty + 8 * kAStages, t_empty = t_full + 8 * kMaxTmemBufs;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + (t_empty + 8 * kMaxTmemBufs - base));

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.pstages; ++i) {
            ptx::mbar_init(p_full + 8 * i, 1);
            ptx::mbar_init(p_empty + 8 * i, kUnpackWarps);
        }
        for (int i = 0; i < kXStages; ++i) {
            ptx::mbar_init(x_full + 8 * i, 1);
            ptx::mbar_init(x_empty + 8 * i, 1);
        }
        for (int i = 0; i < kAStages; ++i) {
            ptx::mbar_init(a_full + 8 * i, kUnpackWarps);
            ptx::mbar_init(a_empty + 8 * i, 1);
        }
        for (int i = 0; i < kMaxTmemBufs; ++i) {
            ptx::mbar_init(t_full + 8 * i, 1);
            ptx::mbar_init(t_empty + 8 * i, kAccWarps);
        }
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), (uint32_t)p.tmem_cols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const uint32_t a_tmem = tmem + (uint32_t)p.a_col;    // code tiles: kAStages x kACols columns
    const uint32_t x_base = base + p.x_off;
    const uint32_t p_base = base + p.p_off;
    const int sps = kBK >> p.lseg_log2;          // segments per stage

    if (warp == 0) {
        // ---------------- TMA producers (lane 0: packed codes, lane 1: x).
        if (lane < 2) {
            const int depth = lane == 0 ? p.pstages : kXStages;
            const uint32_t full = lane == 0 ? p_full : x_full;
            const uint32_t empty = lane == 0 ? p_empty : x_empty;
            const uint64_t pol = ptx::policy_evict_first();
            int issued = 0;
            for (int i = 0; i < nkt; ++i, ++issued) {
                const int kt = kt0 + i;
                const int st = i % depth;
                if (i >= depth && !ptx::mbar_wait(empty + 8 * st, ((i / depth) - 1) & 1, &g_qmm_timeouts))
                    break;
                const uint32_t bar = full + 8 * st;
                if (lane == 0) {
                    ptx::mbar_arrive_expect_tx(bar, kPackedStage);
                    ptx::tma_load_2d_hint(p_base + st * kPackedStage, &wmap, kt * (kBK * BITS / 8), n0, bar, pol);
                } else {
                    const uint32_t xs = x_base + st * p.x_stage;
                    ptx::mbar_arrive_expect_tx(bar, p.x_stage);
                    ptx::tma_load_2d(xs, &xmap, kt * kBK, m0, bar);
                    ptx::tma_load_2d(xs + p.x_stage / 2, &xmap, kt * kBK + 64, m0, bar);
                }
            }
            for (int i = max(0, issued - depth); i < issued; ++i)
                if (!ptx::mbar_wait(full + 8 * (i % depth), (i / depth) & 1, &g_qmm_timeouts)) break;
        }
    } else if (warp < kFirstUnpackWarp) {
        // ---------------- MMA issuers (lane 0 of warps 1 and 2).
        if (lane == 0) {
            static_assert((kXStages & (kXStages - 1)) == 0 && (kAStages & (kAStages - 1)) == 0 && kBK == 128,
                          "ring shapes");
            IssueCtx c;
            c.tmem = tmem;
            c.a_tmem = a_tmem;
            c.x_full = x_full; c.a_full = a_full; c.t_full = t_full; c.t_empty = t_empty;
            c.x_empty = x_empty; c.a_empty = a_empty;
            c.xd0 = ptx::sw128_desc(x_base);
            c.xd_stage = p.x_stage >> 4;
            c.xd_atom = p.x_stage >> 5;
            c.idesc = p.idesc;
            c.nkt = nkt;
            c.nbuf = p.nbuf;
            c.TN = p.TN;
            const int me = warp - 1;
            if (sps == 1) {
                issue_steps<1>(c, me, kIssuers);
            } else if (me == 0) {
                if (sps == 2) issue_steps<2>(c, 0, 1);
                else issue_steps<4>(c, 0, 1);
            }
        }
    } else if (warp < kFirstAccWarp) {
        // ---------------- code unpackers (warps 3..6): thread = one tile row = its TMEM lane.
        const int q = warp & 3;
        // Packed row of this lane in the tile; lane 31 holds the ones row and
        // reads the next quarter's first row (in the tile) only to keep the
        // warp converged.
        const int pr = q * 31 + lane;
        const uint32_t trow = ((uint32_t)(q * 32) << 16);
        bool ok = true;
        for (int kt = 0; kt < nkt && ok; ++kt) {              // kt relative to kt0 here
            const int st = kt % p.pstages, as = kt % kAStages;
            ok = ptx::mbar_wait(p_full + 8 * st, (kt / p.pstages) & 1, &g_qmm_timeouts);
            if (ok && kt >= kAStages)
                ok = ptx::mbar_wait(a_empty + 8 * as, ((kt / kAStages) - 1) & 1, &g_qmm_timeouts);
            if (!ok) break;
            ptx::tc_fence_after();
            const uint8_t *pk = smem + p.p_off + st * kPackedStage + pr * (kBK * BITS / 8);
            const uint32_t adst = a_tmem + trow + (uint32_t)(as * kACols);
            // All four 32-code blocks are loaded before the first tensor-memory
            // store, so that one shared-memory latency covers the step.
            uint32_t w[4][BITS];
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) lds_words<BITS>(pk + blk * (4 * BITS), w[blk]);
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
                uint32_t h[16];
                if constexpr (BITS == 4) {
                    // Four pairs per word in nine instructions: even and odd
                    // nibbles into bytes, bytes into code order, and each
                    // pair of codes beside the magic byte 0x43.
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t t = w[blk][i] & 0x0F0F0F0Fu, u = (w[blk][i] >> 4) & 0x0F0F0F0Fu;
                        const uint32_t v0 = ptx::prmt(t, u, 0x5140u), v1 = ptx::prmt(t, u, 0x7362u);
                        h[4 * i] = ptx::prmt(v0, 0x43434343u, 0x4140u);
                        h[4 * i + 1] = ptx::prmt(v0, 0x43434343u, 0x4342u);
                        h[4 * i + 2] = ptx::prmt(v1, 0x43434343u, 0x4140u);
                        h[4 * i + 3] = ptx::prmt(v1, 0x43434343u, 0x4342u);
                    }
                } else {
                    [&]<int... J>(std::integer_sequence<int, J...>) {
                        ((h[J] = code_pair<BITS, J>(w[blk])), ...);
                    }(std::make_integer_sequence<int, 16>{});
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) h[j] = lane == 31 ? 0x3F803F80u : h[j];   // bf16 (1, 1)
                ptx::tmem_st16(adst + (uint32_t)(blk * 16), h);
            }
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                ptx::mbar_arrive(p_empty + 8 * st);
                ptx::mbar_arrive(a_full + 8 * as);
            }
        }
    } else {
        // ---------------- accumulators (warps 7..14).
        const int q = warp & 3;                          // tensor-memory lane quarter
        const int h = (warp - kFirstAccWarp) >> 2;       // which half of the 16-column chunks
        const int n = n0 + q * 31 + lane;                // TMEM lane 32q + lane; lane 31 is a ones row
        const bool row_ok = lane < 31 && n < p.N;
        const int nrow = min(n, p.N - 1);
        const int nchunk = p.TN / 16;
        float2 acc[4][8];                                // chunks h, h+2, h+4, h+6
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[c][j] = make_float2(0.f, 0.f);
        bool ok = true;
        const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
        // Scale and zero of segment seg+2 are fetched while segment seg is processed.
        const uint16_t *srow = p.s + (int64_t)nrow * p.G, *zrow = p.z + (int64_t)nrow * p.G;
        const int seg0 = kt0 * sps, nseg = nkt * sps;   // this CTA's segments
        auto seg_group = [&](int sg) { return min(((seg0 + sg) << p.lseg_log2) >> p.log2g, p.G - 1); };
        uint16_t s0 = __ldg(srow + seg_group(0)), s1 = __ldg(srow + seg_group(1));
        uint16_t z0 = __ldg(zrow + seg_group(0)), z1 = __ldg(zrow + seg_group(1));
        // Buffer of the segment and the parity of its t_full phase, advanced by
        // counters: two integer divisions by the buffer count per segment cost
        // ~8% of the kernel's time.
        int b = 0;
        uint32_t par = 0;
        for (int seg = 0; seg < nseg; ++seg) {
            const float sv = half_bits_to_float(s0);
            const float zv = half_bits_to_float(z0);
            s0 = s1;
            z0 = z1;
            s1 = __ldg(srow + seg_group(seg + 2));
            z1 = __ldg(zrow + seg_group(seg + 2));
            const float2 s2 = make_float2(sv, sv);
            const float zc = fmaf(-128.f, sv, zv);      // zero minus the codes' +128 offset
            const float2 z2 = make_float2(zc, zc);
            if (ok) ok = ptx::mbar_wait(t_full + 8 * b, par, &g_qmm_timeouts);
            ptx::tc_fence_after();
            bool released = false;                        // one t_empty arrival per warp per segment
#pragma unroll
            for (int c = 0; c < 4; ++c) {                // one 16-column chunk per tensor-memory wait
                const int ch = h + 2 * c;
                uint32_t v[16];
                if (ch < nchunk) ptx::tmem_ld16(trow + (uint32_t)(b * p.TN + ch * 16), v);
                ptx::tmem_ld_wait();
                if (!released && (c + 1 >= 4 || h + 2 * (c + 1) >= nchunk)) {
                    // Last tensor-memory read of this segment: hand the buffer back.
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(t_empty + 8 * b);
                    released = true;
                }
                // The group sums X_g of the chunk's columns sit in lane 31 (the
                // ones row) and are broadcast by shuffles.
                if (ch < nchunk) {
#pragma unroll
                    for (int j = 0; j < 16; j += 2) {
                        const float x0 = __shfl_sync(0xFFFFFFFFu, __uint_as_float(v[j]), 31);
                        const float x1 = __shfl_sync(0xFFFFFFFFu, __uint_as_float(v[j + 1]), 31);
                        float2 &a = acc[c][j / 2];
                        ptx::ffma2(a, make_float2(__uint_as_float(v[j]), __uint_as_float(v[j + 1])), s2, a);
                        ptx::ffma2(a, make_float2(x0, x1), z2, a);
                    }
                }
            }
            if (++b == p.nbuf) {
                b = 0;
                par ^= 1u;
            }
        }
        if (ks == 1) {
            if (ok && row_ok) store_rows(p, acc, h, nchunk, n, m0, -1, 1);
        } else {
            // Split K: chunk c of every thread belongs to CTA c % ks of the
            // cluster.  After every CTA of the cluster has left its pipeline,
            // each sends the chunks it does not own to their owners' shared
            // memory; after a second cluster barrier each owner adds the ks
            // partial sums in rank order (the same order on every run) and
            // stores the rows.
            const int at = threadIdx.x - kFirstAccWarp * 32;           // 0..255
            const int J = (4 + ks - 1) / ks;                           // owned chunks per CTA
            ptx::cluster_sync();
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int ch = h + 2 * c, owner = c % ks;
                if (ch < nchunk && owner != rank) {
                    const uint32_t off = base + p.recv_off + (uint32_t)(((rank * J + c / ks) * 256 + at) * 64);
                    const uint32_t dst = ptx::mapa_shared(off, (uint32_t)owner);
#pragma unroll
                    for (int j = 0; j < 8; j += 2)
                        ptx::st_cluster_v4(dst + j * 8, acc[c][j].x, acc[c][j].y, acc[c][j + 1].x, acc[c][j + 1].y);
                }
            }
            ptx::cluster_sync();
            if (ok && row_ok) store_rows(p, acc, h, nchunk, n, m0, rank, ks, smem + p.recv_off, at);
        }
    }
    if (ks > 1 && warp < kFirstAccWarp) {
        // The other roles take part in the accumulators' two cluster barriers.
        __syncwarp();
        ptx::cluster_sync();
        ptx::cluster_sync();
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) ptx::tmem_dealloc(tmem, (uint32_t)p.tmem_cols);
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------

template <int BITS>
cudaError_t launch_bits(const uint16_t *x, const uint8_t *w, const uint16_t *s, const uint16_t *z,
                        const uint16_t *bias, uint16_t *y, int M, int K, int N, int group,
                        cudaStream_t stream) {
    QmmParams q{};
    q.s = s; q.z = z; q.bias = bias; q.y = y;
    q.M = M; q.N = N; q.K = K; q.G = K / group; q.log2g = __builtin_ctz((unsigned)group);
    q.TN = M >= 128 ? 128 : ((M + 15) / 16) * 16;
    q.nbuf = std::min(kMaxTmemBufs, (512 - kAStages * kACols) / q.TN);
    q.a_col = q.nbuf * q.TN;
    const int cols = q.a_col + kAStages * kACols;
    q.tmem_cols = cols <= 32 ? 32 : (cols <= 64 ? 64 : (cols <= 128 ? 128 : (cols <= 256 ? 256 : 512)));
    q.ktiles = K / kBK;
    q.lseg_log2 = std::min(q.log2g, 7);
    q.nseg = K >> q.lseg_log2;
    q.x_stage = (uint32_t)q.TN * kBK * 2u;
    const uint32_t packed = kBM * (kBK * BITS / 8);
    q.x_off = 1024;                                   // after the barriers
    q.p_off = q.x_off + kXStages * q.x_stage;
    const uint32_t budget = 226u * 1024u - 1024u;     // minus alignment slack
    q.pstages = (int)std::min<uint32_t>(kMaxPStages, (budget - q.p_off) / packed);
    const uint32_t smem = 1024u + q.p_off + q.pstages * packed;
    q.idesc = (1u << 4)                        // accumulate in fp32
            | (1u << 7) | (1u << 10)           // A and B are bf16
            | ((uint32_t)(q.TN >> 3) << 17)    // N
            | ((uint32_t)(kBM >> 4) << 24);    // M = 128

    CUtensorMap xmap, wmap;
    {
        const uint64_t dims[2] = {(uint64_t)K, (uint64_t)M};
        const uint64_t strides[1] = {(uint64_t)K * 2};
        const uint32_t box[2] = {64, (uint32_t)q.TN};
        if (!encode_tiled(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    {
        const uint64_t row_bytes = (uint64_t)K * BITS / 8;
        const uint64_t dims[2] = {row_bytes, (uint64_t)N};
        const uint64_t strides[1] = {row_bytes};
        const uint32_t box[2] = {(uint32_t)(kBK * BITS / 8), (uint32_t)kBM};
        if (!encode_tiled(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, w, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    }
    const void *kfn = reinterpret_cast<const void *>(&qmm_kernel<BITS>);
    const int dev = current_device();
    const int sms = dev < 0 ? 0 : device_sm_count(dev);
    if (sms <= 0) return cudaErrorInvalidDevice;
    if (const cudaError_t e = raise_smem_limit(kfn, dev, 227 * 1024); e != cudaSuccess) return e;
    // Split K over a cluster when the row and batch tiles alone leave SMs idle:
    // as many CTAs per tile as fill the SMs (at most 8, whole groups each),
    // provided every cluster can be resident at once and the partial sums fit
    // in the (by then idle) x and code rings.
    const int ntiles = (N + kRowsOut - 1) / kRowsOut, mtiles = (M + q.TN - 1) / q.TN;
    const int tiles = ntiles * mtiles;
    q.kt_unit = std::max(1, group / kBK);
    const int units = q.ktiles / q.kt_unit;
    q.recv_off = q.x_off;
    int ks = 1;
    if (tiles < sms) ks = std::min(std::min(8, sms / tiles), units);
    while (ks > 1) {
        const uint32_t need = (uint32_t)(ks * ((4 + ks - 1) / ks)) * 256u * 64u;
        if (q.recv_off + need <= smem - 1024u && clusters_at_once(kfn, dev, ks, kThreads, smem) >= tiles) break;
        --ks;
    }
    q.ksplit = ks;
    const dim3 grid(ntiles * ks, mtiles);
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)ks;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = ks > 1 ? 2 : 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, qmm_kernel<BITS>, xmap, wmap, q);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

bool qmm_supported(int64_t K, const void *x, const void *w) {
    return K % kBK == 0 && (reinterpret_cast<uintptr_t>(x) & 15u) == 0 &&
           (reinterpret_cast<uintptr_t>(w) & 15u) == 0;
}

uint32_t qmm_timeouts(bool reset) {
    unsigned int v = 0;
    cudaMemcpyFromSymbol(&v, g_qmm_timeouts, sizeof(v));
    if (reset) {
        const unsigned int zero = 0;
        cudaMemcpyToSymbol(g_qmm_timeouts, &zero, sizeof(zero));
    }
    return v;
}

cudaError_t launch_qmm(const uint16_t *x, const uint8_t *w, const uint16_t *scales,
                       const uint16_t *zeros, const uint16_t *bias, uint16_t *y, int64_t M,
                       int64_t K, int64_t N, int bits, int group, cudaStream_t stream) {
    const int k = (int)K, n = (int)N;
    // Grid y is limited to 65535 tiles of up to 128 rows: chunk very large M.
    for (int64_t m0 = 0; m0 < M; m0 += (int64_t)65535 * 128) {
        const int mc = (int)std::min<int64_t>(M - m0, (int64_t)65535 * 128);
        const uint16_t *xc = x + m0 * K;
        uint16_t *yc = y + m0 * N;
        cudaError_t e;
        switch (bits) {
            case 1: e = launch_bits<1>(xc, w, scales, zeros, bias, yc, mc, k, n, group, stream); break;
            case 2: e = launch_bits<2>(xc, w, scales, zeros, bias, yc, mc, k, n, group, stream); break;
            case 3: e = launch_bits<3>(xc, w, scales, zeros, bias, yc, mc, k, n, group, stream); break;
            case 4: e = launch_bits<4>(xc, w, scales, zeros, bias, yc, mc, k, n, group, stream); break;
            case 5: e = launch_bits<5>(xc, w, scales, zeros, bias, yc, mc, k, n, group, stream); break;
            case 6: e = launch_bits<6>(xc, w, scales, zeros, bias, yc, mc, k, n, group, stream); break;
            case 7: e = launch_bits<7>(xc, w, scales, zeros, bias, yc, mc, k, n, group, stream); break;
            default: return cudaErrorInvalidValue;
        }
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace lowbit
