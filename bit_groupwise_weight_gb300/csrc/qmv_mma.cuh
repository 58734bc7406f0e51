// qmv_mma.cuh -- the decode kernel (M <= 8 per launch) on the warp-level
// tensor cores: the weights are streamed once, the b-bit codes become exact
// fp16 tensor-core operands with one LOP3 per code pair, and the fp32
// accumulation of x * q happens inside mma.sync.
//
// Method: ao PR #2167 "metal lowbit kernels: qmv_fast optimization" (Summary,
// bullets 1-3: N x num_groups scales and zeros, codes stored contiguously,
// a fast matrix-vector kernel); torchchat PR #1415 fixes b = 1..7 and
// g = 32..256.  Per output
//     y[m,n] = sum_g s[n,g] * (sum_{k in g} q[n,k] x[m,k]) + z[n,g] * (sum_{k in g} x[m,k]) + bias[n].
//
// Exact tensor-core operands.
//   A (weights): a code q placed at mantissa bit p of the fp16 pattern 0x6400
//   (1024.0) is the fp16 value 1024 + 2^p q, exact for 2^p q < 1024.  A
//   compile-time plan (make_plan) covers a 32-code block with 16 register
//   "pairs" (two fp16 halves = two MMA k-slots); most pairs come from one
//   32-bit window of the block's bit stream with one LOP3 (mask + OR of the
//   magic), the window being a word or one funnel shift.
//   B (x): x is scaled by an exact power of two 2^e per warp and row of x so
//   that its largest magnitude lies in [2^14, 2^15), then multiplied by 2^-p
//   for the slot's code position and rounded to fp16.  This is exact for
//   every x within 2^31 of the largest (smaller ones round to fp16's
//   subnormal grid, an absolute error below 2^-39 of the largest |x|, far
//   under the fp32 rounding of the sum).
//   The product (1024 + 2^p q) * 2^-p x' = q x' + 1024 2^-p x', so for every
//   group the tensor cores return P' = sum q x' + O with O = sum 1024 2^-p x'
//   (computed once per warp from the same fp16 B fragments, on the tensor
//   cores as well: group_sums), and
//     y = 2^-e * sum_g [ s (P' - O) + z X ],   X = sum x' over the group.
//
// Work split.  A consumer warp owns a 256-code slice of K (its B fragments
// stay in registers for the whole kernel) and walks row tiles of 16 weight
// rows (the MMA's 16 rows).  Thread t of a row group holds the codes of two
// 32-code blocks of the slice, at slice codes 128*beta + 32*t + [0, 32).
// The MMA's 8 columns carry (group, row of x) pairs: column c = j*MP + m with
// j a group of the slice (or of the slice's 128-code half, DB = 2) and m a row
// of x; B is zero where a k-slot's code is outside column c's group, so one
// chain of MMAs over the slice yields every group's P' at once and the
// scale/zero epilogue runs once per slice and row tile.
//
// CTA = W consumer warps (K/ks = 256 W, W <= 16), one producer warp and one
// finishing warp.  The producer copies each 16-row tile with 2D TMA tensor
// copies (one box per part of the CTA's K range, as wide as the part plus its
// row padding) into a ring of shared-memory stages (mbarrier completion).
// Consumers reduce a tile's partial sums over the four lanes of a row group
// with shuffles and store them, per warp, into a reduction buffer of the
// cluster's first CTA (DSMEM); its finishing warp adds the ks * W partials of
// every output in a fixed order, adds the bias, rounds once to bf16 and stores
// y (with 4 or 8 rows of x and at most two stages the first CTA's consumers
// finish the last stage together).  When K > 4096 the K range is split over
// the ks CTAs of a thread-block cluster; no global scratch memory is used.
//
// Every mbarrier wait is bounded (about one second) and counts a timeout
// instead of hanging.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <utility>

#include "common.cuh"
#include "ptx.cuh"

namespace lowbit {
namespace mma {

constexpr int kSlice = 256;                  // codes of K per consumer warp
constexpr int kMaxW = 16;                    // consumer warps per CTA
constexpr int kTile = 16;                    // weight rows per tile (MMA M)
constexpr int kMaxStages = 6;
constexpr int kRedBufs = 4;                  // reduction buffers (stages the consumers may run ahead)
constexpr uint32_t kScrRow = 144;            // bytes per lane quarter in the B-fragment table (64 fp16 + pad)
constexpr uint32_t kScrBytes = 4 * kScrRow;
constexpr int kThreads = (kMaxW + 2) * 32;   // consumers + producer + finisher
constexpr uint32_t kMagic = 0x64006400u;     // fp16 pair (1024, 1024)

// ---------------------------------------------------------------------------
// Compile-time unpack plan for a block of 32 b-bit codes (b 32-bit words).
// A window is the 32 bits of the block's stream starting at bit `off` (a word
// when off % 32 == 0, else one funnel shift; negative offsets shift left).  A
// pair is a register of two fp16 halves: the low half holds code lo_code at
// mantissa bit lo_p of window lo_off, the high half code hi_code at bit
// 16 + hi_p of window hi_off (0 <= p <= 10 - b).
// ---------------------------------------------------------------------------
struct PairSpec {
    int lo_off, lo_code, lo_p, hi_off, hi_code, hi_p;
};

template <int B>
struct Plan {
    PairSpec pr[16];
    int p_of[32];
    bool ok;
};

template <int B>
constexpr Plan<B> make_plan() {
    Plan<B> pl{};
    constexpr int lim = 10 - B;
    bool used[32] = {};
    bool win[32 * 7 + 64] = {};              // windows in use, index off + 32
    int np = 0;
    // Greedy: take the window that yields the most single-LOP3 pairs
    // (preferring words and windows already formed), until none is left.
    for (;;) {
        int bk = 0, bpref = -1, bo = 0;
        for (int o = -32; o < 32 * B; ++o) {
            int nl = 0, nh = 0;
            for (int i = 0; i < 32; ++i) {
                if (used[i]) continue;
                const int pl_ = B * i - o, ph = B * i - o - 16;
                if (pl_ >= 0 && pl_ <= lim) ++nl;
                if (ph >= 0 && ph <= lim) ++nh;
            }
            const int k = nl < nh ? nl : nh;
            if (k == 0) continue;
            const int pref = (o % 32 == 0 || win[o + 32]) ? 1 : 0;
            if (k > bk || (k == bk && pref > bpref)) {
                bk = k;
                bpref = pref;
                bo = o;
            }
        }
        if (bk == 0) break;
        win[bo + 32] = true;
        int lows[32] = {}, highs[32] = {}, nl = 0, nh = 0;
        for (int i = 0; i < 32; ++i) {
            if (used[i]) continue;
            const int pl_ = B * i - bo, ph = B * i - bo - 16;
            if (pl_ >= 0 && pl_ <= lim) lows[nl++] = i;
            if (ph >= 0 && ph <= lim) highs[nh++] = i;
        }
        for (int q = 0; q < bk; ++q) {
            pl.pr[np++] = PairSpec{bo, lows[q], B * lows[q] - bo, bo, highs[q], B * highs[q] - bo - 16};
            used[lows[q]] = true;
            used[highs[q]] = true;
        }
    }
    // The rest in twos, each half from its own window (two LOP3).
    int left[32] = {}, nleft = 0;
    for (int i = 0; i < 32; ++i)
        if (!used[i]) left[nleft++] = i;
    for (int q = 0; q + 1 < nleft; q += 2) {
        const int i = left[q], j = left[q + 1];
        int ol = B * i, oh = B * j - 16;
        for (int o = -32; o < 32 * B; ++o)
            if (win[o + 32] && B * i - o >= 0 && B * i - o <= lim) { ol = o; break; }
        for (int o = -32; o < 32 * B; ++o)
            if (win[o + 32] && B * j - o - 16 >= 0 && B * j - o - 16 <= lim) { oh = o; break; }
        win[ol + 32] = true;
        win[oh + 32] = true;
        pl.pr[np++] = PairSpec{ol, i, B * i - ol, oh, j, B * j - oh - 16};
    }
    bool seen[32] = {};
    bool ok = np == 16 && nleft % 2 == 0;
    for (int k = 0; k < np && k < 16; ++k) {
        const PairSpec &s = pl.pr[k];
        if (seen[s.lo_code] || seen[s.hi_code] || s.lo_p < 0 || s.lo_p > lim || s.hi_p < 0 || s.hi_p > lim)
            ok = false;
        seen[s.lo_code] = true;
        seen[s.hi_code] = true;
        pl.p_of[s.lo_code] = s.lo_p;
        pl.p_of[s.hi_code] = s.hi_p;
    }
    for (int i = 0; i < 32; ++i) ok = ok && seen[i];
    pl.ok = ok;
    return pl;
}

template <int B>
inline constexpr Plan<B> kPlan = make_plan<B>();

// The 32 k-slots of a block in fragment order (pair k: slot 2k low half,
// 2k + 1 high half): the code each holds and its mantissa position, packed
// 5 + 4 bits per slot into 16-bit entries of four 64-bit words.
template <int B>
constexpr uint64_t slot_table(int word) {
    uint64_t v = 0;
    for (int i = 0; i < 4; ++i) {
        const int slot = 4 * word + i, k = slot >> 1;
        const PairSpec &s = kPlan<B>.pr[k];
        const int code = (slot & 1) ? s.hi_code : s.lo_code;
        const int pos = (slot & 1) ? s.hi_p : s.lo_p;
        v |= (uint64_t)(code | (pos << 5)) << (16 * i);
    }
    return v;
}

// For codes 8w .. 8w + 7 of a block: the k-slot (fragment order) each one
// occupies, one byte per code, and its mantissa position, 4 bits per code.
template <int B>
constexpr uint64_t code_slots(int w) {
    uint64_t v = 0;
    for (int k = 0; k < 16; ++k) {
        const PairSpec &s = kPlan<B>.pr[k];
        if (s.lo_code / 8 == w) v |= (uint64_t)(2 * k) << (8 * (s.lo_code % 8));
        if (s.hi_code / 8 == w) v |= (uint64_t)(2 * k + 1) << (8 * (s.hi_code % 8));
    }
    return v;
}
template <int B>
constexpr uint32_t code_pos(int w) {
    uint32_t v = 0;
    for (int i = 0; i < 8; ++i) v |= (uint32_t)kPlan<B>.p_of[8 * w + i] << (4 * i);
    return v;
}

// Mantissa positions of the 32 codes, 4 bits each (two 64-bit words), for
// runtime lookups by code index.
template <int B>
constexpr uint64_t p_table(int half) {
    uint64_t v = 0;
    for (int i = 0; i < 16; ++i) v |= (uint64_t)kPlan<B>.p_of[16 * half + i] << (4 * i);
    return v;
}

// Bits [O, O + 32) of the block's little-endian stream (zeros outside it).
template <int B, int O>
__device__ __forceinline__ uint32_t window(const uint32_t (&w)[B]) {
    if constexpr (O <= -32 || O >= 32 * B) {
        return 0u;
    } else if constexpr (O < 0) {
        return w[0] << (-O);
    } else {
        constexpr int wi = O / 32, sh = O % 32;
        if constexpr (sh == 0) return w[wi];
        else if constexpr (wi + 1 < B) return __funnelshift_r(w[wi], w[wi + 1], sh);
        else return w[wi] >> sh;
    }
}

// Pair K of the plan: two codes as the fp16 pair (1024 + 2^plo qlo, 1024 + 2^phi qhi).
template <int B, int K>
__device__ __forceinline__ uint32_t code_pair(const uint32_t (&w)[B]) {
    constexpr PairSpec s = kPlan<B>.pr[K];
    constexpr uint32_t cm = (1u << B) - 1u;
    if constexpr (s.lo_off == s.hi_off) {
        return ptx::and_or_imm<(cm << s.lo_p) | (cm << (16 + s.hi_p))>(window<B, s.lo_off>(w), kMagic);
    } else {
        const uint32_t lo = ptx::and_or_imm<(cm << s.lo_p)>(window<B, s.lo_off>(w), kMagic);
        return ptx::and_or_imm<(cm << (16 + s.hi_p))>(window<B, s.hi_off>(w), lo);
    }
}

// Pair K of the plan as the fp16 pair (2^plo, 2^phi): against B = x' 2^-p in
// the same k-slots the tensor cores return sum x' (the codes' positions undone).
template <int B, int K>
constexpr uint32_t pos_pair() {
    constexpr PairSpec s = kPlan<B>.pr[K];
    return ((uint32_t)(15 + s.hi_p) << 26) | ((uint32_t)(15 + s.lo_p) << 10);
}

// ---------------------------------------------------------------------------
// Launch parameters.
// ---------------------------------------------------------------------------
struct Params {
    const uint16_t *x;
    const uint8_t *w;
    const uint16_t *s;
    const uint16_t *z;
    const uint16_t *bias;
    uint16_t *y;
    int M, N, K, G, log2g;
    int F;               // gated: F outputs; rows [0, F) gate, [F, 2F) up.  0: plain
    int MP;              // x rows per column set (1, 2, 4 or 8), >= M
    int DB;              // column sets per slice: 1, or 2 (one per 128-code half)
    int ks;              // CTAs of a cluster that split K
    int W;               // consumer warps per CTA
    int Kc;              // K per CTA = 256 W
    int RS;              // row tiles per stage
    int NS;              // ring stages
    int tiles;           // row tiles in all (gated: gate and up tiles interleaved)
    int unit;            // tiles per scheduling unit (2 when gated)
    int units_base, units_extra;   // units per cluster: base (+1 for the first `extra`)
    uint32_t row_bytes;  // K * b / 8
    uint32_t crow_bytes; // Kc * b / 8 (one CTA's part of a row)
    int P;               // parts of a CTA's row range, one TMA box of 16 rows each
    uint32_t part_bytes; // crow_bytes / P (whole warp slices)
    uint32_t sstride;    // shared-memory bytes per staged row of a part (padded)
    uint32_t tile_bytes; // one staged tile: P parts x 16 rows x sstride
    uint32_t sz_off;     // within a stage: scales of its tiles (16 x spg fp16 per tile), then zeros
    uint32_t z_off;
    int spg;             // fp16 per staged row of scales / zeros (a padded box row)
    int gcta;            // groups a CTA fetches from: rank * gcta (0: whole rows from group 0)
    uint32_t stage_bytes;
    uint32_t red_off, ring_off;
    uint32_t scr_off;    // per consumer warp: the B-fragment table of one row of x (kScrBytes)
    uint32_t red_floats; // floats of one reduction buffer
};

// Bounded waits that gave up; one counter per translation unit (each bit
// width is compiled on its own), read by mma_timeouts_bits<BITS>.
namespace {
__device__ unsigned int g_mma_timeouts;

uint32_t read_timeouts(bool reset) {
    unsigned int v = 0;
    cudaMemcpyFromSymbol(&v, g_mma_timeouts, sizeof(v));
    if (reset) {
        const unsigned int zero = 0;
        cudaMemcpyToSymbol(g_mma_timeouts, &zero, sizeof(zero));
    }
    return v;
}
}  // namespace

// The b words of a 32-code block from shared memory (byte address + OFF),
// with the widest loads its alignment allows (block offsets are multiples of
// 4 b bytes).
template <int BITS, int OFF>
__device__ __forceinline__ void lds_block_bits(uint32_t addr, uint32_t (&w)[BITS]) {
    if constexpr (BITS == 4) {
        ptx::lds_v4<OFF>(addr, w[0], w[1], w[2], w[3]);
    } else if constexpr (BITS == 2 || BITS == 6) {
        [&]<int... I>(std::integer_sequence<int, I...>) {
            (ptx::lds_v2<OFF + 8 * I>(addr, w[2 * I], w[2 * I + 1]), ...);
        }(std::make_integer_sequence<int, BITS / 2>{});
    } else {
        [&]<int... I>(std::integer_sequence<int, I...>) {
            ((w[I] = ptx::lds_u32_off<OFF + 4 * I>(addr)), ...);
        }(std::make_integer_sequence<int, BITS>{});
    }
}

// First global row of tile lt.
__device__ __forceinline__ int64_t tile_row0(const Params &p, int lt) {
    return p.F == 0 ? (int64_t)lt * kTile : (int64_t)((lt & 1) ? p.F : 0) + (int64_t)(lt >> 1) * kTile;
}

// 8 bf16 of x (one 16-byte load) as fp32.
__device__ __forceinline__ void x8_to_float(const uint4 &u, float (&v)[8]) {
    const uint32_t a[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = bf16_lo(a[i]);
        v[2 * i + 1] = bf16_hi(a[i]);
    }
}

__device__ __forceinline__ float pow2f(int e) {   // 2^e for -126 <= e <= 127
    return __int_as_float((127 + e) << 23);
}

__device__ __forceinline__ uint32_t half2_bits(float lo, float hi) {
    return (uint32_t)__half_as_ushort(__float2half_rn(lo)) |
           ((uint32_t)__half_as_ushort(__float2half_rn(hi)) << 16);
}

__device__ __forceinline__ float lo_half(uint32_t v) { return half_bits_to_float((uint16_t)(v & 0xFFFFu)); }
__device__ __forceinline__ float hi_half(uint32_t v) { return half_bits_to_float((uint16_t)(v >> 16)); }

// 16 MMAs of one staged row tile over the warp's slice: block BETA of rows
// gid (rowa) and gid + 8 (rowb).  With one column set the MMAs alternate
// between two accumulators (shorter dependency chains); with two, block BETA
// accumulates into its own.
template <int BITS, bool DB2, int BETA>
__device__ __forceinline__ void tile_block(uint32_t rowa, uint32_t rowb, const uint32_t (&bq)[16][2],
                                           float (&d0)[4], float (&d1)[4]) {
    uint32_t wa[BITS], wb[BITS];
    lds_block_bits<BITS, BETA * 16 * BITS>(rowa, wa);
    lds_block_bits<BITS, BETA * 16 * BITS>(rowb, wb);
    [&]<int... C>(std::integer_sequence<int, C...>) {
        ((void)[&] {
            const uint32_t a0 = code_pair<BITS, 2 * C>(wa), a1 = code_pair<BITS, 2 * C>(wb);
            const uint32_t a2 = code_pair<BITS, 2 * C + 1>(wa), a3 = code_pair<BITS, 2 * C + 1>(wb);
            constexpr int c = 8 * BETA + C;
            if constexpr ((DB2 ? BETA : (C & 1)) == 0) ptx::mma_16816_f16(d0, a0, a1, a2, a3, bq[c][0], bq[c][1]);
            else ptx::mma_16816_f16(d1, a0, a1, a2, a3, bq[c][0], bq[c][1]);
        }(), ...);
    }(std::make_integer_sequence<int, 8>{});
}

// The group sums of every B column with the B fragments alone: A rows 0..7
// hold 2^p per k-slot (D = X = sum x'), rows 8..15 hold 1024 (D = O = sum
// 1024 2^-p x', the offset P' carries).  Thread (gid, t) thus receives X and
// O of exactly its accumulator columns 2t, 2t + 1, in the same column sets
// as tile_block's d0 / d1.
template <int BITS, bool DB2, int BETA>
__device__ __forceinline__ void group_sums(const uint32_t (&bq)[16][2], float (&d0)[4], float (&d1)[4]) {
    [&]<int... C>(std::integer_sequence<int, C...>) {
        ((void)[&] {
            constexpr uint32_t a0 = pos_pair<BITS, 2 * C>(), a2 = pos_pair<BITS, 2 * C + 1>();
            constexpr int c = 8 * BETA + C;
            if constexpr ((DB2 ? BETA : (C & 1)) == 0) ptx::mma_16816_f16(d0, a0, kMagic, a2, kMagic, bq[c][0], bq[c][1]);
            else ptx::mma_16816_f16(d1, a0, kMagic, a2, kMagic, bq[c][0], bq[c][1]);
        }(), ...);
    }(std::make_integer_sequence<int, 8>{});
}

// Sum of the nsrc partials of one output (stride `step` floats in the
// reduction buffer) as eight independent chains combined in a fixed order:
// the result is the same on every call, and the loads are not serialised
// behind the adds (a cluster of 8 CTAs has up to 128 partials per output).
__device__ __forceinline__ float sum_partials(const float *red, int nsrc, int step) {
    float c[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    int src = 0;
    for (; src + 8 <= nsrc; src += 8) {
#pragma unroll
        for (int j = 0; j < 8; ++j) c[j] += red[(src + j) * step];
    }
    for (; src < nsrc; ++src) c[0] += red[src * step];
    return ((c[0] + c[1]) + (c[2] + c[3])) + ((c[4] + c[5]) + (c[6] + c[7]));
}

// The outputs of one reduction stage (tiles lta .. lta + nts - 1), summed over
// their nsrc partials by threads th = 0 .. nth - 1 (nth a multiple of 32), add
// the bias, round once to bf16 and store y.  When threads outnumber outputs,
// Q = 2, 4 or 8 neighbouring lanes share an output: lane q of the group adds
// partials q, q + Q, ... and a butterfly combines the group.  Every warp runs
// the same number of passes (the shuffles need whole warps); the order of the
// additions is fixed, so results are the same on every call.
template <int MP>
__device__ __forceinline__ void finish_stage(const Params &p, const float *red, int lta, int nts, int nsrc,
                                             int th, int nth) {
    const int step = p.RS * kTile * MP;                       // floats between two sources' partials
    const bool gated = p.F != 0;
    const int nout = (gated ? nts / 2 : nts) * kTile * MP;
    int Q = 1;
    while (Q < 8 && 2 * Q <= nsrc && 2 * Q * nout <= nth) Q *= 2;
    const int lane = th & 31, q = lane & (Q - 1);
    auto psum = [&](const float *a0) {
        float a;
        if (Q == 1) {
            a = sum_partials(a0, nsrc, step);
        } else {
            a = 0.f;
            for (int src = q; src < nsrc; src += Q) a += a0[src * step];
            for (int o = 1; o < Q; o <<= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
        }
        return a;
    };
    for (int ob = (th >> 5) * (32 / Q); ob < nout; ob += nth / Q) {
        const int o = ob + lane / Q;
        const bool valid = o < nout && q == 0;
        const int oo = o < nout ? o : 0;
        const int rr = oo / MP, m = oo % MP;
        if (!gated) {
            const int row = (lta + rr / kTile) * kTile + rr % kTile;
            float a = psum(red + rr * MP + m);
            if (valid && m < p.M && row < p.N) {
                if (p.bias != nullptr) a += half_bits_to_float(p.bias[row]);
                p.y[(int64_t)m * p.N + row] = float_to_bf16_bits(a);
            }
        } else {
            // Tile 2i of the stage is a gate tile, 2i + 1 its up tile.
            const int ip = rr / kTile, r = rr % kTile;
            const int f = ((lta >> 1) + ip) * kTile + r;
            const int ra = (2 * ip) * kTile + r, ru = ra + kTile;
            float a = psum(red + ra * MP + m);
            float u = psum(red + ru * MP + m);
            if (valid && m < p.M && f < p.F) {
                if (p.bias != nullptr) {
                    a += half_bits_to_float(p.bias[f]);
                    u += half_bits_to_float(p.bias[p.F + f]);
                }
                p.y[(int64_t)m * p.F + f] = float_to_bf16_bits(silu_mul(a, u));
            }
        }
    }
}

// Bounded waits and arrivals on the reduction barriers: cluster scope when
// the K range is split over a cluster, CTA scope (no fence) otherwise.
__device__ __forceinline__ bool red_wait(bool cluster, uint32_t bar, uint32_t parity) {
    return cluster ? ptx::mbar_wait_cluster(bar, parity, &g_mma_timeouts)
                   : ptx::mbar_wait(bar, parity, &g_mma_timeouts);
}
__device__ __forceinline__ void red_arrive(bool cluster, uint32_t bar) {
    if (cluster) ptx::mbar_arrive_cluster(bar);
    else ptx::mbar_arrive(bar);
}

template <int BITS, int MP, bool DB2>
__global__ void __launch_bounds__(kThreads, 1)
qmv_mma_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap smap,
               const __grid_constant__ CUtensorMap zmap, const Params p) {
    static_assert(MP == 1 || MP == 2 || MP == 4 || MP == 8, "rows of x per column set");
    static_assert(!(DB2 && MP == 1), "one row of x always fits one column set");
    constexpr int NB = DB2 ? 2 : 1;                        // column sets per slice
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int W = p.W;
    const uint32_t sb = ptx::smem_u32(smem);
    const uint32_t full0 = sb, empty0 = sb + 8 * kMaxStages;
    const uint32_t rfull0 = sb + 16 * kMaxStages, rfree0 = rfull0 + 8 * kRedBufs;
    const int ks = p.ks;
    const bool clustered = ks > 1;
    const int rank = clustered ? (int)ptx::cluster_ctarank() : 0;
    const int cl = blockIdx.x / ks;
    const int u0 = cl * p.units_base + min(cl, p.units_extra);
    const int nu = p.units_base + (cl < p.units_extra ? 1 : 0);
    const int lt0 = u0 * p.unit;
    const int ntl = max(0, min(nu * p.unit, p.tiles - lt0));    // this cluster's tiles
    const int nst = (ntl + p.RS - 1) / p.RS;                      // and stages
    // With M >= 4 rows of x a stage has 64+ outputs per tile, and the
    // finishing warp's last stage (cold code, once per call) was the call's
    // tail: there the consumers finish the last stage together when a call has
    // at most two stages (o at M = 8: 7.9 -> 6.9 us).  With more stages the
    // finishing warp's code is warm by the last one and it stays faster.
    const bool consumers_finish = MP >= 4 && nst >= 1 && nst <= 2;

    ptx::pdl_launch_dependents();
    if (tid == 0) {
        for (int i = 0; i < p.NS; ++i) {
            ptx::mbar_init(full0 + 8 * i, 1);
            ptx::mbar_init(empty0 + 8 * i, (uint32_t)W);
        }
        for (int b = 0; b < kRedBufs; ++b) {
            ptx::mbar_init(rfull0 + 8 * b, (uint32_t)(ks * W));
            ptx::mbar_init(rfree0 + 8 * b, 1);
        }
        ptx::fence_mbar_init();
    }
    if (clustered) ptx::cluster_sync();
    else __syncthreads();

    if (warp == W) {
        // ---------------- producer: every lane issues row copies.  It reads
        // only packed weights, scales and zeros, which the previous kernel in
        // the stream does not write (the library's interface requires it), so
        // it starts at once: the first stages arrive while the consumers
        // wait for that kernel and prepare x.
        const uint64_t pol = ptx::policy_evict_first();
        int s = 0;
        for (; s < nst; ++s) {
            const int st = s % p.NS;
            if (s >= p.NS && !ptx::mbar_wait(empty0 + 8 * st, ((s / p.NS) - 1) & 1, &g_mma_timeouts)) break;
            const int lta = lt0 + s * p.RS;
            const int nts = min(p.RS, lt0 + ntl - lta);
            const uint32_t full = full0 + 8 * st;
            const uint32_t dst0 = sb + p.ring_off + (uint32_t)st * p.stage_bytes;
            const uint32_t tsz = (uint32_t)(kTile * p.spg * 2);        // bytes of one tile's scales
            // Weights: one 2D tensor copy per part of a tile, a box of 16 rows
            // x sstride bytes (8-byte elements) from byte rank * crow + j *
            // part of the rows: the bytes past the part (the row padding) are
            // the next part's or next row's, or zeros past the matrix, and
            // rows past the matrix read as zero.  Scales and zeros: one 2D
            // tensor copy each per tile, a box of 16 rows x spg fp16 from
            // group rank * gcta (columns past its groups read as zero).
            const uint32_t bytes = (uint32_t)nts * (p.tile_bytes + 2u * tsz);
            if (lane == 0) ptx::mbar_arrive_expect_tx(full, bytes);
            __syncwarp();
            for (int i = 0; i < nts; ++i) {
                const int g0 = (int)tile_row0(p, lta + i);
                if (lane < p.P)
                    ptx::tma_load_2d_hint(dst0 + (uint32_t)i * p.tile_bytes + (uint32_t)(lane * kTile) * p.sstride,
                                          &wmap, (int)((rank * p.crow_bytes + (uint32_t)lane * p.part_bytes) >> 3),
                                          g0, full, pol);
                if (lane == 31) {
                    ptx::tma_load_2d_hint(dst0 + p.sz_off + i * tsz, &smap, rank * p.gcta, g0, full, pol);
                    ptx::tma_load_2d_hint(dst0 + p.z_off + i * tsz, &zmap, rank * p.gcta, g0, full, pol);
                }
            }
        }
        // Stay until this warp's last copies have landed.
        for (int i = max(0, s - p.NS); i < s; ++i)
            if (!ptx::mbar_wait(full0 + 8 * (i % p.NS), (i / p.NS) & 1, &g_mma_timeouts)) break;
    } else if (warp == W + 1) {
        // ---------------- finisher (first CTA of the cluster): sum the partials
        // of every stage (but the last when the consumers finish it).
        ptx::pdl_wait();            // y and bias: only after the previous kernel in the stream
        if (rank == 0) {
            const int nsrc = ks * W;
            const int rows_stage = p.RS * kTile;
            bool ok = true;
            for (int s = 0; s + (consumers_finish ? 1 : 0) < nst; ++s) {
                const int buf = s % kRedBufs;
                if (ok) ok = red_wait(clustered, rfull0 + 8 * buf, (s / kRedBufs) & 1);
                const int lta = lt0 + s * p.RS;
                const int nts = min(p.RS, lt0 + ntl - lta);
                const float *red = reinterpret_cast<const float *>(smem + p.red_off) + (size_t)buf * p.red_floats;
                if (ok && p.F == 0) {
                    for (int o = lane; o < nts * kTile * MP; o += 32) {
                        const int rr = o / MP, m = o % MP;
                        const int row = (lta + rr / kTile) * kTile + rr % kTile;
                        if (m < p.M && row < p.N) {
                            float a = sum_partials(red + rr * MP + m, nsrc, rows_stage * MP);
                            if (p.bias != nullptr) a += half_bits_to_float(p.bias[row]);
                            p.y[(int64_t)m * p.N + row] = float_to_bf16_bits(a);
                        }
                    }
                } else if (ok) {
                    // Gated: tile 2i of the stage is a gate tile, 2i + 1 its up tile.
                    for (int o = lane; o < (nts / 2) * kTile * MP; o += 32) {
                        const int rr = o / MP, m = o % MP;
                        const int ip = rr / kTile, r = rr % kTile;
                        const int f = ((lta >> 1) + ip) * kTile + r;
                        if (m < p.M && f < p.F) {
                            const int ra = (2 * ip) * kTile + r, ru = ra + kTile;
                            float a = sum_partials(red + ra * MP + m, nsrc, rows_stage * MP);
                            float u = sum_partials(red + ru * MP + m, nsrc, rows_stage * MP);
                            if (p.bias != nullptr) {
                                a += half_bits_to_float(p.bias[f]);
                                u += half_bits_to_float(p.bias[p.F + f]);
                            }
                            p.y[(int64_t)m * p.F + f] = float_to_bf16_bits(silu_mul(a, u));
                        }
                    }
                }
                // Hand the buffer back to every CTA of the cluster, when a later
                // stage reuses it (stage s + kRedBufs).  The arrive releases this
                // warp's stores of y as well, so it is not made when nothing
                // waits for it: it would only lengthen the call's tail.
                if (s + kRedBufs < nst) {
                    __syncwarp();
                    if (lane < ks)
                        red_arrive(clustered, clustered ? ptx::mapa_shared(rfree0 + 8 * buf, (uint32_t)lane) : rfree0 + 8 * buf);
                }
            }
        }
    } else {
        // ---------------- consumers.
        ptx::pdl_wait();            // x may come from the previous kernel in the stream
        const int gid = lane >> 2, t = lane & 3;
        const int M = p.M;
        const int kw0 = rank * p.Kc + warp * kSlice;          // first code of this warp's slice
        const int gsl = max(1, kSlice >> p.log2g);            // groups per slice
        const int gpb = max(1, 128 >> p.log2g);               // groups per 128-code half
        const int gpc = DB2 ? gpb : gsl;                      // groups per column set
        const int gw0 = kw0 >> p.log2g;                       // first group of the slice
        const int mcol = gid % MP, jcol = gid / MP;           // this thread's B column
        const bool bvalid = mcol < M && jcol < gpc;

        // Columns 2t + e of this thread's accumulators: x row me[e] and group
        // j = (2t + e) / MP of each column set.  Unused columns read the
        // slice's first groups (finite data) and add zero.
        int gk[NB][2];
        int me[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int col = 2 * t + e;
            me[e] = col % MP;
#pragma unroll
            for (int bb = 0; bb < NB; ++bb) {
                const int j = col / MP;
                gk[bb][e] = gw0 + ((me[e] < M && j < gpc) ? bb * gpb + j : 0);
            }
        }
        // MP == 1: columns 2t, 2t + 1 are adjacent groups (both used or both
        // unused when the slice has two or more groups), read as one word.
        const bool pair_sz = MP == 1 && gsl >= 2;
        const int gbase = rank * p.gcta;                      // first group of a staged scale row
        const int gpair = gw0 - gbase + ((MP == 1 && 2 * t < gsl) ? 2 * t : 0);

        // Per x row m: the scale 2^e of the warp's slice and the B fragments of
        // the threads whose column holds row m.  Lane l converts the slice's
        // codes [8l, 8l + 8) (block l / 16 of lane quarter (l / 4) % 4) and
        // writes them, in fragment order, to the warp's table; a thread reads
        // its 64 fp16 values back as 32 words and keeps the blocks of its
        // column group.  The group sums X and O follow from the fragments on
        // the tensor cores (group_sums).
        float isc[2] = {1.f, 1.f};
        uint32_t bq[16][2];
        uint8_t *scr = smem + p.scr_off + (size_t)warp * kScrBytes;
        const int lw = lane & 3;                               // which 8 codes of the lane's block
        const uint64_t slots = lw == 0 ? code_slots<BITS>(0) : lw == 1 ? code_slots<BITS>(1)
                             : lw == 2 ? code_slots<BITS>(2) : code_slots<BITS>(3);
        const uint32_t poss = lw == 0 ? code_pos<BITS>(0) : lw == 1 ? code_pos<BITS>(1)
                            : lw == 2 ? code_pos<BITS>(2) : code_pos<BITS>(3);
        uint16_t *srow = reinterpret_cast<uint16_t *>(scr + ((lane >> 2) & 3) * kScrRow) + 32 * (lane >> 4);
        // x rows come through a queue of up to four loads in flight (one load
        // latency for M <= 4 instead of M); row m is always xr[0].
        constexpr int kQ = MP < 4 ? MP : 4;
        const uint16_t *xlane = p.x + kw0 + 8 * lane;
        uint4 xr[kQ];
#pragma unroll
        for (int m = 0; m < kQ; ++m)
            xr[m] = m < M ? __ldg(reinterpret_cast<const uint4 *>(xlane + (int64_t)m * p.K)) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll 1
        for (int m = 0; m < MP; ++m) {
            float xv[8];
            x8_to_float(xr[0], xv);
#pragma unroll
            for (int j = 0; j + 1 < kQ; ++j) xr[j] = xr[j + 1];
            if constexpr (MP > kQ)
                xr[kQ - 1] = m + kQ < M ? __ldg(reinterpret_cast<const uint4 *>(xlane + (int64_t)(m + kQ) * p.K))
                                        : make_uint4(0u, 0u, 0u, 0u);
            float mx = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) mx = fmaxf(mx, fabsf(xv[i]));
            // A non-negative float's bits order like its value: one warp-wide
            // integer maximum.
            mx = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(mx)));
            int ex = 0;
            if (mx > 0.f) {
                (void)frexpf(mx, &ex);                   // mx = f 2^ex, f in [0.5, 1)
                ex = min(126, max(-126, 15 - ex));       // mx 2^ex in [2^14, 2^15)
            }
            const float sc = pow2f(ex);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int pp = (int)((poss >> (4 * i)) & 15u);
                srow[(slots >> (8 * i)) & 255u] = __half_as_ushort(__float2half_rn(xv[i] * sc * pow2f(-pp)));
            }
            if (m == me[0]) isc[0] = pow2f(-ex);
            if (m == me[1]) isc[1] = pow2f(-ex);
            __syncwarp();
            if (m == mcol) {
                const uint4 *tb = reinterpret_cast<const uint4 *>(scr + t * kScrRow);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint4 u = tb[i];
                    bq[2 * i][0] = u.x; bq[2 * i][1] = u.y; bq[2 * i + 1][0] = u.z; bq[2 * i + 1][1] = u.w;
                }
            }
            __syncwarp();
        }
        // Keep only the blocks whose codes lie in this thread's column group (a
        // 32-code block never straddles a group).
#pragma unroll
        for (int beta = 0; beta < 2; ++beta) {
            const int jt = (DB2 ? beta * gpb : 0) + jcol;
            const bool keep = bvalid && ((128 * beta + 32 * t) >> p.log2g) == jt;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                bq[8 * beta + c][0] = keep ? bq[8 * beta + c][0] : 0u;
                bq[8 * beta + c][1] = keep ? bq[8 * beta + c][1] : 0u;
            }
        }
        // X and O of this thread's columns (zero for unused columns, whose B
        // fragments are zero).
        float X[NB][2], O[NB][2];
        {
            float g0[4] = {0.f, 0.f, 0.f, 0.f}, g1[4] = {0.f, 0.f, 0.f, 0.f};
            group_sums<BITS, DB2, 0>(bq, g0, g1);
            group_sums<BITS, DB2, 1>(bq, g0, g1);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                if constexpr (DB2) {
                    X[0][e] = g0[e];
                    O[0][e] = g0[2 + e];
                    X[NB - 1][e] = g1[e];
                    O[NB - 1][e] = g1[2 + e];
                } else {
                    X[0][e] = g0[e] + g1[e];
                    O[0][e] = g0[2 + e] + g1[2 + e];
                }
            }
        }

        // Shared-memory byte offsets, fixed per thread: row gid's first block
        // within a staged tile (the warp's slice lies in part warp / (W / P)),
        // row gid + 8 from there, a tile's stride; the
        // scales of rows gid and gid + 8 within a tile's scale box (the zeros
        // sit zdelta bytes after their scales); this thread's slot in a
        // reduction buffer of the cluster's first CTA (this CTA's own when
        // there is no cluster).
        const int wpp = W / p.P;                                  // warps per part
        const uint32_t a_off = (uint32_t)((warp / wpp) * kTile + gid) * p.sstride +
                               (uint32_t)(warp % wpp) * (kSlice * BITS / 8) + (uint32_t)((32 * t * BITS) >> 3);
        const uint32_t b_off = 8u * p.sstride;
        const uint32_t t_str = p.tile_bytes;
        const uint32_t tsz = (uint32_t)(kTile * p.spg * 2);
        const uint32_t zdelta = p.z_off - p.sz_off;
        const uint32_t r8 = (uint32_t)(16 * p.spg);                      // 8 scale rows, bytes
        const uint32_t srow0 = (uint32_t)(2 * gid * p.spg);
        uint32_t so[NB][2];
#pragma unroll
        for (int bb = 0; bb < NB; ++bb)
#pragma unroll
            for (int e = 0; e < 2; ++e) so[bb][e] = srow0 + 2u * (uint32_t)(gk[bb][e] - gbase);
        const uint32_t so_pair = srow0 + 2u * (uint32_t)gpair;
        const uint32_t red_base = (clustered ? ptx::mapa_shared(sb + p.red_off, 0u) : sb + p.red_off) +
                                  4u * (uint32_t)((rank * W + warp) * p.RS * kTile * MP);
        const uint32_t red_buf_bytes = 4u * p.red_floats;
        const uint32_t rfull_leader = clustered ? ptx::mapa_shared(rfull0, 0u) : rfull0;

        bool ok = true;
        uint32_t stage = sb + p.ring_off, fpar = 0;       // ring stage of step s, its index and parity
        int st = 0;
        for (int s = 0; s < nst; ++s) {
            const int buf = s % kRedBufs;
            if (ok) ok = ptx::mbar_wait(full0 + 8 * st, fpar, &g_mma_timeouts);
            if (ok && s >= kRedBufs) ok = red_wait(clustered, rfree0 + 8 * buf, ((s / kRedBufs) - 1) & 1);
            const int nts = min(p.RS, ntl - s * p.RS);
            uint32_t tile = stage + a_off, sz = stage + p.sz_off;
            uint32_t red = red_base + (uint32_t)buf * red_buf_bytes;
            for (int i = 0; i < nts && ok; ++i, tile += t_str, sz += tsz, red += 4u * kTile * MP) {
                // Scales and zeros of rows gid, gid + 8 (read before the MMAs).
                float sv[2][NB][2], zv[2][NB][2];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const uint32_t rs = sz + (r ? r8 : 0u);
                    if (pair_sz) {
                        const uint32_t s2 = ptx::lds_u32(rs + so_pair);
                        const uint32_t z2 = ptx::lds_u32(rs + so_pair + zdelta);
                        sv[r][0][0] = lo_half(s2); sv[r][0][1] = hi_half(s2);
                        zv[r][0][0] = lo_half(z2); zv[r][0][1] = hi_half(z2);
                    } else {
#pragma unroll
                        for (int bb = 0; bb < NB; ++bb)
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                if (MP >= 2 && e == 1) {      // same group as column 2t
                                    sv[r][bb][1] = sv[r][bb][0];
                                    zv[r][bb][1] = zv[r][bb][0];
                                } else {
                                    sv[r][bb][e] = half_bits_to_float(ptx::lds_u16(rs + so[bb][e]));
                                    zv[r][bb][e] = half_bits_to_float(ptx::lds_u16(rs + so[bb][e] + zdelta));
                                }
                            }
                    }
                }
                float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
                tile_block<BITS, DB2, 0>(tile, tile + b_off, bq, d0, d1);
                tile_block<BITS, DB2, 1>(tile, tile + b_off, bq, d0, d1);
                float acc[2][2];
#pragma unroll
                for (int r = 0; r < 2; ++r)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        if constexpr (DB2) {
                            acc[r][e] = fmaf(sv[r][0][e], d0[2 * r + e] - O[0][e],
                                        fmaf(zv[r][0][e], X[0][e],
                                        fmaf(sv[r][1][e], d1[2 * r + e] - O[1][e], zv[r][1][e] * X[1][e])));
                        } else {
                            acc[r][e] = fmaf(sv[r][0][e], (d0[2 * r + e] + d1[2 * r + e]) - O[0][e],
                                             zv[r][0][e] * X[0][e]);
                        }
                    }
                // Sum over the lanes that hold the same (row, x row), then store
                // this warp's partial sums, in units of x (times 2^-e).
                auto put = [&](int row, int m, float v) {
                    const uint32_t a = red + 4u * (uint32_t)(row * MP + m);
                    if (clustered) ptx::st_cluster_f32(a, v);
                    else ptx::sts_f32(a, v);
                };
                if constexpr (MP == 1) {
                    float v0 = acc[0][0] + acc[0][1], v1 = acc[1][0] + acc[1][1];
                    v0 += __shfl_xor_sync(0xffffffffu, v0, 1);
                    v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
                    v0 += __shfl_xor_sync(0xffffffffu, v0, 2);
                    v1 += __shfl_xor_sync(0xffffffffu, v1, 2);
                    if (t < 2) put(gid + 8 * t, 0, (t ? v1 : v0) * isc[0]);
                } else if constexpr (MP == 2) {
#pragma unroll
                    for (int r = 0; r < 2; ++r)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            acc[r][e] += __shfl_xor_sync(0xffffffffu, acc[r][e], 1);
                            acc[r][e] += __shfl_xor_sync(0xffffffffu, acc[r][e], 2);
                        }
                    const int r = t >> 1, e = t & 1;
                    const float v = r ? (e ? acc[1][1] : acc[1][0]) : (e ? acc[0][1] : acc[0][0]);
                    put(gid + 8 * r, e, v * isc[e]);
                } else if constexpr (MP == 4) {
#pragma unroll
                    for (int r = 0; r < 2; ++r)
#pragma unroll
                        for (int e = 0; e < 2; ++e) acc[r][e] += __shfl_xor_sync(0xffffffffu, acc[r][e], 2);
                    const int r = t >> 1;
#pragma unroll
                    for (int e = 0; e < 2; ++e) put(gid + 8 * r, me[e], (r ? acc[1][e] : acc[0][e]) * isc[e]);
                } else {
#pragma unroll
                    for (int r = 0; r < 2; ++r)
#pragma unroll
                        for (int e = 0; e < 2; ++e) put(gid + 8 * r, me[e], acc[r][e] * isc[e]);
                }
            }
            __syncwarp();
            if (lane == 0) {
                ptx::mbar_arrive(empty0 + 8 * st);
                red_arrive(clustered, rfull_leader + 8 * buf);
            }
            stage += p.stage_bytes;
            if (++st == p.NS) {
                st = 0;
                stage = sb + p.ring_off;
                fpar ^= 1u;
            }
        }
        // The last stage, when the consumers finish it: the first CTA's
        // consumers meet at a named barrier (the CTA's own partials are then
        // written, and no warp polls while others still compute), await a
        // cluster's other CTAs on the stage's barrier, and sum the stage's
        // outputs together.  No stage follows, so its buffer is not handed
        // back.
        if (consumers_finish && rank == 0) {
            const int s = nst - 1, buf = s % kRedBufs;
            ptx::named_sync(1, (uint32_t)W * 32u);
            if (ok && clustered) ok = red_wait(true, rfull0 + 8 * buf, (s / kRedBufs) & 1);
            ok = __all_sync(0xffffffffu, ok);
            const int lta = lt0 + s * p.RS;
            const int nts = min(p.RS, lt0 + ntl - lta);
            const float *red = reinterpret_cast<const float *>(smem + p.red_off) + (size_t)buf * p.red_floats;
            if (ok) finish_stage<MP>(p, red, lta, nts, ks * W, warp * 32 + lane, W * 32);
        }
    }
    if (clustered) ptx::cluster_sync();
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
struct LaunchPlan {
    bool ok = false;
    Params prm{};
    CUtensorMap wmap, smap, zmap;
    int grid = 0;
    int threads = 0;
    uint32_t smem = 0;
};

// Largest rows of x one launch takes for group size g (columns = groups x rows <= 8 per column set).
inline int max_rows(int group) { return group == 32 ? 2 : (group == 64 ? 4 : 8); }

// Shared-memory padding after each staged row: the smallest modelled bank
// conflicts for the consumers' reads (row gid of lane 4 gid + t reads its two
// blocks at slice bytes (128 beta + 32 t) b / 8).
uint32_t row_pad(int bits, uint32_t crow_bytes);
// Padded length (fp16) of a staged row of `groups` scales, from a model of the
// epilogue's reads (see qmv_mma_host.cu), and 2D tensor-map encoding.
int sz_pitch(int groups, int gsl, int MP, int W);
bool encode_2d(CUtensorMap *map, CUtensorMapDataType type, const void *base, uint64_t inner, uint64_t rows,
               uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows);

// Clusters of ks CTAs (smem bytes, `threads` threads each) resident at once on device dev.
int max_clusters(const void *fn, int dev, int ks, uint32_t smem, int threads);

// Kernel variant for x rows per column set and column sets per slice.
template <int BITS>
const void *kernel_ptr(int MP, bool db2) {
    switch (MP) {
        case 1: return db2 ? nullptr : reinterpret_cast<const void *>(&qmv_mma_kernel<BITS, 1, false>);
        case 2: return db2 ? reinterpret_cast<const void *>(&qmv_mma_kernel<BITS, 2, true>)
                           : reinterpret_cast<const void *>(&qmv_mma_kernel<BITS, 2, false>);
        case 4: return db2 ? reinterpret_cast<const void *>(&qmv_mma_kernel<BITS, 4, true>)
                           : reinterpret_cast<const void *>(&qmv_mma_kernel<BITS, 4, false>);
        case 8: return db2 ? reinterpret_cast<const void *>(&qmv_mma_kernel<BITS, 8, true>)
                           : reinterpret_cast<const void *>(&qmv_mma_kernel<BITS, 8, false>);
        default: return nullptr;
    }
}
template <int BITS>
LaunchPlan plan_launch(const uint16_t *x, const uint8_t *w, const uint16_t *s, const uint16_t *z,
                       const uint16_t *bias, uint16_t *y, int M, int K, int N, int group, int F) {
    LaunchPlan pl;
    static_assert(kPlan<BITS>.ok, "unpack plan must cover every code exactly once");
    if (M < 1 || M > max_rows(group) || K % kSlice != 0) return pl;
    if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(w) & 15u) ||
        (reinterpret_cast<uintptr_t>(s) & 15u) || (reinterpret_cast<uintptr_t>(z) & 15u))
        return pl;
    if (F != 0 && F % kTile != 0) return pl;
    Params &q = pl.prm;
    q.x = x; q.w = w; q.s = s; q.z = z; q.bias = bias; q.y = y;
    q.M = M; q.N = N; q.K = K; q.G = K / group; q.log2g = __builtin_ctz((unsigned)group);
    q.F = F;
    q.MP = M <= 1 ? 1 : (M <= 2 ? 2 : (M <= 4 ? 4 : 8));
    const int gsl = std::max(1, kSlice / group);
    q.DB = gsl * q.MP <= 8 ? 1 : 2;
    int ks = 0;
    for (int k = 1; k <= 8; ++k)
        if (K % (kSlice * k) == 0 && K / k <= kSlice * kMaxW) { ks = k; break; }
    if (ks == 0) return pl;
    q.ks = ks;
    q.Kc = K / ks;
    q.W = q.Kc / kSlice;
    q.unit = F != 0 ? 2 : 1;
    q.tiles = F != 0 ? 2 * (F / kTile) : (N + kTile - 1) / kTile;
    q.row_bytes = (uint32_t)((int64_t)K * BITS / 8);
    q.crow_bytes = (uint32_t)((int64_t)q.Kc * BITS / 8);
    // A part of a CTA's row range is whole warp slices and, with its padding,
    // fits one TMA box row (at most 256 elements of 8 bytes): the fewest parts.
    for (int pp = 1; pp <= q.W && q.P == 0; ++pp) {
        if (q.W % pp != 0) continue;
        const uint32_t part = q.crow_bytes / (uint32_t)pp;
        const uint32_t pad = row_pad(BITS, part);
        if (part + pad <= 256u * 8u) {
            q.P = pp;
            q.part_bytes = part;
            q.sstride = part + pad;
        }
    }
    if (q.P == 0) return pl;
    q.tile_bytes = (uint32_t)q.P * kTile * q.sstride;
    // Scales and zeros: a CTA fetches its own groups when they start on a
    // 16-byte boundary, else whole rows; the box row is padded (over-read)
    // so that the epilogue's reads of 16 rows fall into distinct banks.
    if ((q.G * 2) % 16 != 0) return pl;                     // rows of scales must be 16-byte multiples
    const int gc = q.Kc / group;
    q.gcta = (ks == 1 || (gc * 2) % 16 == 0) ? gc : 0;
    q.spg = sz_pitch(q.gcta != 0 ? gc : q.G, std::max(1, kSlice / group), q.MP, q.W);
    if (q.spg > 256) return pl;
    constexpr uint32_t kBudget = 227u * 1024u;
    constexpr uint32_t kBars = 16u * kMaxStages + 16u * kRedBufs;
    for (int rs = 8; rs >= q.unit; rs -= q.unit) {
        const uint32_t stage = (uint32_t)rs * (q.tile_bytes + kTile * 4u * (uint32_t)q.spg);
        // Larger stages cost fewer per-stage barrier round trips: up to 80 KB
        // (two b = 4 tiles at K = 4096 as two stages measured 8% faster than
        // one-tile stages as five).
        if (rs > q.unit && stage > 80u * 1024u) continue;
        const uint32_t red_floats = (uint32_t)(ks * q.W * rs * kTile * q.MP);
        const uint32_t red_off = (kBars + 127u) & ~127u;
        const uint32_t scr_off = (red_off + (uint32_t)kRedBufs * red_floats * 4u + 127u) & ~127u;
        const uint32_t ring_off = (scr_off + (uint32_t)q.W * kScrBytes + 127u) & ~127u;
        if (ring_off >= kBudget) continue;
        const int ns = (int)std::min<uint32_t>(kMaxStages, (kBudget - ring_off) / stage);
        if (ns < 2) continue;
        q.RS = rs;
        q.NS = ns;
        q.stage_bytes = stage;
        q.sz_off = (uint32_t)rs * q.tile_bytes;
        q.z_off = q.sz_off + (uint32_t)rs * kTile * (uint32_t)q.spg * 2u;
        q.red_floats = red_floats;
        q.red_off = red_off;
        q.scr_off = scr_off;
        q.ring_off = ring_off;
        pl.smem = ring_off + (uint32_t)ns * stage;
        break;
    }
    if (q.RS == 0) return pl;
    const int rows_total = F != 0 ? 2 * F : N;
    if (!encode_2d(&pl.wmap, CU_TENSOR_MAP_DATA_TYPE_UINT64, w, (uint64_t)(q.row_bytes / 8u), (uint64_t)rows_total,
                   (uint64_t)q.row_bytes, q.sstride / 8u, kTile) ||
        !encode_2d(&pl.smap, CU_TENSOR_MAP_DATA_TYPE_UINT16, s, (uint64_t)q.G, (uint64_t)rows_total,
                   (uint64_t)q.G * 2, (uint32_t)q.spg, kTile) ||
        !encode_2d(&pl.zmap, CU_TENSOR_MAP_DATA_TYPE_UINT16, z, (uint64_t)q.G, (uint64_t)rows_total,
                   (uint64_t)q.G * 2, (uint32_t)q.spg, kTile))
        return pl;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return pl;
    const void *fn = kernel_ptr<BITS>(q.MP, q.DB == 2);
    if (fn == nullptr) return pl;
    if (raise_smem_limit(fn, dev, 227 * 1024) != cudaSuccess) return pl;
    const int units = q.tiles / q.unit;
    pl.threads = (q.W + 2) * 32;
    const int maxc = max_clusters(fn, dev, ks, pl.smem, pl.threads);
    if (maxc < 1) return pl;
    const int clusters = std::max(1, std::min(units, maxc));
    q.units_base = units / clusters;
    q.units_extra = units % clusters;
    pl.grid = clusters * ks;
    pl.ok = true;
    return pl;
}

template <int BITS>
cudaError_t launch_plan(const LaunchPlan &pl, cudaStream_t stream) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(pl.grid);
    cfg.blockDim = dim3(pl.threads);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)pl.prm.ks;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pl.prm.ks > 1 ? 2 : 1;
    using KFn = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const Params);
    const KFn fn = reinterpret_cast<KFn>(const_cast<void *>(kernel_ptr<BITS>(pl.prm.MP, pl.prm.DB == 2)));
    if (fn == nullptr) return cudaErrorInvalidValue;
    cudaError_t e = cudaLaunchKernelEx(&cfg, fn, pl.wmap, pl.smap, pl.zmap, pl.prm);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// y = x W^T (+ bias) for M rows of x, in launches of up to max_rows(group)
// rows; F > 0: the gated form.  Returns cudaErrorNotSupported (nothing
// launched) when the shape is not one this kernel takes.
template <int BITS>
cudaError_t launch_rows(const uint16_t *x, const uint8_t *w, const uint16_t *s, const uint16_t *z,
                        const uint16_t *bias, uint16_t *y, int64_t M, int K, int N, int group, int F,
                        cudaStream_t stream) {
    const int64_t ys = F != 0 ? F : N;
    const int chunk = max_rows(group);
    LaunchPlan first = plan_launch<BITS>(x, w, s, z, bias, y, (int)std::min<int64_t>(M, chunk), K, N, group, F);
    if (!first.ok) return cudaErrorNotSupported;
    for (int64_t m0 = 0; m0 < M; m0 += chunk) {
        const int mc = (int)std::min<int64_t>(chunk, M - m0);
        LaunchPlan pl = plan_launch<BITS>(x + m0 * K, w, s, z, bias, y + m0 * ys, mc, K, N, group, F);
        if (!pl.ok) return cudaErrorNotSupported;
        cudaError_t e = launch_plan<BITS>(pl, stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace mma
}  // namespace lowbit
