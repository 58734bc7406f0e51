// quantize.cu -- groupwise asymmetric quantisation of a weight matrix, fused
// with packing.
//
// The pages name a `_quantize` function producing the codes and the
// N x num_groups scales and zeros (ao PR #2167 "metal lowbit kernels:
// qmv_fast optimization", Summary, bullet 1) without defining it; the
// min/max reading used throughout this library:
//   zero  = fp16 rounded toward -inf of min(w over the group)
//   scale = fp16 rounded toward +inf of (max - zero) / (2^b - 1)
//   q     = clamp(round-half-even((w - zero) / scale), 0, 2^b - 1)
//   a constant group (max == min): scale = 2^-14 (smallest fp16 normal), q = 0.
// The result is defined by fp64 arithmetic on the exact inputs.  The kernel
// reaches the same bits with fp32 arithmetic wherever fp32 provably decides
// the same way, and falls back to fp64 where it cannot tell:
//   - min and max are exact in fp32 (the inputs are fp32, bf16 or fp16);
//   - the fp64 scale quotient lies between (max - zero) rounded down times
//     1/qmax rounded down, and the same rounded up (every step rounded
//     outward), so when both bounds round up to the same fp16 that fp16 is
//     the scale (the fp64 quotient is the fp64 value nearest the exact one,
//     and no fp32 bound can lie between the two); when they round to two
//     adjacent fp16 values, the sign of an exact fp32 residual picks one;
//   - (w - zero) / scale in fp32 differs from the fp64 quotient by less than
//     3 * 2^-24 * 2^7 < 2^-15 (it is at most 2^7 and carries three roundings
//     of 2^-24 relative), so its round-half-even agrees with fp64's unless it
//     lies within that distance of a half-integer; those codes are decided by
//     the sign of an exact fp32 residual against that half-integer;
//   - fp64 itself only where w - zero or max - zero is not exact in fp32.
// The codes need no clamping: zero <= min and scale >= (max - zero) / qmax,
// so the exact quotient lies in [0, qmax], and the fp32 and fp64 quotients
// stay within [0, qmax + 2^-15].
// The codes are written packed (contiguous, LSB-first, ao PR #2167 Summary
// bullet 2).
//
// Work unit: one warp per chunk of 1024 consecutive weights of a row.  Lane l
// takes weights [32l, 32l+32); a group of g weights spans g/32 lanes (one lane
// for g = 32), whose min/max is a segmented shuffle reduction; the lane's 32
// codes are four octets, written as 4b bytes at byte 4lb of the chunk's packed
// bytes.  (Eight weights a lane cost 240 instructions per 256 weights, more
// than half of them per chunk rather than per weight: prefetch bookkeeping, the
// group reductions, the scale and its broadcast, indices and stores.)  The
// weights arrive through a per-warp ring in shared memory of 4 chunks (16-bit
// inputs) or 2 (fp32), filled with 16-byte asynchronous copies (cp.async) that
// many chunks ahead of the one being coded, less one, so that each warp keeps
// several KB of loads in flight; a lane reads its weights from the ring twice
// (for the group's min/max, then for the codes) rather than holding 32 values.
#include "common.cuh"

namespace lowbit {
namespace {

constexpr int kPerLane = 32;         // weights per lane per step
constexpr int kOct = kPerLane / 8;   // octets (blocks of 8 weights) per lane
constexpr int kChunk = 32 * kPerLane; // weights per warp per step
constexpr int kRingBytes = 8192;     // a warp's shared-memory ring: 4 chunks of 16-bit weights, 2 of fp32
constexpr int kWarps = 8;            // warps per block

struct W8 {
    float v[8];
};

// A lane's 8 weights from their raw bytes (16 for 16-bit inputs, 32 for
// fp32), converted exactly to fp32.
__device__ __forceinline__ W8 convert8(int dtype, uint4 u, uint4 u2) {
    W8 r;
    if (dtype == LOWBIT_DTYPE_F32) {
        r.v[0] = __uint_as_float(u.x); r.v[1] = __uint_as_float(u.y);
        r.v[2] = __uint_as_float(u.z); r.v[3] = __uint_as_float(u.w);
        r.v[4] = __uint_as_float(u2.x); r.v[5] = __uint_as_float(u2.y);
        r.v[6] = __uint_as_float(u2.z); r.v[7] = __uint_as_float(u2.w);
    } else {
        const uint32_t words[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (dtype == LOWBIT_DTYPE_BF16) {
                r.v[2 * i] = __uint_as_float(words[i] << 16);
                r.v[2 * i + 1] = __uint_as_float(words[i] & 0xFFFF0000u);
            } else {
                r.v[2 * i] = __half2float(__ushort_as_half((uint16_t)(words[i] & 0xFFFFu)));
                r.v[2 * i + 1] = __half2float(__ushort_as_half((uint16_t)(words[i] >> 16)));
            }
        }
    }
    return r;
}

// Packed minimum / maximum of two bf16 or two fp16 pairs: exact, and a NaN
// input yields the other input, as fminf / fmaxf do.
__device__ __forceinline__ uint32_t min_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("min.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t max_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t min_f16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("min.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t max_f16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// 16 bytes of shared memory, loaded where it is written (volatile: the
// weights are read twice from the ring, rather than held in registers).
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// 16-byte asynchronous copy global -> shared (L2 only); src_bytes 0 fills zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }


// fp16 scale: rounded toward +inf of fl64(fl64(mx - z) / qmax).  rq_lo and
// rq_hi are 1/qmax rounded down and up.  When the two bounds round up to
// different fp16 values lo < hi (adjacent: the bounds are a few fp32 ulps
// apart), the scale is lo if the quotient is at most lo and hi otherwise.
// With mx - z exact in fp32, fma(-lo, qmax, mx - z) has the sign of the
// exact (mx - z) - lo qmax (lo qmax has at most 18 significant bits); a
// nonzero difference is at least 2^-23 of it, far above the fp64 quotient's
// rounding, so fp64 lies on the same side of lo.  Otherwise fp64 decides.
__device__ __forceinline__ uint16_t scale_bits(float mx, float z, float qmax, float rq_lo, float rq_hi) {
    const float d_lo = __fsub_rd(mx, z), d_hi = __fsub_ru(mx, z);
    const uint16_t lo = __half_as_ushort(__float2half_ru(__fmul_rd(d_lo, rq_lo)));
    const uint16_t hi = __half_as_ushort(__float2half_ru(__fmul_ru(d_hi, rq_hi)));
    if (lo == hi) return lo;
    if (d_lo == d_hi && hi == lo + 1u) {
        const float res = fmaf(-__half2float(__ushort_as_half(lo)), qmax, d_lo);
        return res <= 0.0f ? lo : hi;
    }
    const double t = ((double)mx - (double)z) / (double)qmax;
    // Directed rounding to fp16 through fp32 in the same direction equals
    // directed rounding to fp16 directly: every fp16 is an fp32.
    return __half_as_ushort(__float2half_ru(__double2float_ru(t)));
}

// fp16 scale of a constant group (every weight equal to mn, all codes 0):
// the larger of 2^-14 and fp16 rounded toward +inf of 2 (mn - z), so that
// mn - z <= scale / 2.  mn - z is exact in fp32: z is mn rounded down to fp16,
// so the two lie within a factor of two, or z is a multiple of mn's ulp.
__device__ __forceinline__ uint16_t flat_scale_bits(float mn, float z) {
    const uint32_t cover = __half_as_ushort(__float2half_ru(2.0f * __fsub_rn(mn, z)));
    return (uint16_t)max(cover, 0x0400u);
}

// Packed fp32 pairs (IEEE round-to-nearest, subnormals kept).
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
    unsigned long long r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r)
        : "l"(*reinterpret_cast<unsigned long long *>(&a)), "l"(*reinterpret_cast<unsigned long long *>(&b)));
    return *reinterpret_cast<float2 *>(&r);
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    unsigned long long r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r)
        : "l"(*reinterpret_cast<unsigned long long *>(&a)), "l"(*reinterpret_cast<unsigned long long *>(&b)));
    return *reinterpret_cast<float2 *>(&r);
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    unsigned long long r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r)
        : "l"(*reinterpret_cast<unsigned long long *>(&a)), "l"(*reinterpret_cast<unsigned long long *>(&b)));
    return *reinterpret_cast<float2 *>(&r);
}

// Code of a weight whose fp32 quotient r lies within 2^-14 of the half-integer
// h = rint(r) + 1/2 sign(r - rint(r)); the fp64 quotient is then h - 1/2 or
// h + 1/2 after rounding.  When v - z is exact in fp32 (its downward and
// upward roundings agree), fma(-h, s, v - z) has the sign of the exact
// (v - z) - h s: h s has at most 19 significant bits, so the fma rounds once.
// A nonzero residual is at least 2^-23 h s (its last bit is that of v - z or
// of h s), far above the fp64 quotient's rounding, so fp64 rounds to the
// same side; a zero residual is an exact tie, which fp64 rounds to even.
// Otherwise fp64 decides.
__device__ __noinline__ uint32_t code_near_tie(float v, float z, float s, uint32_t q, float d) {
    const float lo = __fsub_rd(v, z), hi = __fsub_ru(v, z);
    if (lo != hi) return (uint32_t)rint(((double)v - (double)z) / (double)s);
    const float h = d > 0.0f ? (float)q + 0.5f : (float)q - 0.5f;
    const float res = fmaf(-h, s, lo);
    const uint32_t below = (uint32_t)(h - 0.5f);
    if (res > 0.0f) return below + 1u;
    if (res < 0.0f) return below;
    return below + (below & 1u);                      // exact tie: to even
}

// Codes of a lane's 8 weights: rint(fl64(fl64(v - z) / s)) (see the header).
// r = (v - z) * (1/s) in fp32; t = r + 2^23 rounds r to the nearest integer,
// ties to even, into t's low mantissa bits (0 <= r < 2^22), so t's bits are
// 0x4B000000 + code and the code is t's bits under the b-bit mask (0x4B000000
// has none of them; a NaN weight's bits give the same masked code as before);
// r - (t - 2^23) is exact.  Weights whose r lies within 2^-14 of a
// half-integer are recomputed in fp64.
__device__ __forceinline__ void codes8(const float (&v)[8], float z, float s, float inv_s, uint32_t mask,
                                       uint32_t (&q)[8]) {
    const float2 z2 = make_float2(z, z), is2 = make_float2(inv_s, inv_s);
    const float2 big = make_float2(8388608.0f, 8388608.0f);
    float2 d[4];
    bool near_tie = false;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 r = mul2(sub2(make_float2(v[2 * i], v[2 * i + 1]), z2), is2);
        const float2 t = add2(r, big);
        d[i] = sub2(r, sub2(t, big));
        q[2 * i] = __float_as_uint(t.x) & mask;
        q[2 * i + 1] = __float_as_uint(t.y) & mask;
        near_tie |= fmaxf(fabsf(d[i].x), fabsf(d[i].y)) > 0.5f - 1.0f / 16384.0f;
    }
    if (near_tie) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float di = (i & 1) ? d[i / 2].y : d[i / 2].x;
            if (fabsf(di) > 0.5f - 1.0f / 16384.0f) q[i] = code_near_tie(v[i], z, s, q[i], di);
        }
    }
}

// Lane-held octet of 8 b-bit codes: code i at bits [b*i, b*i+b) of (lo, hi).
// The fields are disjoint and q < 2^b, so adding a code equals OR-ing it in
// (and is one shift-add).
template <int BITS>
struct Octet {
    uint32_t lo = 0, hi = 0;
    __device__ __forceinline__ void put(int i, uint32_t q) {
        const int b = BITS * i;
        if (b < 32) {
            lo += q << b;
            if (b + BITS > 32) hi += q >> (32 - b);
        } else {
            hi += q << (b - 32);
        }
    }
    __device__ __forceinline__ uint8_t byte(int i) const {
        return (uint8_t)(i < 4 ? lo >> (8 * i) : hi >> (8 * (i - 4)));
    }
};

// GL = lanes per group (g / 32): 1, 2, 4 or 8.  WIDE: the packed matrix is
// aligned for the 16- and 32-bit stores of b = 2, 4, 6 (it may have any
// alignment; otherwise every byte is stored on its own).
template <int BITS, int GL, bool WIDE>
__global__ void __launch_bounds__(256, 3)
quantize_kernel(const void *__restrict__ w, int dtype, uint8_t *__restrict__ packed,
                uint16_t *__restrict__ scales, uint16_t *__restrict__ zeros, int64_t N, int K) {
    constexpr int group = GL * kPerLane;
    constexpr float qmax = (float)((1 << BITS) - 1);
    const float rq_lo = __frcp_rd(qmax), rq_hi = __frcp_ru(qmax);
    const int lane = threadIdx.x & 31;
    const int G = K / group;
    const int cpr = (K + kChunk - 1) / kChunk;               // chunks per row
    const int64_t chunks = N * cpr;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
    const int64_t row_bytes = (int64_t)K * BITS / 8;

    // The warp's ring: R slots of 32 lanes x 32 weights (R = 4 for 16-bit
    // inputs, 2 for fp32).
    __shared__ __align__(16) uint8_t ring[kWarps][kRingBytes];
    const int wib = threadIdx.x >> 5;
    const int esz = dtype == LOWBIT_DTYPE_F32 ? 4 : 2;
    const int lane_bytes = kPerLane * esz;
    const int R = kRingBytes / (32 * lane_bytes);
    const uint32_t ring0 = (uint32_t)__cvta_generic_to_shared(&ring[wib][lane * lane_bytes]);

    int64_t c = (int64_t)blockIdx.x * (blockDim.x / 32) + wib;
    if (c >= chunks) return;                                 // whole warp leaves together
    // Chunk c is row c / cpr, chunk c % cpr of the row; the warp strides by
    // `warps` chunks, i.e. dn rows and dc chunks with a carry.
    const int64_t dn = warps / cpr;
    const int dc = (int)(warps % cpr);
    int64_t n = c / cpr;
    int kc = (int)(c - n * cpr);
    int k = kc * kChunk + lane * kPerLane;
    // Prefetch cursor: R - 1 chunks ahead of (c, n, kc), each copy group
    // committed whether or not it copies anything, so that waiting for all but
    // the newest R - 1 groups always means "this chunk has landed".
    int64_t cp_c = c, cp_n = n;
    int cp_kc = kc;
    auto issue = [&](int slot) {
        const int kk = cp_kc * kChunk + lane * kPerLane;
        if (cp_c < chunks) {
            const uint8_t *src = reinterpret_cast<const uint8_t *>(w) + (cp_n * K + kk) * esz;
            const uint32_t nb = kk < K ? 16u : 0u;
            const uint32_t dst = ring0 + (uint32_t)(slot * 32 * lane_bytes);
            for (int j = 0; j < lane_bytes; j += 16) cp_async16(dst + j, kk < K ? src + j : w, nb);
        }
        cp_async_commit();
        cp_c += warps;
        cp_n += dn;
        cp_kc += dc;
        if (cp_kc >= cpr) { cp_kc -= cpr; ++cp_n; }
    };
    for (int j = 0; j < R - 1; ++j) issue(j);
    int slot = 0;                                        // ring slot of this chunk
    for (; c < chunks; c += warps) {
        issue(slot == 0 ? R - 1 : slot - 1);             // into the slot read last iteration
        if (esz == 4) cp_async_wait<1>();                // this chunk's copies have landed
        else cp_async_wait<3>();
        const uint32_t mine = ring0 + (uint32_t)(slot * 32 * lane_bytes);
        if (++slot == R) slot = 0;
        // Block h of the lane's weights: 8 weights from the ring (16 or 32 bytes).
        auto block = [&](int h) {
            if (esz == 4) return convert8(dtype, lds128(mine + 32u * h), lds128(mine + 32u * h + 16u));
            const uint4 a = lds128(mine + 16u * h);
            return convert8(dtype, a, a);
        };
        int64_t n2 = n + dn;
        int kc2 = kc + dc;
        if (kc2 >= cpr) { kc2 -= cpr; ++n2; }
        const int k2 = kc2 * kChunk + lane * kPerLane;
        // A group lies wholly inside or wholly outside the row (K % group == 0),
        // so lanes past the row end only ever reduce among themselves.
        float mn, mx;
        if (esz == 2) {
            // 16-bit weights: packed minimum and maximum of the raw pairs,
            // then of the two halves (the signs of zeros do not matter here:
            // a zero minimum's sign is settled below, and the maximum only
            // enters as max - zero).
            const uint4 u0 = lds128(mine), u1 = lds128(mine + 16u), u2 = lds128(mine + 32u), u3 = lds128(mine + 48u);
            const uint32_t wd[16] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w,
                                     u2.x, u2.y, u2.z, u2.w, u3.x, u3.y, u3.z, u3.w};
            uint32_t lo2 = wd[0], hi2 = wd[0];
            if (dtype == LOWBIT_DTYPE_BF16) {
#pragma unroll
                for (int i = 1; i < 16; ++i) {
                    lo2 = min_bf16x2(lo2, wd[i]);
                    hi2 = max_bf16x2(hi2, wd[i]);
                }
                mn = fminf(__uint_as_float(lo2 << 16), __uint_as_float(lo2 & 0xFFFF0000u));
                mx = fmaxf(__uint_as_float(hi2 << 16), __uint_as_float(hi2 & 0xFFFF0000u));
            } else {
#pragma unroll
                for (int i = 1; i < 16; ++i) {
                    lo2 = min_f16x2(lo2, wd[i]);
                    hi2 = max_f16x2(hi2, wd[i]);
                }
                mn = fminf(__half2float(__ushort_as_half((uint16_t)(lo2 & 0xFFFFu))),
                           __half2float(__ushort_as_half((uint16_t)(lo2 >> 16))));
                mx = fmaxf(__half2float(__ushort_as_half((uint16_t)(hi2 & 0xFFFFu))),
                           __half2float(__ushort_as_half((uint16_t)(hi2 >> 16))));
            }
        } else {
            const W8 b0 = block(0);
            mn = b0.v[0];
            mx = b0.v[0];
#pragma unroll
            for (int i = 1; i < 8; ++i) {
                mn = fminf(mn, b0.v[i]);
                mx = fmaxf(mx, b0.v[i]);
            }
#pragma unroll
            for (int h = 1; h < kOct; ++h) {
                const W8 bh = block(h);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    mn = fminf(mn, bh.v[i]);
                    mx = fmaxf(mx, bh.v[i]);
                }
            }
        }
#pragma unroll
        for (int o = 1; o < GL; o <<= 1) {
            mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        }
        // A zero minimum takes the sign of the group's first zero (the first
        // minimum a left-to-right scan meets).
        if (__any_sync(0xffffffffu, mn == 0.0f)) {
            uint32_t key = 0xFFFFFFFFu;                       // (position << 1) | sign
#pragma unroll
            for (int h = 0; h < kOct; ++h) {
                const W8 bh = block(h);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (bh.v[i] == 0.0f)
                        key = min(key, ((uint32_t)(lane * kPerLane + 8 * h + i) << 1) | (__float_as_uint(bh.v[i]) >> 31));
            }
#pragma unroll
            for (int o = 1; o < GL; o <<= 1)
                key = min(key, __shfl_xor_sync(0xffffffffu, key, o));
            if (mn == 0.0f) mn = (key & 1u) ? -0.0f : 0.0f;
        }
        const uint16_t zh = __half_as_ushort(__float2half_rd(mn));
        const float z = __half2float(__ushort_as_half(zh));
        const bool flat = (mx == mn);
        // The first lane of each group computes the scale (two directed
        // divisions); a group is an aligned run of GL lanes, so a shuffle
        // hands it to the others.
        uint32_t sh32 = 0x0400u;
        if ((lane & (GL - 1)) == 0) sh32 = flat ? flat_scale_bits(mn, z) : scale_bits(mx, z, qmax, rq_lo, rq_hi);
        const uint16_t sh = (uint16_t)__shfl_sync(0xffffffffu, sh32, lane & ~(GL - 1));
        if (k < K) {
            const float s = __half2float(__ushort_as_half(sh));
            const float inv_s = __frcp_rn(s);
            Octet<BITS> o[kOct];
            if (!flat) {
#pragma unroll
                for (int h = 0; h < kOct; ++h) {
                    uint32_t q[8];
                    codes8(block(h).v, z, s, inv_s, (1u << BITS) - 1u, q);
#pragma unroll
                    for (int i = 0; i < 8; ++i) o[h].put(i, q[i]);
                }
            }
            uint8_t *dst = packed + n * row_bytes + (int64_t)(k / 8) * BITS;
            // kOct b bytes at byte (k / 8) b of the row, octet after octet:
            // 32-bit stores for b = 4, 16-bit stores for b = 2 and 6 (row and
            // octet offsets are multiples of 4 and 2 bytes), bytes otherwise or
            // when the matrix is not aligned.
#pragma unroll
            for (int h = 0; h < kOct; ++h) {
                uint8_t *dh = dst + h * BITS;
                if constexpr (WIDE && BITS == 4) {
                    *reinterpret_cast<uint32_t *>(dh) = o[h].lo;
                } else if constexpr (WIDE && BITS == 2) {
                    *reinterpret_cast<uint16_t *>(dh) = (uint16_t)o[h].lo;
                } else if constexpr (WIDE && BITS == 6) {
                    uint16_t *d16 = reinterpret_cast<uint16_t *>(dh);
                    d16[0] = (uint16_t)o[h].lo;
                    d16[1] = (uint16_t)(o[h].lo >> 16);
                    d16[2] = (uint16_t)o[h].hi;
                } else {
#pragma unroll
                    for (int i = 0; i < BITS; ++i) dh[i] = o[h].byte(i);
                }
            }
            if ((lane & (GL - 1)) == 0) {
                const int64_t gi = n * G + k / group;
                scales[gi] = sh;
                zeros[gi] = zh;
            }
        }
        n = n2;
        kc = kc2;
        k = k2;
    }
}

// One resident wave: as many blocks as fit on the device at once (each warp
// then strides over chunks), or fewer when there are fewer chunks.
template <int BITS, int GL, bool WIDE>
cudaError_t launch_one(const void *w, int dtype, uint8_t *packed, uint16_t *scales,
                       uint16_t *zeros, int64_t N, int K, cudaStream_t stream) {
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, quantize_kernel<BITS, GL, WIDE>, 256, 0);
    if (e != cudaSuccess) return e;
    const int64_t chunks = N * ((K + kChunk - 1) / kChunk);
    const int64_t want = (chunks + 7) / 8;
    const int64_t wave = (int64_t)sms * (per_sm > 0 ? per_sm : 1);
    const unsigned blocks = (unsigned)(want < wave ? want : wave);
    quantize_kernel<BITS, GL, WIDE><<<blocks, kWarps * 32, 0, stream>>>(w, dtype, packed, scales, zeros, N, K);
    return cudaGetLastError();
}

template <int BITS, bool WIDE>
cudaError_t launch_group(const void *w, int dtype, uint8_t *packed, uint16_t *scales,
                         uint16_t *zeros, int64_t N, int K, int group, cudaStream_t stream) {
    switch (group) {
        case 32: return launch_one<BITS, 1, WIDE>(w, dtype, packed, scales, zeros, N, K, stream);
        case 64: return launch_one<BITS, 2, WIDE>(w, dtype, packed, scales, zeros, N, K, stream);
        case 128: return launch_one<BITS, 4, WIDE>(w, dtype, packed, scales, zeros, N, K, stream);
        case 256: return launch_one<BITS, 8, WIDE>(w, dtype, packed, scales, zeros, N, K, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <int BITS>
cudaError_t launch_bits(const void *w, int dtype, uint8_t *packed, uint16_t *scales,
                        uint16_t *zeros, int64_t N, int K, int group, cudaStream_t stream) {
    // Only b = 2, 4, 6 have wide stores; they need 2- or 4-byte alignment.
    constexpr uintptr_t need = BITS == 4 ? 4 : 2;
    if constexpr (BITS == 2 || BITS == 4 || BITS == 6) {
        if ((reinterpret_cast<uintptr_t>(packed) & (need - 1)) == 0)
            return launch_group<BITS, true>(w, dtype, packed, scales, zeros, N, K, group, stream);
    }
    return launch_group<BITS, false>(w, dtype, packed, scales, zeros, N, K, group, stream);
}

}  // namespace

cudaError_t launch_quantize(const void *w, int dtype, uint8_t *packed, uint16_t *scales,
                            uint16_t *zeros, int64_t N, int64_t K, int bits, int group,
                            cudaStream_t stream) {
    const int k = (int)K;
    switch (bits) {
        case 1: return launch_bits<1>(w, dtype, packed, scales, zeros, N, k, group, stream);
        case 2: return launch_bits<2>(w, dtype, packed, scales, zeros, N, k, group, stream);
        case 3: return launch_bits<3>(w, dtype, packed, scales, zeros, N, k, group, stream);
        case 4: return launch_bits<4>(w, dtype, packed, scales, zeros, N, k, group, stream);
        case 5: return launch_bits<5>(w, dtype, packed, scales, zeros, N, k, group, stream);
        case 6: return launch_bits<6>(w, dtype, packed, scales, zeros, N, k, group, stream);
        case 7: return launch_bits<7>(w, dtype, packed, scales, zeros, N, k, group, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace lowbit
