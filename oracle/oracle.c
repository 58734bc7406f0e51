/*
 * oracle.c -- plain, slow, obviously-correct CPU oracle for the weight-only,
 * groupwise, asymmetric low-bit linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this code.  It shares no code, header,
 * table or helper with the CUDA library, and the CUDA library never calls it.
 *
 * What it computes (all sources are the pages about "linear:afpwx" low-bit
 * weights in torchao / torchchat):
 *   - torchchat PR #1415 "Add torchao mps ops": weights only are quantized,
 *     groupwise, bit width 1..7, group size 32/64/128/256; activations stay
 *     floating point.
 *   - ao PR #2167 "metal lowbit kernels: qmv_fast optimization", Summary:
 *       bullet 1: scales and zeros have shape N x num_groups;
 *       bullet 2: codes are stored contiguously, a code continuing into the
 *                 next byte once the current byte is full.
 *   - ao issue #3446 "Revamp int4 MPS support in torchao": bias requested.
 * The dequantised weight is  W[n,k] = scale[n, k/g] * q[n,k] + zero[n, k/g]
 * and the layer is  y[m,n] = sum_k x[m,k] * W[n,k] + bias[n].
 *
 * Readings where the pages are silent (each stated again where it is used):
 *   - "zero" is an additive offset (W = s*q + z), not s*(q - zp);
 *   - the bit stream of a row is little-endian: stream bit j is bit (j % 8)
 *     of byte (j / 8), and code bit 0 goes to the lowest stream position;
 *   - each row of the weight matrix is its own stream of K*b/8 bytes
 *     (K is a multiple of g >= 32, so K*b/8 is a whole number of bytes);
 *   - group index of column k is floor(k / g);
 *   - codes >= 2^b are masked to their low b bits.
 *
 * Everything is computed in fp64: fp16 and bf16 inputs convert to double
 * exactly, so the only rounding is in the fp64 sum.
 *
 * PLANT_* macros: each plants one plausible mistake.  They exist only so the
 * pin tests can show that every such mistake fails at least one pin; the
 * default build defines none of them.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL 1

/* ------------------------------------------------------------------------ */
/* Number formats, decoded from their IEEE-754 bit layouts.                  */
/* ------------------------------------------------------------------------ */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* zero or subnormal */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
#ifdef PLANT_HALF_BIAS
        v = ldexp(1024.0 + (double)f, e - 24);
#else
        v = ldexp(1024.0 + (double)f, e - 25);     /* (1 + f/1024) * 2^(e-15) */
#endif
    return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of a binary32 (1 sign, 8 exponent bits with
 * bias 127, 7 fraction bits). */
double oracle_bf16_to_double(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int f = b & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);                /* zero or subnormal */
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp(128.0 + (double)f, e - 134);     /* (1 + f/128) * 2^(e-127) */
    return sign ? -v : v;
}

/* Rounding modes for oracle_double_to_half. */
#define ORACLE_RN 0   /* to nearest, ties to even */
#define ORACLE_RD 1   /* toward -infinity */
#define ORACLE_RU 2   /* toward +infinity */

/* Encode a non-negative magnitude that is exactly representable in binary16
 * (or is +infinity) into its bit pattern. */
static uint16_t encode_half_magnitude(double a)
{
    if (isinf(a) || a > 65504.0)
        return 0x7c00;
    if (a < ldexp(1.0, -14))                        /* subnormal or zero */
        return (uint16_t)(a / ldexp(1.0, -24));
    int E;
    double fr = frexp(a, &E);                      /* a = fr * 2^E, fr in [0.5,1) */
    int e = E - 1;                                 /* a = (2 fr) * 2^e          */
    double mant = (2.0 * fr - 1.0) * 1024.0;       /* exact integer 0..1023      */
    return (uint16_t)(((e + 15) << 10) | (int)mant);
}

/* Round a double to binary16 with the given mode. */
uint16_t oracle_double_to_half(double v, int mode)
{
    if (isnan(v))
        return 0x7e00;
    int neg = signbit(v) ? 1 : 0;
    double a = fabs(v);
    if (a == 0.0)
        return (uint16_t)(neg << 15);
    /* Rounding the magnitude: toward -inf on a negative value rounds the
     * magnitude up, and so on. */
    int up;              /* 1: magnitude rounds away from zero, 0: toward, -1: nearest */
    if (mode == ORACLE_RN) up = -1;
    else if (mode == ORACLE_RD) up = neg ? 1 : 0;
    else up = neg ? 0 : 1;

    double quantum;
    if (a < ldexp(1.0, -14)) {
        quantum = ldexp(1.0, -24);
    } else {
        int E;
        frexp(a, &E);
        quantum = ldexp(1.0, (E - 1) - 10);
    }
    double q = a / quantum;                        /* exact: power-of-two scale */
    double lo = floor(q);
    double r;
    if (q == lo) r = lo;
    else if (up == 1) r = lo + 1.0;
    else if (up == 0) r = lo;
    else {
        double frac = q - lo;
        if (frac > 0.5) r = lo + 1.0;
        else if (frac < 0.5) r = lo;
        else r = (fmod(lo, 2.0) == 0.0) ? lo : lo + 1.0;
    }
    double mag = r * quantum;
    uint16_t bits;
    if (mag > 65504.0) {
        /* Past the largest finite value: nearest rounds to infinity beyond
         * 65520; toward zero stays at 65504. */
        if (up == 0) bits = 0x7bff;
        else if (up == 1) bits = 0x7c00;
        else bits = (a >= 65520.0) ? 0x7c00 : 0x7bff;
    } else {
        bits = encode_half_magnitude(mag);
    }
    return (uint16_t)((neg << 15) | bits);
}

/* ------------------------------------------------------------------------ */
/* Packing: one bit at a time (ao PR #2167, Summary, bullet 2).             */
/* ------------------------------------------------------------------------ */

static int bits_ok(int bits) { return bits >= 1 && bits <= 7; }
static int group_ok(int g) { return g == 32 || g == 64 || g == 128 || g == 256; }

/* Bytes of one packed row: K codes of b bits each. */
int64_t oracle_row_bytes(int64_t K, int bits) { return K * bits / 8; }

/* Stream bit index of bit i of code k. */
static int64_t stream_bit(int64_t k, int bits, int i)
{
#ifdef PLANT_CODE_MSB
    return k * bits + (bits - 1 - i);
#else
    return k * bits + i;
#endif
}

/* Bit position inside its byte of stream bit j. */
static int bit_in_byte(int64_t j)
{
#ifdef PLANT_STREAM_MSB
    return 7 - (int)(j % 8);
#else
    return (int)(j % 8);
#endif
}

/* Write code c (masked to b bits) at bit position k*b of a zeroed row stream. */
static void put_code(uint8_t *row, int64_t k, int bits, unsigned c)
{
    for (int i = 0; i < bits; ++i) {
        int64_t j = stream_bit(k, bits, i);
        if ((c >> i) & 1u)
            row[j / 8] |= (uint8_t)(1u << bit_in_byte(j));
    }
}

static unsigned get_code(const uint8_t *row, int64_t k, int bits)
{
    unsigned c = 0;
    for (int i = 0; i < bits; ++i) {
        int64_t j = stream_bit(k, bits, i);
        unsigned bit = (row[j / 8] >> bit_in_byte(j)) & 1u;
        c |= bit << i;
    }
    return c;
}

/* codes: [N, K], one code per byte.  packed: [N, K*bits/8].  K*bits must be a
 * multiple of 8 so that every row is a whole number of bytes. */
int oracle_pack(const uint8_t *codes, uint8_t *packed, int64_t N, int64_t K, int bits)
{
    if (!bits_ok(bits) || N < 0 || K < 0 || (K * bits) % 8 != 0)
        return ORACLE_EINVAL;
    int64_t rb = oracle_row_bytes(K, bits);
    memset(packed, 0, (size_t)(N * rb));
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            put_code(packed + n * rb, k, bits, codes[n * K + k]);
    return ORACLE_OK;
}

int oracle_unpack(const uint8_t *packed, uint8_t *codes, int64_t N, int64_t K, int bits)
{
    if (!bits_ok(bits) || N < 0 || K < 0 || (K * bits) % 8 != 0)
        return ORACLE_EINVAL;
    int64_t rb = oracle_row_bytes(K, bits);
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            codes[n * K + k] = (uint8_t)get_code(packed + n * rb, k, bits);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Dequantisation and the linear layer.                                     */
/* ------------------------------------------------------------------------ */

static int shape_ok(int64_t M, int64_t K, int64_t N, int bits, int group)
{
    return bits_ok(bits) && group_ok(group) && M >= 0 && N >= 0 && K > 0 && K % group == 0;
}

/* Dequantise row n into w[0..K): W[n,k] = scale[n,k/g]*q[n,k] + zero[n,k/g]
 * (ao PR #2167 Summary bullet 1 for the N x num_groups layout). */
static void dequant_row(const uint8_t *packed, const uint16_t *scales, const uint16_t *zeros,
                        int64_t n, int64_t N, int64_t K, int bits, int group, double *w)
{
    int64_t rb = oracle_row_bytes(K, bits);
    int64_t G = K / group;
    const uint8_t *row = packed + n * rb;
    (void)N;
    for (int64_t k = 0; k < K; ++k) {
#ifdef PLANT_GROUP_MOD
        int64_t gi = k % G;
#else
        int64_t gi = k / group;
#endif
#ifdef PLANT_SZ_TRANSPOSED
        int64_t at = gi * N + n;                   /* the older num_groups x N layout */
#else
        int64_t at = n * G + gi;
#endif
        double s = oracle_half_to_double(scales[at]);
        double z = oracle_half_to_double(zeros[at]);
        double q = (double)get_code(row, k, bits);
#if defined(PLANT_DROP_ZERO)
        w[k] = s * q;
#elif defined(PLANT_ZERO_POINT)
        w[k] = s * (q - z);
#else
        w[k] = s * q + z;
#endif
    }
}

/* One output: sum_k x[m,k] * w[k] + b, in order k = 0..K-1. */
static double dot_row(const uint16_t *x, int64_t m, int64_t M, int64_t K, const double *w, double b)
{
    double acc = 0.0;
    (void)M;
#ifdef PLANT_LAST_K
    for (int64_t k = 0; k < K - 1; ++k)
#else
    for (int64_t k = 0; k < K; ++k)
#endif
    {
#ifdef PLANT_X_TRANSPOSED
        acc += oracle_bf16_to_double(x[k * M + m]) * w[k];
#else
        acc += oracle_bf16_to_double(x[m * K + k]) * w[k];
#endif
    }
#ifdef PLANT_DROP_BIAS
    (void)b;
    return acc;
#else
    return acc + b;
#endif
}

/* W: [N, K] fp64. */
int oracle_dequant(const uint8_t *packed, const uint16_t *scales, const uint16_t *zeros,
                   int64_t N, int64_t K, int bits, int group, double *W)
{
    if (!shape_ok(1, K, N, bits, group))
        return ORACLE_EINVAL;
    for (int64_t n = 0; n < N; ++n)
        dequant_row(packed, scales, zeros, n, N, K, bits, group, W + n * K);
    return ORACLE_OK;
}

/* y[m, j] = sum_k x[m,k] * W[rows[j], k] + bias[rows[j]] for the listed rows,
 * summed in order k = 0..K-1 in fp64.  x: [M, K] bf16 bits; bias: [N] fp16
 * bits or NULL; y: [M, nrows] fp64; w_tmp: K doubles of caller scratch. */
int oracle_linear_rows(const uint16_t *x, const uint8_t *packed, const uint16_t *scales,
                       const uint16_t *zeros, const uint16_t *bias,
                       int64_t M, int64_t K, int64_t N, int bits, int group,
                       const int64_t *rows, int64_t nrows, double *y, double *w_tmp)
{
    if (!shape_ok(M, K, N, bits, group))
        return ORACLE_EINVAL;
    for (int64_t j = 0; j < nrows; ++j) {
        int64_t n = rows[j];
        if (n < 0 || n >= N)
            return ORACLE_EINVAL;
        dequant_row(packed, scales, zeros, n, N, K, bits, group, w_tmp);
        double b = bias ? oracle_half_to_double(bias[n]) : 0.0;
        for (int64_t m = 0; m < M; ++m)
            y[m * nrows + j] = dot_row(x, m, M, K, w_tmp, b);
    }
    return ORACLE_OK;
}

/* Full layer: y [M, N] fp64. */
int oracle_linear(const uint16_t *x, const uint8_t *packed, const uint16_t *scales,
                  const uint16_t *zeros, const uint16_t *bias,
                  int64_t M, int64_t K, int64_t N, int bits, int group,
                  double *y, double *w_tmp)
{
    if (!shape_ok(M, K, N, bits, group))
        return ORACLE_EINVAL;
    for (int64_t n = 0; n < N; ++n) {
        dequant_row(packed, scales, zeros, n, N, K, bits, group, w_tmp);
        double b = bias ? oracle_half_to_double(bias[n]) : 0.0;
        for (int64_t m = 0; m < M; ++m)
            y[m * N + n] = dot_row(x, m, M, K, w_tmp, b);
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Gated activation of a gate/up projection pair.  The pages time Llama     */
/* token generation (torchchat PR #1415, ao PR #2167 decode tables), whose  */
/* MLP multiplies silu of the gate projection by the up projection; the     */
/* pages do not write it out, so the plain reading is used:                 */
/*   h[m,f] = silu(a) * u,  a = y[m, f],  u = y[m, F + f],                   */
/*   silu(a) = a / (1 + exp(-a)),                                           */
/* on the unrounded fp64 outputs y [M, 2F] of a layer whose first F rows    */
/* are the gate projection and last F rows the up projection.               */
/* ------------------------------------------------------------------------ */
int oracle_silu_mul(const double *y, int64_t M, int64_t F, double *h)
{
    if (M < 0 || F < 0)
        return ORACLE_EINVAL;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t f = 0; f < F; ++f) {
#ifdef PLANT_SILU_SWAP
            double a = y[m * 2 * F + F + f];
            double u = y[m * 2 * F + f];
#else
            double a = y[m * 2 * F + f];
            double u = y[m * 2 * F + F + f];
#endif
#ifdef PLANT_SILU_SIGN
            double e = exp(a);
#else
            double e = exp(-a);
#endif
            h[m * F + f] = a / (1.0 + e) * u;
        }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Reference quantiser.  The pages name a `_quantize` function that produces */
/* the codes and the N x num_groups scales and zeros (ao PR #2167, Summary,  */
/* bullet 1) but do not define it.  Reading used here (min/max asymmetric):  */
/*   zero  = fp16 rounded toward -inf of min(w over the group);              */
/*   scale = fp16 rounded toward +inf of (max - zero) / (2^b - 1);           */
/*   q     = clamp(round-half-even((w - zero) / scale), 0, 2^b - 1);         */
/*   the minimum of a group holding both zeros is the first zero met in k    */
/*   order (its sign survives into the zero);                                */
/*   a constant group (max == min) gets q = 0 and scale = the larger of the  */
/*   smallest fp16 normal and fp16 rounded toward +inf of 2 (min - zero), so */
/*   that |w - (scale q + zero)| <= scale / 2 there as everywhere.           */
/* min - zero is exact in fp64 (zero is min rounded down to fp16, so the two */
/* lie within a factor of two, or zero is a multiple of min's ulp).          */
/* ------------------------------------------------------------------------ */
int oracle_quantize(const double *w, int64_t N, int64_t K, int bits, int group,
                    uint8_t *codes, uint16_t *scales, uint16_t *zeros)
{
    if (!shape_ok(1, K, N, bits, group))
        return ORACLE_EINVAL;
    int64_t G = K / group;
    double qmax = (double)((1 << bits) - 1);
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t gi = 0; gi < G; ++gi) {
            const double *wg = w + n * K + gi * group;
            double mn = wg[0], mx = wg[0];
            for (int i = 1; i < group; ++i) {
#ifdef PLANT_MIN_LAST
                if (wg[i] <= mn) mn = wg[i];
#else
                if (wg[i] < mn) mn = wg[i];
#endif
                if (wg[i] > mx) mx = wg[i];
            }
            uint16_t zh = oracle_double_to_half(mn, ORACLE_RD);
            double z = oracle_half_to_double(zh);
            uint16_t sh;
            if (mx == mn) {
#ifdef PLANT_CONST_SCALE_FLOOR
                sh = 0x0400;
#else
                uint16_t cover = oracle_double_to_half(2.0 * (mn - z), ORACLE_RU);
                sh = cover > 0x0400 ? cover : 0x0400;   /* 2^-14 at least */
#endif
            } else {
                sh = oracle_double_to_half((mx - z) / qmax, ORACLE_RU);
            }
            double s = oracle_half_to_double(sh);
            scales[n * G + gi] = sh;
            zeros[n * G + gi] = zh;
            for (int i = 0; i < group; ++i) {
#ifdef PLANT_ROUND_HALF_AWAY
                double q = (mx == mn) ? 0.0 : round((wg[i] - z) / s);
#else
                double q = (mx == mn) ? 0.0 : nearbyint((wg[i] - z) / s);
#endif
                if (q < 0.0) q = 0.0;
                if (q > qmax) q = qmax;
                codes[n * K + gi * group + i] = (uint8_t)q;
            }
        }
    }
    return ORACLE_OK;
}
