/*
 * lowbit.h -- C ABI of liblowbit, a GB300 (sm_103a) library for the
 * weight-only, groupwise, asymmetric low-bit linear layer
 *
 *     y[m,n] = sum_k x[m,k] * W[n,k] + bias[n],
 *     W[n,k] = scale[n, k/g] * q[n,k] + zero[n, k/g],
 *
 * with q an unsigned b-bit code, b = 1..7, and group size g in {32,64,128,256}.
 *
 * Sources (web pages about low-bit weights in torchao / torchchat):
 *   - torchchat PR #1415 "Add torchao mps ops": the scheme quantises only the
 *     weights, groupwise, with bit width 1..7 and group size 32..256;
 *     activations stay floating point.
 *   - ao PR #2167 "metal lowbit kernels: qmv_fast optimization", Summary:
 *     bullet 1 -- scales and zeros are N x num_groups; bullet 2 -- the codes
 *     are stored contiguously, continuing into the next byte once the current
 *     byte is full; bullet 3 -- a fast matrix-vector kernel (qmv) for decode.
 *     A reviewer on the same page asks whether it carries over to gemm (qmm).
 *   - ao issue #3446 "Revamp int4 MPS support in torchao": bias support, and
 *     the per-bit-width packing op `_pack_weight_{n}bit`.
 *
 * Conventions for every entry point:
 *   - All data pointers are DEVICE pointers owned by the caller.  The library
 *     keeps no pointer after a call returns and allocates no device memory.
 *   - Calls only enqueue work on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream) and return without synchronising.  A launch error is
 *     reported as LOWBIT_ECUDA; an error in the kernel itself surfaces at the
 *     caller's next synchronisation, as for any CUDA kernel.
 *   - Arguments are checked on the host before anything is launched; a call
 *     that returns anything but LOWBIT_OK has launched nothing.
 *   - Overlap with the previous kernel in the stream: the linear entry points
 *     launch with programmatic dependent launch, and the decode kernel starts
 *     reading the packed weights, scales and zeros before the previous kernel
 *     in the stream has finished, when that kernel allows it (this library's
 *     linear kernels do, as soon as they start).  x and bias are read, and y
 *     written, only after the previous kernel has completed.  So the packed
 *     weights, scales and zeros of a linear call must not be written by the
 *     kernel immediately before it in the stream if that kernel is one of
 *     this library's linear kernels (which write only y) or another kernel
 *     that allows early launch.  Ordinary kernels and copies, and this
 *     library's packing and quantising kernels, do not allow it: weights they
 *     produce are always seen complete.
 *   - 16-bit floats are passed as their bit patterns (uint16_t): bf16 for x and
 *     y, IEEE binary16 (fp16) for scales, zeros and bias.
 *   - The library holds no global handle; calls from several host threads are
 *     safe as long as they do not write the same output buffer.
 *
 * Packed layout (ao PR #2167, Summary, bullet 2, read LSB-first): row n of the
 * packed matrix is a byte string of K*b/8 bytes; code k of that row occupies
 * bits [k*b, k*b+b) of the row's little-endian bit stream, where stream bit j
 * is bit (j % 8) of byte (j / 8) and bit 0 of the code comes first.  A code
 * that does not fit in the current byte continues in the next one.  Rows are
 * stored one after another, so the matrix is [N, K*b/8] row-major.
 */
#ifndef LOWBIT_H
#define LOWBIT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define LOWBIT_API __attribute__((visibility("default")))
#else
#define LOWBIT_API
#endif

/* A cudaStream_t (struct CUstream_st *) without pulling in the CUDA headers. */
typedef struct CUstream_st *lowbit_stream_t;

typedef enum {
    LOWBIT_OK = 0,
    LOWBIT_EINVAL = 1,       /* an argument is out of range, null or misaligned   */
    LOWBIT_EUNSUPPORTED = 2, /* the current device is not an sm_103 (GB300) GPU   */
    LOWBIT_ECUDA = 3         /* a CUDA runtime call or a kernel launch failed     */
} lowbit_status;

/* Which kernel lowbit_linear_ex runs. */
typedef enum {
    LOWBIT_PATH_AUTO = 0,    /* what lowbit_linear picks (see lowbit_select_path)  */
    LOWBIT_PATH_QMV = 1,     /* decode (matrix-vector) kernels, any M (in chunks)  */
    LOWBIT_PATH_QMM = 2      /* tensor-core (tcgen05) matrix-matrix kernel, any M  */
} lowbit_path;

/* Element type of a floating-point input that is not fixed by the method. */
typedef enum {
    LOWBIT_DTYPE_F32 = 0,    /* IEEE binary32                                     */
    LOWBIT_DTYPE_BF16 = 1,   /* bfloat16 bit patterns (uint16_t)                  */
    LOWBIT_DTYPE_F16 = 2     /* IEEE binary16 bit patterns (uint16_t)             */
} lowbit_dtype;

/* Human-readable name of a status code.  Never NULL. */
LOWBIT_API const char *lowbit_status_string(lowbit_status status);

/* Bytes of a packed [N, K] matrix of b-bit codes: N * K * bits / 8.
 * Returns 0 when bits is not in 1..7, N or K is negative, or K*bits is not a
 * multiple of 8 (ao PR #2167, Summary, bullet 2: rows are contiguous bit
 * streams, so a row only ends on a byte boundary when K*b % 8 == 0). */
LOWBIT_API size_t lowbit_packed_bytes(int64_t N, int64_t K, int bits);

/* Pack one-code-per-byte codes into the contiguous b-bit layout
 * (ao PR #2167, Summary, bullet 2; the `_pack_weight_{n}bit` op of
 * ao issue #3446, one function here for every bit width).
 *   codes   [N, K] uint8, row-major, device, 8-byte aligned.  Only the low
 *           `bits` bits of each byte are used; higher bits are ignored.
 *   packed  [N, K*bits/8] uint8, row-major, device, written in full.
 *   N >= 0, K >= 0 with K % 8 == 0, bits in 1..7.
 * Errors: LOWBIT_EINVAL for a bad size, bit width, null pointer (when the
 * matrix is not empty) or misaligned `codes`; LOWBIT_EUNSUPPORTED on a device
 * that is not sm_103; LOWBIT_ECUDA when the launch fails.  N == 0 or K == 0
 * is a valid empty call that launches nothing. */
LOWBIT_API lowbit_status lowbit_pack_weights(const uint8_t *codes, uint8_t *packed,
                                  int64_t N, int64_t K, int bits, lowbit_stream_t stream);

/* Inverse of lowbit_pack_weights: one code per output byte (0 .. 2^bits-1).
 * Same layouts, sizes, alignment and errors as lowbit_pack_weights, with
 * `codes` the output (8-byte aligned). */
LOWBIT_API lowbit_status lowbit_unpack_weights(const uint8_t *packed, uint8_t *codes,
                                    int64_t N, int64_t K, int bits, lowbit_stream_t stream);

/* Quantise a floating-point weight matrix groupwise and write it in the
 * packed layout, with its scales and zeros (the `_quantize` step of
 * ao PR #2167, Summary, bullet 1, which produces N x num_groups scales and
 * zeros; the pages do not define it, so this is the min/max asymmetric reading):
 *     zero  = fp16 rounded toward -inf of min(w over the group)
 *     scale = fp16 rounded toward +inf of (max - zero) / (2^bits - 1)
 *     q     = clamp(round-half-to-even((w - zero) / scale), 0, 2^bits - 1)
 * The minimum of a group holding both signed zeros is the first zero in k
 * order.  A constant group (max == min) gets q = 0 and scale = the larger of
 * 2^-14 and fp16 rounded toward +inf of 2 (min - zero).  Every decision is
 * taken in fp64, so the outputs are fully determined by w.
 * Then |w - (scale*q + zero)| <= scale/2 for every weight.
 *   w        [N, K] of `dtype`, row-major, device, 16-byte aligned.
 *            Values must be finite with magnitude at most 32752, so that a
 *            group's zero and range fit fp16.
 *   packed   [N, K*bits/8] uint8, device, written in full (any alignment).
 *   scales   [N, K/group] fp16, row-major, device, 2-byte aligned.
 *   zeros    [N, K/group] fp16, row-major, device, 2-byte aligned.
 *   N >= 0, K > 0, group in {32, 64, 128, 256}, K % group == 0, bits in 1..7.
 *   N == 0 is a valid empty call.  Outputs must not overlap w or each other.
 * Errors: LOWBIT_EINVAL for a bad size, bit width, group, dtype, null or
 * misaligned pointer; LOWBIT_EUNSUPPORTED on a device that is not sm_103;
 * LOWBIT_ECUDA when the launch fails. */
LOWBIT_API lowbit_status lowbit_quantize_weights(const void *w, lowbit_dtype dtype,
                                      uint8_t *packed, uint16_t *scales, uint16_t *zeros,
                                      int64_t N, int64_t K, int bits, int group,
                                      lowbit_stream_t stream);

/* The quantised linear layer (torchchat PR #1415; ao PR #2167 Summary
 * bullets 1-3; bias per ao issue #3446):
 *     y[m,n] = bf16_rn( sum_k x[m,k] * (scale[n,k/g]*q[n,k] + zero[n,k/g]) + bias[n] )
 * accumulated in fp32.
 *   x        [M, K] bf16, row-major, device, 16-byte aligned.
 *   packed_w [N, K*bits/8] uint8 in the packed layout above, 16-byte aligned.
 *   scales   [N, K/group] fp16, row-major, device, 2-byte aligned.
 *   zeros    [N, K/group] fp16, row-major, device, 2-byte aligned.  The zero
 *            is an additive offset: W = scale*q + zero.
 *   bias     [N] fp16 or NULL (no bias), 2-byte aligned.
 *   y        [M, N] bf16, row-major, device, 2-byte aligned; written in full.
 *            y must not overlap any input.
 *   M >= 0, N >= 0, K > 0, group in {32, 64, 128, 256}, K % group == 0,
 *   bits in 1..7.  M == 0 or N == 0 is a valid empty call.
 * The kernel is picked by lowbit_select_path.
 * Errors: LOWBIT_EINVAL for a bad size, bit width, group, null pointer or
 * misaligned pointer; LOWBIT_EUNSUPPORTED on a device that is not sm_103;
 * LOWBIT_ECUDA when a launch fails. */
LOWBIT_API lowbit_status lowbit_linear(const uint16_t *x, const uint8_t *packed_w,
                            const uint16_t *scales, const uint16_t *zeros,
                            const uint16_t *bias, uint16_t *y,
                            int64_t M, int64_t K, int64_t N, int bits, int group,
                            lowbit_stream_t stream);

/* lowbit_linear with the kernel chosen by the caller (both kernels are
 * correct for every M; this is how each is tested and timed on its own).
 * Same arguments and errors as lowbit_linear, plus LOWBIT_EINVAL for an
 * unknown `path` and LOWBIT_EUNSUPPORTED when LOWBIT_PATH_QMM is asked for a
 * shape the tensor-core kernel does not take (K not a multiple of 128). */
LOWBIT_API lowbit_status lowbit_linear_ex(const uint16_t *x, const uint8_t *packed_w,
                               const uint16_t *scales, const uint16_t *zeros,
                               const uint16_t *bias, uint16_t *y,
                               int64_t M, int64_t K, int64_t N, int bits, int group,
                               lowbit_path path, lowbit_stream_t stream);

/* Gate and up projections of a gated MLP fused into one decode call: with the
 * packed matrix holding 2F rows -- rows [0, F) the gate projection, rows
 * [F, 2F) the up projection, each quantised as for lowbit_linear --
 *     a[m,f] = sum_k x[m,k] W[f,k]   + bias[f]
 *     u[m,f] = sum_k x[m,k] W[F+f,k] + bias[F+f]
 *     y[m,f] = silu(a[m,f]) * u[m,f],   silu(a) = a / (1 + e^-a),
 * computed in fp32 and rounded once to bf16 (a and u are never rounded).
 * This is the decode step the pages time (torchchat PR #1415 and ao PR #2167
 * measure Llama token generation, whose MLP applies this activation to its
 * gate and up projections); it saves one launch and one pass over a and u.
 * It runs the decode kernels for every M (up to 8 rows of x per launch on the
 * tensor-core decode kernel, two on the CUDA-core one), so it is meant for
 * decode-sized M.
 *   x        [M, K] bf16, as for lowbit_linear.
 *   packed_w [2F, K*bits/8], scales and zeros [2F, K/group], bias NULL or
 *            [2F] fp16: layouts, alignment and ownership as for lowbit_linear
 *            with N = 2F.
 *   y        [M, F] bf16, device, 2-byte aligned, written in full.
 *   F >= 0; every other size limit as for lowbit_linear.  M == 0 or F == 0 is
 *   a valid empty call.
 * Errors: as for lowbit_linear (LOWBIT_EINVAL also for F < 0). */
LOWBIT_API lowbit_status lowbit_linear_swiglu(const uint16_t *x, const uint8_t *packed_w,
                                   const uint16_t *scales, const uint16_t *zeros,
                                   const uint16_t *bias, uint16_t *y,
                                   int64_t M, int64_t K, int64_t F, int bits, int group,
                                   lowbit_stream_t stream);

/* The kernel lowbit_linear runs for this problem, from crossovers measured on
 * GB300: LOWBIT_PATH_QMV when the tensor-core decode kernel takes the shape
 * (K a multiple of 256 up to 32768 with K/group a multiple of 8; one launch
 * per 2 rows of x for group 32, 4 for group 64, 8 for groups 128 and 256) in
 * at most 128/group launches (one for groups 128 and 256), twice as many when
 * N >= 24576 and group <= 128, and, when K > 8192, for M <= 4 (groups 128,
 * 256), 6 (64) or 8 (32); for other K, M <= 2, or M <= 6 when N >= 9424; and
 * whenever K is not a multiple of 128.
 * LOWBIT_PATH_QMM otherwise.  The choice assumes x, the packed weights,
 * scales and zeros 16-byte aligned (the decode path still runs, slower,
 * when they are not).
 * Host-only; never touches the GPU.  Returns LOWBIT_PATH_AUTO for arguments
 * lowbit_linear would reject. */
LOWBIT_API lowbit_path lowbit_select_path(int64_t M, int64_t K, int64_t N, int bits, int group);

/* Every wait inside the library's kernels (a stage of streamed weights, a
 * tensor-core completion) is bounded: one that has not completed after about
 * one second gives up, the kernel finishes without that data (its outputs are
 * then unspecified) and a device-side counter is incremented.  This returns
 * the counter for the current device in *count (0 in normal operation) and
 * clears it when `reset` is non-zero.  Synchronises the current device.
 * Errors: LOWBIT_EINVAL for a NULL `count`; LOWBIT_EUNSUPPORTED on a device
 * that is not sm_103; LOWBIT_ECUDA when the synchronisation or the read
 * fails (for instance after an earlier kernel fault). */
LOWBIT_API lowbit_status lowbit_wait_timeouts(uint32_t *count, int reset);

/* Self-test of the bounded waits: enqueues one single-thread kernel that waits,
 * through the library's bounded-wait helper, on a barrier nothing completes.
 * After the wait limit (about one second) it gives up, writes 1 to *gave_up
 * and counts one timeout (seen by lowbit_wait_timeouts); the kernel then
 * returns normally, so the device stays usable.
 *   gave_up  device pointer to one uint32_t, 4-byte aligned, written by the kernel.
 * Errors: LOWBIT_EINVAL for a NULL or misaligned pointer; LOWBIT_EUNSUPPORTED
 * on a device that is not sm_103; LOWBIT_ECUDA when the launch fails. */
LOWBIT_API lowbit_status lowbit_selftest_wait_timeout(uint32_t *gave_up, lowbit_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LOWBIT_H */
