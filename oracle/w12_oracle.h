/*
 * W12 oracle — TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, scalar C restatement of the W12 v1 weight format and of the
 * GEMM it feeds.  Only the test suite, the smoke check and the CPU-baseline leg
 * of the benchmark may load it.  It shares no code, header, table or helper with
 * the product library (the CUDA kernels and the host encoder); the two are
 * written independently and compared against each other.
 *
 * What the pages fix (SpecPilot, three pages):
 *   - "StargazerX0/SpecPilot" (hotrepo.ai), §What it is: W12 is a 12-bit weight
 *     format that decodes bit-exactly inside the GEMM.
 *   - "SpecPilot" (fasttoolhub.com), §Differentiation: a general, lossless
 *     12-bit weight format.
 *   - "SpecPilot: an agent doubled speculative decoding speed, and the 10.87x
 *     needs context" (ai.jakubjirak.com), §The mechanisms it found: about
 *     12.01-12.02 bits per weight on dense models, decoded in GEMM registers;
 *     reading 12 instead of 16 bits cuts weight traffic by a quarter.
 * The pages give no bit layout, so the concrete layout (W12 v1: sign + 7-bit
 * mantissa byte, 4-bit code into a per-segment table of 15 frequent exponents,
 * escape code 15 with a side list of raw exponents) is the one this project
 * defines; every step below follows that definition in its own order.
 *
 * Pins (tests that tie this file to something other than itself):
 *   encode/decode : exhaustive round trip of all 65536 BF16 patterns (the
 *                   "lossless"/"bit-exactly" property), a hand-worked 2x2
 *                   example, a hand-worked blob with five escapes over two
 *                   quarters, two chunks and two segments (escape bytes,
 *                   bases, counts and masks listed by hand),
 *                   table-optimality and escape-mass invariants, the
 *                   size closed form, normal-CDF escape rate on Gaussian data.
 *   gemm_f64      : numpy float64 matmul, one-hot and small-integer exact cases.
 *   q8 encode     : a hand-worked row, the scale/range invariants, the
 *                   half-step rounding bound, ties to even.
 *   q8 product    : one-hot and small-integer products worked by hand.
 */
#ifndef W12_ORACLE_H
#define W12_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Total size in bytes of the W12 v1 blob for the N x K BF16 matrix w
 * (row-major, bit patterns).  Returns -1 on bad arguments. */
int64_t oracle_w12_size(const uint16_t *w, int64_t N, int64_t K);

/* Encode w into blob (cap bytes).  Returns the blob size, or -1 if cap is too
 * small or the arguments are bad. */
int64_t oracle_w12_encode(const uint16_t *w, int64_t N, int64_t K,
                          uint8_t *blob, int64_t cap);

/* Decode a blob of len bytes into w_out (N x K, N and K read from the header).
 * Returns 0 on success, -1 if the blob is malformed. */
int oracle_w12_decode(const uint8_t *blob, int64_t len, uint16_t *w_out);

/* Read N and K from a blob header; returns 0 on success. */
int oracle_w12_dims(const uint8_t *blob, int64_t len, int64_t *N, int64_t *K);

/* y[m*N + n] = sum_k x[m*K + k] * w[n*K + k], every term and the sum in
 * double precision; x and w are BF16 bit patterns. */
void oracle_gemm_f64(const uint16_t *x, const uint16_t *w, int64_t M,
                     int64_t N, int64_t K, double *y);

/* The same GEMM over the weights held in a W12 blob: decode rows one by one,
 * then take the fp64 dot products.  Used as the CPU baseline.  Runs on
 * `threads` OpenMP threads when built with OpenMP (<= 0: the runtime default).
 * Returns 0 on success, -1 on a malformed blob. */
int oracle_w12_gemm_f64(const uint16_t *x, const uint8_t *blob, int64_t len,
                        int64_t M, double *y, int threads);

/* Number of OpenMP threads a parallel region would use (1 without OpenMP). */
int oracle_max_threads(int threads);

/* Q8 weight copy (see w12_oracle.c for the scheme and layout).  Size of the
 * Q8 v1 blob of an N x K matrix (-1 on bad arguments). */
int64_t oracle_q8_size(int64_t N, int64_t K);

/* Quantize w (N x K BF16 bit patterns) into blob; returns the size, or -1 on
 * bad arguments, a short buffer or a non-finite weight. */
int64_t oracle_q8_encode(const uint16_t *w, int64_t N, int64_t K, uint8_t *blob, int64_t cap);

/* Read scales[N] and q[N*K] (row-major) back from a Q8 blob; 0 on success. */
int oracle_q8_decode(const uint8_t *blob, int64_t len, float *scales, int8_t *q);

#ifdef __cplusplus
}
#endif
#endif
