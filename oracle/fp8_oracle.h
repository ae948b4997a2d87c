/*
 * fp8_oracle.h -- plain, slow CPU oracle for scaled FP8 quantisation and the
 * FP8 GEMM that consumes it.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this code: only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark use it.  It shares no code, header, table or constant with the
 * CUDA library; the two agree only because both follow the same definitions.
 *
 * Source pages (cited by title and section):
 *   [fp8_parity]  "fp8_parity.py" (mlinterviewnotes.com, FP8 numerics lab):
 *                 constants E4M3_MAX / E5M2_MAX, function scaled_roundtrip,
 *                 class FP8Matmul, smoke steps 1-4.
 *   [te_blog]     "How to Optimize Transformer-Based Models for Low-Precision
 *                 Training" (NVIDIA blog repost): Fprop/Dgrad/Wgrad GEMM shapes,
 *                 delayed scaling with an amax history.
 *
 * Every function is single-threaded, takes fp32 or bf16 input and computes in
 * the precision the definition states (fp32 for scale and quotient, double for
 * GEMM sums).  Build with -ffp-contract=off so that no a*b+c is fused.
 *
 * Pinning (the tests that tie this oracle to something other than itself):
 *   encode/decode  -> torch CPU float8 casts, exhaustive over bf16 and all bytes
 *   quantize_*     -> the pages' scaled_roundtrip run on torch CPU ops, and the
 *                     smoke-step bounds printed on the fp8_parity page
 *   delayed        -> brute-force ring bookkeeping on short histories
 *   gemm           -> exact rational brute force on tiny shapes, numpy float64
 *                     matmul of decoded operands, closed forms (one-hot rows)
 *   MX (MXFP8)     -> torch's CPU float8_e8m0fnu decode of every scale byte,
 *                     the defining bracket of the shared exponent checked in
 *                     exact rationals, brute-force nearest-value search over
 *                     all 256 element codes, torch's CPU float8 casts
 * No function here is "parity unpinned".
 */
#ifndef FP8_ORACLE_H
#define FP8_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Format tags.  E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits, no
 * infinity, NaN = S.1111.111, largest finite 448.  E5M2: 1 sign, 5 exponent
 * (bias 15), 2 mantissa bits, IEEE-style Inf/NaN, largest finite 57344. */
#define ORC_E4M3 0
#define ORC_E5M2 1

/* Input element types. */
#define ORC_IN_F32 0
#define ORC_IN_BF16 1

/* Scale granularities (GEMM operand description). */
#define ORC_SCALE_TENSOR 0
#define ORC_SCALE_TILE 1   /* one scale per row per 128-wide K block */
#define ORC_SCALE_BLOCK 2  /* one scale per 128x128 block            */
#define ORC_SCALE_ROW 3    /* one scale per row over all of K         */
#define ORC_SCALE_MX 4     /* one E8M0 scale per row per 32-wide K block */

double orc_fmax(int fmt);

/* Widen element i of an fp32 or bf16 array to fp32 (exact). */
float orc_load(const void *x, int in_dtype, int64_t i);

/* FP8 byte -> value (NaN / +-Inf where the format has them). */
double orc_fp8_decode(uint8_t code, int fmt);

/* fp32 value -> FP8 byte, round to nearest, ties to even.
 * saturate == 0: magnitudes that round above the largest finite value become
 *                NaN (E4M3) or Inf (E5M2), as a plain cast does.
 * saturate != 0: they clamp to +-fmax.
 * NaN -> 0x7F with the NaN's sign bit, in both formats and both modes. */
uint8_t orc_fp8_encode(float v, int fmt, int saturate);

/* max |x| over n elements; NaN if any element is NaN. */
float orc_amax(const void *x, int in_dtype, int64_t n);

/* s = fl32(amax / fmax), then clamped below at fl32(1e-12). */
float orc_scale_from_amax(float amax, int fmt);

/* q[i] = encode(fl32(x[i] / s)) over n elements. */
void orc_cast(const void *x, int in_dtype, int64_t n, float s, int fmt,
              int saturate, uint8_t *q);

/* Per-tensor quantisation of a row-major [rows, cols] matrix with a given
 * scale.  q (nullable) is [rows, cols]; q_t (nullable) is [cols, rows]. */
void orc_quantize_tensor(const void *x, int in_dtype, int64_t rows,
                         int64_t cols, float s, int fmt, int saturate,
                         uint8_t *q, uint8_t *q_t);

/* 1x128 tiles along each row: tile (r, kb) covers columns
 * [128 kb, min(cols, 128 kb + 128)).  q is [rows, cols];
 * scales is [ceil(cols/128), rows]: scale(r, kb) = scales[kb * rows + r]. */
void orc_quantize_tile_rows(const void *x, int in_dtype, int64_t rows,
                            int64_t cols, int fmt, int saturate, uint8_t *q,
                            float *scales);

/* 128x1 tiles down each column, written transposed: q_t is [cols, rows] and
 * scales is [ceil(rows/128), cols]: scale(c, rb) = scales[rb * cols + c].
 * This is exactly orc_quantize_tile_rows applied to the transpose. */
void orc_quantize_tile_cols(const void *x, int in_dtype, int64_t rows,
                            int64_t cols, int fmt, int saturate, uint8_t *q_t,
                            float *scales);

/* 128x128 blocks: scales is [ceil(rows/128), ceil(cols/128)] row-major.
 * q and q_t (each nullable) as in orc_quantize_tensor. */
void orc_quantize_block(const void *x, int in_dtype, int64_t rows,
                        int64_t cols, int fmt, int saturate, uint8_t *q,
                        uint8_t *q_t, float *scales);

/* Row-wise scaling (the fp8_parity page's torchao "rowwise" recipe, read as
 * one scale per row of each K-major GEMM operand): either or both of
 *   q [rows, cols] with q_scales[rows]: row r scaled by its own amax over
 *     all columns;
 *   q_t [cols, rows] with qt_scales[cols]: column c of x (row c of x^T)
 *     scaled by its own amax over all rows.
 * Each pair may be NULL. */
void orc_quantize_rowwise(const void *x, int in_dtype, int64_t rows,
                          int64_t cols, int fmt, int saturate, uint8_t *q,
                          float *q_scales, uint8_t *q_t, float *qt_scales);

/* Delayed scaling with an amax history ring of hist_len entries.
 * s = max(history) / fmax (clamped as orc_scale_from_amax); x is cast with s;
 * then amax(x) overwrites history[*next] and *next advances modulo hist_len.
 * Returns s. */
float orc_quantize_delayed(const void *x, int in_dtype, int64_t rows,
                           int64_t cols, int fmt, int saturate, float *history,
                           int32_t hist_len, int32_t *next, uint8_t *q,
                           uint8_t *q_t);

/* d[i] = fl32(decode(q[i]) * s). */
void orc_dequantize(const uint8_t *q, int64_t n, int fmt, float s, float *d);

/* ------------------------------------------------------------------ MXFP8
 * The Transformer Engine recipe "mxfp8" that the SpikingJelly precision page
 * lists (fp8_recipe) and that the low-precision-training blog repost uses as
 * its Blackwell baseline.  The pages give no encoding, so these functions
 * follow the public OCP Microscaling Formats (MX) Specification v1.0:
 *   - a block is ORC_MX_BLOCK = 32 consecutive elements along a row (the
 *     contraction dimension of the GEMM operand); the last block of a row
 *     may be shorter;
 *   - the block's shared scale X is an E8M0 byte: unsigned 8-bit exponent,
 *     bias 127, X = 2^(code - 127); code 0xFF is NaN; there is no zero;
 *   - elements are FP8 E4M3 or E5M2 (MXFP8);
 *   - conversion (the specification's vector-to-MX algorithm):
 *       shared_exp = floor(log2(max_i |V_i|)) - emax_elem, where emax_elem is
 *       the exponent of the element format's largest normal (8 for E4M3,
 *       whose largest value is 448 = 1.75 * 2^8; 15 for E5M2, 57344 =
 *       1.75 * 2^15), clamped to the E8M0 range [-127, 127];
 *       X = 2^shared_exp;
 *       P_i = V_i / X rounded to nearest, ties to even, into the element
 *       format, with finite magnitudes beyond its largest normal clamped to
 *       it.
 * Readings where the specification leaves a case open:
 *   - a block whose elements are all zero has max 0, floor(log2 0) = -inf,
 *     which the clamp takes to -127: code 0x00, elements +-0;
 *   - a block holding a NaN or an infinity gets the NaN scale 0xFF; the
 *     whole block then decodes to NaN whatever its elements hold, and every
 *     element byte is written as 0x7F (a NaN code in both formats).
 * V_i / X is exact (X is a power of two and the quotient is formed in
 * double), so the element rounding is the only rounding. */
#define ORC_MX_BLOCK 32

/* E8M0 byte -> 2^(code - 127), or NaN for 0xFF. */
double orc_e8m0_decode(uint8_t code);

/* E8M0 code of the shared scale of a block whose max |V_i| is amax. */
uint8_t orc_mx_scale_code(float amax, int fmt);

/* 1x32 blocks along each row: q [rows, cols], scales [rows, ceil(cols/32)]
 * row-major: scale(r, j) = scales[r * ceil(cols/32) + j] for the block of
 * columns [32 j, min(cols, 32 j + 32)). */
void orc_quantize_mx_rows(const void *x, int in_dtype, int64_t rows,
                          int64_t cols, int fmt, uint8_t *q, uint8_t *scales);

/* 32x1 blocks down each column, written transposed: q_t [cols, rows],
 * scales [cols, ceil(rows/32)].  Exactly orc_quantize_mx_rows of x^T. */
void orc_quantize_mx_cols(const void *x, int in_dtype, int64_t rows,
                          int64_t cols, int fmt, uint8_t *q_t, uint8_t *scales);

/* One GEMM operand: data is row-major [rows, K] FP8 bytes.
 *   TENSOR: scale[0]
 *   TILE:   scale[kb * stride_k + row * stride_row]
 *   BLOCK:  scale[(row / 128) * stride_row + kb * stride_k]
 *   ROW:    scale[row * stride_row]
 *   MX:     e8m0_decode(mx_scale[row * stride_row + (k / 32) * stride_k])
 * with kb = k / 128. */
typedef struct {
  const uint8_t *data;
  int32_t fmt;
  int32_t scaling;
  const float *scale;
  int64_t stride_row;
  int64_t stride_k;
  const uint8_t *mx_scale; /* MX only: E8M0 codes */
} orc_operand;

/* Scale of element (row, k) of an operand, as defined above (every E8M0
 * value is exact in double; 2^-127 is an fp32 subnormal, so double is the
 * return type). */
double orc_operand_scale(const orc_operand *op, int64_t row, int64_t k);

/* Reference GEMM on a list of output positions:
 *   y[i]     = sum_k decode(A[m,k]) sA(m,k) * decode(B[n,k]) sB(n,k)
 *   absum[i] = sum_k |same product|
 * with (m, n) = (ms[i], ns[i]), accumulated in double. */
void orc_gemm_points(const orc_operand *A, const orc_operand *B, int64_t K,
                     int64_t npts, const int64_t *ms, const int64_t *ns,
                     double *y, double *absum);

/* The same over a dense block of rows [m0, m1) x all n in [0, N):
 * y and absum are [(m1 - m0), N] row-major. */
void orc_gemm_rows(const orc_operand *A, const orc_operand *B, int64_t N,
                   int64_t K, int64_t m0, int64_t m1, double *y,
                   double *absum);

#ifdef __cplusplus
}
#endif
#endif
