/*
 * fp8_oracle.c -- see fp8_oracle.h.  TEST INFRASTRUCTURE ONLY.
 *
 * Each function restates a definition from the pages in the most literal
 * form available; speed is irrelevant.  The arithmetic happens in the
 * precision named in the comments, never in anything wider by accident
 * (compile with -ffp-contract=off; FLT_EVAL_METHOD is 0 on x86-64 and
 * aarch64).
 */
#include "fp8_oracle.h"

#include <math.h>
#include <string.h>

/* ---------------------------------------------------------------- formats */

/* Field layout of the two FP8 formats ([fp8_parity] docstring: E4M3 has 3
 * mantissa bits and range 448, E5M2 has 2 mantissa bits and range 57344;
 * smallest normals 2^-6 and 2^-14 in smoke step 1). */
typedef struct {
  int exp_bits;
  int man_bits;
  int bias;
  double fmax;
  int has_inf; /* E5M2 reserves exponent 31 for Inf/NaN; E4M3 only S.1111.111 */
} fmt_desc;

static fmt_desc describe(int fmt) {
  fmt_desc d;
  if (fmt == ORC_E4M3) {
    d.exp_bits = 4;
    d.man_bits = 3;
    d.bias = 7;
    d.fmax = 448.0; /* E4M3_MAX in fp8_parity.py */
    d.has_inf = 0;
  } else {
    d.exp_bits = 5;
    d.man_bits = 2;
    d.bias = 15;
    d.fmax = 57344.0; /* E5M2_MAX in fp8_parity.py */
    d.has_inf = 1;
  }
  return d;
}

double orc_fmax(int fmt) { return describe(fmt).fmax; }

float orc_load(const void *x, int in_dtype, int64_t i) {
  if (in_dtype == ORC_IN_F32) return ((const float *)x)[i];
  /* bf16 is the top half of an fp32 bit pattern: widening appends 16 zero
   * bits and is exact. */
  uint32_t bits = (uint32_t)((const uint16_t *)x)[i] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return f;
}

double orc_fp8_decode(uint8_t code, int fmt) {
  fmt_desc d = describe(fmt);
  int sign = code >> 7;
  int e = (code >> d.man_bits) & ((1 << d.exp_bits) - 1);
  int m = code & ((1 << d.man_bits) - 1);
  int e_all_ones = (1 << d.exp_bits) - 1;
  double v;
  if (d.has_inf && e == e_all_ones) {
    v = (m == 0) ? INFINITY : NAN;
  } else if (!d.has_inf && e == e_all_ones && m == (1 << d.man_bits) - 1) {
    v = NAN;
  } else if (e == 0) {
    /* subnormal: 0.m * 2^(1 - bias) */
    v = ldexp((double)m, 1 - d.bias - d.man_bits);
  } else {
    /* normal: 1.m * 2^(e - bias) */
    v = ldexp((double)((1 << d.man_bits) + m), e - d.bias - d.man_bits);
  }
  return sign ? -v : v;
}

/* Round a non-negative finite magnitude to the FP8 grid of `d`, ignoring the
 * upper end of the range (the caller checks overflow on the result).  The
 * grid spacing in the binade [2^e, 2^(e+1)) is 2^(e - man_bits); below the
 * smallest normal 2^(1-bias) the spacing stays at the subnormal quantum. */
static double round_to_grid(double a, fmt_desc d) {
  if (a == 0.0) return 0.0;
  int ex;
  frexp(a, &ex); /* a = f * 2^ex with f in [0.5, 1) -> binade exponent ex-1 */
  int e = ex - 1;
  int emin = 1 - d.bias;
  if (e < emin) e = emin;
  double quantum = ldexp(1.0, e - d.man_bits);
  double n = a / quantum;   /* exact: division by a power of two */
  double r = floor(n);
  double frac = n - r;      /* exact */
  if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
  return r * quantum;       /* exact */
}

/* Round-to-nearest-even of a double into the format (see orc_fp8_encode);
 * every fp32 value is exact in double, so the fp32 entry point is this one. */
static uint8_t encode_double(double v, int fmt, int saturate) {
  fmt_desc d = describe(fmt);
  uint8_t sign = signbit(v) ? 0x80 : 0x00;
  if (isnan(v)) return (uint8_t)(sign | 0x7F);

  uint8_t max_code = (uint8_t)(fmt == ORC_E4M3 ? 0x7E : 0x7B);
  uint8_t ovf_code = (uint8_t)(fmt == ORC_E4M3 ? 0x7F : 0x7C); /* NaN / Inf */

  double a = fabs((double)v);
  double mag = isinf(a) ? INFINITY : round_to_grid(a, d);
  if (mag > d.fmax) return (uint8_t)(sign | (saturate ? max_code : ovf_code));
  if (mag == 0.0) return sign;

  int ex;
  frexp(mag, &ex);
  int e = ex - 1;
  int emin = 1 - d.bias;
  int biased, mant;
  if (e < emin) {
    biased = 0;
    mant = (int)(mag / ldexp(1.0, emin - d.man_bits));
  } else {
    biased = e + d.bias;
    mant = (int)(mag / ldexp(1.0, e - d.man_bits)) - (1 << d.man_bits);
  }
  return (uint8_t)(sign | (biased << d.man_bits) | mant);
}

uint8_t orc_fp8_encode(float v, int fmt, int saturate) {
  return encode_double((double)v, fmt, saturate);
}

/* ------------------------------------------------------------ amax / scale */

/* amax = max |x| ([fp8_parity] scaled_roundtrip: x.abs().max()).  A NaN
 * anywhere makes the result NaN, as torch's max does. */
float orc_amax(const void *x, int in_dtype, int64_t n) {
  float m = 0.0f;
  for (int64_t i = 0; i < n; ++i) {
    float a = fabsf(orc_load(x, in_dtype, i));
    if (isnan(a)) return a;
    if (a > m) m = a;
  }
  return m;
}

/* s = (amax / fmax).clamp_min(1e-12) in fp32 ([fp8_parity] scaled_roundtrip).
 * A NaN amax stays NaN (clamp_min propagates NaN). */
float orc_scale_from_amax(float amax, int fmt) {
  float s = amax / (float)describe(fmt).fmax;
  const float floor_s = (float)1e-12;
  if (s < floor_s) s = floor_s;
  return s;
}

/* ------------------------------------------------------------------- casts */

/* q = (x / scale).to(fp8) ([fp8_parity] scaled_roundtrip): an fp32 IEEE
 * division, then one round-to-nearest-even into the format.
 * NaN (the pages never meet one; IEEE 754 leaves the sign of a NaN result
 * open and x86 and aarch64 disagree on it): a NaN input keeps its sign, as
 * the plain cast does (0x7F | sign); a NaN that the division itself creates
 * (NaN scale, Inf / Inf) is encoded 0x7F. */
static uint8_t cast_one(float xv, float s, int fmt, int saturate) {
  if (isnan(xv)) return (uint8_t)(0x7F | (signbit(xv) ? 0x80 : 0x00));
  float v = xv / s;
  if (isnan(v)) return 0x7F;
  return orc_fp8_encode(v, fmt, saturate);
}

void orc_cast(const void *x, int in_dtype, int64_t n, float s, int fmt,
              int saturate, uint8_t *q) {
  for (int64_t i = 0; i < n; ++i)
    q[i] = cast_one(orc_load(x, in_dtype, i), s, fmt, saturate);
}

void orc_quantize_tensor(const void *x, int in_dtype, int64_t rows,
                         int64_t cols, float s, int fmt, int saturate,
                         uint8_t *q, uint8_t *q_t) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) {
      uint8_t b = cast_one(orc_load(x, in_dtype, r * cols + c), s, fmt, saturate);
      if (q) q[r * cols + c] = b;
      if (q_t) q_t[c * rows + r] = b;
    }
}

/* [fp8_parity] smoke step 4 applies scaled_roundtrip to each 1x128 piece of a
 * row independently: one amax, one scale, one cast per tile. */
void orc_quantize_tile_rows(const void *x, int in_dtype, int64_t rows,
                            int64_t cols, int fmt, int saturate, uint8_t *q,
                            float *scales) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c0 = 0; c0 < cols; c0 += 128) {
      int64_t c1 = c0 + 128 < cols ? c0 + 128 : cols;
      float amax = 0.0f;
      int nan_seen = 0;
      for (int64_t c = c0; c < c1; ++c) {
        float a = fabsf(orc_load(x, in_dtype, r * cols + c));
        if (isnan(a)) nan_seen = 1;
        else if (a > amax) amax = a;
      }
      if (nan_seen) amax = NAN;
      float s = orc_scale_from_amax(amax, fmt);
      scales[(c0 / 128) * rows + r] = s;
      for (int64_t c = c0; c < c1; ++c)
        q[r * cols + c] = cast_one(orc_load(x, in_dtype, r * cols + c), s, fmt, saturate);
    }
}

void orc_quantize_tile_cols(const void *x, int in_dtype, int64_t rows,
                            int64_t cols, int fmt, int saturate, uint8_t *q_t,
                            float *scales) {
  for (int64_t c = 0; c < cols; ++c)
    for (int64_t r0 = 0; r0 < rows; r0 += 128) {
      int64_t r1 = r0 + 128 < rows ? r0 + 128 : rows;
      float amax = 0.0f;
      int nan_seen = 0;
      for (int64_t r = r0; r < r1; ++r) {
        float a = fabsf(orc_load(x, in_dtype, r * cols + c));
        if (isnan(a)) nan_seen = 1;
        else if (a > amax) amax = a;
      }
      if (nan_seen) amax = NAN;
      float s = orc_scale_from_amax(amax, fmt);
      scales[(r0 / 128) * cols + c] = s;
      for (int64_t r = r0; r < r1; ++r)
        q_t[c * rows + r] = cast_one(orc_load(x, in_dtype, r * cols + c), s, fmt, saturate);
    }
}

void orc_quantize_block(const void *x, int in_dtype, int64_t rows,
                        int64_t cols, int fmt, int saturate, uint8_t *q,
                        uint8_t *q_t, float *scales) {
  int64_t ncb = (cols + 127) / 128;
  for (int64_t r0 = 0; r0 < rows; r0 += 128)
    for (int64_t c0 = 0; c0 < cols; c0 += 128) {
      int64_t r1 = r0 + 128 < rows ? r0 + 128 : rows;
      int64_t c1 = c0 + 128 < cols ? c0 + 128 : cols;
      float amax = 0.0f;
      int nan_seen = 0;
      for (int64_t r = r0; r < r1; ++r)
        for (int64_t c = c0; c < c1; ++c) {
          float a = fabsf(orc_load(x, in_dtype, r * cols + c));
          if (isnan(a)) nan_seen = 1;
          else if (a > amax) amax = a;
        }
      if (nan_seen) amax = NAN;
      float s = orc_scale_from_amax(amax, fmt);
      scales[(r0 / 128) * ncb + c0 / 128] = s;
      for (int64_t r = r0; r < r1; ++r)
        for (int64_t c = c0; c < c1; ++c) {
          uint8_t b = cast_one(orc_load(x, in_dtype, r * cols + c), s, fmt, saturate);
          if (q) q[r * cols + c] = b;
          if (q_t) q_t[c * rows + r] = b;
        }
    }
}

/* Row-wise scaling: scaled_roundtrip applied to each whole row (and, for the
 * transposed copy, to each whole column). */
void orc_quantize_rowwise(const void *x, int in_dtype, int64_t rows,
                          int64_t cols, int fmt, int saturate, uint8_t *q,
                          float *q_scales, uint8_t *q_t, float *qt_scales) {
  if (q) {
    for (int64_t r = 0; r < rows; ++r) {
      float amax = 0.0f;
      int nan_seen = 0;
      for (int64_t c = 0; c < cols; ++c) {
        float a = fabsf(orc_load(x, in_dtype, r * cols + c));
        if (isnan(a)) nan_seen = 1;
        else if (a > amax) amax = a;
      }
      if (nan_seen) amax = NAN;
      float s = orc_scale_from_amax(amax, fmt);
      q_scales[r] = s;
      for (int64_t c = 0; c < cols; ++c)
        q[r * cols + c] = cast_one(orc_load(x, in_dtype, r * cols + c), s, fmt, saturate);
    }
  }
  if (q_t) {
    for (int64_t c = 0; c < cols; ++c) {
      float amax = 0.0f;
      int nan_seen = 0;
      for (int64_t r = 0; r < rows; ++r) {
        float a = fabsf(orc_load(x, in_dtype, r * cols + c));
        if (isnan(a)) nan_seen = 1;
        else if (a > amax) amax = a;
      }
      if (nan_seen) amax = NAN;
      float s = orc_scale_from_amax(amax, fmt);
      qt_scales[c] = s;
      for (int64_t r = 0; r < rows; ++r)
        q_t[c * rows + r] = cast_one(orc_load(x, in_dtype, r * cols + c), s, fmt, saturate);
    }
  }
}

/* Delayed scaling ([fp8_parity] smoke step 3; [te_blog] "FP8 DelayedScaling
 * ... relies on an amax history"): the scale comes from the history only, so
 * the tensor being cast does not see its own amax; its amax is recorded for
 * the calls that follow. */
float orc_quantize_delayed(const void *x, int in_dtype, int64_t rows,
                           int64_t cols, int fmt, int saturate, float *history,
                           int32_t hist_len, int32_t *next, uint8_t *q,
                           uint8_t *q_t) {
  float hmax = 0.0f;
  int nan_seen = 0;
  for (int32_t i = 0; i < hist_len; ++i) {
    if (isnan(history[i])) nan_seen = 1;
    else if (history[i] > hmax) hmax = history[i];
  }
  if (nan_seen) hmax = NAN;
  float s = orc_scale_from_amax(hmax, fmt);
  orc_quantize_tensor(x, in_dtype, rows, cols, s, fmt, saturate, q, q_t);
  history[*next] = orc_amax(x, in_dtype, rows * cols);
  *next = (*next + 1) % hist_len;
  return s;
}

/* (q).float() * scale ([fp8_parity] scaled_roundtrip), in fp32. */
void orc_dequantize(const uint8_t *q, int64_t n, int fmt, float s, float *d) {
  for (int64_t i = 0; i < n; ++i) d[i] = (float)orc_fp8_decode(q[i], fmt) * s;
}

/* ------------------------------------------------------------------ MXFP8 */

double orc_e8m0_decode(uint8_t code) {
  if (code == 0xFF) return NAN;
  return ldexp(1.0, (int)code - 127);
}

/* emax_elem: the exponent of the element format's largest normal value
 * (E4M3: 448 = 1.75 * 2^8; E5M2: 57344 = 1.75 * 2^15). */
static int mx_emax_elem(int fmt) {
  int ex;
  frexp(describe(fmt).fmax, &ex); /* fmax = f * 2^ex, f in [0.5, 1) */
  return ex - 1;
}

/* OCP MX v1.0 conversion, shared exponent: floor(log2(amax)) - emax_elem,
 * clamped to E8M0's [-127, 127]. */
uint8_t orc_mx_scale_code(float amax, int fmt) {
  if (isnan(amax) || isinf(amax)) return 0xFF;
  int e;
  if (amax == 0.0f) {
    e = -127; /* floor(log2 0) = -inf, clamped */
  } else {
    int ex;
    frexp((double)amax, &ex); /* amax = f * 2^ex, f in [0.5, 1): floor(log2) = ex-1 */
    e = (ex - 1) - mx_emax_elem(fmt);
    if (e < -127) e = -127;
    if (e > 127) e = 127;
  }
  return (uint8_t)(e + 127);
}

/* One block of n elements x[i * stride], i < n: its scale code and bytes. */
static uint8_t mx_block(const void *x, int in_dtype, int64_t first, int64_t stride,
                        int64_t n, int fmt, uint8_t *out, int64_t out_stride) {
  float amax = 0.0f;
  int nonfinite = 0;
  for (int64_t i = 0; i < n; ++i) {
    float a = fabsf(orc_load(x, in_dtype, first + i * stride));
    if (isnan(a) || isinf(a)) nonfinite = 1;
    else if (a > amax) amax = a;
  }
  uint8_t code = nonfinite ? (uint8_t)0xFF : orc_mx_scale_code(amax, fmt);
  for (int64_t i = 0; i < n; ++i) {
    if (code == 0xFF) {
      out[i * out_stride] = 0x7F;
    } else {
      /* V / X = V * 2^-(code - 127): exact in double; saturating RNE */
      double v = ldexp((double)orc_load(x, in_dtype, first + i * stride), 127 - (int)code);
      out[i * out_stride] = encode_double(v, fmt, 1);
    }
  }
  return code;
}

void orc_quantize_mx_rows(const void *x, int in_dtype, int64_t rows,
                          int64_t cols, int fmt, uint8_t *q, uint8_t *scales) {
  int64_t nb = (cols + ORC_MX_BLOCK - 1) / ORC_MX_BLOCK;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t j = 0; j < nb; ++j) {
      int64_t c0 = j * ORC_MX_BLOCK;
      int64_t n = cols - c0 < ORC_MX_BLOCK ? cols - c0 : ORC_MX_BLOCK;
      scales[r * nb + j] = mx_block(x, in_dtype, r * cols + c0, 1, n, fmt, q + r * cols + c0, 1);
    }
}

void orc_quantize_mx_cols(const void *x, int in_dtype, int64_t rows,
                          int64_t cols, int fmt, uint8_t *q_t, uint8_t *scales) {
  int64_t nb = (rows + ORC_MX_BLOCK - 1) / ORC_MX_BLOCK;
  for (int64_t c = 0; c < cols; ++c)
    for (int64_t j = 0; j < nb; ++j) {
      int64_t r0 = j * ORC_MX_BLOCK;
      int64_t n = rows - r0 < ORC_MX_BLOCK ? rows - r0 : ORC_MX_BLOCK;
      scales[c * nb + j] =
          mx_block(x, in_dtype, r0 * cols + c, cols, n, fmt, q_t + c * rows + r0, 1);
    }
}

/* -------------------------------------------------------------------- GEMM */

double orc_operand_scale(const orc_operand *op, int64_t row, int64_t k) {
  int64_t kb = k / 128;
  if (op->scaling == ORC_SCALE_MX)
    return orc_e8m0_decode(op->mx_scale[row * op->stride_row + (k / ORC_MX_BLOCK) * op->stride_k]);
  if (op->scaling == ORC_SCALE_TENSOR) return op->scale[0];
  if (op->scaling == ORC_SCALE_TILE)
    return op->scale[kb * op->stride_k + row * op->stride_row];
  if (op->scaling == ORC_SCALE_ROW) return op->scale[row * op->stride_row];
  return op->scale[(row / 128) * op->stride_row + kb * op->stride_k];
}

/* y = x_deq @ w_deq.T ([fp8_parity] FP8Matmul.forward: xq @ wq.T) where each
 * dequantised element is decode(byte) * its scale.  The products and the sum
 * are taken in double; decode(a) * sA is exact in double (4 + 24 significant
 * bits), so the only rounding is in the double products and sums. */
static void gemm_one(const orc_operand *A, const orc_operand *B, int64_t K,
                     int64_t m, int64_t n, double *y, double *absum) {
  double acc = 0.0, aacc = 0.0;
  for (int64_t k = 0; k < K; ++k) {
    double a = orc_fp8_decode(A->data[m * K + k], A->fmt) * orc_operand_scale(A, m, k);
    double b = orc_fp8_decode(B->data[n * K + k], B->fmt) * orc_operand_scale(B, n, k);
    acc += a * b;
    aacc += fabs(a * b);
  }
  *y = acc;
  *absum = aacc;
}

void orc_gemm_points(const orc_operand *A, const orc_operand *B, int64_t K,
                     int64_t npts, const int64_t *ms, const int64_t *ns,
                     double *y, double *absum) {
  for (int64_t i = 0; i < npts; ++i) gemm_one(A, B, K, ms[i], ns[i], &y[i], &absum[i]);
}

void orc_gemm_rows(const orc_operand *A, const orc_operand *B, int64_t N,
                   int64_t K, int64_t m0, int64_t m1, double *y,
                   double *absum) {
  for (int64_t m = m0; m < m1; ++m)
    for (int64_t n = 0; n < N; ++n)
      gemm_one(A, B, K, m, n, &y[(m - m0) * N + n], &absum[(m - m0) * N + n]);
}
