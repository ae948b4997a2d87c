/*
 * fp8q.h -- C ABI of the scaled FP8 quantize -> FP8 GEMM library (libfp8q.so)
 * for NVIDIA GB300 (sm_103a).
 *
 * What it computes (sources cited by page title and section):
 *   [fp8_parity]  "fp8_parity.py", FP8 numerics lab (mlinterviewnotes.com):
 *                 scaled_roundtrip, FP8Matmul, smoke steps 1-4.
 *   [te_blog]     "How to Optimize Transformer-Based Models for Low-Precision
 *                 Training" (repost of the NVIDIA blog): autocast vs
 *                 pre-quantized GEMM timing, Fprop/Dgrad/Wgrad shapes,
 *                 DelayedScaling with an amax history.
 *   [sj_precision] SpikingJelly "Training and Inference Precision": FP8 Linear
 *                 alignment (input dim % 16, output dim % 8), and "raises
 *                 rather than falling back" when hardware or recipe is missing.
 *
 * Conventions shared by every entry point
 *   - Every pointer argument that names tensor data is DEVICE memory owned by
 *     the caller; the library never allocates, frees or retains it.  Host
 *     pointers are only the small parameter structs (fp8q_operand) and the
 *     optional host array of fp8q_history_init.
 *   - Matrices are row-major and dense: element (r, c) of an [R, C] matrix is
 *     at offset r * C + c.  bf16 is passed as raw 16-bit patterns.
 *   - FP8 bytes: E4M3 (1-4-3, bias 7, no Inf, NaN = S.1111.111, max 448) and
 *     E5M2 (1-5-2, bias 15, IEEE Inf/NaN, max 57344) ([fp8_parity] constants
 *     E4M3_MAX / E5M2_MAX).
 *   - Scales are fp32 DEQUANT multipliers: value = decode(byte) * s, and the
 *     cast is byte = RNE_fp8(fl32(x / s)) with s = max(fl32(amax / fmax),
 *     fl32(1e-12)) ([fp8_parity] scaled_roundtrip).  The quotient is the
 *     correctly rounded fp32 division, as the definition states.
 *   - saturate == 0: a quotient whose magnitude rounds above fmax becomes NaN
 *     (E4M3) or Inf (E5M2), as a plain cast does ([fp8_parity] smoke step 2);
 *     saturate != 0 clamps it to +-fmax.  NaN inputs stay NaN (0x7F | sign).
 *   - Calls are asynchronous on `stream` (0 = legacy default stream).  A
 *     return of FP8Q_OK means the arguments were valid and the work was
 *     enqueued.  A kernel whose wait on a hardware barrier lasts two seconds
 *     gives up, records FP8Q_ERR_TIMEOUT in a device error word that
 *     fp8q_device_status() reports after the stream completes, and returns
 *     after letting the copies and MMAs it issued finish (each of those
 *     drains waits at most 0.2 s more).
 *   - The library runs only on compute capability 10.3 (GB300).  Any other
 *     device gives FP8Q_ERR_ARCH; there is no fallback path of any kind.
 *   - Alignment: every device pointer must be 16-byte aligned
 *     (FP8Q_ERR_MISALIGNED otherwise).  Inner (contiguous) dimensions must be
 *     multiples of 16 where stated (FP8Q_ERR_INVALID_ARG otherwise).
 *   - Diagnostics: with the environment variable FP8Q_LOG set (to anything
 *     but "0") every call and every kernel launch prints one line to stderr
 *     naming the kernel that serves it, its tile or unit shape and its grid or
 *     raster.  The variable is read once per process.
 *   - Threads and devices: every entry point works on the calling thread's
 *     current CUDA device and may be called from several host threads at
 *     once, in a process that drives one device or several; each kernel's
 *     one-time launch set-up (its shared-memory size attribute, an occupancy
 *     query) runs once per device.  Work that shares a buffer, an amax
 *     history or a workspace must be ordered by the caller (one stream, or
 *     events).
 */
#ifndef FP8Q_H
#define FP8Q_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------ codes */

typedef enum fp8q_status {
  FP8Q_OK = 0,
  FP8Q_ERR_INVALID_ARG = 1,     /* null where required, negative size, bad enum,
                                   inner dimension not a multiple of 16, sizes
                                   whose byte counts do not fit in int64 */
  FP8Q_ERR_MISALIGNED = 2,      /* a device pointer is not 16-byte aligned */
  FP8Q_ERR_ARCH = 3,            /* current device is not compute capability 10.3 */
  FP8Q_ERR_WORKSPACE = 4,       /* workspace missing or smaller than required */
  FP8Q_ERR_TIMEOUT = 5,         /* a kernel's bounded wait expired (device-side) */
  FP8Q_ERR_CUDA = 6,            /* a CUDA runtime/driver call failed */
  FP8Q_ERR_NOT_IMPLEMENTED = 7  /* valid request this build does not support */
} fp8q_status;

typedef enum fp8q_dtype {
  FP8Q_DT_F32 = 0,
  FP8Q_DT_BF16 = 1
} fp8q_dtype;

typedef enum fp8q_format {
  FP8Q_E4M3 = 0,  /* activations and weights ([fp8_parity] FP8Matmul.forward) */
  FP8Q_E5M2 = 1   /* output gradients ([fp8_parity] FP8Matmul.backward) */
} fp8q_format;

typedef enum fp8q_scaling {
  FP8Q_SCALE_TENSOR = 0,      /* one scale for the whole operand */
  FP8Q_SCALE_TILE_1x128 = 1,  /* one scale per row per 128-wide K block */
  FP8Q_SCALE_BLOCK_128x128 = 2, /* one scale per 128x128 block */
  FP8Q_SCALE_ROW = 3,           /* one scale per row over all of K */
  FP8Q_SCALE_MX_1x32 = 4        /* MXFP8: one E8M0 scale per row per 32 K */
} fp8q_scaling;

typedef enum fp8q_recipe {
  FP8Q_RECIPE_TENSOR_CURRENT = 0, /* per-tensor, scale from this tensor's amax */
  FP8Q_RECIPE_TENSOR_DELAYED = 1, /* per-tensor, scale from an amax history */
  FP8Q_RECIPE_BLOCK = 2,          /* 1x128 tiles on x, 128x128 blocks on w */
  FP8Q_RECIPE_MXFP8 = 3           /* MXFP8 1x32 blocks on x and w */
} fp8q_recipe;

/* Length of the delayed-scaling amax history ([fp8_parity] smoke step 3 keeps
 * 16 past amaxes). */
#define FP8Q_HISTORY_LEN 16

/* Delayed-scaling state, in DEVICE memory, owned by the caller (80 bytes,
 * 16-byte aligned).  It is plain data: copy it as raw bytes to checkpoint.
 *   amax[]     the last FP8Q_HISTORY_LEN amax values (a ring)
 *   next       index of the ring slot the next call overwrites
 *   scale      the scale the most recent call used
 *   pending, arrivals
 *              zero between calls; used by a call in flight to combine the
 *              per-block amax values.  Two calls on one state must not run
 *              concurrently. */
typedef struct fp8q_amax_history {
  float amax[FP8Q_HISTORY_LEN];
  int32_t next;
  float scale;
  uint32_t pending;
  uint32_t arrivals;
} fp8q_amax_history;

/* ------------------------------------------------------------ diagnostics */

/* Human-readable name of a status code (static storage). */
const char *fp8q_status_string(int status);

/* Reads and clears the device error word of the current device after
 * synchronising the device.  Returns FP8Q_OK, FP8Q_ERR_TIMEOUT (a kernel's
 * bounded barrier wait expired; its outputs are undefined) or FP8Q_ERR_CUDA. */
int fp8q_device_status(void);

/* 1 if the current device is compute capability 10.3, else 0. */
int fp8q_device_supported(void);

/* Self-test of the failure path: launches one warp that waits, through the
 * library's bounded barrier wait, on an mbarrier nothing arrives at.  After
 * the wait limit (about two seconds) the kernel records a timeout and
 * returns; fp8q_device_status() then reports FP8Q_ERR_TIMEOUT once and the
 * context stays usable.  Asynchronous on `stream`.
 * Errors: ARCH, CUDA. */
int fp8q_selftest_barrier_timeout(cudaStream_t stream);

/* --------------------------------------------------------------- step a1 */

/* amax = max |x| over n elements ([fp8_parity] scaled_roundtrip:
 * x.abs().max()).  A NaN anywhere makes amax NaN; n == 0 gives 0.
 *   x       device, n elements of in_dtype, 16-byte aligned
 *   amax    device, one float, overwritten with the result (the kernel's
 *           last CTA writes it; nothing else touches it)
 * Errors: INVALID_ARG (null, n < 0, bad dtype), MISALIGNED, ARCH, CUDA. */
int fp8_amax(const void *x, int in_dtype, int64_t n, float *amax,
             cudaStream_t stream);

/* ----------------------------------------------------------- steps a2, a3 */

/* Per-tensor current scaling ([fp8_parity] scaled_roundtrip with
 * scale=None): s = max(fl32(*amax / fmax), 1e-12), q = RNE(x / s).
 *   x          device [rows, cols] of in_dtype; cols % 16 == 0
 *   amax       device float holding max|x| (from fp8_amax, or any value the
 *              caller chooses: the cast uses it as given)
 *   scale_out  device float or NULL: receives s
 *   q          device [rows, cols] FP8 bytes or NULL
 *   q_t        device [cols, rows] FP8 bytes (the transpose) or NULL;
 *              requires rows % 16 == 0.  At least one of q, q_t non-NULL
 *              unless the matrix is empty (then only *scale_out is written).
 * Errors: INVALID_ARG, MISALIGNED, ARCH, CUDA. */
int fp8_quantize_tensor(const void *x, int in_dtype, int64_t rows,
                        int64_t cols, int format, const float *amax,
                        float *scale_out, uint8_t *q, uint8_t *q_t,
                        int saturate, cudaStream_t stream);

/* Per-tensor current scaling in one call: *amax_out = max |x| (as fp8_amax),
 * then the cast of fp8_quantize_tensor with that amax ([fp8_parity]
 * scaled_roundtrip with scale=None: amax, scale and cast together).  Results
 * are those of fp8_amax followed by fp8_quantize_tensor, bit for bit.
 *   When x holds at most 8 MiB both run in one cooperative launch: the amax
 *   pass reads x, a grid-wide barrier publishes the amax, and the cast
 *   re-reads x from the L2 cache.  Larger inputs run the two kernels, which
 *   are faster there.
 *   amax_out   device float, 4-byte aligned: receives max |x| (zeroed on
 *              `stream` first)
 *   the other arguments as fp8_quantize_tensor.
 * Errors: INVALID_ARG, MISALIGNED, ARCH, CUDA (including a cooperative
 * launch the device refuses). */
int fp8_quantize_tensor_current(const void *x, int in_dtype, int64_t rows,
                                int64_t cols, int format, float *amax_out,
                                float *scale_out, uint8_t *q, uint8_t *q_t,
                                int saturate, cudaStream_t stream);

/* Per-tensor delayed scaling ([fp8_parity] smoke step 3; [te_blog]
 * DelayedScaling, which keeps a history of amax values): s = max(fl32(max(hist->amax) /
 * fmax), 1e-12) is computed from the history alone, x is cast with s, then
 * amax(x) -- found in the same pass over x -- overwrites hist->amax[hist->next]
 * and hist->next advances modulo FP8Q_HISTORY_LEN.  hist->scale receives s.
 *   hist        device state (see fp8q_amax_history); exclusive to this call
 *   scale_out, q, q_t, rows/cols rules as fp8_quantize_tensor
 * Errors: INVALID_ARG, MISALIGNED, ARCH, CUDA. */
int fp8_quantize_delayed(const void *x, int in_dtype, int64_t rows,
                         int64_t cols, int format, fp8q_amax_history *hist,
                         float *scale_out, uint8_t *q, uint8_t *q_t,
                         int saturate, cudaStream_t stream);

/* Writes a fresh history: amax[] from `initial` (HOST array of
 * FP8Q_HISTORY_LEN floats) or zeros when NULL; next = 0, scale = 0, scratch
 * words zero.  Synchronous with respect to the host. */
int fp8q_history_init(fp8q_amax_history *hist, const float *initial,
                      cudaStream_t stream);

/* 1x128 tile scaling ([fp8_parity] smoke step 4 scales each 1x128 piece of a
 * row on its own).  One read of x produces either or both of
 *   row tiles:    q [rows, cols], q_scales [ceil(cols/128), rows] with
 *                 scale(r, kb) = q_scales[kb * rows + r]  (tile = row r,
 *                 columns [128 kb, 128 kb + 128))
 *   column tiles: q_t [cols, rows] (the transpose), qt_scales
 *                 [ceil(rows/128), cols] with scale(c, rb) =
 *                 qt_scales[rb * cols + c] (tile = column c, rows
 *                 [128 rb, 128 rb + 128)); i.e. 1x128 row tiles of x^T.
 * Column tiles are what Wgrad needs: its contraction runs over x's rows.
 * Partial edge tiles are allowed.  cols % 16 == 0; rows % 16 == 0 when the
 * column-tile pair is requested.  Each pair is both-or-neither; at least one.
 * Errors: INVALID_ARG, MISALIGNED, ARCH, CUDA. */
int fp8_quantize_tile1x128(const void *x, int in_dtype, int64_t rows,
                           int64_t cols, int format, uint8_t *q,
                           float *q_scales, uint8_t *q_t, float *qt_scales,
                           int saturate, cudaStream_t stream);

/* Row-wise scaling, the torchao "rowwise" recipe the fp8_parity page offers
 * (argument --recipe), read as one scale per row of each K-major GEMM operand
 * over its whole contraction: from two reads of x, either or both of
 *   q [rows, cols] with q_scales [rows]: row r cast with its own scale;
 *   q_t [cols, rows] with qt_scales [cols]: column c of x (row c of x^T) cast
 *     with its own scale (what Dgrad's and Wgrad's operands need).
 * Scales as everywhere: max(fl32(amax / fmax), 1e-12).  cols % 16 == 0;
 * rows % 16 == 0 when the column pair is requested.  Each pair is
 * both-or-neither; at least one.  The scale arrays also serve as the amax
 * accumulators of the first read (the call zeroes them on `stream`).
 * Errors: INVALID_ARG, MISALIGNED, ARCH, CUDA. */
int fp8_quantize_rowwise(const void *x, int in_dtype, int64_t rows,
                         int64_t cols, int format, uint8_t *q, float *q_scales,
                         uint8_t *q_t, float *qt_scales, int saturate,
                         cudaStream_t stream);

/* MXFP8 ([sj_precision] lists "mxfp8" among Transformer Engine's fp8_recipe
 * choices; [te_blog] "Decoding the results for a real model" uses MXFP8 as its
 * Blackwell baseline).  The pages give no encoding; this follows the OCP
 * Microscaling Formats (MX) Specification v1.0:
 *   - blocks of 32 consecutive elements share one E8M0 scale byte
 *     X = 2^(code - 127) (0xFF = NaN);
 *   - code = floor(log2(max |x|)) - emax + 127, clamped to [0, 254], with
 *     emax = 8 (E4M3, 448 = 1.75 * 2^8) or 15 (E5M2, 57344 = 1.75 * 2^15);
 *     an all-zero block gets code 0;
 *   - byte = RNE(x / X) into `format`, saturating at +-fmax (exact: X is a
 *     power of two);
 *   - a block holding a NaN or an infinity gets code 0xFF and every byte
 *     0x7F (it decodes to NaN whatever its bytes).
 * One read of x produces either or both of
 *   q [rows, cols] with 1x32 blocks along each row (q_scales), and
 *   q_t [cols, rows] (the transpose) with 32x1 blocks down each column of x,
 *     i.e. 1x32 blocks along each row of q_t (qt_scales) -- the operand
 *     Dgrad's and Wgrad's contractions need.
 * Scale layout ("atoms", what the MXFP8 GEMM copies to the tensor cores as
 * is): for an operand [R, K] (q: R = rows, K = cols; q_t: R = cols,
 * K = rows), one 512-byte atom per 128-row x 128-K tile; the atom of row
 * block rb and K block kb starts at byte (rb * ceil(K/128) + kb) * 512, and
 * the scale of row 128 rb + r, 32-wide K block 4 kb + j (r < 128, j < 4) is
 * byte (r % 32) * 16 + (r / 32) * 4 + j of it.  Rows and K blocks past the
 * matrix hold code 0.  Each array takes fp8q_mx_scale_bytes(rows, cols).
 * cols % 16 == 0; rows % 16 == 0 when the q_t pair is requested.  Each pair
 * is both-or-neither; at least one.  Scale arrays 16-byte aligned.
 * Errors: INVALID_ARG, MISALIGNED, ARCH, CUDA. */
int fp8_quantize_mxfp8(const void *x, int in_dtype, int64_t rows, int64_t cols,
                       int format, uint8_t *q, uint8_t *q_scales, uint8_t *q_t,
                       uint8_t *qt_scales, cudaStream_t stream);

/* Bytes of one orientation's MXFP8 scale atoms for an [rows, cols] matrix:
 * ceil(rows/128) * ceil(cols/128) * 512 (the same for the transpose); 0 for
 * negative sizes. */
size_t fp8q_mx_scale_bytes(int64_t rows, int64_t cols);

/* 128x128 block scaling for weights ([te_blog] "2D block scaling for
 * weights"): one scale per block, block_scales [ceil(rows/128),
 * ceil(cols/128)] row-major; q [rows, cols] and/or q_t [cols, rows] (the same
 * bytes transposed -- a block's scale serves both orientations).
 * cols % 16 == 0; rows % 16 == 0 when q_t is requested.
 * Errors: INVALID_ARG, MISALIGNED, ARCH, CUDA. */
int fp8_quantize_block128x128(const void *x, int in_dtype, int64_t rows,
                              int64_t cols, int format, uint8_t *q,
                              uint8_t *q_t, float *block_scales, int saturate,
                              cudaStream_t stream);

/* ----------------------------------------------------------- steps a4, a5 */

/* One FP8 GEMM operand: `data` is a device [rows, K] row-major byte matrix
 * (K contiguous, K % 16 == 0, 16-byte aligned).  The scale of element
 * (row, k), kb = k / 128, is
 *   FP8Q_SCALE_TENSOR:        scale[0]
 *   FP8Q_SCALE_TILE_1x128:    scale[kb * scale_stride_k + row * scale_stride_row]
 *   FP8Q_SCALE_BLOCK_128x128: scale[(row/128) * scale_stride_row + kb * scale_stride_k]
 *   FP8Q_SCALE_ROW:           scale[row * scale_stride_row]
 *   FP8Q_SCALE_MX_1x32:       2^(mx_scale byte of (row, k / 32) - 127), the
 *                             byte found through the atom layout of
 *                             fp8_quantize_mxfp8 (strides unused, 0)
 * (scale in device memory).  The quantize calls above produce:
 *   tile scales of an [R, K] matrix:   stride_row = 1, stride_k = R
 *   block scales of an [R, K] matrix:  stride_row = ceil(K/128), stride_k = 1
 *   block scales used for the transpose [K, R]: stride_row = 1,
 *                                      stride_k = ceil(K/128)
 *   row scales:                        stride_row = 1
 * fp8_gemm and fp8_gemm_amax take any non-negative strides (the caller keeps
 * every index inside its scale array); the role wrappers fp8_gemm_fprop /
 * _dgrad / _wgrad accept only the layouts listed here, for the operand's own
 * shape, and return FP8Q_ERR_INVALID_ARG for any other. */
typedef struct fp8q_operand {
  const uint8_t *data;
  int32_t format;
  int32_t scaling;
  union {
    const float *scale;       /* TENSOR, TILE_1x128, BLOCK_128x128, ROW */
    const uint8_t *mx_scale;  /* MX_1x32: E8M0 atoms (fp8_quantize_mxfp8
                                 layout for this [rows, K] operand), 16-byte
                                 aligned; both strides must be 0 */
  };
  int64_t scale_stride_row;
  int64_t scale_stride_k;
} fp8q_operand;

/* C[m, n] = sum_k A(m, k) * B(n, k) with each factor dequantised by its own
 * scale, accumulated in fp32 on the tensor cores, then written as out_dtype
 * (bf16, round-to-nearest-even, or fp32) to device C [M, N] row-major
 * ([fp8_parity] FP8Matmul.forward: xq @ wq.T).  With TILE/BLOCK scaling the
 * partial sum of every 128-wide K block is promoted into the fp32 result with
 * that block's scale product.
 *   A: [M, K], B: [N, K]; N % 16 == 0, K % 16 == 0; M >= 0 any.
 *   M == 0 or N == 0: nothing to do.  K == 0: C is zero.
 * Supported combinations: TENSOR/ROW with TENSOR/ROW (scales applied in the
 * epilogue), A TILE with B TILE or BLOCK (promoted per K block), and MX_1x32
 * with MX_1x32 (the tensor cores apply the E8M0 scales per 32 K; MX atoms of
 * K blocks past K must hold finite codes, as fp8_quantize_mxfp8 writes).
 * Errors: INVALID_ARG, MISALIGNED, ARCH, NOT_IMPLEMENTED (other combinations),
 * CUDA. */
int fp8_gemm(const fp8q_operand *A, const fp8q_operand *B, void *C,
             int out_dtype, int64_t M, int64_t N, int64_t K,
             cudaStream_t stream);

/* fp8_gemm, and in the same launch amax_out[0] = max |C[m, n]| over the
 * values as stored (after the bf16 rounding for bf16 output); NaN propagates
 * as in fp8_amax.  This is amax fused into the producer of the next
 * quantisation: [te_blog] "Decoding the results for a real model" lists the
 * extra memory pass that per-tensor amax needs among the overheads outside
 * the GEMMs, and feeding amax_out to fp8_quantize_tensor as its `amax` spares
 * the separate fp8_amax read of C.
 *   amax_out: one device float, 4-byte aligned.  The call zeroes it on
 *   `stream` first, so it holds exactly amax(C) when the GEMM is done
 *   (0 when M, N or K is 0).
 * Arguments, layout and errors otherwise as fp8_gemm (INVALID_ARG also for a
 * null amax_out, MISALIGNED for an unaligned one). */
int fp8_gemm_amax(const fp8q_operand *A, const fp8q_operand *B, void *C,
                  int out_dtype, int64_t M, int64_t N, int64_t K,
                  float *amax_out, cudaStream_t stream);

/* The three GEMMs of a linear layer y = x w^T with x [M, K] (tokens x input
 * features), w [N, K], grad_out g [M, N] ([fp8_parity] FP8Matmul; [te_blog],
 * which times the Fprop, Dgrad and Wgrad shapes one by one).  M, N, K
 * are always the LAYER's sizes; each call maps them onto fp8_gemm:
 *   fprop: y [M, N]  = x [M, K] . w [N, K]^T        (contraction K)
 *   dgrad: dx [M, K] = g [M, N] . w                 (contraction N;
 *          pass w_t = w^T as a [K, N] operand, e.g. q_t of the weight)
 *   wgrad: dw [N, K] = g^T . x                      (contraction M;
 *          pass g_t [N, M] and x_t [K, M], e.g. column-tile / q_t outputs)
 * Alignment: the contraction and the output column count must be multiples
 * of 16 (so M % 16 == 0 for wgrad).  Each operand's scale strides must be one
 * of the layouts listed with fp8q_operand for its [rows, contraction] shape.
 * Errors as fp8_gemm, INVALID_ARG also for a scale layout outside that list. */
int fp8_gemm_fprop(const fp8q_operand *x, const fp8q_operand *w, void *y,
                   int out_dtype, int64_t M, int64_t N, int64_t K,
                   cudaStream_t stream);
int fp8_gemm_dgrad(const fp8q_operand *g, const fp8q_operand *w_t, void *dx,
                   int out_dtype, int64_t M, int64_t N, int64_t K,
                   cudaStream_t stream);
int fp8_gemm_wgrad(const fp8q_operand *g_t, const fp8q_operand *x_t, void *dw,
                   int out_dtype, int64_t M, int64_t N, int64_t K,
                   cudaStream_t stream);

/* Up to FP8Q_GEMM_GROUP_MAX independent GEMMs in one call, for example one
 * linear's Fprop, Dgrad and Wgrad ([te_blog] the layer's 12 GEMMs, three per
 * linear).  Each C_i [M_i, N_i] = A_i [M_i, K_i] . B_i [N_i, K_i]^T is
 * computed exactly as fp8_gemm computes it, bit for bit.
 *   When every GEMM has per-tensor scales on both operands, N_i > 128 and no
 *   size is 0, the group runs as one persistent launch whose output tiles are
 *   numbered GEMM after GEMM, so only the group's last wave of tiles is
 *   partial instead of each GEMM's.
 *   Otherwise the GEMMs are launched one after another, in order.
 *   descs: host array of `count` entries (0 <= count <= FP8Q_GEMM_GROUP_MAX);
 *   every operand is checked as by fp8_gemm, and its scale layout as by the
 *   role wrappers (the layouts the quantize calls write).  The outputs must
 *   not overlap one another or any operand.
 * Errors: as fp8_gemm, for the first GEMM that fails a check (nothing is
 * launched then); FP8Q_ERR_INVALID_ARG for a count out of range or null
 * descs. */
#define FP8Q_GEMM_GROUP_MAX 3
typedef struct fp8q_gemm_desc {
  fp8q_operand A;  /* [M, K] */
  fp8q_operand B;  /* [N, K] */
  void *C;         /* [M, N], out_dtype */
  int64_t M, N, K;
} fp8q_gemm_desc;
int fp8_gemm_grouped(const fp8q_gemm_desc *descs, int count, int out_dtype,
                     cudaStream_t stream);

/* ----------------------------------------------------- the whole forward */

/* Bytes of workspace fp8_linear_autocast needs for this recipe and shape
 * (rounded up to 256-byte pieces); 0 for negative sizes and for sizes whose
 * element counts M*K or N*K would overflow int64 (which the forward calls
 * reject with FP8Q_ERR_INVALID_ARG). */
size_t fp8q_linear_workspace_size(int recipe, int64_t M, int64_t N, int64_t K);

/* Autocast forward of a linear layer ([te_blog] autocast mode: the inputs are
 * quantised on the fly ahead of every GEMM and the timing includes that): with
 * x [M, K] and w [N, K] in in_dtype, quantizes both to E4M3 under `recipe`
 * and computes y [M, N] = x w^T in out_dtype, all on `stream`, without
 * synchronising.
 *   TENSOR_CURRENT: amax(x), amax(w), cast x, cast w, per-tensor GEMM
 *   TENSOR_DELAYED: casts with hist_x / hist_w (device state, required)
 *   BLOCK:          1x128 row tiles of x, 128x128 blocks of w, promoted GEMM
 *   MXFP8:          1x32 MXFP8 blocks of x and w, block-scaled MMA
 *   workspace  device scratch of at least fp8q_linear_workspace_size bytes,
 *              256-byte aligned; holds the FP8 copies, scales and amaxes
 * Alignment: K % 16 == 0, N % 16 == 0.
 * Errors: INVALID_ARG, MISALIGNED, WORKSPACE, ARCH, CUDA. */
int fp8_linear_autocast(const void *x, const void *w, int in_dtype, int64_t M,
                        int64_t N, int64_t K, int recipe,
                        fp8q_amax_history *hist_x, fp8q_amax_history *hist_w,
                        void *y, int out_dtype, void *workspace,
                        size_t ws_bytes, cudaStream_t stream);

/* ----------------------------------------- a linear layer's whole step */

/* Bytes of workspace fp8_linear_train needs: the FP8 copies of x, w and
 * grad_out in both orientations plus the recipe's scales (256-byte pieces);
 * 0 for negative sizes, sizes whose element counts overflow, or a bad recipe. */
size_t fp8q_linear_train_workspace_size(int recipe, int64_t M, int64_t N, int64_t K);

/* The three GEMMs of one linear layer in training, each operand quantized
 * on the fly ([fp8_parity] FP8Matmul: the forward quantizes x and w to E4M3
 * and returns xq @ wq.T; the backward quantizes grad_out to E5M2 and returns
 * gq @ wq and gq.T @ xq; [te_blog] autocast mode: the inputs are quantised
 * on the fly ahead of every GEMM):
 *   y  [M, N] = x [M, K] . w [N, K]^T      (Fprop)
 *   dx [M, K] = g [M, N] . w               (Dgrad)
 *   dw [N, K] = g^T . x                    (Wgrad)
 * with x, w and grad_out g (device, in_dtype) quantized under `recipe`, each
 * into both orientations (the transposed copies feed Dgrad and Wgrad):
 *   TENSOR_CURRENT: per-tensor scales from each tensor's own amax
 *   TENSOR_DELAYED: per-tensor scales from hist_x / hist_w / hist_g (device
 *                   state, required; each is updated as fp8_quantize_delayed
 *                   does)
 *   BLOCK:          1x128 tiles on x and g (row tiles for Fprop / Dgrad,
 *                   column tiles for Wgrad), 128x128 blocks on w
 *   MXFP8:          1x32 MXFP8 blocks on all three, in both orientations
 * Outputs y, dx, dw are device out_dtype.  All work is enqueued on `stream`.
 *   workspace: device, >= fp8q_linear_train_workspace_size, 256-byte aligned
 * Alignment: M, N, K multiples of 16.
 * Errors: INVALID_ARG, MISALIGNED, WORKSPACE, ARCH, CUDA. */
int fp8_linear_train(const void *x, const void *w, const void *g, int in_dtype,
                     int64_t M, int64_t N, int64_t K, int recipe,
                     fp8q_amax_history *hist_x, fp8q_amax_history *hist_w,
                     fp8q_amax_history *hist_g, void *y, void *dx, void *dw,
                     int out_dtype, void *workspace, size_t ws_bytes,
                     cudaStream_t stream);

/* Bytes of device workspace fp8_linear_train_host needs: that of
 * fp8_linear_train plus device copies of x, w, g (in_dtype) and of y, dx, dw
 * (out_dtype); 0 for invalid arguments. */
size_t fp8q_linear_train_host_workspace_size(int recipe, int in_dtype, int out_dtype,
                                             int64_t M, int64_t N, int64_t K);

/* fp8_linear_train from and to HOST buffers: x_h, w_h, g_h and y_h, dx_h,
 * dw_h are host memory (page-locked for the copies to overlap), copied in and
 * out inside the call's work.  The copies run on two streams the library
 * owns (one per direction, created on the first call on a device and kept
 * until the process exits), ordered against `stream` by events:
 *   - the copies in start after the work already queued on `stream`;
 *   - x and w are quantized while g is still being copied in;
 *   - y is copied out during the Dgrad, dx during the Wgrad;
 *   - `stream` waits for the last copy out, so work queued on it after this
 *     call sees the host outputs filled (synchronise `stream` before reading
 *     them on the host).
 * Calls from several host threads on one device are serialised internally
 * while they enqueue.  The workspace must not be in use by other work.
 *   workspace: device, >= fp8q_linear_train_host_workspace_size, 256-byte
 *              aligned
 * Arguments, alignment and errors otherwise as fp8_linear_train. */
int fp8_linear_train_host(const void *x_h, const void *w_h, const void *g_h,
                          int in_dtype, int64_t M, int64_t N, int64_t K,
                          int recipe, fp8q_amax_history *hist_x,
                          fp8q_amax_history *hist_w, fp8q_amax_history *hist_g,
                          void *y_h, void *dx_h, void *dw_h, int out_dtype,
                          void *workspace, size_t ws_bytes, cudaStream_t stream);

/* ------------------------------------------ forward without a workspace */

/* Size of the static scratch used by fp8_linear_autocast_noalloc. */
#define FP8Q_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/* fp8_linear_autocast for callers that cannot call cudaMalloc: for example a
 * plugin hosted by an application that owns all device memory and passes in
 * only the tensors, a serving loop that forbids allocation after start-up, or
 * code under another allocator's accounting that may not grow the device
 * footprint.  Such callers cannot provide the workspace fp8_linear_autocast
 * needs, so this variant keeps it in one file-scope device array of
 * FP8Q_NOALLOC_SCRATCH_BYTES (64 MiB) inside the library.  The source pages
 * have no counterpart to this entry point.
 *   - It allocates nothing: no cudaMalloc, cudaFree or allocating library
 *     routine.  Every GPU on which the library's device code is loaded holds
 *     the 64 MiB array until the process exits.
 *   - Sizes whose scratch, fp8q_linear_workspace_size(recipe, M, N, K),
 *     exceeds FP8Q_NOALLOC_SCRATCH_BYTES are rejected with
 *     FP8Q_ERR_WORKSPACE before any device work.
 *   - The first call on a device, with that device current, looks up the
 *     array's device address (cudaGetSymbolAddress); make that first call
 *     before any stream capture.
 *   - All calls on a device share the one array, which keeps the last call's
 *     contents.  Each call clears what must start at zero (the amax words)
 *     itself.  Calls whose work overlaps on the GPU (other streams, other
 *     host threads) race on the array: serialise them.
 * Arguments, results and the other errors are those of fp8_linear_autocast. */
int fp8_linear_autocast_noalloc(const void *x, const void *w, int in_dtype,
                                int64_t M, int64_t N, int64_t K, int recipe,
                                fp8q_amax_history *hist_x,
                                fp8q_amax_history *hist_w, void *y,
                                int out_dtype, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* FP8Q_H */
