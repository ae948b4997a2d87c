// The extern "C" boundary of libfp8q.so (declared in include/fp8q.h):
// argument validation, device checks, and dispatch to the kernels.  No entry
// point allocates device memory; none synchronises except the diagnostics
// and fp8q_history_init.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <mutex>

#include "fp8q_internal.h"
#include "fp8q_ptx.cuh"

namespace fp8q {
namespace {

constexpr int kMaxDevices = 64;

// Word set by kernels whose bounded waits expire.  One copy per device (the
// module is loaded per context); its address is looked up per device.
__device__ unsigned int g_error_word = 0;

struct DeviceInfo {
  std::once_flag once;
  int supported = 0;
  int sms = 0;
  unsigned int *err = nullptr;
};
DeviceInfo g_dev[kMaxDevices];

DeviceInfo *current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  DeviceInfo *d = &g_dev[dev];
  std::call_once(d->once, [d, dev] {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return;
    d->supported = (prop.major == 10 && prop.minor == 3) ? 1 : 0;
    d->sms = prop.multiProcessorCount;
    void *p = nullptr;
    if (d->supported && cudaGetSymbolAddress(&p, g_error_word) == cudaSuccess)
      d->err = static_cast<unsigned int *>(p);
  });
  return d;
}


int check_device() {
  DeviceInfo *d = current_device();
  if (d == nullptr) return FP8Q_ERR_CUDA;
  return d->supported ? FP8Q_OK : FP8Q_ERR_ARCH;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool valid_dtype(int d) { return d == FP8Q_DT_F32 || d == FP8Q_DT_BF16; }
bool valid_format(int f) { return f == FP8Q_E4M3 || f == FP8Q_E5M2; }

int from_cuda(cudaError_t e) { return e == cudaSuccess ? FP8Q_OK : FP8Q_ERR_CUDA; }

// Shared validation of the quantize calls.
int check_quant(const void *x, int in_dtype, int64_t rows, int64_t cols, int format,
                bool want_t) {
  if (!valid_dtype(in_dtype) || !valid_format(format)) return FP8Q_ERR_INVALID_ARG;
  if (rows < 0 || cols < 0) return FP8Q_ERR_INVALID_ARG;
  // the byte size of x (4-byte elements at most) must fit in int64
  if (rows > 0 && cols > INT64_MAX / 4 / rows) return FP8Q_ERR_INVALID_ARG;
  if (cols % 16 != 0) return FP8Q_ERR_INVALID_ARG;
  if (want_t && rows % 16 != 0) return FP8Q_ERR_INVALID_ARG;
  if (rows > 0 && cols > 0) {
    if (x == nullptr) return FP8Q_ERR_INVALID_ARG;
    if (!aligned16(x)) return FP8Q_ERR_MISALIGNED;
  }
  return FP8Q_OK;
}

int check_ptr(const void *p, bool required) {
  if (p == nullptr) return required ? FP8Q_ERR_INVALID_ARG : FP8Q_OK;
  return aligned16(p) ? FP8Q_OK : FP8Q_ERR_MISALIGNED;
}

int check_operand(const fp8q_operand *op, int64_t rows, int64_t K) {
  if (op == nullptr || !valid_format(op->format)) return FP8Q_ERR_INVALID_ARG;
  if (op->scaling != FP8Q_SCALE_TENSOR && op->scaling != FP8Q_SCALE_TILE_1x128 &&
      op->scaling != FP8Q_SCALE_BLOCK_128x128 && op->scaling != FP8Q_SCALE_ROW &&
      op->scaling != FP8Q_SCALE_MX_1x32)
    return FP8Q_ERR_INVALID_ARG;
  if (op->scale == nullptr) return FP8Q_ERR_INVALID_ARG;
  if (op->scaling == FP8Q_SCALE_MX_1x32) {
    // atoms are fetched with 16-byte bulk copies; the layout has no strides
    if (!aligned16(op->mx_scale)) return FP8Q_ERR_MISALIGNED;
    if (op->scale_stride_row != 0 || op->scale_stride_k != 0) return FP8Q_ERR_INVALID_ARG;
  }
  if ((reinterpret_cast<uintptr_t>(op->scale) & 3u) != 0) return FP8Q_ERR_MISALIGNED;
  if (op->scaling != FP8Q_SCALE_TENSOR && (op->scale_stride_row < 0 || op->scale_stride_k < 0))
    return FP8Q_ERR_INVALID_ARG;
  if (rows > 0 && K > 0) {
    if (op->data == nullptr) return FP8Q_ERR_INVALID_ARG;
    if (!aligned16(op->data)) return FP8Q_ERR_MISALIGNED;
  }
  return FP8Q_OK;
}

// The role wrappers know every operand's shape, so they accept only the
// scale layouts the quantize calls write (documented with fp8q_operand): any
// other stride would index past the scale array on the device.
//   TILE_1x128 of an [R, K] operand:      stride_row 1, stride_k R
//   BLOCK_128x128 of an [R, K] operand:   stride_row ceil(K/128), stride_k 1
//   BLOCK_128x128 read transposed:        stride_row 1, stride_k ceil(R/128)
//   ROW:                                  stride_row 1
int check_layout(const fp8q_operand *op, int64_t rows, int64_t K) {
  const int64_t kb = (K + 127) / 128, rb = (rows + 127) / 128;
  switch (op->scaling) {
    case FP8Q_SCALE_TENSOR:
      return FP8Q_OK;
    case FP8Q_SCALE_TILE_1x128:
      return (op->scale_stride_row == 1 && op->scale_stride_k == rows) ? FP8Q_OK
                                                                       : FP8Q_ERR_INVALID_ARG;
    case FP8Q_SCALE_BLOCK_128x128:
      return ((op->scale_stride_row == kb && op->scale_stride_k == 1) ||
              (op->scale_stride_row == 1 && op->scale_stride_k == rb))
                 ? FP8Q_OK
                 : FP8Q_ERR_INVALID_ARG;
    case FP8Q_SCALE_ROW:
      return op->scale_stride_row == 1 ? FP8Q_OK : FP8Q_ERR_INVALID_ARG;
    case FP8Q_SCALE_MX_1x32:
      return (op->scale_stride_row == 0 && op->scale_stride_k == 0) ? FP8Q_OK
                                                                     : FP8Q_ERR_INVALID_ARG;
  }
  return FP8Q_ERR_INVALID_ARG;
}

GemmOperandDev to_dev(const fp8q_operand *op) {
  GemmOperandDev d;
  d.data = op->data;
  d.format = op->format;
  d.scaling = op->scaling;
  d.scale = op->scale;
  d.mx_scale = op->scaling == FP8Q_SCALE_MX_1x32 ? op->mx_scale : nullptr;
  d.stride_row = op->scale_stride_row;
  d.stride_k = op->scale_stride_k;
  return d;
}

size_t round256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

// Self-test of the failure path: one warp waits, through the same bounded
// wait the GEMM and quantize kernels use, on an mbarrier that nothing ever
// arrives at.  After the wait's time limit it records the timeout in the
// device error word and the kernel returns normally.
__global__ void selftest_timeout_kernel(unsigned int *err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bar), 1);
    abort_flag = 0;
    ptx::fence_barrier_init();
  }
  __syncthreads();
  (void)ptx::wait_bounded_warp(ptx::smem_u32(&bar), 0, &abort_flag, err);
}

}  // namespace

// Sizes of a linear layer whose element counts M*K and N*K do not overflow.
bool linear_dims_ok(int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N < 0 || K < 0) return false;
  const int64_t lim = INT64_MAX / 4;  // room for the byte sums of the workspace
  if (K > 0 && (M > lim / K || N > lim / K)) return false;
  return true;
}

unsigned int *device_error_word() {
  DeviceInfo *d = current_device();
  return d ? d->err : nullptr;
}

int sm_count() {
  DeviceInfo *d = current_device();
  return (d && d->sms > 0) ? d->sms : kNumSMsHint;
}

bool log_enabled() {
  static const bool on = [] {   // initialised once, thread-safe
    const char *e = getenv("FP8Q_LOG");
    return e != nullptr && e[0] != '\0' && e[0] != '0';
  }();
  return on;
}

}  // namespace fp8q

using namespace fp8q;

extern "C" {

const char *fp8q_status_string(int status) {
  switch (status) {
    case FP8Q_OK: return "ok";
    case FP8Q_ERR_INVALID_ARG: return "invalid argument";
    case FP8Q_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case FP8Q_ERR_ARCH: return "device is not compute capability 10.3 (GB300)";
    case FP8Q_ERR_WORKSPACE: return "workspace missing or too small";
    case FP8Q_ERR_TIMEOUT: return "kernel barrier wait timed out";
    case FP8Q_ERR_CUDA: return "CUDA error";
    case FP8Q_ERR_NOT_IMPLEMENTED: return "not implemented";
  }
  return "unknown status";
}

int fp8q_device_supported(void) { return check_device() == FP8Q_OK ? 1 : 0; }

int fp8q_device_status(void) {
  int rc = check_device();
  if (rc != FP8Q_OK) return rc;
  if (cudaDeviceSynchronize() != cudaSuccess) return FP8Q_ERR_CUDA;
  unsigned int *w = device_error_word();
  if (w == nullptr) return FP8Q_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpy(&v, w, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return FP8Q_ERR_CUDA;
  if (v != 0) {
    unsigned int zero = 0;
    if (cudaMemcpy(w, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
      return FP8Q_ERR_CUDA;
    return FP8Q_ERR_TIMEOUT;
  }
  return FP8Q_OK;
}

int fp8q_selftest_barrier_timeout(cudaStream_t stream) {
  int rc = check_device();
  if (rc != FP8Q_OK) return rc;
  unsigned int *err = device_error_word();
  if (err == nullptr) return FP8Q_ERR_CUDA;
  selftest_timeout_kernel<<<1, 32, 0, stream>>>(err);
  return from_cuda(cudaGetLastError());
}

int fp8_amax(const void *x, int in_dtype, int64_t n, float *amax, cudaStream_t stream) {
  if (!valid_dtype(in_dtype) || n < 0 || n > INT64_MAX / 4 || amax == nullptr)
    return FP8Q_ERR_INVALID_ARG;
  if (n > 0 && x == nullptr) return FP8Q_ERR_INVALID_ARG;
  if (n > 0 && !aligned16(x)) return FP8Q_ERR_MISALIGNED;
  if ((reinterpret_cast<uintptr_t>(amax) & 3u) != 0) return FP8Q_ERR_MISALIGNED;
  int rc = check_device();
  if (rc != FP8Q_OK) return rc;
  return from_cuda(launch_amax(x, in_dtype, n, amax, stream));
}

int fp8_quantize_tensor(const void *x, int in_dtype, int64_t rows, int64_t cols, int format,
                        const float *amax, float *scale_out, uint8_t *q, uint8_t *q_t,
                        int saturate, cudaStream_t stream) {
  int rc = check_quant(x, in_dtype, rows, cols, format, q_t != nullptr);
  if (rc != FP8Q_OK) return rc;
  if (amax == nullptr) return FP8Q_ERR_INVALID_ARG;
  if (rows > 0 && cols > 0 && q == nullptr && q_t == nullptr) return FP8Q_ERR_INVALID_ARG;
  if ((rc = check_ptr(q, false)) != FP8Q_OK || (rc = check_ptr(q_t, false)) != FP8Q_OK) return rc;
  if ((rc = check_device()) != FP8Q_OK) return rc;
  QuantParams p{};
  p.x = x;
  p.rows = rows;
  p.cols = cols;
  p.in_dtype = in_dtype;
  p.format = format;
  p.saturate = saturate;
  p.mode = kModeTensorCurrent;
  p.err = device_error_word();
  p.amax_in = amax;
  p.scale_out = scale_out;
  p.q = q;
  p.q_t = q_t;
  if (log_enabled())
    fprintf(stderr, "[fp8q] quantize_tensor %lldx%lld fmt=%d q=%d q_t=%d\n", (long long)rows,
            (long long)cols, format, q != nullptr, q_t != nullptr);
  return from_cuda(launch_quant2d(p, stream));
}

int fp8_quantize_tensor_current(const void *x, int in_dtype, int64_t rows, int64_t cols,
                                int format, float *amax_out, float *scale_out, uint8_t *q,
                                uint8_t *q_t, int saturate, cudaStream_t stream) {
  int rc = check_quant(x, in_dtype, rows, cols, format, q_t != nullptr);
  if (rc != FP8Q_OK) return rc;
  if (amax_out == nullptr) return FP8Q_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(amax_out) & 3u) return FP8Q_ERR_MISALIGNED;
  if (rows > 0 && cols > 0 && q == nullptr && q_t == nullptr) return FP8Q_ERR_INVALID_ARG;
  if ((rc = check_ptr(q, false)) != FP8Q_OK || (rc = check_ptr(q_t, false)) != FP8Q_OK) return rc;
  if ((rc = check_device()) != FP8Q_OK) return rc;
  const int64_t bytes = rows * cols * (in_dtype == FP8Q_DT_BF16 ? 2 : 4);
  if (rows == 0 || cols == 0 || bytes > kFusedTensorMaxBytes) {
    if ((rc = fp8_amax(x, in_dtype, rows * cols, amax_out, stream)) != FP8Q_OK) return rc;
    return fp8_quantize_tensor(x, in_dtype, rows, cols, format, amax_out, scale_out, q, q_t,
                               saturate, stream);
  }
  if (cudaMemsetAsync(amax_out, 0, sizeof(float), stream) != cudaSuccess) return FP8Q_ERR_CUDA;
  QuantParams p{};
  p.x = x;
  p.rows = rows;
  p.cols = cols;
  p.in_dtype = in_dtype;
  p.format = format;
  p.saturate = saturate;
  p.mode = kModeTensorFused;
  p.err = device_error_word();
  p.amax_out = amax_out;
  p.scale_out = scale_out;
  p.q = q;
  p.q_t = q_t;
  return from_cuda(launch_quant2d(p, stream));
}

int fp8_quantize_delayed(const void *x, int in_dtype, int64_t rows, int64_t cols, int format,
                         fp8q_amax_history *hist, float *scale_out, uint8_t *q, uint8_t *q_t,
                         int saturate, cudaStream_t stream) {
  int rc = check_quant(x, in_dtype, rows, cols, format, q_t != nullptr);
  if (rc != FP8Q_OK) return rc;
  if (hist == nullptr) return FP8Q_ERR_INVALID_ARG;
  if (rows > 0 && cols > 0 && q == nullptr && q_t == nullptr) return FP8Q_ERR_INVALID_ARG;
  if ((rc = check_ptr(hist, true)) != FP8Q_OK) return rc;
  if ((rc = check_ptr(q, false)) != FP8Q_OK || (rc = check_ptr(q_t, false)) != FP8Q_OK) return rc;
  if ((rc = check_device()) != FP8Q_OK) return rc;
  QuantParams p{};
  p.x = x;
  p.rows = rows;
  p.cols = cols;
  p.in_dtype = in_dtype;
  p.format = format;
  p.saturate = saturate;
  p.mode = kModeTensorDelayed;
  p.err = device_error_word();
  p.hist = hist;
  p.scale_out = scale_out;
  p.q = q;
  p.q_t = q_t;
  return from_cuda(launch_quant2d(p, stream));
}

int fp8q_history_init(fp8q_amax_history *hist, const float *initial, cudaStream_t stream) {
  if (hist == nullptr) return FP8Q_ERR_INVALID_ARG;
  if (!aligned16(hist)) return FP8Q_ERR_MISALIGNED;
  int rc = check_device();
  if (rc != FP8Q_OK) return rc;
  fp8q_amax_history h{};
  if (initial != nullptr)
    for (int i = 0; i < FP8Q_HISTORY_LEN; ++i) h.amax[i] = initial[i];
  if (cudaMemcpyAsync(hist, &h, sizeof h, cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return FP8Q_ERR_CUDA;
  return from_cuda(cudaStreamSynchronize(stream));
}

int fp8_quantize_tile1x128(const void *x, int in_dtype, int64_t rows, int64_t cols, int format,
                           uint8_t *q, float *q_scales, uint8_t *q_t, float *qt_scales,
                           int saturate, cudaStream_t stream) {
  const bool want_row = q != nullptr || q_scales != nullptr;
  const bool want_col = q_t != nullptr || qt_scales != nullptr;
  int rc = check_quant(x, in_dtype, rows, cols, format, want_col);
  if (rc != FP8Q_OK) return rc;
  if (rows > 0 && cols > 0) {
    if (!want_row && !want_col) return FP8Q_ERR_INVALID_ARG;
    if (want_row && (q == nullptr || q_scales == nullptr)) return FP8Q_ERR_INVALID_ARG;
    if (want_col && (q_t == nullptr || qt_scales == nullptr)) return FP8Q_ERR_INVALID_ARG;
  }
  if ((rc = check_ptr(q, false)) != FP8Q_OK || (rc = check_ptr(q_t, false)) != FP8Q_OK) return rc;
  if ((q_scales && (reinterpret_cast<uintptr_t>(q_scales) & 3u)) ||
      (qt_scales && (reinterpret_cast<uintptr_t>(qt_scales) & 3u)))
    return FP8Q_ERR_MISALIGNED;
  if ((rc = check_device()) != FP8Q_OK) return rc;
  if (rows == 0 || cols == 0) return FP8Q_OK;
  QuantParams p{};
  p.x = x;
  p.rows = rows;
  p.cols = cols;
  p.in_dtype = in_dtype;
  p.format = format;
  p.saturate = saturate;
  p.mode = kModeTile;
  p.err = device_error_word();
  p.q = want_row ? q : nullptr;
  p.q_scales = want_row ? q_scales : nullptr;
  p.q_t = want_col ? q_t : nullptr;
  p.qt_scales = want_col ? qt_scales : nullptr;
  if (log_enabled())
    fprintf(stderr, "[fp8q] quantize_tile1x128 %lldx%lld fmt=%d rows=%d cols=%d\n",
            (long long)rows, (long long)cols, format, want_row, want_col);
  return from_cuda(launch_quant2d(p, stream));
}

int fp8_quantize_rowwise(const void *x, int in_dtype, int64_t rows, int64_t cols, int format,
                         uint8_t *q, float *q_scales, uint8_t *q_t, float *qt_scales,
                         int saturate, cudaStream_t stream) {
  const bool want_row = q != nullptr || q_scales != nullptr;
  const bool want_col = q_t != nullptr || qt_scales != nullptr;
  int rc = check_quant(x, in_dtype, rows, cols, format, want_col);
  if (rc != FP8Q_OK) return rc;
  if (rows > 0 && cols > 0) {
    if (!want_row && !want_col) return FP8Q_ERR_INVALID_ARG;
    if (want_row && (q == nullptr || q_scales == nullptr)) return FP8Q_ERR_INVALID_ARG;
    if (want_col && (q_t == nullptr || qt_scales == nullptr)) return FP8Q_ERR_INVALID_ARG;
  }
  if ((rc = check_ptr(q, false)) != FP8Q_OK || (rc = check_ptr(q_t, false)) != FP8Q_OK) return rc;
  if ((q_scales && (reinterpret_cast<uintptr_t>(q_scales) & 3u)) ||
      (qt_scales && (reinterpret_cast<uintptr_t>(qt_scales) & 3u)))
    return FP8Q_ERR_MISALIGNED;
  if ((rc = check_device()) != FP8Q_OK) return rc;
  if (rows == 0 || cols == 0) return FP8Q_OK;
  // pass 1 gathers the amaxes in the scale arrays, so they start at zero
  if (want_row && cudaMemsetAsync(q_scales, 0, sizeof(float) * (size_t)rows, stream) != cudaSuccess)
    return FP8Q_ERR_CUDA;
  if (want_col && cudaMemsetAsync(qt_scales, 0, sizeof(float) * (size_t)cols, stream) != cudaSuccess)
    return FP8Q_ERR_CUDA;
  QuantParams p{};
  p.x = x;
  p.rows = rows;
  p.cols = cols;
  p.in_dtype = in_dtype;
  p.format = format;
  p.saturate = saturate;
  p.err = device_error_word();
  p.q_scales = want_row ? q_scales : nullptr;
  p.qt_scales = want_col ? qt_scales : nullptr;
  p.mode = kModeRowAmax;
  if ((rc = from_cuda(launch_quant2d(p, stream))) != FP8Q_OK) return rc;
  p.mode = kModeRowCast;
  p.q = want_row ? q : nullptr;
  p.q_t = want_col ? q_t : nullptr;
  if ((rc = from_cuda(launch_quant2d(p, stream))) != FP8Q_OK) return rc;
  if (want_row && (rc = from_cuda(launch_amax_to_scale(q_scales, rows, format, stream))) != FP8Q_OK)
    return rc;
  if (want_col && (rc = from_cuda(launch_amax_to_scale(qt_scales, cols, format, stream))) != FP8Q_OK)
    return rc;
  return FP8Q_OK;
}

size_t fp8q_mx_scale_bytes(int64_t rows, int64_t cols) {
  if (rows < 0 || cols < 0) return 0;
  return (size_t)((rows + 127) / 128) * (size_t)((cols + 127) / 128) * 512u;
}

int fp8_quantize_mxfp8(const void *x, int in_dtype, int64_t rows, int64_t cols, int format,
                       uint8_t *q, uint8_t *q_scales, uint8_t *q_t, uint8_t *qt_scales,
                       cudaStream_t stream) {
  const bool want_row = q != nullptr || q_scales != nullptr;
  const bool want_col = q_t != nullptr || qt_scales != nullptr;
  int rc = check_quant(x, in_dtype, rows, cols, format, want_col);
  if (rc != FP8Q_OK) return rc;
  if (rows > 0 && cols > 0) {
    if (!want_row && !want_col) return FP8Q_ERR_INVALID_ARG;
    if (want_row && (q == nullptr || q_scales == nullptr)) return FP8Q_ERR_INVALID_ARG;
    if (want_col && (q_t == nullptr || qt_scales == nullptr)) return FP8Q_ERR_INVALID_ARG;
  }
  if ((rc = check_ptr(q, false)) != FP8Q_OK || (rc = check_ptr(q_t, false)) != FP8Q_OK ||
      (rc = check_ptr(q_scales, false)) != FP8Q_OK || (rc = check_ptr(qt_scales, false)) != FP8Q_OK)
    return rc;
  if ((rc = check_device()) != FP8Q_OK) return rc;
  if (rows == 0 || cols == 0) return FP8Q_OK;
  QuantParams p{};
  p.x = x;
  p.rows = rows;
  p.cols = cols;
  p.in_dtype = in_dtype;
  p.format = format;
  p.saturate = 1;
  p.mode = kModeMx;
  p.err = device_error_word();
  p.q = want_row ? q : nullptr;
  p.mx_scales = want_row ? q_scales : nullptr;
  p.q_t = want_col ? q_t : nullptr;
  p.mxt_scales = want_col ? qt_scales : nullptr;
  if (log_enabled())
    fprintf(stderr, "[fp8q] quantize_mxfp8 %lldx%lld fmt=%d rows=%d cols=%d\n", (long long)rows,
            (long long)cols, format, want_row, want_col);
  return from_cuda(launch_quant2d(p, stream));
}

int fp8_quantize_block128x128(const void *x, int in_dtype, int64_t rows, int64_t cols,
                              int format, uint8_t *q, uint8_t *q_t, float *block_scales,
                              int saturate, cudaStream_t stream) {
  int rc = check_quant(x, in_dtype, rows, cols, format, q_t != nullptr);
  if (rc != FP8Q_OK) return rc;
  if (rows > 0 && cols > 0 && (block_scales == nullptr || (q == nullptr && q_t == nullptr)))
    return FP8Q_ERR_INVALID_ARG;
  if ((rc = check_ptr(q, false)) != FP8Q_OK || (rc = check_ptr(q_t, false)) != FP8Q_OK) return rc;
  if (reinterpret_cast<uintptr_t>(block_scales) & 3u) return FP8Q_ERR_MISALIGNED;
  if ((rc = check_device()) != FP8Q_OK) return rc;
  if (rows == 0 || cols == 0) return FP8Q_OK;
  QuantParams p{};
  p.x = x;
  p.rows = rows;
  p.cols = cols;
  p.in_dtype = in_dtype;
  p.format = format;
  p.saturate = saturate;
  p.mode = kModeBlock;
  p.err = device_error_word();
  p.q = q;
  p.q_t = q_t;
  p.q_scales = block_scales;
  return from_cuda(launch_quant2d(p, stream));
}

namespace {

int gemm_common(const fp8q_operand *A, const fp8q_operand *B, void *C, int out_dtype, int64_t M,
                int64_t N, int64_t K, float *amax_out, cudaStream_t stream) {
  if (M < 0 || N < 0 || K < 0 || !valid_dtype(out_dtype)) return FP8Q_ERR_INVALID_ARG;
  // operand bytes M K and N K, and output bytes (4 per element at most), fit in int64
  if ((M > 0 && K > INT64_MAX / M) || (N > 0 && K > INT64_MAX / N) ||
      (M > 0 && N > INT64_MAX / 4 / M))
    return FP8Q_ERR_INVALID_ARG;
  if (N % 16 != 0 || K % 16 != 0) return FP8Q_ERR_INVALID_ARG;
  int rc;
  if ((rc = check_operand(A, M, K)) != FP8Q_OK) return rc;
  if ((rc = check_operand(B, N, K)) != FP8Q_OK) return rc;
  if (M > 0 && N > 0) {
    if (C == nullptr) return FP8Q_ERR_INVALID_ARG;
    if (!aligned16(C)) return FP8Q_ERR_MISALIGNED;
  }
  if ((rc = check_device()) != FP8Q_OK) return rc;
  if (log_enabled())
    fprintf(stderr, "[fp8q] gemm M=%lld N=%lld K=%lld A(fmt=%d,scale=%d) B(fmt=%d,scale=%d) out=%d\n",
            (long long)M, (long long)N, (long long)K, A->format, A->scaling, B->format,
            B->scaling, out_dtype);
  if (amax_out != nullptr &&
      cudaMemsetAsync(amax_out, 0, sizeof(float), stream) != cudaSuccess)
    return FP8Q_ERR_CUDA;
  return launch_gemm(to_dev(A), to_dev(B), C, out_dtype, M, N, K, stream, amax_out);
}

}  // namespace

int fp8_gemm(const fp8q_operand *A, const fp8q_operand *B, void *C, int out_dtype, int64_t M,
             int64_t N, int64_t K, cudaStream_t stream) {
  return gemm_common(A, B, C, out_dtype, M, N, K, nullptr, stream);
}

int fp8_gemm_amax(const fp8q_operand *A, const fp8q_operand *B, void *C, int out_dtype,
                  int64_t M, int64_t N, int64_t K, float *amax_out, cudaStream_t stream) {
  if (amax_out == nullptr) return FP8Q_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(amax_out) & 3u) return FP8Q_ERR_MISALIGNED;
  return gemm_common(A, B, C, out_dtype, M, N, K, amax_out, stream);
}

namespace {

// C [m, n] = A [m, k] . B [n, k]^T for one role, with both operands' scale
// layouts checked against their shapes first.
int gemm_role(const fp8q_operand *A, const fp8q_operand *B, void *C, int out_dtype, int64_t m,
              int64_t n, int64_t k, cudaStream_t stream) {
  if (A == nullptr || B == nullptr || m < 0 || n < 0 || k < 0) return FP8Q_ERR_INVALID_ARG;
  int rc;
  if ((rc = check_layout(A, m, k)) != FP8Q_OK || (rc = check_layout(B, n, k)) != FP8Q_OK)
    return rc;
  return fp8_gemm(A, B, C, out_dtype, m, n, k, stream);
}

}  // namespace

int fp8_gemm_grouped(const fp8q_gemm_desc *descs, int count, int out_dtype,
                     cudaStream_t stream) {
  if (count < 0 || count > FP8Q_GEMM_GROUP_MAX || (count > 0 && descs == nullptr) ||
      !valid_dtype(out_dtype))
    return FP8Q_ERR_INVALID_ARG;
  GemmOperandDev A[FP8Q_GEMM_GROUP_MAX], B[FP8Q_GEMM_GROUP_MAX];
  void *C[FP8Q_GEMM_GROUP_MAX];
  int64_t M[FP8Q_GEMM_GROUP_MAX], N[FP8Q_GEMM_GROUP_MAX], K[FP8Q_GEMM_GROUP_MAX];
  for (int i = 0; i < count; ++i) {
    const fp8q_gemm_desc &d = descs[i];
    if (d.M < 0 || d.N < 0 || d.K < 0 || d.N % 16 != 0 || d.K % 16 != 0)
      return FP8Q_ERR_INVALID_ARG;
    int rc;
    if ((rc = check_operand(&d.A, d.M, d.K)) != FP8Q_OK) return rc;
    if ((rc = check_operand(&d.B, d.N, d.K)) != FP8Q_OK) return rc;
    if ((rc = check_layout(&d.A, d.M, d.K)) != FP8Q_OK) return rc;
    if ((rc = check_layout(&d.B, d.N, d.K)) != FP8Q_OK) return rc;
    if (d.M > 0 && d.N > 0) {
      if (d.C == nullptr) return FP8Q_ERR_INVALID_ARG;
      if (!aligned16(d.C)) return FP8Q_ERR_MISALIGNED;
    }
    A[i] = to_dev(&d.A);
    B[i] = to_dev(&d.B);
    C[i] = d.C;
    M[i] = d.M;
    N[i] = d.N;
    K[i] = d.K;
  }
  if (count == 0) return FP8Q_OK;
  int rc;
  if ((rc = check_device()) != FP8Q_OK) return rc;
  return launch_gemm_group(A, B, C, M, N, K, count, out_dtype, stream);
}

int fp8_gemm_fprop(const fp8q_operand *x, const fp8q_operand *w, void *y, int out_dtype,
                   int64_t M, int64_t N, int64_t K, cudaStream_t stream) {
  // y [M, N] = x [M, K] . w [N, K]^T
  return gemm_role(x, w, y, out_dtype, M, N, K, stream);
}

int fp8_gemm_dgrad(const fp8q_operand *g, const fp8q_operand *w_t, void *dx, int out_dtype,
                   int64_t M, int64_t N, int64_t K, cudaStream_t stream) {
  // dx [M, K] = g [M, N] . (w_t [K, N])^T, contraction over N
  return gemm_role(g, w_t, dx, out_dtype, M, K, N, stream);
}

int fp8_gemm_wgrad(const fp8q_operand *g_t, const fp8q_operand *x_t, void *dw, int out_dtype,
                   int64_t M, int64_t N, int64_t K, cudaStream_t stream) {
  // dw [N, K] = g_t [N, M] . (x_t [K, M])^T, contraction over M
  return gemm_role(g_t, x_t, dw, out_dtype, N, K, M, stream);
}

size_t fp8q_linear_workspace_size(int recipe, int64_t M, int64_t N, int64_t K) {
  if (!linear_dims_ok(M, N, K)) return 0;
  size_t b = round256((size_t)(M * K)) + round256((size_t)(N * K));  // FP8 copies of x, w
  b += 2 * round256(sizeof(float)) * 2;                               // amax + scale for x, w
  if (recipe == FP8Q_RECIPE_BLOCK) {
    b += round256(sizeof(float) * (size_t)(((K + 127) / 128) * M));    // x tile scales
    b += round256(sizeof(float) * (size_t)(((N + 127) / 128) * ((K + 127) / 128)));
  } else if (recipe == FP8Q_RECIPE_MXFP8) {
    b += round256(fp8q_mx_scale_bytes(M, K)) + round256(fp8q_mx_scale_bytes(N, K));
  }
  return b;
}

int fp8_linear_autocast(const void *x, const void *w, int in_dtype, int64_t M, int64_t N,
                        int64_t K, int recipe, fp8q_amax_history *hist_x,
                        fp8q_amax_history *hist_w, void *y, int out_dtype, void *workspace,
                        size_t ws_bytes, cudaStream_t stream) {
  if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype)) return FP8Q_ERR_INVALID_ARG;
  if (!linear_dims_ok(M, N, K) || K % 16 != 0 || N % 16 != 0) return FP8Q_ERR_INVALID_ARG;
  if (recipe != FP8Q_RECIPE_TENSOR_CURRENT && recipe != FP8Q_RECIPE_TENSOR_DELAYED &&
      recipe != FP8Q_RECIPE_BLOCK && recipe != FP8Q_RECIPE_MXFP8)
    return FP8Q_ERR_INVALID_ARG;
  if (recipe == FP8Q_RECIPE_TENSOR_DELAYED && (hist_x == nullptr || hist_w == nullptr))
    return FP8Q_ERR_INVALID_ARG;
  const size_t need = fp8q_linear_workspace_size(recipe, M, N, K);
  if (workspace == nullptr || ws_bytes < need) return FP8Q_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FP8Q_ERR_MISALIGNED;
  int rc = check_device();
  if (rc != FP8Q_OK) return rc;

  uint8_t *ws = static_cast<uint8_t *>(workspace);
  uint8_t *qx = ws;
  ws += round256((size_t)(M * K));
  uint8_t *qw = ws;
  ws += round256((size_t)(N * K));
  float *amax_x = reinterpret_cast<float *>(ws);
  ws += round256(sizeof(float));
  float *amax_w = reinterpret_cast<float *>(ws);
  ws += round256(sizeof(float));
  float *sx = reinterpret_cast<float *>(ws);
  ws += round256(sizeof(float));
  float *sw = reinterpret_cast<float *>(ws);
  ws += round256(sizeof(float));

  fp8q_operand A{}, B{};
  A.data = qx;
  A.format = FP8Q_E4M3;
  B.data = qw;
  B.format = FP8Q_E4M3;
  if (recipe == FP8Q_RECIPE_BLOCK) {
    float *x_scales = reinterpret_cast<float *>(ws);
    ws += round256(sizeof(float) * (size_t)(((K + 127) / 128) * M));
    float *w_scales = reinterpret_cast<float *>(ws);
    if ((rc = fp8_quantize_tile1x128(x, in_dtype, M, K, FP8Q_E4M3, qx, x_scales, nullptr, nullptr,
                                     0, stream)) != FP8Q_OK)
      return rc;
    if ((rc = fp8_quantize_block128x128(w, in_dtype, N, K, FP8Q_E4M3, qw, nullptr, w_scales, 0,
                                        stream)) != FP8Q_OK)
      return rc;
    A.scaling = FP8Q_SCALE_TILE_1x128;
    A.scale = x_scales;
    A.scale_stride_row = 1;
    A.scale_stride_k = M;
    B.scaling = FP8Q_SCALE_BLOCK_128x128;
    B.scale = w_scales;
    B.scale_stride_row = (K + 127) / 128;
    B.scale_stride_k = 1;
  } else if (recipe == FP8Q_RECIPE_MXFP8) {
    uint8_t *x_atoms = ws;
    ws += round256(fp8q_mx_scale_bytes(M, K));
    uint8_t *w_atoms = ws;
    if ((rc = fp8_quantize_mxfp8(x, in_dtype, M, K, FP8Q_E4M3, qx, x_atoms, nullptr, nullptr,
                                 stream)) != FP8Q_OK)
      return rc;
    if ((rc = fp8_quantize_mxfp8(w, in_dtype, N, K, FP8Q_E4M3, qw, w_atoms, nullptr, nullptr,
                                 stream)) != FP8Q_OK)
      return rc;
    A.scaling = FP8Q_SCALE_MX_1x32;
    A.mx_scale = x_atoms;
    B.scaling = FP8Q_SCALE_MX_1x32;
    B.mx_scale = w_atoms;
  } else {
    if (recipe == FP8Q_RECIPE_TENSOR_CURRENT) {
      if ((rc = fp8_amax(x, in_dtype, M * K, amax_x, stream)) != FP8Q_OK) return rc;
      if ((rc = fp8_amax(w, in_dtype, N * K, amax_w, stream)) != FP8Q_OK) return rc;
      if ((rc = fp8_quantize_tensor(x, in_dtype, M, K, FP8Q_E4M3, amax_x, sx, qx, nullptr, 0,
                                    stream)) != FP8Q_OK)
        return rc;
      if ((rc = fp8_quantize_tensor(w, in_dtype, N, K, FP8Q_E4M3, amax_w, sw, qw, nullptr, 0,
                                    stream)) != FP8Q_OK)
        return rc;
    } else {
      if ((rc = fp8_quantize_delayed(x, in_dtype, M, K, FP8Q_E4M3, hist_x, sx, qx, nullptr, 0,
                                     stream)) != FP8Q_OK)
        return rc;
      if ((rc = fp8_quantize_delayed(w, in_dtype, N, K, FP8Q_E4M3, hist_w, sw, qw, nullptr, 0,
                                     stream)) != FP8Q_OK)
        return rc;
    }
    A.scaling = FP8Q_SCALE_TENSOR;
    A.scale = sx;
    B.scaling = FP8Q_SCALE_TENSOR;
    B.scale = sw;
  }
  return fp8_gemm_fprop(&A, &B, y, out_dtype, M, N, K, stream);
}

}  // extern "C"

// ----------------------------------------------------- a linear's whole step

namespace {

// Workspace carving of fp8_linear_train: FP8 copies of x, w, g in both
// orientations, then the recipe's scales (256-byte aligned pieces).
struct TrainLayout {
  size_t qx, qxt, qw, qwt, qg, qgt;        // byte offsets of the FP8 copies
  size_t sx, sxt, sw, swt, sg, sgt;        // scale arrays (or per-tensor scalars)
  size_t ax, aw, ag;                       // per-tensor amax words
  size_t total;
};

TrainLayout train_layout(int recipe, int64_t M, int64_t N, int64_t K) {
  TrainLayout L{};
  size_t o = 0;
  auto take = [&](size_t bytes) { const size_t at = o; o += round256(bytes); return at; };
  L.qx = take((size_t)(M * K));
  L.qxt = take((size_t)(M * K));
  L.qw = take((size_t)(N * K));
  L.qwt = take((size_t)(N * K));
  L.qg = take((size_t)(M * N));
  L.qgt = take((size_t)(M * N));
  const size_t f = sizeof(float);
  if (recipe == FP8Q_RECIPE_BLOCK) {
    L.sx = take(f * (size_t)(((K + 127) / 128) * M));          // x row tiles
    L.sxt = take(f * (size_t)(((M + 127) / 128) * K));         // x column tiles
    L.sw = take(f * (size_t)(((N + 127) / 128) * ((K + 127) / 128)));
    L.sg = take(f * (size_t)(((N + 127) / 128) * M));          // g row tiles
    L.sgt = take(f * (size_t)(((M + 127) / 128) * N));         // g column tiles
  } else if (recipe == FP8Q_RECIPE_MXFP8) {
    L.sx = take(fp8q_mx_scale_bytes(M, K));
    L.sxt = take(fp8q_mx_scale_bytes(K, M));
    L.sw = take(fp8q_mx_scale_bytes(N, K));
    L.swt = take(fp8q_mx_scale_bytes(K, N));
    L.sg = take(fp8q_mx_scale_bytes(M, N));
    L.sgt = take(fp8q_mx_scale_bytes(N, M));
  } else {
    L.sx = take(f);
    L.sw = take(f);
    L.sg = take(f);
    L.ax = take(f);
    L.aw = take(f);
    L.ag = take(f);
  }
  L.total = o;
  return L;
}

bool valid_recipe(int r) {
  return r == FP8Q_RECIPE_TENSOR_CURRENT || r == FP8Q_RECIPE_TENSOR_DELAYED ||
         r == FP8Q_RECIPE_BLOCK || r == FP8Q_RECIPE_MXFP8;
}

int check_train_args(int in_dtype, int out_dtype, int64_t M, int64_t N, int64_t K, int recipe,
                     fp8q_amax_history *hx, fp8q_amax_history *hw, fp8q_amax_history *hg) {
  if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype) || !valid_recipe(recipe))
    return FP8Q_ERR_INVALID_ARG;
  if (!linear_dims_ok(M, N, K) || M % 16 != 0 || N % 16 != 0 || K % 16 != 0)
    return FP8Q_ERR_INVALID_ARG;
  if (recipe == FP8Q_RECIPE_TENSOR_DELAYED && (hx == nullptr || hw == nullptr || hg == nullptr))
    return FP8Q_ERR_INVALID_ARG;
  return FP8Q_OK;
}

// Library-owned streams and events of fp8_linear_train_host, per device,
// created on first use and kept until the process exits.  The mutex keeps
// the record / wait sequences of concurrent host threads apart.
struct HostStepRes {
  std::once_flag once;
  std::mutex mu;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t ev[8] = {};
  bool ok = false;
};
HostStepRes g_host_step[kMaxDevices];

HostStepRes *host_step_res() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  HostStepRes *r = &g_host_step[dev];
  std::call_once(r->once, [r] {
    bool ok = cudaStreamCreateWithFlags(&r->in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&r->out, cudaStreamNonBlocking) == cudaSuccess;
    for (int i = 0; ok && i < 8; ++i)
      ok = cudaEventCreateWithFlags(&r->ev[i], cudaEventDisableTiming) == cudaSuccess;
    r->ok = ok;
  });
  return r->ok ? r : nullptr;
}

}  // namespace

extern "C" {

size_t fp8q_linear_train_workspace_size(int recipe, int64_t M, int64_t N, int64_t K) {
  if (!linear_dims_ok(M, N, K) || !valid_recipe(recipe)) return 0;
  return train_layout(recipe, M, N, K).total;
}

}  // extern "C"

namespace {

// The body of fp8_linear_train, with three optional events for the
// host-buffer variant: the stream waits for g_ready before quantising g, and
// records y_done after the Fprop and dx_done after the Dgrad.  Arguments are
// validated by the callers.
int train_impl(const void *x, const void *w, const void *g, int in_dtype, int64_t M, int64_t N,
               int64_t K, int recipe, fp8q_amax_history *hist_x, fp8q_amax_history *hist_w,
               fp8q_amax_history *hist_g, void *y, void *dx, void *dw, int out_dtype,
               uint8_t *ws, cudaStream_t stream, cudaEvent_t g_ready, cudaEvent_t y_done,
               cudaEvent_t dx_done) {
  int rc;
  const TrainLayout L = train_layout(recipe, M, N, K);
  auto wait_g = [&]() {
    return g_ready == nullptr || cudaStreamWaitEvent(stream, g_ready, 0) == cudaSuccess;
  };
  uint8_t *qx = ws + L.qx, *qxt = ws + L.qxt, *qw = ws + L.qw, *qwt = ws + L.qwt;
  uint8_t *qg = ws + L.qg, *qgt = ws + L.qgt;
  auto fp = [&](size_t off) { return reinterpret_cast<float *>(ws + off); };
  fp8q_operand fx{}, fw{}, dg{}, dwt{}, wgt{}, wxt{};   // fprop A/B, dgrad A/B, wgrad A/B
  fx.data = qx;   fx.format = FP8Q_E4M3;
  fw.data = qw;   fw.format = FP8Q_E4M3;
  dg.data = qg;   dg.format = FP8Q_E5M2;
  dwt.data = qwt; dwt.format = FP8Q_E4M3;
  wgt.data = qgt; wgt.format = FP8Q_E5M2;
  wxt.data = qxt; wxt.format = FP8Q_E4M3;
  if (recipe == FP8Q_RECIPE_BLOCK) {
    if ((rc = fp8_quantize_tile1x128(x, in_dtype, M, K, FP8Q_E4M3, qx, fp(L.sx), qxt, fp(L.sxt),
                                     0, stream)) != FP8Q_OK ||
        (rc = fp8_quantize_block128x128(w, in_dtype, N, K, FP8Q_E4M3, qw, qwt, fp(L.sw), 0,
                                        stream)) != FP8Q_OK)
      return rc;
    if (!wait_g()) return FP8Q_ERR_CUDA;
    if ((rc = fp8_quantize_tile1x128(g, in_dtype, M, N, FP8Q_E5M2, qg, fp(L.sg), qgt, fp(L.sgt),
                                     0, stream)) != FP8Q_OK)
      return rc;
    const int64_t kbk = (K + 127) / 128;
    fx.scaling = FP8Q_SCALE_TILE_1x128;   fx.scale = fp(L.sx);   fx.scale_stride_row = 1;
    fx.scale_stride_k = M;
    fw.scaling = FP8Q_SCALE_BLOCK_128x128; fw.scale = fp(L.sw); fw.scale_stride_row = kbk;
    fw.scale_stride_k = 1;
    dg.scaling = FP8Q_SCALE_TILE_1x128;   dg.scale = fp(L.sg);   dg.scale_stride_row = 1;
    dg.scale_stride_k = M;
    dwt.scaling = FP8Q_SCALE_BLOCK_128x128; dwt.scale = fp(L.sw); dwt.scale_stride_row = 1;
    dwt.scale_stride_k = kbk;
    wgt.scaling = FP8Q_SCALE_TILE_1x128;  wgt.scale = fp(L.sgt); wgt.scale_stride_row = 1;
    wgt.scale_stride_k = N;
    wxt.scaling = FP8Q_SCALE_TILE_1x128;  wxt.scale = fp(L.sxt); wxt.scale_stride_row = 1;
    wxt.scale_stride_k = K;
  } else if (recipe == FP8Q_RECIPE_MXFP8) {
    if ((rc = fp8_quantize_mxfp8(x, in_dtype, M, K, FP8Q_E4M3, qx, ws + L.sx, qxt, ws + L.sxt,
                                 stream)) != FP8Q_OK ||
        (rc = fp8_quantize_mxfp8(w, in_dtype, N, K, FP8Q_E4M3, qw, ws + L.sw, qwt, ws + L.swt,
                                 stream)) != FP8Q_OK)
      return rc;
    if (!wait_g()) return FP8Q_ERR_CUDA;
    if ((rc = fp8_quantize_mxfp8(g, in_dtype, M, N, FP8Q_E5M2, qg, ws + L.sg, qgt, ws + L.sgt,
                                 stream)) != FP8Q_OK)
      return rc;
    fp8q_operand *ops[6] = {&fx, &fw, &dg, &dwt, &wgt, &wxt};
    const size_t offs[6] = {L.sx, L.sw, L.sg, L.swt, L.sgt, L.sxt};
    for (int i = 0; i < 6; ++i) {
      ops[i]->scaling = FP8Q_SCALE_MX_1x32;
      ops[i]->mx_scale = ws + offs[i];
    }
  } else {
    const bool delayed = recipe == FP8Q_RECIPE_TENSOR_DELAYED;
    const void *src[3] = {x, w, g};
    const int64_t rr[3] = {M, N, M}, cc[3] = {K, K, N};
    const int fmt[3] = {FP8Q_E4M3, FP8Q_E4M3, FP8Q_E5M2};
    uint8_t *q[3] = {qx, qw, qg}, *qt[3] = {qxt, qwt, qgt};
    const size_t so[3] = {L.sx, L.sw, L.sg}, ao[3] = {L.ax, L.aw, L.ag};
    fp8q_amax_history *h[3] = {hist_x, hist_w, hist_g};
    for (int i = 0; i < 3; ++i) {
      if (i == 2 && !wait_g()) return FP8Q_ERR_CUDA;
      if (delayed)
        rc = fp8_quantize_delayed(src[i], in_dtype, rr[i], cc[i], fmt[i], h[i], fp(so[i]), q[i],
                                  qt[i], 0, stream);
      else
        rc = fp8_quantize_tensor_current(src[i], in_dtype, rr[i], cc[i], fmt[i], fp(ao[i]),
                                         fp(so[i]), q[i], qt[i], 0, stream);
      if (rc != FP8Q_OK) return rc;
    }
    fx.scaling = fw.scaling = dg.scaling = dwt.scaling = wgt.scaling = wxt.scaling =
        FP8Q_SCALE_TENSOR;
    fx.scale = wxt.scale = fp(L.sx);
    fw.scale = dwt.scale = fp(L.sw);
    dg.scale = wgt.scale = fp(L.sg);
  }
  if ((rc = fp8_gemm_fprop(&fx, &fw, y, out_dtype, M, N, K, stream)) != FP8Q_OK) return rc;
  if (y_done != nullptr && cudaEventRecord(y_done, stream) != cudaSuccess) return FP8Q_ERR_CUDA;
  if ((rc = fp8_gemm_dgrad(&dg, &dwt, dx, out_dtype, M, N, K, stream)) != FP8Q_OK) return rc;
  if (dx_done != nullptr && cudaEventRecord(dx_done, stream) != cudaSuccess) return FP8Q_ERR_CUDA;
  return fp8_gemm_wgrad(&wgt, &wxt, dw, out_dtype, M, N, K, stream);
}

}  // namespace

extern "C" {

int fp8_linear_train(const void *x, const void *w, const void *g, int in_dtype, int64_t M,
                     int64_t N, int64_t K, int recipe, fp8q_amax_history *hist_x,
                     fp8q_amax_history *hist_w, fp8q_amax_history *hist_g, void *y, void *dx,
                     void *dw, int out_dtype, void *workspace, size_t ws_bytes,
                     cudaStream_t stream) {
  int rc = check_train_args(in_dtype, out_dtype, M, N, K, recipe, hist_x, hist_w, hist_g);
  if (rc != FP8Q_OK) return rc;
  if (workspace == nullptr || ws_bytes < train_layout(recipe, M, N, K).total)
    return FP8Q_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FP8Q_ERR_MISALIGNED;
  if ((rc = check_device()) != FP8Q_OK) return rc;
  return train_impl(x, w, g, in_dtype, M, N, K, recipe, hist_x, hist_w, hist_g, y, dx, dw,
                    out_dtype, static_cast<uint8_t *>(workspace), stream, nullptr, nullptr,
                    nullptr);
}

size_t fp8q_linear_train_host_workspace_size(int recipe, int in_dtype, int out_dtype, int64_t M,
                                             int64_t N, int64_t K) {
  if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype)) return 0;
  const size_t base = fp8q_linear_train_workspace_size(recipe, M, N, K);
  if (base == 0) return 0;
  const size_t ib = in_dtype == FP8Q_DT_BF16 ? 2 : 4, ob = out_dtype == FP8Q_DT_BF16 ? 2 : 4;
  return base + round256(ib * (size_t)(M * K)) + round256(ib * (size_t)(N * K)) +
         round256(ib * (size_t)(M * N)) + round256(ob * (size_t)(M * N)) +
         round256(ob * (size_t)(M * K)) + round256(ob * (size_t)(N * K));
}

int fp8_linear_train_host(const void *x_h, const void *w_h, const void *g_h, int in_dtype,
                          int64_t M, int64_t N, int64_t K, int recipe,
                          fp8q_amax_history *hist_x, fp8q_amax_history *hist_w,
                          fp8q_amax_history *hist_g, void *y_h, void *dx_h, void *dw_h,
                          int out_dtype, void *workspace, size_t ws_bytes, cudaStream_t stream) {
  int rc = check_train_args(in_dtype, out_dtype, M, N, K, recipe, hist_x, hist_w, hist_g);
  if (rc != FP8Q_OK) return rc;
  const size_t need = fp8q_linear_train_host_workspace_size(recipe, in_dtype, out_dtype, M, N, K);
  if (workspace == nullptr || ws_bytes < need) return FP8Q_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FP8Q_ERR_MISALIGNED;
  const bool any = M > 0 && N > 0 && K > 0;
  if (any && (x_h == nullptr || w_h == nullptr || g_h == nullptr || y_h == nullptr ||
              dx_h == nullptr || dw_h == nullptr))
    return FP8Q_ERR_INVALID_ARG;
  if ((rc = check_device()) != FP8Q_OK) return rc;
  HostStepRes *r = host_step_res();
  if (r == nullptr) return FP8Q_ERR_CUDA;
  const size_t ib = in_dtype == FP8Q_DT_BF16 ? 2 : 4, ob = out_dtype == FP8Q_DT_BF16 ? 2 : 4;
  const size_t bx = ib * (size_t)(M * K), bw = ib * (size_t)(N * K), bg = ib * (size_t)(M * N);
  const size_t by = ob * (size_t)(M * N), bdx = ob * (size_t)(M * K), bdw = ob * (size_t)(N * K);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  const size_t base = fp8q_linear_train_workspace_size(recipe, M, N, K);
  uint8_t *dxin = ws + base, *dwin = dxin + round256(bx), *dgin = dwin + round256(bw);
  uint8_t *dy = dgin + round256(bg), *ddx = dy + round256(by), *ddw = ddx + round256(bdx);
  std::lock_guard<std::mutex> lock(r->mu);
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  cudaEvent_t *ev = r->ev;
  // copies in: after everything already on the caller's stream (the
  // workspace may still be in use there); x and w first, g after
  if (!ok(cudaEventRecord(ev[0], stream)) || !ok(cudaStreamWaitEvent(r->in, ev[0], 0)) ||
      !ok(cudaMemcpyAsync(dxin, x_h, bx, cudaMemcpyHostToDevice, r->in)) ||
      !ok(cudaMemcpyAsync(dwin, w_h, bw, cudaMemcpyHostToDevice, r->in)) ||
      !ok(cudaEventRecord(ev[1], r->in)) ||
      !ok(cudaMemcpyAsync(dgin, g_h, bg, cudaMemcpyHostToDevice, r->in)) ||
      !ok(cudaEventRecord(ev[2], r->in)) || !ok(cudaStreamWaitEvent(stream, ev[1], 0)))
    return FP8Q_ERR_CUDA;
  // the step on the caller's stream: x and w are quantised while g is still
  // being copied in (the stream waits for it only before quantising g)
  if ((rc = train_impl(dxin, dwin, dgin, in_dtype, M, N, K, recipe, hist_x, hist_w, hist_g, dy,
                       ddx, ddw, out_dtype, ws, stream, ev[2], ev[3], ev[4])) != FP8Q_OK)
    return rc;
  // copies out on the library's out stream as each output is done (y during
  // the Dgrad, dx during the Wgrad), then the caller's stream waits for the
  // last, so work queued after this call sees the host buffers filled
  if (!ok(cudaStreamWaitEvent(r->out, ev[3], 0)) ||
      !ok(cudaMemcpyAsync(y_h, dy, by, cudaMemcpyDeviceToHost, r->out)) ||
      !ok(cudaStreamWaitEvent(r->out, ev[4], 0)) ||
      !ok(cudaMemcpyAsync(dx_h, ddx, bdx, cudaMemcpyDeviceToHost, r->out)) ||
      !ok(cudaEventRecord(ev[5], stream)) || !ok(cudaStreamWaitEvent(r->out, ev[5], 0)) ||
      !ok(cudaMemcpyAsync(dw_h, ddw, bdw, cudaMemcpyDeviceToHost, r->out)) ||
      !ok(cudaEventRecord(ev[6], r->out)) || !ok(cudaStreamWaitEvent(stream, ev[6], 0)))
    return FP8Q_ERR_CUDA;
  return FP8Q_OK;
}

}  // extern "C"
