// Host-side declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/fp8q.h"

namespace fp8q {

constexpr int kNumSMsHint = 152;

// One-time set-up of a kernel launch (its shared-memory attribute, an
// occupancy query), run once per device and safe against concurrent first
// calls: get() runs init() on the first call from the current device and
// returns that call's result from then on.  Function attributes are
// per-device state, so a process that drives several devices sets each one.
class PerDeviceOnce {
 public:
  template <typename F>
  int get(F &&init) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return init();
    std::call_once(flag_[dev], [&] { value_[dev] = init(); });
    return value_[dev];
  }

 private:
  static constexpr int kMaxDevices = 64;
  std::once_flag flag_[kMaxDevices];
  int value_[kMaxDevices] = {};
};

// Device error word of the current device (set by kernels whose bounded
// waits expire).  Defined in fp8q_api.cu.
unsigned int *device_error_word();

// SM count of the current device (cached).
int sm_count();

// True when the environment sets FP8Q_LOG (to anything but "0"): every entry
// point and every kernel launch then prints one line to stderr naming what
// it runs, so a caller can see which kernel served each call.
bool log_enabled();

// True when M, N, K are non-negative and M*K, N*K (and the byte sums of a
// linear layer's workspace) fit in int64.  Defined in fp8q_api.cu.
bool linear_dims_ok(int64_t M, int64_t N, int64_t K);

// 2D tiled tensor map over a row-major matrix (outer rows of `inner`
// elements, rows row_stride_bytes apart); out-of-bounds elements read as
// zero.  False if the driver entry point is missing or rejects the shape.
bool make_tmap_2d(CUtensorMap *m, const void *base, CUtensorMapDataType dtype, uint64_t inner,
                  uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner,
                  uint32_t box_outer, CUtensorMapSwizzle swizzle);

enum QuantMode : int {
  kModeTensorCurrent = 0,  // s from a device amax
  kModeTensorDelayed = 1,  // s from a device amax history, amax(x) pushed
  kModeTile = 2,           // 1x128 row tiles and/or 128x1 column tiles
  kModeBlock = 3,          // 128x128 blocks
  kModeRowAmax = 4,        // row-wise pass 1: per-row / per-column amax into the scale arrays
  kModeRowCast = 5,        // row-wise pass 2: cast with per-row / per-column scales
  kModeTensorFused = 6,    // amax and per-tensor cast in one cooperative launch
  kModeMx = 7              // MXFP8: 1x32 row blocks and/or 32x1 column blocks, E8M0 scales
};

struct QuantParams {
  const void *x;
  int64_t rows, cols;
  int in_dtype;   // FP8Q_DT_*
  int format;     // FP8Q_E4M3 / FP8Q_E5M2
  int saturate;
  int mode;       // QuantMode
  const float *amax_in;        // kModeTensorCurrent
  fp8q_amax_history *hist;     // kModeTensorDelayed
  float *scale_out;            // tensor modes, nullable
  float *amax_out;             // kModeTensorFused: max |x| (zero on entry)
  uint8_t *q;                  // [rows, cols] or null
  uint8_t *q_t;                // [cols, rows] or null
  float *q_scales;             // tile: [ceil(cols/128), rows]; block: [nrb, ncb]
  float *qt_scales;            // tile: [ceil(rows/128), cols]
  uint8_t *mx_scales;          // MX: E8M0 atoms of q (see fp8_quantize_mxfp8)
  uint8_t *mxt_scales;         // MX: E8M0 atoms of q_t
  unsigned int *err;           // device error word (bounded waits)
  int work_slot;               // tile-scheduling slot (set at launch)
  int dynamic;                 // 1: tiles past the first few are claimed (set at launch)
};

cudaError_t launch_amax(const void *x, int in_dtype, int64_t n, float *amax,
                        cudaStream_t stream);
cudaError_t launch_quant2d(const QuantParams &p, cudaStream_t stream);
// Largest input (bytes) quantised by kModeTensorFused.  Up to here the one
// launch saves more than its grid barrier costs (4 and 8 MiB: 0.2-2 us
// faster); from 16 MiB the amax and cast kernels are 1.6-5 us faster, and the
// input must in any case stay in L2 between the two passes.
constexpr int64_t kFusedTensorMaxBytes = 8ll << 20;
// Row-wise pass 3: s[i] = max(fl32(s[i] / fmax), 1e-12) in place.
cudaError_t launch_amax_to_scale(float *s, int64_t n, int format, cudaStream_t stream);

struct GemmOperandDev {
  const uint8_t *data;
  int format;
  int scaling;
  const float *scale;
  const uint8_t *mx_scale;   // FP8Q_SCALE_MX_1x32: E8M0 atoms
  int64_t stride_row;
  int64_t stride_k;
};

// C[M,N] = A[M,K] . B[N,K]^T with dequantising scales.  With amax_out (one
// fp32, zero on entry) the epilogue also folds max |C| over the stored values
// into it.
int launch_gemm(const GemmOperandDev &A, const GemmOperandDev &B, void *C,
                int out_dtype, int64_t M, int64_t N, int64_t K,
                cudaStream_t stream, float *amax_out = nullptr);

// Independent GEMMs (count <= 3) in one launch where the CTA-pair kernel runs
// them all, else one launch each; arguments already validated.
int launch_gemm_group(const GemmOperandDev *A, const GemmOperandDev *B, void *const *C,
                      const int64_t *M, const int64_t *N, const int64_t *K, int count,
                      int out_dtype, cudaStream_t stream);

}  // namespace fp8q
