// fp8_linear_autocast_noalloc: the autocast forward for callers that cannot
// allocate device memory.
//
// Some callers of this library may not call cudaMalloc: a plugin hosted by an
// application that owns all device memory and hands it only the tensors, a
// serving loop that forbids allocation after start-up, or code that runs
// under another allocator's accounting and may not grow the process's device
// footprint.  They cannot provide the workspace that fp8_linear_autocast
// needs for the FP8 copies of x and w, their amaxes and scales.  This entry
// point keeps that workspace in one file-scope device array of a fixed size
// instead, and otherwise runs exactly fp8_linear_autocast.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "fp8q_internal.h"

namespace fp8q {
namespace {

// The shared scratch.  Every GPU on which this library's device code is
// loaded holds it until the process exits.
static __device__ __align__(256) uint8_t g_noalloc_scratch[FP8Q_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxNoallocDevices = 64;

struct ScratchSlot {
  std::once_flag once;
  void *ptr = nullptr;
  cudaError_t err = cudaSuccess;
};
ScratchSlot g_slots[kMaxNoallocDevices];

// Device address of the array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device, with that device current, and the return code checked.
int scratch_address(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxNoallocDevices)
    return FP8Q_ERR_CUDA;
  ScratchSlot *s = &g_slots[dev];
  std::call_once(s->once, [s] {
    void *p = nullptr;
    s->err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (s->err == cudaSuccess) s->ptr = p;
  });
  if (s->err != cudaSuccess || s->ptr == nullptr) return FP8Q_ERR_CUDA;
  *out = s->ptr;
  return FP8Q_OK;
}

}  // namespace
}  // namespace fp8q

extern "C" int fp8_linear_autocast_noalloc(const void *x, const void *w, int in_dtype,
                                           int64_t M, int64_t N, int64_t K, int recipe,
                                           fp8q_amax_history *hist_x,
                                           fp8q_amax_history *hist_w, void *y, int out_dtype,
                                           cudaStream_t stream) {
  // Negative sizes, or sizes whose byte counts overflow, never reach the
  // size check below (whose result could otherwise wrap under the limit).
  if (!fp8q::linear_dims_ok(M, N, K)) return FP8Q_ERR_INVALID_ARG;
  // Reject sizes whose scratch does not fit before touching the device.
  const size_t need = fp8q_linear_workspace_size(recipe, M, N, K);
  if (need > (size_t)FP8Q_NOALLOC_SCRATCH_BYTES) return FP8Q_ERR_WORKSPACE;
  if (fp8q_device_supported() != 1) return FP8Q_ERR_ARCH;
  void *scratch = nullptr;
  const int rc = fp8q::scratch_address(&scratch);
  if (rc != FP8Q_OK) return rc;
  // The amax words that must start at zero are cleared inside (fp8_amax
  // zeroes its output on the stream before reducing into it).
  return fp8_linear_autocast(x, w, in_dtype, M, N, K, recipe, hist_x, hist_w, y, out_dtype,
                             scratch, (size_t)FP8Q_NOALLOC_SCRATCH_BYTES, stream);
}
