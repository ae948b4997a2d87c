"""The boundary without Python: a C program that includes include/fp8q.h,
links libfp8q.so and the CUDA runtime, and runs amax -> per-tensor cast ->
Fprop GEMM on device buffers it allocates itself.  Its FP8 bytes must equal
the oracle's and its bf16 output must lie within the GEMM bound of the
oracle's result for the same inputs."""
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_SOURCE = r"""
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "fp8q.h"

#define CHECK_FP8Q(call)                                                  \
  do {                                                                    \
    int rc_ = (call);                                                     \
    if (rc_ != FP8Q_OK) {                                                 \
      fprintf(stderr, "%s: %s\n", #call, fp8q_status_string(rc_));        \
      return 1;                                                           \
    }                                                                     \
  } while (0)
#define CHECK_CUDA(call)                                                  \
  do {                                                                    \
    cudaError_t e_ = (call);                                              \
    if (e_ != cudaSuccess) {                                              \
      fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));         \
      return 1;                                                           \
    }                                                                     \
  } while (0)

static int load(const char *dir, const char *name, void *dst, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE *f = fopen(path, "rb");
  if (!f) return 1;
  size_t got = fread(dst, 1, bytes, f);
  fclose(f);
  return got == bytes ? 0 : 1;
}

static int save(const char *dir, const char *name, const void *src, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/%s", dir, name);
  FILE *f = fopen(path, "wb");
  if (!f) return 1;
  size_t put = fwrite(src, 1, bytes, f);
  fclose(f);
  return put == bytes ? 0 : 1;
}

int main(int argc, char **argv) {
  if (argc != 5) return 2;
  const char *dir = argv[1];
  const int64_t M = atoll(argv[2]), N = atoll(argv[3]), K = atoll(argv[4]);
  const size_t xb = (size_t)(M * K) * 2, wb = (size_t)(N * K) * 2, yb = (size_t)(M * N) * 2;
  if (!fp8q_device_supported()) return 3;
  void *hx = malloc(xb), *hw = malloc(wb), *hy = malloc(yb), *hq = malloc(xb / 2);
  if (!hx || !hw || !hy || !hq) return 4;
  if (load(dir, "x.bin", hx, xb) || load(dir, "w.bin", hw, wb)) return 5;

  void *x, *w, *y;
  uint8_t *qx, *qw;
  float *amax, *scale;   /* [0]: x, [1]: w */
  CHECK_CUDA(cudaMalloc(&x, xb));
  CHECK_CUDA(cudaMalloc(&w, wb));
  CHECK_CUDA(cudaMalloc(&y, yb));
  CHECK_CUDA(cudaMalloc((void **)&qx, xb / 2));
  CHECK_CUDA(cudaMalloc((void **)&qw, wb / 2));
  CHECK_CUDA(cudaMalloc((void **)&amax, 256));
  CHECK_CUDA(cudaMalloc((void **)&scale, 256));
  CHECK_CUDA(cudaMemcpy(x, hx, xb, cudaMemcpyHostToDevice));
  CHECK_CUDA(cudaMemcpy(w, hw, wb, cudaMemcpyHostToDevice));

  cudaStream_t s;
  CHECK_CUDA(cudaStreamCreate(&s));
  CHECK_FP8Q(fp8_amax(x, FP8Q_DT_BF16, M * K, amax, s));
  CHECK_FP8Q(fp8_amax(w, FP8Q_DT_BF16, N * K, amax + 4, s));
  CHECK_FP8Q(fp8_quantize_tensor(x, FP8Q_DT_BF16, M, K, FP8Q_E4M3, amax, scale, qx, NULL, 0, s));
  CHECK_FP8Q(fp8_quantize_tensor(w, FP8Q_DT_BF16, N, K, FP8Q_E4M3, amax + 4, scale + 4, qw,
                                 NULL, 0, s));
  fp8q_operand a, b;
  a.data = qx;
  a.format = FP8Q_E4M3;
  a.scaling = FP8Q_SCALE_TENSOR;
  a.scale = scale;
  a.scale_stride_row = 0;
  a.scale_stride_k = 0;
  b = a;
  b.data = qw;
  b.scale = scale + 4;
  CHECK_FP8Q(fp8_gemm_fprop(&a, &b, y, FP8Q_DT_BF16, M, N, K, s));
  CHECK_CUDA(cudaStreamSynchronize(s));
  CHECK_FP8Q(fp8q_device_status());

  CHECK_CUDA(cudaMemcpy(hy, y, yb, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(hq, qx, xb / 2, cudaMemcpyDeviceToHost));
  if (save(dir, "y.bin", hy, yb) || save(dir, "qx.bin", hq, xb / 2)) return 6;
  printf("ok\n");
  return 0;
}
"""


def test_c_program_runs_the_path(tmp_path):
    from scaled_quantize_fp8_warp_gb300 import build_lib
    lib = build_lib.build()
    src = tmp_path / "use_fp8q.c"
    src.write_text(C_SOURCE)
    exe = tmp_path / "use_fp8q"
    subprocess.run([build_lib.nvcc(), "-O2", "-I", os.path.join(ROOT, "include"), "-o", str(exe),
                    str(src), lib, "-Xlinker", "-rpath", "-Xlinker", os.path.dirname(lib)],
                   check=True, capture_output=True, text=True)

    M, N, K = 256, 272, 384          # CTA-pair kernel, ragged N tile
    x = workloads.normal((M, K), 1.0, 90)
    w = workloads.normal((N, K), 0.02, 91)
    xb, wb = (t.view(torch.int16).numpy().view(np.uint16) for t in (x, w))
    xb.tofile(tmp_path / "x.bin")
    wb.tofile(tmp_path / "w.bin")
    r = subprocess.run([str(exe), str(tmp_path), str(M), str(N), str(K)], capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stderr)

    rq, _, rs = oracle.quantize_tensor(xb, oracle.E4M3)
    assert np.array_equal(np.fromfile(tmp_path / "qx.bin", dtype=np.uint8).reshape(M, K), rq)
    rqw, _, rsw = oracle.quantize_tensor(wb, oracle.E4M3)
    y_ref, absum = oracle.gemm_rows(oracle.GemmOperand.tensor(rq, oracle.E4M3, rs),
                                    oracle.GemmOperand.tensor(rqw, oracle.E4M3, rsw))
    bits = np.fromfile(tmp_path / "y.bin", dtype=np.uint16).reshape(M, N)
    y = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.all(np.abs(y - y_ref) <= oracle.gemm_bound(y_ref, absum, True))
