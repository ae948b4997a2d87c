// Device-side pieces shared by the GEMM kernels (fp8q_gemm.cu,
// fp8q_gemm_block.cu, fp8q_gemm_mx.cu): tile constants, the launch argument
// block, the persistent raster, the TMA producer loop for plain K blocks, the
// output stores and the fused amax of C; plus the per-family launch entry
// points the host dispatch in fp8q_gemm.cu calls.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fp8q_internal.h"
#include "fp8q_ptx.cuh"

namespace fp8q {
namespace gemm {

using namespace ptx;

constexpr int kBM = 128;
constexpr int kBK = 128;            // bytes = FP8 elements per K block
constexpr int kUmmaK = 32;          // K per tcgen05.mma for 8-bit inputs
// Per-tensor / row scaling at N > 128 runs on CTA pairs (cta_group::2) with
// kPairAcc TMEM accumulators of 256 columns each and a ring of kPairStages
// 32 KB stages per CTA.
constexpr int kPairAcc = 2;
constexpr int kPairStages = 6;
// Tile width and promotion warpgroups of the tile/block-scaled kernel.
constexpr int kBlockScaledBN = 256;
constexpr int kBlockScaledWG = 2;
constexpr int kMxBN = 256;   // N per tile of the MXFP8 kernel
// Raster of the block-scaled kernel: groups of 16 M tiles, M fastest.  Its
// promotion warps use the constant (no registers to spare for a runtime
// raster); the host passes the same values in GemmArgs for its producer.
constexpr int kBlockGroupM = 16;

struct GemmArgs {
  int64_t M, N, K;
  int num_m_tiles, num_n_tiles, num_k_blocks;
  uint32_t idesc;
  void *C;
  // per-tensor scales (device scalars)
  const float *scale_a;
  const float *scale_b;
  // tile / block / row scales
  int64_t a_stride_row, a_stride_k;
  int64_t b_stride_row, b_stride_k;
  int a_row, b_row;   // per-tensor kernel: 1 = one scale per row (ROW), 0 = scalar
  int group, along_n;  // raster (tile_coords)
  unsigned int *amax;  // max |C| over the stored values (fp32 bit pattern), or null
  unsigned int *err;
  // MXFP8: E8M0 scale atoms, 512 bytes per 128 rows x 128 K, atom (rb, kb) at
  // byte (rb * num_k_blocks + kb) * 512
  const uint8_t *mx_a;
  const uint8_t *mx_b;
};

// Raster of the persistent tile loop.  Units are visited in groups of
// `group` rows along M (p.along_n == 0: M fastest inside a group, then the
// group sweeps every N column) or of `group` columns along N (along_n == 1,
// roles swapped).  The host picks the orientation and the group so that the
// group's panels of the swept-across operand stay resident in L2 while the
// other operand streams past (see raster_for).
__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int &mt, int &nt,
                                            int group, int along_n) {
  const int num_a = along_n ? num_n : num_m;   // the grouped dimension
  const int num_b = along_n ? num_m : num_n;
  const int per_group = group * num_b;
  const int g = tile / per_group;
  const int first = g * group;
  const int gsize = min(num_a - first, group);
  const int local = tile - g * per_group;
  const int a = first + local % gsize, b = local / gsize;
  mt = along_n ? b : a;
  nt = along_n ? a : b;
}

// A 128-byte K block is staged with 128-byte swizzling: 8-row atoms of 1024
// bytes, shared-memory descriptor swizzle mode 2.
constexpr uint32_t kSwzMode = 2;
constexpr uint32_t kSwzSBO = 1024;

template <int BN, int STAGES>
struct Layout {
  static constexpr int kABytes = kBM * kBK;
  static constexpr int kBBytes = BN * kBK;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kRingBytes = STAGES * kStageBytes;
  static constexpr int kBarBytes = 8 * (2 * STAGES + 5);  // full, empty, acc full/empty x2, drain
  static constexpr int kSmemBytes = kRingBytes + kBarBytes + 16 + 1024;  // + align slack
};

// Producer loop shared by both kernels: one 128 x 128-byte A box and one
// BN x 128-byte B box per K block, into the next ring slot once the MMAs
// have released it.
template <int BN, int STAGES>
__device__ __forceinline__ void producer_loop(const CUtensorMap *ta, const CUtensorMap *tb,
                                              const GemmArgs &p, uint32_t ring, uint32_t bars,
                                              volatile int *abort_flag) {
  using L = Layout<BN, STAGES>;
  const int total = p.num_m_tiles * p.num_n_tiles;
  uint32_t it = 0;
  bool ok = true;
  for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
    int mt, nt;
    tile_coords(u, p.num_m_tiles, p.num_n_tiles, mt, nt, p.group, p.along_n);
    for (int kb = 0; kb < p.num_k_blocks; ++kb, ++it) {
      const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
      const uint32_t full = bars + 8 * s, empty = bars + 8 * (STAGES + s);
      if (!wait_bounded(empty, ph ^ 1u, abort_flag, p.err)) {
        ok = false;
        break;
      }
      const uint32_t sa = ring + s * L::kStageBytes;
      mbar_arrive_expect_tx(full, L::kStageBytes);
      tma_load_2d(sa, ta, kb * kBK, mt * kBM, full);
      tma_load_2d(sa + L::kABytes, tb, kb * kBK, nt * BN, full);
    }
  }
  if (!ok) {
    // Let the copies already issued land before the CTA goes away.
    const uint32_t n = it < (uint32_t)STAGES ? it : (uint32_t)STAGES;
    for (uint32_t j = 0; j < n; ++j) {
      const uint32_t jj = it - 1 - j;
      const uint32_t s = jj % STAGES, ph = (jj / STAGES) & 1u;
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(bars + 8 * s, ph) && globaltimer_ns() - t0 < 200000000ull) {
      }
    }
  }
}

// MMAs of one K block held in ring slot `s` (BK / 32 MMAs of K = 32).
template <int BN, int STAGES>
__device__ __forceinline__ void issue_kblock(uint32_t ring, uint32_t s, uint32_t d_tmem,
                                             uint32_t idesc, bool accumulate_first) {
  using L = Layout<BN, STAGES>;
  const uint32_t a0 = ring + s * L::kStageBytes;
  const uint32_t b0 = a0 + L::kABytes;
#pragma unroll
  for (int k = 0; k < kBK / kUmmaK; ++k) {
    const uint64_t ad = sdesc_k(a0 + k * kUmmaK, kSwzSBO, kSwzMode);
    const uint64_t bd = sdesc_k(b0 + k * kUmmaK, kSwzSBO, kSwzMode);
    mma_f8f6f4(d_tmem, ad, bd, idesc, (accumulate_first || k > 0) ? 1u : 0u);
  }
}

__device__ __forceinline__ void drain_mma(uint32_t drain_bar, volatile int *abort_flag) {
  // Completion of everything this thread issued: commit to a private barrier
  // and wait for its first phase (bounded).
  mma_commit(drain_bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(drain_bar, 0) && globaltimer_ns() - t0 < 200000000ull) {
  }
  (void)abort_flag;
}

// Store 32 consecutive fp32 results (already scaled) of row m starting at
// column n0; columns >= N are skipped in groups of 8 (N % 16 == 0).  The
// stores are streaming (evict-first in L2): C is written once and never read
// here, while the L2 still holds operand panels that other tiles re-read.
// Returns
// max |value| over what was stored, as it was stored (bf16 rounded or fp32),
// as an fp32 bit pattern; NaN patterns sort above Inf.
template <bool OUT_BF16>
__device__ __forceinline__ uint32_t store32(void *C, int64_t N, int64_t m, int64_t n0,
                                            const float (&v)[32]) {
  uint32_t mx = 0;
  if (OUT_BF16) {
    __nv_bfloat16 *row = static_cast<__nv_bfloat16 *>(C) + m * N;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      if (n0 + 8 * g < N) {
        uint32_t w[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          __nv_bfloat162 b = __floats2bfloat162_rn(v[8 * g + 2 * h], v[8 * g + 2 * h + 1]);
          w[h] = *reinterpret_cast<uint32_t *>(&b);
        }
        __stcs(reinterpret_cast<uint4 *>(row + n0 + 8 * g), make_uint4(w[0], w[1], w[2], w[3]));
        const uint32_t k = 0x7FFF7FFFu;
        const uint32_t p = __vmaxu2(__vmaxu2(w[0] & k, w[1] & k), __vmaxu2(w[2] & k, w[3] & k));
        mx = max(mx, max(p & 0xFFFFu, p >> 16) << 16);
      }
    }
  } else {
    float *row = static_cast<float *>(C) + m * N;
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      if (n0 + 4 * g < N) {
        __stcs(reinterpret_cast<float4 *>(row + n0 + 4 * g),
               make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]));
#pragma unroll
        for (int j = 0; j < 4; ++j) mx = max(mx, __float_as_uint(v[4 * g + j]) & 0x7FFFFFFFu);
      }
    }
  }
  return mx;
}

// One atomicMax per warp of the lanes' running output maxima (the warp is
// converged here), when the caller asked for amax(C).
__device__ __forceinline__ void publish_amax(unsigned int *amax, uint32_t run_max) {
  if (amax == nullptr) return;
  const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, run_max);
  if ((threadIdx.x & 31) == 0 && m != 0) atomicMax(amax, m);
}

template <typename KernelT>
cudaError_t set_smem(KernelT kernel, int bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

// Launch entry points of the three kernel families (host side).
int run_tensor_family(const CUtensorMap &ta, const CUtensorMap &tb, const GemmArgs &a, int grid,
                      int BN, bool bf16, bool vec, cudaStream_t stream);
int run_blockscaled_family(const CUtensorMap &ta, const CUtensorMap &tb, const GemmArgs &a,
                           int grid, bool bf16, bool b_tile, cudaStream_t stream);
int run_mx_family(const CUtensorMap &ta, const CUtensorMap &tb, const GemmArgs &a, int grid,
                  bool bf16, cudaStream_t stream);

}  // namespace gemm
}  // namespace fp8q
