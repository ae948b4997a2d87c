// The MXFP8 GEMM ("mxfp8", OCP Microscaling Formats v1.0: one E8M0 scale per
// 32 K elements of each operand row), on the tensor cores' own block scaling.
#include "fp8q_gemm_common.cuh"

namespace fp8q {
namespace gemm {
namespace {

// ------------------------------------------------------------------------
// MXFP8 GEMM (tcgen05.mma kind::mxf8f6f4 with block scaling): the tensor
// cores apply each operand's E8M0 scale per 32 K themselves, so the whole K
// range accumulates in TMEM and the epilogue only converts.  One SM per
// 128 x 256 tile.  A ring stage holds A (16 KB), B (32 KB) and the K block's
// scale atoms (512 bytes for A's 128 rows, two for B's 256 rows), which the
// MMA thread copies into a per-stage slot of tensor memory (tcgen05.cp,
// ordered before its MMAs) right before the K block's four MMAs.  Tensor
// memory: the accumulator in columns [0, 256), then one 16-column scale slot
// per ring stage (A's atom in 4 columns, B's two in 8): the slot the MMA
// reads for scale row i is column i / 32, byte = the MMA's K step, lane
// i % 32 of the lane quarter.  With no room for a second 256-column
// accumulator, the eight epilogue warps load the accumulator into registers
// and release it at once, so the next tile's MMAs overlap the conversion and
// the stores.
// ------------------------------------------------------------------------
constexpr int kMxStages = 4;
struct MxLayout {
  static constexpr int kABytes = kBM * kBK;            // 16 KB
  static constexpr int kBBytes = kMxBN * kBK;          // 32 KB
  static constexpr int kSfaOff = kABytes + kBBytes;    // A's scale atom
  static constexpr int kSfbOff = kSfaOff + 512;        // B's two atoms
  static constexpr int kStageBytes = 50 * 1024;        // a multiple of 1024: stages stay aligned
  static constexpr int kRingBytes = kMxStages * kStageBytes;
  static constexpr int kBarBytes = 8 * (2 * kMxStages + 3);  // full, empty, acc full/empty, drain
  static constexpr int kSmemBytes = kRingBytes + kBarBytes + 16 + 1024;
  static constexpr uint32_t kSfCol0 = 256;             // first scale slot
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kSfbOff + 1024 <= kStageBytes, "a stage holds tiles and atoms");
  static_assert(kSfCol0 + 16 * kMxStages <= kTmemCols, "scale slots fit in TMEM");
};

template <bool OUT_BF16>
__global__ void __launch_bounds__(320, 1)
    gemm_mx_kernel(const __grid_constant__ CUtensorMap ta,
                   const __grid_constant__ CUtensorMap tb, const GemmArgs p) {
  using L = MxLayout;
  constexpr int STAGES = kMxStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t ring = (raw + 1023u) & ~1023u;
  const uint32_t bars = ring + L::kRingBytes;
  const uint32_t full0 = bars, empty0 = bars + 8 * STAGES;
  const uint32_t accf = bars + 8 * (2 * STAGES), acce = accf + 8, drain = acce + 8;
  const uint32_t slot = bars + L::kBarBytes;
  uint8_t *slot_ptr = smem_raw + (slot - raw);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(slot_ptr + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    mbar_init(accf, 1);
    mbar_init(acce, 8);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
    prefetch_tmap(&ta);
    prefetch_tmap(&tb);
  }
  if (warp == 1) {
    tmem_alloc(slot, L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(slot_ptr);
  const int total = p.num_m_tiles * p.num_n_tiles;
  const int num_nb = (int)((p.N + 127) / 128);   // 128-row blocks of B

  if (warp == 0) {
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
        int mt, nt;
        tile_coords(u, p.num_m_tiles, p.num_n_tiles, mt, nt, p.group, p.along_n);
        const int nb0 = 2 * nt;
        const int nbv = min(2, num_nb - nb0);   // B's row blocks inside the matrix
        for (int kb = 0; kb < p.num_k_blocks; ++kb, ++it) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
          const uint32_t full = full0 + 8 * s;
          if (!wait_bounded(empty0 + 8 * s, ph ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          const uint32_t sa = ring + s * L::kStageBytes;
          mbar_arrive_expect_tx(full, L::kABytes + L::kBBytes + 512u * (1u + (uint32_t)nbv));
          tma_load_2d(sa, &ta, kb * kBK, mt * kBM, full);
          tma_load_2d(sa + L::kABytes, &tb, kb * kBK, nt * kMxBN, full);
          bulk_load(sa + L::kSfaOff, p.mx_a + ((int64_t)mt * p.num_k_blocks + kb) * 512, 512,
                    full);
          for (int h = 0; h < nbv; ++h)
            bulk_load(sa + L::kSfbOff + 512 * h,
                      p.mx_b + ((int64_t)(nb0 + h) * p.num_k_blocks + kb) * 512, 512, full);
        }
      }
      if (!ok) {
        // Let the copies already issued land before the CTA goes away.
        const uint32_t n = it < (uint32_t)STAGES ? it : (uint32_t)STAGES;
        for (uint32_t j = 0; j < n; ++j) {
          const uint32_t jj = it - 1 - j;
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(full0 + 8 * (jj % STAGES), (jj / STAGES) & 1u) &&
                 globaltimer_ns() - t0 < 200000000ull) {
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t it = 0, acc_it = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < total && ok; u += gridDim.x, ++acc_it) {
        if (!wait_bounded(acce, (acc_it & 1u) ^ 1u, abort_flag, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < p.num_k_blocks; ++kb, ++it) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
          if (!wait_bounded(full0 + 8 * s, ph, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = ring + s * L::kStageBytes;
          const uint32_t sf = tmem_base + L::kSfCol0 + 16u * s;
          tmem_cp_32x128b_x4(sf, sdesc_plain(sa + L::kSfaOff, 128));
          tmem_cp_32x128b_x4(sf + 4, sdesc_plain(sa + L::kSfbOff, 128));
          tmem_cp_32x128b_x4(sf + 8, sdesc_plain(sa + L::kSfbOff + 512, 128));
#pragma unroll
          for (int k = 0; k < kBK / kUmmaK; ++k) {
            const uint64_t ad = sdesc_k(sa + k * kUmmaK, kSwzSBO, kSwzMode);
            const uint64_t bd = sdesc_k(sa + L::kABytes + k * kUmmaK, kSwzSBO, kSwzMode);
            // K step k uses byte k of each scale word (32-wide block 4 kb + k)
            mma_mxf8f6f4(tmem_base, ad, bd, p.idesc | ((uint32_t)k << 29) | ((uint32_t)k << 4),
                         sf, sf + 4, (kb > 0 || k > 0) ? 1u : 0u);
          }
          mma_commit(empty0 + 8 * s);
        }
        if (!ok) break;
        mma_commit(accf);
      }
      drain_mma(drain, abort_flag);
    }
    __syncwarp();
  } else {
    // Warps 2..9: warp w drains TMEM lane quarter w % 4, columns
    // [128 h, 128 h + 128) with h = (w - 2) / 4.
    const int quarter = warp & 3, half = (warp - 2) >> 2;
    uint32_t acc_it = 0, run_max = 0;
    for (int u = blockIdx.x; u < total; u += gridDim.x, ++acc_it) {
      int mt, nt;
      tile_coords(u, p.num_m_tiles, p.num_n_tiles, mt, nt, p.group, p.along_n);
      if (!wait_bounded_warp(accf, acc_it & 1u, abort_flag, p.err)) break;
      tc_fence_after();
      uint32_t r[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c)
        tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(quarter * 32) << 16) + half * 128 + c * 32,
                           r[c]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce);   // the accumulator is free for the next tile
      const int64_t m = (int64_t)mt * kBM + quarter * 32 + lane;
      if (m < p.M) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int64_t n0 = (int64_t)nt * kMxBN + half * 128 + c * 32;
          if (n0 < p.N) {
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[c][j]);
            run_max = max(run_max, store32<OUT_BF16>(p.C, p.N, m, n0, v));
          }
        }
      }
    }
    publish_amax(p.amax, run_max);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, L::kTmemCols);
}

template <bool OUT_BF16>
int run_mx(const CUtensorMap &ta, const CUtensorMap &tb, const GemmArgs &a, int grid,
           cudaStream_t stream) {
  auto kernel = gemm_mx_kernel<OUT_BF16>;
  static PerDeviceOnce setup;  // per instantiation
  if (setup.get([&] { return set_smem(kernel, MxLayout::kSmemBytes) == cudaSuccess ? 1 : 0; }) !=
      1)
    return FP8Q_ERR_CUDA;
  kernel<<<grid, 320, MxLayout::kSmemBytes, stream>>>(ta, tb, a);
  return cudaGetLastError() == cudaSuccess ? FP8Q_OK : FP8Q_ERR_CUDA;
}

}  // namespace

int run_mx_family(const CUtensorMap &ta, const CUtensorMap &tb, const GemmArgs &a, int grid,
                  bool bf16, cudaStream_t stream) {
  return bf16 ? run_mx<true>(ta, tb, a, grid, stream) : run_mx<false>(ta, tb, a, grid, stream);
}

}  // namespace gemm
}  // namespace fp8q
