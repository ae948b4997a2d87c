// Steps a4-a5 of the path: the FP8 GEMM C = A . B^T with dequantising scales
// ("fp8_parity.py", FP8Matmul: xq @ wq.T; the blog repost's Fprop / Dgrad /
// Wgrad shapes), on the 5th-generation tensor cores.
//
// Persistent, warp-specialised kernels over output tiles, in three files:
//   this file            the per-tensor / row-scaled kernels and the host
//                        dispatch (launch_gemm):
//     gemm_tensor_pair_kernel  N > 128: a CTA pair (cta_group::2) computes
//                        256 x 256 tiles, each CTA staging its own 128 rows
//                        of A and of B;
//     gemm_tensor_kernel       N <= 128: one SM per 128 x BN tile (BN = 64,
//                        128);
//   fp8q_gemm_block.cu   gemm_blockscaled_kernel, 1x128 / 128x128 scales
//                        promoted per K block in fp32 registers;
//   fp8q_gemm_mx.cu      gemm_mx_kernel, MXFP8 with the tensor cores' own
//                        block scaling.
// Roles: warp 0 is the TMA producer (128-byte swizzled boxes into a
// shared-memory ring with full/empty mbarriers); warp 1 allocates TMEM and
// issues tcgen05.mma from one thread (K = 32 per instruction, four per
// 128-byte K block), with tcgen05.commit releasing ring slots and handing
// accumulators on; the remaining warps drain TMEM (tcgen05.ld), scale,
// convert and store.  Every TMA load fetches into the issuing CTA's own
// shared memory.  Per-tensor scaling accumulates the whole K range in TMEM
// (two accumulator buffers so one tile's epilogue overlaps the next tile's
// MMAs) and applies s_A s_B once.
//
// Every mbarrier wait is bounded (about two seconds of wall time); on expiry
// the kernel records FP8Q_ERR_TIMEOUT in the device error word, drains what
// it issued, frees its TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <stdio.h>

#include <algorithm>
#include <mutex>

#include "fp8q_gemm_common.cuh"

namespace fp8q {
namespace gemm {
namespace {

// ------------------------------------------------------------------------
// Per-tensor scaled GEMM: 6 warps (producer, MMA, 4 epilogue warps).
// ------------------------------------------------------------------------
template <int BN, int STAGES, bool OUT_BF16, bool VEC>
__global__ void __launch_bounds__(192, 1)
    gemm_tensor_kernel(const __grid_constant__ CUtensorMap ta,
                       const __grid_constant__ CUtensorMap tb, const GemmArgs p) {
  using L = Layout<BN, STAGES>;
  constexpr uint32_t kTmemCols = (2 * BN < 32) ? 32 : 2 * BN;  // 128, 256 or 512
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t ring = (raw + 1023u) & ~1023u;
  const uint32_t bars = ring + L::kRingBytes;
  const uint32_t full0 = bars, empty0 = bars + 8 * STAGES;
  const uint32_t accf0 = bars + 8 * (2 * STAGES), acce0 = accf0 + 16;
  const uint32_t drain = acce0 + 16;
  const uint32_t slot = bars + L::kBarBytes;  // TMEM base address written here
  uint8_t *slot_ptr = smem_raw + (slot - raw);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(slot_ptr + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf0 + 8 * b, 1);
      mbar_init(acce0 + 8 * b, 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
    prefetch_tmap(&ta);
    prefetch_tmap(&tb);
  }
  if (warp == 1) {
    tmem_alloc(slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(slot_ptr);
  const int total = p.num_m_tiles * p.num_n_tiles;
  const int unit0 = blockIdx.x, unit_step = gridDim.x;

  if (warp == 0) {
    if (lane == 0) producer_loop<BN, STAGES>(&ta, &tb, p, ring, bars, abort_flag);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t it = 0, acc_it = 0;
      bool ok = true;
      for (int u = unit0; u < total && ok; u += unit_step, ++acc_it) {
        const uint32_t buf = acc_it & 1u, aph = (acc_it >> 1) & 1u;
        if (!wait_bounded(acce0 + 8 * buf, aph ^ 1u, abort_flag, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * BN;
        for (int kb = 0; kb < p.num_k_blocks; ++kb, ++it) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
          if (!wait_bounded(full0 + 8 * s, ph, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_kblock<BN, STAGES>(ring, s, d_tmem, p.idesc, kb > 0);
          mma_commit(empty0 + 8 * s);
        }
        if (!ok) break;
        mma_commit(accf0 + 8 * buf);
      }
      drain_mma(drain, abort_flag);
    }
    __syncwarp();
  } else {
    // Epilogue warps 2..5 -> TMEM lane quarters 2, 3, 0, 1.
    const int quarter = warp & 3;
    // Per-tensor: one product s_A s_B.  With row scales (VEC): s_A of this
    // thread's row times s_B of each column, applied the same way.
    const float scale = VEC ? 0.0f : __fmul_rn(p.scale_a[0], p.scale_b[0]);
    uint32_t acc_it = 0, run_max = 0;
    for (int u = unit0; u < total; u += unit_step, ++acc_it) {
      int mt, nt;
      tile_coords(u, p.num_m_tiles, p.num_n_tiles, mt, nt, p.group, p.along_n);
      const uint32_t buf = acc_it & 1u, aph = (acc_it >> 1) & 1u;
      if (!wait_bounded_warp(accf0 + 8 * buf, aph, abort_flag, p.err)) break;
      tc_fence_after();
      const int64_t m = (int64_t)mt * kBM + quarter * 32 + lane;
      float sa = 0.0f;
      if (VEC)
        sa = p.a_row ? (m < p.M ? p.scale_a[m * p.a_stride_row] : 0.0f) : p.scale_a[0];
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(quarter * 32) << 16) + buf * BN + c * 32, r);
        tmem_ld_wait();
        float v[32];
        const int64_t n0 = (int64_t)nt * BN + c * 32;
        if (VEC) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float sb = p.b_row ? (n0 + j < p.N ? p.scale_b[(n0 + j) * p.b_stride_row] : 0.0f)
                                     : p.scale_b[0];
            v[j] = __fmul_rn(__uint_as_float(r[j]), __fmul_rn(sa, sb));
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __fmul_rn(__uint_as_float(r[j]), scale);
        }
        if (m < p.M && n0 < p.N) run_max = max(run_max, store32<OUT_BF16>(p.C, p.N, m, n0, v));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce0 + 8 * buf);
    }
    publish_amax(p.amax, run_max);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

// ------------------------------------------------------------------------
// Per-tensor (or row) scaled GEMM on CTA pairs: tcgen05.mma.cta_group::2.
// A cluster of two CTAs computes one 256 x 256 tile.  Each CTA stages its
// own 128 rows of A and its own 128 of the tile's 256 B rows per K block
// (32 KB a stage instead of 48 KB for a 128 x 256 tile on one SM, so six
// stages fit where four did); the even CTA's MMA thread issues M = 256,
// N = 256 MMAs that read both CTAs' shared memory and write rows 0-127 of D
// into its own TMEM and rows 128-255 into the peer's.  Both CTAs' loads
// count on the even CTA's full barriers; its commits release the slots of
// both CTAs and hand each CTA's epilogue its half of D; both epilogues
// release the accumulator on the even CTA's barrier (8 warps).
// ------------------------------------------------------------------------
// A group of up to kMaxGroup independent GEMMs (for example a linear's
// Fprop, Dgrad and Wgrad) run by one persistent launch: their 256 x 256 units
// are numbered one problem after the other, so only the group's last wave is
// partial instead of each GEMM's.  A single GEMM is a group of one.
constexpr int kMaxGroup = 3;
struct PairGroup {
  int n;                       // problems in the group
  int unit_end[kMaxGroup];     // cumulative unit counts
  GemmArgs prob[kMaxGroup];
};
struct PairMaps {
  CUtensorMap a[kMaxGroup];
  CUtensorMap b[kMaxGroup];
};

// The problem of group unit u.  A launch of one GEMM (GROUPED = false) reads
// problem 0 at constant offsets, as a plain single-GEMM kernel would.
template <bool GROUPED>
__device__ __forceinline__ int group_of(const PairGroup &g, int u) {
  if (!GROUPED) return 0;
  int q = 0;
  while (q + 1 < g.n && u >= g.unit_end[q]) ++q;
  return q;
}

// Problem q and unit coordinates (unit row mu, column nt) of group unit u.
template <bool GROUPED>
__device__ __forceinline__ void group_coords(const PairGroup &g, int u, int &q, int &mu, int &nt) {
  q = group_of<GROUPED>(g, u);
  const int lu = u - (q > 0 ? g.unit_end[q - 1] : 0);
  const GemmArgs &p = g.prob[q];
  tile_coords(lu, (p.num_m_tiles + 1) / 2, p.num_n_tiles, mu, nt, p.group, p.along_n);
}

template <int STAGES>
struct PairLayout {
  static constexpr int kABytes = kBM * kBK;        // this CTA's 128 rows of A
  static constexpr int kBBytes = 128 * kBK;        // this CTA's 128 rows of B
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kRingBytes = STAGES * kStageBytes;
  static constexpr int kBarBytes = 8 * (2 * STAGES + 5);
  static constexpr int kSmemBytes = kRingBytes + kBarBytes + 16 + 1024;
};

template <int STAGES, int ACC, bool OUT_BF16, bool VEC, bool GROUPED>
__global__ void __launch_bounds__(192, 1)
    gemm_tensor_pair_kernel(const __grid_constant__ PairMaps maps,
                            const __grid_constant__ PairGroup g) {
  constexpr int BN = 256;
  using L = PairLayout<STAGES>;
  constexpr uint32_t kTmemCols = ACC * BN;
  constexpr uint16_t kBoth = 3;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t ring = (raw + 1023u) & ~1023u;
  const uint32_t bars = ring + L::kRingBytes;
  const uint32_t full0 = bars, empty0 = bars + 8 * STAGES;
  const uint32_t accf0 = bars + 8 * (2 * STAGES), acce0 = accf0 + 16;
  const uint32_t drain = acce0 + 16;
  const uint32_t slot = bars + L::kBarBytes;
  uint8_t *slot_ptr = smem_raw + (slot - raw);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(slot_ptr + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();   // 0: issues the pair's MMAs
  unsigned int *const err = g.prob[0].err;
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf0 + 8 * b, 1);
      mbar_init(acce0 + 8 * b, 8);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
    for (int q = 0; q < (GROUPED ? g.n : 1); ++q) {
      prefetch_tmap(&maps.a[q]);
      prefetch_tmap(&maps.b[q]);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(slot, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(slot_ptr);
  // One allocation serves the pair: both CTAs must hold the same address.
  // Otherwise neither does any work (a symmetric decision, no waiting).
  const bool paired = ld_shared_cluster_u32(mapa_shared(slot, rank ^ 1u)) == tmem_base;
  if (!paired && threadIdx.x == 0) atomicOr(err, 4u);

  const int total = g.unit_end[GROUPED ? g.n - 1 : 0];
  const int unit0 = blockIdx.x / 2, unit_step = gridDim.x / 2;

  if (!paired) {
  } else if (warp == 0) {
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int u = unit0; u < total && ok; u += unit_step) {
        int q, mu, nt;
        group_coords<GROUPED>(g, u, q, mu, nt);
        const int nkb = g.prob[q].num_k_blocks;
        // past the last M tile (odd count): re-read that tile's A, store nothing
        const int mt = min(2 * mu + (int)rank, g.prob[q].num_m_tiles - 1);
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
          if (!wait_bounded(empty0 + 8 * s, ph ^ 1u, abort_flag, err)) {
            ok = false;
            break;
          }
          const uint32_t sa = ring + s * L::kStageBytes;
          const uint32_t full_even = mapa_shared(full0 + 8 * s, 0);
          if (rank == 0) mbar_arrive_expect_tx(full0 + 8 * s, 2 * L::kStageBytes);
          tma_load_2d_pair(sa, &maps.a[q], kb * kBK, mt * kBM, full_even);
          tma_load_2d_pair(sa + L::kABytes, &maps.b[q], kb * kBK, nt * BN + (int)rank * 128,
                           full_even);
        }
      }
      // every slot's last release (the even CTA's commits) has arrived here
      for (uint32_t j = 0, jt = it; ok && j < (uint32_t)STAGES; ++j, ++jt)
        ok = wait_bounded(empty0 + 8 * (jt % STAGES), ((jt / STAGES) & 1u) ^ 1u, abort_flag,
                          err);
      if (!ok) {
        // aborting: give copies already issued (their barrier may be the
        // other CTA's) a millisecond to land before the CTA can leave
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 1000000ull) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      uint32_t it = 0, acc_it = 0;
      bool ok = true;
      for (int u = unit0; u < total && ok; u += unit_step, ++acc_it) {
        const uint32_t buf = ACC == 2 ? (acc_it & 1u) : 0u;
        const uint32_t aph = ACC == 2 ? ((acc_it >> 1) & 1u) : (acc_it & 1u);
        if (!wait_bounded(acce0 + 8 * buf, aph ^ 1u, abort_flag, err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * BN;
        const int q = group_of<GROUPED>(g, u);
        const int nkb = g.prob[q].num_k_blocks;
        const uint32_t idesc = g.prob[q].idesc;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
          if (!wait_bounded(full0 + 8 * s, ph, abort_flag, err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = ring + s * L::kStageBytes, b0 = a0 + L::kABytes;
#pragma unroll
          for (int k = 0; k < kBK / kUmmaK; ++k) {
            const uint64_t ad = sdesc_k(a0 + k * kUmmaK, kSwzSBO, kSwzMode);
            const uint64_t bd = sdesc_k(b0 + k * kUmmaK, kSwzSBO, kSwzMode);
            mma_f8f6f4_pair(d_tmem, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
          }
          mma_commit_pair_multicast(empty0 + 8 * s, kBoth);
        }
        if (!ok) break;
        mma_commit_pair_multicast(accf0 + 8 * buf, kBoth);
      }
      mma_commit_pair(drain);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(drain, 0) && globaltimer_ns() - t0 < 200000000ull) {
      }
    }
    __syncwarp();
  } else {
    // Epilogue warps 2..5 -> TMEM lane quarters 2, 3, 0, 1 of this CTA's
    // 128 rows of the pair tile.
    const int quarter = warp & 3;
    const uint32_t acce_even0 = mapa_shared(acce0, 0);
    uint32_t acc_it = 0, run_max0 = 0, run_max1 = 0, run_max2 = 0;   // per problem
    for (int u = unit0; u < total; u += unit_step, ++acc_it) {
      int q, mu, nt;
      group_coords<GROUPED>(g, u, q, mu, nt);
      // this unit's problem, read from the parameter block once (a reference
      // into it would be re-read after every asm statement)
      const GemmArgs p = g.prob[q];
      const float scale = VEC ? 0.0f : __fmul_rn(p.scale_a[0], p.scale_b[0]);
      uint32_t run_max = 0;
      const int mt = 2 * mu + (int)rank;   // >= num_m_tiles: nothing to store
      const uint32_t buf = ACC == 2 ? (acc_it & 1u) : 0u;
      const uint32_t aph = ACC == 2 ? ((acc_it >> 1) & 1u) : (acc_it & 1u);
      if (!wait_bounded_warp(accf0 + 8 * buf, aph, abort_flag, err)) break;
      tc_fence_after();
      const int64_t m = (int64_t)mt * kBM + quarter * 32 + lane;
      float sa = 0.0f;
      if (VEC)
        sa = p.a_row ? (m < p.M ? p.scale_a[m * p.a_stride_row] : 0.0f) : p.scale_a[0];
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(quarter * 32) << 16) + buf * BN + c * 32, r);
        tmem_ld_wait();
        float v[32];
        const int64_t n0 = (int64_t)nt * BN + c * 32;
        if (VEC) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float sb = p.b_row ? (n0 + j < p.N ? p.scale_b[(n0 + j) * p.b_stride_row] : 0.0f)
                                     : p.scale_b[0];
            v[j] = __fmul_rn(__uint_as_float(r[j]), __fmul_rn(sa, sb));
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __fmul_rn(__uint_as_float(r[j]), scale);
        }
        if (m < p.M && n0 < p.N) run_max = max(run_max, store32<OUT_BF16>(p.C, p.N, m, n0, v));
      }
      if (q == 0) run_max0 = max(run_max0, run_max);
      else if (q == 1) run_max1 = max(run_max1, run_max);
      else run_max2 = max(run_max2, run_max);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0)
          mbar_arrive(acce0 + 8 * buf);
        else
          mbar_arrive_cluster(acce_even0 + 8 * buf);
      }
    }
    publish_amax(g.prob[0].amax, run_max0);
    if (GROUPED && g.n > 1) publish_amax(g.prob[1].amax, run_max1);
    if (GROUPED && g.n > 2) publish_amax(g.prob[2].amax, run_max2);
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // neither CTA leaves while the other may still signal it
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, kTmemCols);
}

template <int STAGES, int ACC, bool OUT_BF16, bool VEC, bool GROUPED>
int run_tensor_pair(const PairMaps &maps, const PairGroup &grp, cudaStream_t stream) {
  using L = PairLayout<STAGES>;
  auto kernel = gemm_tensor_pair_kernel<STAGES, ACC, OUT_BF16, VEC, GROUPED>;
  static PerDeviceOnce setup;  // per instantiation: the pairs that fit at once, 0 on failure
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.blockDim = dim3(192, 1, 1);
  cfg.dynamicSmemBytes = L::kSmemBytes;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int max_clusters = setup.get([&] {
    if (set_smem(kernel, L::kSmemBytes) != cudaSuccess) return 0;
    cudaLaunchConfig_t q = cfg;
    q.gridDim = dim3(2 * (sm_count() / 2), 1, 1);
    int n = 0;
    return cudaOccupancyMaxActiveClusters(&n, kernel, &q) == cudaSuccess ? n : 0;
  });
  if (max_clusters < 1) return FP8Q_ERR_CUDA;
  const int units = grp.unit_end[grp.n - 1];
  if (units <= 0) return FP8Q_OK;
  cfg.gridDim = dim3(2 * (units < max_clusters ? units : max_clusters), 1, 1);
  if (cudaLaunchKernelEx(&cfg, kernel, maps, grp) != cudaSuccess) return FP8Q_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? FP8Q_OK : FP8Q_ERR_CUDA;
}

// One problem of a pair group: the pair instruction descriptor (M = N = 256)
// and the problem's unit count.
void add_pair_problem(PairMaps &maps, PairGroup &grp, const CUtensorMap &ta,
                      const CUtensorMap &tb, const GemmArgs &a) {
  const int q = grp.n++;
  maps.a[q] = ta;
  maps.b[q] = tb;
  grp.prob[q] = a;
  grp.prob[q].idesc = ptx::idesc_f8f6f4((a.idesc >> 7) & 7u, (a.idesc >> 10) & 7u, 256, 256);
  const int units = ((a.num_m_tiles + 1) / 2) * a.num_n_tiles;
  grp.unit_end[q] = (q > 0 ? grp.unit_end[q - 1] : 0) + units;
}

template <int STAGES, int ACC, bool OUT_BF16, bool VEC>
int run_tensor_pair(const CUtensorMap &ta, const CUtensorMap &tb, const GemmArgs &a,
                    cudaStream_t stream) {
  PairMaps maps;
  PairGroup grp{};
  add_pair_problem(maps, grp, ta, tb, a);
  return run_tensor_pair<STAGES, ACC, OUT_BF16, VEC, false>(maps, grp, stream);
}

template <int BN, int STAGES, bool OUT_BF16, bool VEC>
int run_tensor(const CUtensorMap &ta, const CUtensorMap &tb, const GemmArgs &a, int grid,
               cudaStream_t stream) {
  using L = Layout<BN, STAGES>;
  auto kernel = gemm_tensor_kernel<BN, STAGES, OUT_BF16, VEC>;
  static PerDeviceOnce setup;  // per instantiation
  if (setup.get([&] { return set_smem(kernel, L::kSmemBytes) == cudaSuccess ? 1 : 0; }) != 1)
    return FP8Q_ERR_CUDA;
  kernel<<<grid, 192, L::kSmemBytes, stream>>>(ta, tb, a);
  return cudaGetLastError() == cudaSuccess ? FP8Q_OK : FP8Q_ERR_CUDA;
}

}  // namespace

// A group of per-tensor-scaled problems (row scales are never grouped).
int run_tensor_pair_group(const PairMaps &maps, const PairGroup &grp, bool bf16,
                          cudaStream_t stream) {
  constexpr int PS = kPairStages, PA = kPairAcc;
  return bf16 ? run_tensor_pair<PS, PA, true, false, true>(maps, grp, stream)
              : run_tensor_pair<PS, PA, false, false, true>(maps, grp, stream);
}

int run_tensor_family(const CUtensorMap &ta, const CUtensorMap &tb, const GemmArgs &a, int grid,
                      int BN, bool bf16, bool vec, cudaStream_t stream) {
  constexpr int PS = kPairStages, PA = kPairAcc;
  if (vec) {
    if (BN == 64)
      return bf16 ? run_tensor<64, 8, true, true>(ta, tb, a, grid, stream)
                  : run_tensor<64, 8, false, true>(ta, tb, a, grid, stream);
    if (BN == 128)
      return bf16 ? run_tensor<128, 6, true, true>(ta, tb, a, grid, stream)
                  : run_tensor<128, 6, false, true>(ta, tb, a, grid, stream);
    return bf16 ? run_tensor_pair<PS, PA, true, true>(ta, tb, a, stream)
                : run_tensor_pair<PS, PA, false, true>(ta, tb, a, stream);
  }
  if (BN == 64)
    return bf16 ? run_tensor<64, 8, true, false>(ta, tb, a, grid, stream)
                : run_tensor<64, 8, false, false>(ta, tb, a, grid, stream);
  if (BN == 128)
    return bf16 ? run_tensor<128, 6, true, false>(ta, tb, a, grid, stream)
                : run_tensor<128, 6, false, false>(ta, tb, a, grid, stream);
  return bf16 ? run_tensor_pair<PS, PA, true, false>(ta, tb, a, stream)
              : run_tensor_pair<PS, PA, false, false>(ta, tb, a, stream);
}

namespace {
// Row-major [rows, K] byte matrix, box = 128 bytes of K x box_rows, 128-byte
// swizzle, out-of-bounds elements read as zero.
bool make_tmap(CUtensorMap *m, const void *base, uint64_t rows, uint64_t K, uint32_t box_rows) {
  return make_tmap_2d(m, base, CU_TENSOR_MAP_DATA_TYPE_UINT8, K, rows, K, kBK, box_rows,
                      CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

}  // namespace gemm

using namespace gemm;

// Raster for a persistent grid over units of unit_m x unit_n output
// elements (the two operands' panels are unit_m x K and unit_n x K bytes).
// Grouping along M with g units per group keeps those g A panels resident
// while the group sweeps all of N: A is read from DRAM once and B once per
// group; grouping along N is the mirror image.  g is as large as fits in
// kRasterBudget of L2 (the rest holds the streaming operand's panels and the
// output passing through), and the orientation with the smaller modelled
// DRAM traffic wins.
static void raster_for(int num_mu, int num_nu, int64_t unit_m, int64_t unit_n, int64_t K,
                       int &group, int &along_n) {
  constexpr int64_t kRasterBudget = 40ll << 20;
  const int64_t pa = unit_m * K, pb = unit_n * K;
  const int64_t ga = std::max<int64_t>(1, std::min<int64_t>(num_mu, kRasterBudget / pa));
  const int64_t gb = std::max<int64_t>(1, std::min<int64_t>(num_nu, kRasterBudget / pb));
  const int64_t a_bytes = pa * num_mu, b_bytes = pb * num_nu;
  const int64_t along_m_traffic = a_bytes + b_bytes * ((num_mu + ga - 1) / ga);
  const int64_t along_n_traffic = b_bytes + a_bytes * ((num_nu + gb - 1) / gb);
  if (along_n_traffic < along_m_traffic) {
    group = (int)gb;
    along_n = 1;
  } else {
    group = (int)ga;
    along_n = 0;
  }
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool make_tmap_2d(CUtensorMap *m, const void *base, CUtensorMapDataType dtype, uint64_t inner,
                  uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner,
                  uint32_t box_outer, CUtensorMapSwizzle swizzle) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t gdim[2] = {inner, outer};
  cuuint64_t gstride[1] = {row_stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estride[2] = {1, 1};
  CUresult r = fn(m, dtype, 2, const_cast<void *>(base), gdim, gstride, box, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The launch arguments every kernel family shares.
static void fill_args(GemmArgs &a, const GemmOperandDev &A, const GemmOperandDev &B, void *C,
                      int64_t M, int64_t N, int64_t K, int BN, float *amax_out) {
  a = GemmArgs{};
  a.M = M;
  a.N = N;
  a.K = K;
  a.num_m_tiles = (int)((M + kBM - 1) / kBM);
  a.num_n_tiles = (int)((N + BN - 1) / BN);
  a.num_k_blocks = (int)((K + kBK - 1) / kBK);
  a.idesc = ptx::idesc_f8f6f4((uint32_t)A.format, (uint32_t)B.format, kBM, (uint32_t)BN);
  a.C = C;
  a.scale_a = A.scale;
  a.scale_b = B.scale;
  a.a_stride_row = A.stride_row;
  a.a_stride_k = A.stride_k;
  a.b_stride_row = B.stride_row;
  a.b_stride_k = B.stride_k;
  a.a_row = A.scaling == FP8Q_SCALE_ROW ? 1 : 0;
  a.b_row = B.scaling == FP8Q_SCALE_ROW ? 1 : 0;
  a.amax = reinterpret_cast<unsigned int *>(amax_out);
  a.mx_a = A.mx_scale;
  a.mx_b = B.mx_scale;
  a.err = device_error_word();
}

int launch_gemm(const GemmOperandDev &A, const GemmOperandDev &B, void *C, int out_dtype,
                int64_t M, int64_t N, int64_t K, cudaStream_t stream, float *amax_out) {
  const bool bf16 = out_dtype == FP8Q_DT_BF16;
  if (M == 0 || N == 0) return FP8Q_OK;
  if (K == 0) {
    return cudaMemsetAsync(C, 0, (size_t)(M * N) * (bf16 ? 2 : 4), stream) == cudaSuccess
               ? FP8Q_OK
               : FP8Q_ERR_CUDA;
  }
  // TENSOR and ROW scales are constant along K: the whole sum accumulates in
  // TMEM and the scales are applied in the epilogue.
  const bool a_ep = A.scaling == FP8Q_SCALE_TENSOR || A.scaling == FP8Q_SCALE_ROW;
  const bool b_ep = B.scaling == FP8Q_SCALE_TENSOR || B.scaling == FP8Q_SCALE_ROW;
  const bool tensor = a_ep && b_ep;
  const bool vec = tensor && (A.scaling == FP8Q_SCALE_ROW || B.scaling == FP8Q_SCALE_ROW);
  const bool mx = A.scaling == FP8Q_SCALE_MX_1x32 && B.scaling == FP8Q_SCALE_MX_1x32;
  if (!tensor && !mx) {
    if (A.scaling != FP8Q_SCALE_TILE_1x128 ||
        (B.scaling != FP8Q_SCALE_TILE_1x128 && B.scaling != FP8Q_SCALE_BLOCK_128x128))
      return FP8Q_ERR_NOT_IMPLEMENTED;
  }
  int BN = mx ? kMxBN : kBlockScaledBN;
  if (tensor) BN = N <= 64 ? 64 : (N <= 128 ? 128 : 256);
  // BN = 256 runs on CTA pairs: each CTA loads 128 of the tile's B rows.
  const int b_box_rows = BN == 256 && tensor ? 128 : BN;
  CUtensorMap ta, tb;
  if (!make_tmap(&ta, A.data, (uint64_t)M, (uint64_t)K, kBM) ||
      !make_tmap(&tb, B.data, (uint64_t)N, (uint64_t)K, (uint32_t)b_box_rows))
    return FP8Q_ERR_CUDA;

  GemmArgs a;
  fill_args(a, A, B, C, M, N, K, BN, amax_out);
  if (a.err == nullptr) return FP8Q_ERR_CUDA;
  const int64_t tiles = (int64_t)a.num_m_tiles * a.num_n_tiles;
  if (tiles > INT32_MAX / 2) return FP8Q_ERR_INVALID_ARG;
  if (tensor && BN == 256) {         // CTA pairs: 256 x 256 units
    raster_for((a.num_m_tiles + 1) / 2, a.num_n_tiles, 256, 256, K, a.group, a.along_n);
  } else if (tensor || mx) {
    raster_for(a.num_m_tiles, a.num_n_tiles, kBM, BN, K, a.group, a.along_n);
  } else {
    // the promoted block-scaled kernel keeps a fixed raster: groups of 16 M
    // tiles measured 15% faster on its Wgrads than the traffic model's
    a.group = kBlockGroupM;
    a.along_n = 0;
  }
  int grid = sm_count();
  if (tiles < grid) grid = (int)tiles;
  if (log_enabled()) {
    const char *kernel = tensor ? (BN == 256 ? "gemm_tensor_pair_kernel" : "gemm_tensor_kernel")
                                : (mx ? "gemm_mx_kernel" : "gemm_blockscaled_kernel");
    const int unit_m = tensor && BN == 256 ? 256 : kBM;
    fprintf(stderr,
            "[fp8q] launch %s unit %dx%d units %lld k_blocks %d raster %d%s scales %s out %s\n",
            kernel, unit_m, BN, (long long)(unit_m == 256 ? (int64_t)((a.num_m_tiles + 1) / 2) *
                                                                a.num_n_tiles
                                                          : tiles),
            a.num_k_blocks, a.group, a.along_n ? " along N" : " along M",
            vec ? "row" : (tensor ? "tensor" : (mx ? "mx" : "promoted per K block")),
            bf16 ? "bf16" : "fp32");
  }

  if (tensor) return run_tensor_family(ta, tb, a, grid, BN, bf16, vec, stream);
  if (mx) {
    a.idesc = ptx::idesc_mxf8f6f4((uint32_t)A.format, (uint32_t)B.format, kBM, kMxBN, 0, 0);
    return run_mx_family(ta, tb, a, grid, bf16, stream);
  }
  return run_blockscaled_family(ta, tb, a, grid, bf16, B.scaling == FP8Q_SCALE_TILE_1x128,
                                stream);
}

int launch_gemm_group(const GemmOperandDev *A, const GemmOperandDev *B, void *const *C,
                      const int64_t *M, const int64_t *N, const int64_t *K, int count,
                      int out_dtype, cudaStream_t stream) {
  // One launch when every problem runs on the CTA-pair kernel with per-tensor
  // scales (N > 128, nothing empty).  Row scales keep one launch per GEMM: the
  // grouped form of their per-element scale epilogue measured 17% slower on
  // the layer's GEMMs.
  bool pair = count >= 1 && count <= kMaxGroup;
  for (int i = 0; i < count && pair; ++i) {
    if (A[i].scaling != FP8Q_SCALE_TENSOR || B[i].scaling != FP8Q_SCALE_TENSOR || N[i] <= 128 ||
        M[i] == 0 || K[i] == 0)
      pair = false;
  }
  if (!pair) {
    if (log_enabled())
      fprintf(stderr, "[fp8q] grouped call of %d GEMMs: one launch per GEMM\n", count);
    for (int i = 0; i < count; ++i) {
      const int rc = launch_gemm(A[i], B[i], C[i], out_dtype, M[i], N[i], K[i], stream, nullptr);
      if (rc != FP8Q_OK) return rc;
    }
    return FP8Q_OK;
  }
  PairMaps maps;
  PairGroup grp{};
  int64_t units = 0;
  for (int i = 0; i < count; ++i) {
    CUtensorMap ta, tb;
    if (!make_tmap(&ta, A[i].data, (uint64_t)M[i], (uint64_t)K[i], kBM) ||
        !make_tmap(&tb, B[i].data, (uint64_t)N[i], (uint64_t)K[i], 128))
      return FP8Q_ERR_CUDA;
    GemmArgs a;
    fill_args(a, A[i], B[i], C[i], M[i], N[i], K[i], 256, nullptr);
    if (a.err == nullptr) return FP8Q_ERR_CUDA;
    units += (int64_t)((a.num_m_tiles + 1) / 2) * a.num_n_tiles;
    if (units > INT32_MAX / 2) return FP8Q_ERR_INVALID_ARG;
    raster_for((a.num_m_tiles + 1) / 2, a.num_n_tiles, 256, 256, K[i], a.group, a.along_n);
    add_pair_problem(maps, grp, ta, tb, a);
  }
  if (log_enabled())
    fprintf(stderr, "[fp8q] launch gemm_tensor_pair_kernel grouped: %d GEMMs, %lld units 256x256\n",
            count, (long long)units);
  return run_tensor_pair_group(maps, grp, out_dtype == FP8Q_DT_BF16, stream);
}

}  // namespace fp8q
