// Steps a4-a5 of the path: the FP8 GEMM C = A . B^T with dequantising scales
// ("fp8_parity.py", FP8Matmul: xq @ wq.T; the blog repost's Fprop / Dgrad /
// Wgrad shapes), on the 5th-generation tensor cores.
//
// Three persistent, warp-specialised kernels (static round-robin over output
// tiles, grouped along M for L2 reuse):
//   gemm_tensor_pair_kernel  per-tensor / row scales at N > 128: a CTA pair
//            (cta_group::2) computes 256 x 256 tiles, each CTA staging its own
//            128 rows of A and of B;
//   gemm_tensor_kernel       per-tensor / row scales at N <= 128, one SM per
//            128 x BN tile (BN = 64 or 128);
//   gemm_blockscaled_kernel  1x128 / 128x128 scales, one SM per 128 x 256 tile.
// Roles: warp 0 is the TMA producer (128-byte swizzled boxes into a
// shared-memory ring with full/empty mbarriers); warp 1 allocates TMEM and
// issues tcgen05.mma.kind::f8f6f4 (K = 32 per instruction, four per 128-byte
// K block) from one thread, with tcgen05.commit releasing ring slots and
// handing accumulators on; the remaining warps drain TMEM (tcgen05.ld),
// scale, convert and store.  Every TMA load fetches into the issuing CTA's
// own shared memory.
// Per-tensor scaling accumulates the whole K range in TMEM (two accumulator
// buffers so one tile's epilogue overlaps the next tile's MMAs) and applies
// s_A s_B once.  Tile/block scaling accumulates each 128-wide K block into a
// ping-pong TMEM buffer; the promotion warps add it into fp32 registers with
// that block's s_A(m, kb) s_B(n, kb) (the blocked sum of the definition).
//
// Every mbarrier wait is bounded (about two seconds of wall time); on expiry
// the kernel records FP8Q_ERR_TIMEOUT in the device error word, drains what
// it issued, frees its TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <mutex>

#include "fp8q_internal.h"
#include "fp8q_ptx.cuh"

namespace fp8q {
namespace {

using namespace ptx;

constexpr int kBM = 128;
constexpr int kBK = 128;            // bytes = FP8 elements per K block
constexpr int kUmmaK = 32;          // K per tcgen05.mma for 8-bit inputs
constexpr int kGroupM = 16;         // M-tiles per raster group
// Tile width and promotion warpgroups of the tile/block-scaled kernel.
#ifndef FP8Q_BLOCK_BN
#define FP8Q_BLOCK_BN 256
#define FP8Q_BLOCK_WG 2
#endif
// Per-tensor / row scaling at N > 128 runs on CTA pairs (cta_group::2) with
// kPairAcc TMEM accumulators of 256 columns each and a ring of kPairStages
// 32 KB stages per CTA.
constexpr int kPairAcc = 2;
constexpr int kPairStages = 6;
constexpr int kBlockScaledBN = FP8Q_BLOCK_BN;
constexpr int kBlockScaledWG = FP8Q_BLOCK_WG;

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
  unsigned int *amax;  // max |C| over the stored values (fp32 bit pattern), or null
  unsigned int *err;
  // MXFP8: E8M0 scale atoms, 512 bytes per 128 rows x 128 K, atom (rb, kb) at
  // byte (rb * num_k_blocks + kb) * 512
  const uint8_t *mx_a;
  const uint8_t *mx_b;
};

__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int &mt, int &nt,
                                            int group_m = kGroupM) {
  const int per_group = group_m * num_n;
  const int g = tile / per_group;
  const int first_m = g * group_m;
  const int gsize = min(num_m - first_m, group_m);
  const int local = tile - g * per_group;
  mt = first_m + local % gsize;
  nt = local / gsize;
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
    tile_coords(u, p.num_m_tiles, p.num_n_tiles, mt, nt);
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
// column n0; columns >= N are skipped in groups of 8 (N % 16 == 0).  Returns
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
        *reinterpret_cast<uint4 *>(row + n0 + 8 * g) = make_uint4(w[0], w[1], w[2], w[3]);
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
        *reinterpret_cast<float4 *>(row + n0 + 4 * g) =
            make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
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
      tile_coords(u, p.num_m_tiles, p.num_n_tiles, mt, nt);
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
template <int STAGES>
struct PairLayout {
  static constexpr int kABytes = kBM * kBK;        // this CTA's 128 rows of A
  static constexpr int kBBytes = 128 * kBK;        // this CTA's 128 rows of B
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kRingBytes = STAGES * kStageBytes;
  static constexpr int kBarBytes = 8 * (2 * STAGES + 5);
  static constexpr int kSmemBytes = kRingBytes + kBarBytes + 16 + 1024;
};

template <int STAGES, int ACC, bool OUT_BF16, bool VEC>
__global__ void __launch_bounds__(192, 1)
    gemm_tensor_pair_kernel(const __grid_constant__ CUtensorMap ta,
                            const __grid_constant__ CUtensorMap tb, const GemmArgs p) {
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
    prefetch_tmap(&ta);
    prefetch_tmap(&tb);
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
  if (!paired && threadIdx.x == 0) atomicOr(p.err, 4u);

  const int num_mu = (p.num_m_tiles + 1) / 2;
  const int total = num_mu * p.num_n_tiles;
  const int unit0 = blockIdx.x / 2, unit_step = gridDim.x / 2;

  if (!paired) {
  } else if (warp == 0) {
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int u = unit0; u < total && ok; u += unit_step) {
        int mu, nt;
        tile_coords(u, num_mu, p.num_n_tiles, mu, nt, kGroupM / 2);
        // past the last M tile (odd count): re-read that tile's A, store nothing
        const int mt = min(2 * mu + (int)rank, p.num_m_tiles - 1);
        for (int kb = 0; kb < p.num_k_blocks; ++kb, ++it) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
          if (!wait_bounded(empty0 + 8 * s, ph ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          const uint32_t sa = ring + s * L::kStageBytes;
          const uint32_t full_even = mapa_shared(full0 + 8 * s, 0);
          if (rank == 0) mbar_arrive_expect_tx(full0 + 8 * s, 2 * L::kStageBytes);
          tma_load_2d_pair(sa, &ta, kb * kBK, mt * kBM, full_even);
          tma_load_2d_pair(sa + L::kABytes, &tb, kb * kBK, nt * BN + (int)rank * 128, full_even);
        }
      }
      // every slot's last release (the even CTA's commits) has arrived here
      for (uint32_t j = 0, jt = it; ok && j < (uint32_t)STAGES; ++j, ++jt)
        ok = wait_bounded(empty0 + 8 * (jt % STAGES), ((jt / STAGES) & 1u) ^ 1u, abort_flag,
                          p.err);
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
          const uint32_t a0 = ring + s * L::kStageBytes, b0 = a0 + L::kABytes;
#pragma unroll
          for (int k = 0; k < kBK / kUmmaK; ++k) {
            const uint64_t ad = sdesc_k(a0 + k * kUmmaK, kSwzSBO, kSwzMode);
            const uint64_t bd = sdesc_k(b0 + k * kUmmaK, kSwzSBO, kSwzMode);
            mma_f8f6f4_pair(d_tmem, ad, bd, p.idesc, (kb > 0 || k > 0) ? 1u : 0u);
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
    const float scale = VEC ? 0.0f : __fmul_rn(p.scale_a[0], p.scale_b[0]);
    const uint32_t acce_even0 = mapa_shared(acce0, 0);
    uint32_t acc_it = 0, run_max = 0;
    for (int u = unit0; u < total; u += unit_step, ++acc_it) {
      int mu, nt;
      tile_coords(u, num_mu, p.num_n_tiles, mu, nt, kGroupM / 2);
      const int mt = 2 * mu + (int)rank;   // >= num_m_tiles: nothing to store
      const uint32_t buf = ACC == 2 ? (acc_it & 1u) : 0u;
      const uint32_t aph = ACC == 2 ? ((acc_it >> 1) & 1u) : (acc_it & 1u);
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
      if (lane == 0) {
        if (rank == 0)
          mbar_arrive(acce0 + 8 * buf);
        else
          mbar_arrive_cluster(acce_even0 + 8 * buf);
      }
    }
    publish_amax(p.amax, run_max);
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // neither CTA leaves while the other may still signal it
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, kTmemCols);
}

// ------------------------------------------------------------------------
// Tile/block scaled GEMM.  Warpgroup 0 holds the producer (warp 0) and the MMA
// issuer (warp 1); NWG promotion warpgroups follow, warpgroup g owning tile
// columns [g C, g C + C) with C = BN / NWG.  A carries 1x128 tile scales; B
// carries 128x128 block scales (B_TILE = false) or 1x128 tile scales
// (B_TILE = true).  Each 128-wide K block is accumulated into one of two
// TMEM buffers of BN columns; the promotion warps load their C columns of it
// (64 per round trip), hand the buffer back, and add it into fp32 registers
// with the block's scale product.
//
// Register split (setmaxnreg inside each role's branch): the launch of
// 128 (1 + NWG) threads gets kLaunchRegs per thread; warpgroup 0 drops to
// kLowRegs and the promotion warpgroups rise to kHighRegs, with
// 128 kLowRegs + 128 NWG kHighRegs <= 128 (1 + NWG) kLaunchRegs.  The host
// checks the compiled launch count before the first launch.
// ------------------------------------------------------------------------
template <int BN, int NWG>
struct BSConfig {
  static constexpr int kThreads = 128 * (1 + NWG);
  static constexpr int kCols = BN / NWG;                 // columns per promotion warpgroup
  static constexpr int kStages = BN <= 192 ? 5 : 4;
  static constexpr int kLaunchRegs = (65536 / kThreads) / 8 * 8;
  static constexpr int kLowRegs = NWG == 2 ? 40 : 56;
  static constexpr int kHighRegs = ((65536 - 128 * kLowRegs) / (128 * NWG)) / 8 * 8 > 232
                                       ? 232
                                       : ((65536 - 128 * kLowRegs) / (128 * NWG)) / 8 * 8;
  static constexpr uint32_t kTmemCols = 512;              // two BN-column buffers fit
  static_assert(BN % NWG == 0 && (kCols == 64 || kCols == 128), "64 or 128 columns per WG");
  static_assert(2 * BN <= 512, "two partial-sum buffers must fit in TMEM");
  static_assert(128 * kLowRegs + 128 * NWG * kHighRegs <= kThreads * kLaunchRegs,
                "register split exceeds the launch allocation");
};

template <int BN, int NWG, bool B_TILE, bool OUT_BF16>
__global__ void __launch_bounds__(BSConfig<BN, NWG>::kThreads, 1)
    gemm_blockscaled_kernel(const __grid_constant__ CUtensorMap ta,
                            const __grid_constant__ CUtensorMap tb, const GemmArgs p) {
  using Cfg = BSConfig<BN, NWG>;
  constexpr int STAGES = Cfg::kStages;
  constexpr int C = Cfg::kCols;
  constexpr int NPW = 4 * NWG;   // promotion warps
  using L = Layout<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(16) float sh_bscale[NPW][C];  // per promotion warp: B tile scales

  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t ring = (raw + 1023u) & ~1023u;
  const uint32_t bars = ring + L::kRingBytes;
  const uint32_t full0 = bars, empty0 = bars + 8 * STAGES;
  const uint32_t pf0 = bars + 8 * (2 * STAGES), pe0 = pf0 + 16;
  const uint32_t drain = pe0 + 16;
  const uint32_t slot = bars + L::kBarBytes;
  uint8_t *slot_ptr = smem_raw + (slot - raw);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(slot_ptr + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(pf0 + 8 * b, 1);
      mbar_init(pe0 + 8 * b, NPW);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
    prefetch_tmap(&ta);
    prefetch_tmap(&tb);
  }
  if (warp == 1) {
    tmem_alloc(slot, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(slot_ptr);
  const int total = p.num_m_tiles * p.num_n_tiles;
  const int nkb = p.num_k_blocks;

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(Cfg::kLowRegs));
    if (warp == 0) {
      if (lane == 0) producer_loop<BN, STAGES>(&ta, &tb, p, ring, bars, abort_flag);
      __syncwarp();
    } else if (warp == 1) {
      if (lane == 0) {
        uint32_t it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
          for (int kb = 0; kb < nkb; ++kb, ++it) {
            const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
            const uint32_t pb = it & 1u, pph = (it >> 1) & 1u;
            if (!wait_bounded(pe0 + 8 * pb, pph ^ 1u, abort_flag, p.err) ||
                !wait_bounded(full0 + 8 * s, ph, abort_flag, p.err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_kblock<BN, STAGES>(ring, s, tmem_base + pb * BN, p.idesc, false);
            mma_commit(empty0 + 8 * s);
            mma_commit(pf0 + 8 * pb);
          }
        }
        drain_mma(drain, abort_flag);
      }
      __syncwarp();
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(Cfg::kHighRegs));
    const int pw = warp - 4;              // promotion warp 0 .. NPW-1
    const int wg = pw >> 2;
    const int quarter = warp & 3;         // TMEM lane quarter of this warp
    float *my_bs = sh_bscale[pw];
    constexpr int kPerLane = C / 32;      // B tile scales each lane stages (2 or 4)
    uint32_t it = 0, run_max = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
      int mt, nt;
      tile_coords(tile, p.num_m_tiles, p.num_n_tiles, mt, nt);
      const int64_t m = (int64_t)mt * kBM + quarter * 32 + lane;
      const bool m_ok = m < p.M;
      const int64_t ncol0 = (int64_t)nt * BN + wg * C;   // first column of this warpgroup
      const int64_t nl = ncol0 + lane * kPerLane;         // this lane's B-scale columns
      auto load_sa = [&](int kb) -> float {
        return m_ok ? p.scale_a[kb * p.a_stride_k + m * p.a_stride_row] : 0.0f;
      };
      // Block scales: a warpgroup's C columns may straddle two 128-column
      // blocks when C = 64 only if ncol0 % 128 == 64; both halves of a
      // 64-column group lie in one block, so one scale serves the group.
      auto load_sb = [&](int kb) -> float {
        return ncol0 < p.N ? p.scale_b[(ncol0 / 128) * p.b_stride_row + kb * p.b_stride_k] : 0.0f;
      };
      float acc[C];
#pragma unroll
      for (int j = 0; j < C; ++j) acc[j] = 0.0f;
      float sa_next = load_sa(0);
      float sb_next = B_TILE ? 0.0f : load_sb(0);
      float sbt_next[kPerLane];
      if (B_TILE) {
#pragma unroll
        for (int u = 0; u < kPerLane; ++u)
          sbt_next[u] = (nl + u < p.N) ? p.scale_b[(nl + u) * p.b_stride_row] : 0.0f;
      }
      for (int kb = 0; kb < nkb; ++kb, ++it) {
        const float sa = sa_next;
        const float sb = sb_next;
        if (B_TILE) {
          __syncwarp();
#pragma unroll
          for (int u = 0; u < kPerLane; ++u) my_bs[lane * kPerLane + u] = sbt_next[u];
          __syncwarp();
        }
        if (kb + 1 < nkb) {
          sa_next = load_sa(kb + 1);
          if (B_TILE) {
#pragma unroll
            for (int u = 0; u < kPerLane; ++u)
              sbt_next[u] = (nl + u < p.N)
                                ? p.scale_b[(kb + 1) * p.b_stride_k + (nl + u) * p.b_stride_row]
                                : 0.0f;
          } else {
            sb_next = load_sb(kb + 1);
          }
        }
        const uint32_t pb = it & 1u, pph = (it >> 1) & 1u;
        if (!wait_bounded_warp(pf0 + 8 * pb, pph, abort_flag, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float sab = __fmul_rn(sa, sb);
#pragma unroll
        for (int h = 0; h < C / 64; ++h) {
          // 64 columns per round trip: two 32-column TMEM loads, one wait
          uint32_t r0[32], r1[32];
          const uint32_t col = pb * BN + wg * C + h * 64;
          const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
          tmem_ld_32x32b_x32(tmem_base + lane_base + col, r0);
          tmem_ld_32x32b_x32(tmem_base + lane_base + col + 32, r1);
          tmem_ld_wait();
          if (h == C / 64 - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(pe0 + 8 * pb);
          }
          if (B_TILE) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              acc[h * 64 + j] = __fmaf_rn(__uint_as_float(r0[j]),
                                          __fmul_rn(sa, my_bs[h * 64 + j]), acc[h * 64 + j]);
              acc[h * 64 + 32 + j] =
                  __fmaf_rn(__uint_as_float(r1[j]), __fmul_rn(sa, my_bs[h * 64 + 32 + j]),
                            acc[h * 64 + 32 + j]);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              acc[h * 64 + j] = __fmaf_rn(__uint_as_float(r0[j]), sab, acc[h * 64 + j]);
              acc[h * 64 + 32 + j] = __fmaf_rn(__uint_as_float(r1[j]), sab, acc[h * 64 + 32 + j]);
            }
          }
        }
      }
      if (!ok) break;
      if (m_ok) {
#pragma unroll
        for (int c = 0; c < C / 32; ++c) {
          const int64_t n0 = ncol0 + c * 32;
          if (n0 < p.N) {
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = acc[c * 32 + j];
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
  if (warp == 1) tmem_dealloc(tmem_base, Cfg::kTmemCols);
}

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
constexpr int kMxBN = 256;
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
        tile_coords(u, p.num_m_tiles, p.num_n_tiles, mt, nt);
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
      tile_coords(u, p.num_m_tiles, p.num_n_tiles, mt, nt);
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

// ------------------------------------------------------------------ host

// Row-major [rows, K] byte matrix, box = 128 bytes of K x box_rows, 128-byte
// swizzle, out-of-bounds elements read as zero.
bool make_tmap(CUtensorMap *m, const void *base, uint64_t rows, uint64_t K, uint32_t box_rows) {
  return make_tmap_2d(m, base, CU_TENSOR_MAP_DATA_TYPE_UINT8, K, rows, K, kBK, box_rows,
                      CU_TENSOR_MAP_SWIZZLE_128B);
}

template <typename KernelT>
cudaError_t set_smem(KernelT kernel, int bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <int STAGES, int ACC, bool OUT_BF16, bool VEC>
int run_tensor_pair(const CUtensorMap &ta, const CUtensorMap &tb, const GemmArgs &a,
                    cudaStream_t stream) {
  using L = PairLayout<STAGES>;
  auto kernel = gemm_tensor_pair_kernel<STAGES, ACC, OUT_BF16, VEC>;
  static bool attr_done = false;  // per instantiation
  static int max_clusters = 0;
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
  if (!attr_done) {
    if (set_smem(kernel, L::kSmemBytes) != cudaSuccess) return FP8Q_ERR_CUDA;
    cfg.gridDim = dim3(2 * (sm_count() / 2), 1, 1);
    if (cudaOccupancyMaxActiveClusters(&max_clusters, kernel, &cfg) != cudaSuccess ||
        max_clusters < 1)
      return FP8Q_ERR_CUDA;
    attr_done = true;
  }
  GemmArgs pa = a;
  pa.idesc = ptx::idesc_f8f6f4((a.idesc >> 7) & 7u, (a.idesc >> 10) & 7u, 256, 256);
  const int units = ((a.num_m_tiles + 1) / 2) * a.num_n_tiles;
  cfg.gridDim = dim3(2 * (units < max_clusters ? units : max_clusters), 1, 1);
  if (cudaLaunchKernelEx(&cfg, kernel, ta, tb, pa) != cudaSuccess) return FP8Q_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? FP8Q_OK : FP8Q_ERR_CUDA;
}

template <int BN, int STAGES, bool OUT_BF16, bool VEC>
int run_tensor(const CUtensorMap &ta, const CUtensorMap &tb, const GemmArgs &a, int grid,
               cudaStream_t stream) {
  using L = Layout<BN, STAGES>;
  auto kernel = gemm_tensor_kernel<BN, STAGES, OUT_BF16, VEC>;
  static bool attr_done = false;  // per instantiation
  if (!attr_done) {
    if (set_smem(kernel, L::kSmemBytes) != cudaSuccess) return FP8Q_ERR_CUDA;
    attr_done = true;
  }
  kernel<<<grid, 192, L::kSmemBytes, stream>>>(ta, tb, a);
  return cudaGetLastError() == cudaSuccess ? FP8Q_OK : FP8Q_ERR_CUDA;
}

template <bool OUT_BF16>
int run_mx(const CUtensorMap &ta, const CUtensorMap &tb, const GemmArgs &a, int grid,
           cudaStream_t stream) {
  auto kernel = gemm_mx_kernel<OUT_BF16>;
  static bool attr_done = false;
  if (!attr_done) {
    if (set_smem(kernel, MxLayout::kSmemBytes) != cudaSuccess) return FP8Q_ERR_CUDA;
    attr_done = true;
  }
  kernel<<<grid, 320, MxLayout::kSmemBytes, stream>>>(ta, tb, a);
  return cudaGetLastError() == cudaSuccess ? FP8Q_OK : FP8Q_ERR_CUDA;
}

template <int BN, int NWG, bool B_TILE, bool OUT_BF16>
int run_blockscaled(const CUtensorMap &ta, const CUtensorMap &tb, const GemmArgs &a, int grid,
                    cudaStream_t stream) {
  using Cfg = BSConfig<BN, NWG>;
  using L = Layout<BN, Cfg::kStages>;
  auto kernel = gemm_blockscaled_kernel<BN, NWG, B_TILE, OUT_BF16>;
  static bool attr_done = false;
  if (!attr_done) {
    // The setmaxnreg split is only safe if the kernel launches with at least
    // kLaunchRegs registers per thread; refuse to launch otherwise.
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kernel) != cudaSuccess) return FP8Q_ERR_CUDA;
    if (fa.numRegs < Cfg::kLaunchRegs) return FP8Q_ERR_CUDA;
    if (set_smem(kernel, L::kSmemBytes) != cudaSuccess) return FP8Q_ERR_CUDA;
    attr_done = true;
  }
  kernel<<<grid, Cfg::kThreads, L::kSmemBytes, stream>>>(ta, tb, a);
  return cudaGetLastError() == cudaSuccess ? FP8Q_OK : FP8Q_ERR_CUDA;
}

}  // namespace

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

  GemmArgs a{};
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
  if (a.err == nullptr) return FP8Q_ERR_CUDA;
  const int64_t tiles = (int64_t)a.num_m_tiles * a.num_n_tiles;
  if (tiles > INT32_MAX / 2) return FP8Q_ERR_INVALID_ARG;
  int grid = sm_count();
  if (tiles < grid) grid = (int)tiles;

  if (tensor) {
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
  if (mx) {
    a.idesc = ptx::idesc_mxf8f6f4((uint32_t)A.format, (uint32_t)B.format, kBM, kMxBN, 0, 0);
    return bf16 ? run_mx<true>(ta, tb, a, grid, stream) : run_mx<false>(ta, tb, a, grid, stream);
  }
  const bool b_tile = B.scaling == FP8Q_SCALE_TILE_1x128;
  constexpr int BBN = kBlockScaledBN, BWG = kBlockScaledWG;
  if (b_tile)
    return bf16 ? run_blockscaled<BBN, BWG, true, true>(ta, tb, a, grid, stream)
                : run_blockscaled<BBN, BWG, true, false>(ta, tb, a, grid, stream);
  return bf16 ? run_blockscaled<BBN, BWG, false, true>(ta, tb, a, grid, stream)
              : run_blockscaled<BBN, BWG, false, false>(ta, tb, a, grid, stream);
}

}  // namespace fp8q
