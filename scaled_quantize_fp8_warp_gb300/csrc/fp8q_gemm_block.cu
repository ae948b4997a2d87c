// The tile/block-scaled FP8 GEMM (1x128 tiles on A; 128x128 blocks or 1x128
// tiles on B): each 128-wide K block is accumulated into a ping-pong TMEM
// buffer and promoted into fp32 registers with that block's scale product
// (the blocked sum of the definition; "fp8_parity.py", FP8Matmul, with the
// scales applied per K block).
#include "fp8q_gemm_common.cuh"

namespace fp8q {
namespace gemm {
namespace {

// Named (hardware) barriers, warp-granular: every thread of the calling warp
// executes the instruction; `count` is the number of threads that complete one
// generation.  bar.arrive does not wait; bar.sync waits for the generation.
__device__ __forceinline__ void nbar_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void nbar_arrive(uint32_t id, uint32_t count) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ------------------------------------------------------------------------
// Tile/block scaled GEMM.  Warpgroup 0 holds the producer (warp 0), the MMA
// issuer (warp 1), the scale warp (warp 2) and the relay (warp 3); NWG
// promotion warpgroups follow, warpgroup g owning tile columns [g C, g C + C)
// with C = BN / NWG.  A carries 1x128 tile scales; B carries 128x128 block
// scales (B_TILE = false) or 1x128 tile scales (B_TILE = true).  Each
// 128-wide K block is accumulated into one of two TMEM buffers of BN columns;
// the promotion warps load their C columns of it (64 per round trip), hand
// the buffer back, and add it into fp32 registers with the block's scale
// product.  The handoff runs on named (hardware) barriers: the relay waits
// for each K block's MMA commit and wakes the promotion warps, and they
// release the buffer to the MMA warp, so the promotion loop touches no
// shared-memory barrier on that path (each such operation measured a few
// hundred cycles while the MMAs stream operands through shared memory).
// Every role walks the same sequence of K blocks, also after an abort, so
// the named barriers always balance.  The scales
// reach them through a shared-memory ring that the scale warp fills with
// cp.async, kScaleGroup K blocks per slot and kScaleSlots slots ahead, so no
// global-load latency sits in the promotion loop and its slot handshake
// (two shared-memory barrier operations, each a few hundred cycles while the
// MMAs stream operands through shared memory) is paid once per group.
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
  static constexpr int kScaleGroup = 4;                  // K blocks of scales per ring slot
  static constexpr int kScaleSlots = 4;                  // ring slots
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
  constexpr int SS = Cfg::kScaleSlots;
  constexpr int KG = Cfg::kScaleGroup;
  constexpr int C = Cfg::kCols;
  constexpr int NPW = 4 * NWG;   // promotion warps
  using L = Layout<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  // Scale ring: per K block, the tile's 128 A scales and its B scales (BN
  // column scales, or one 128x128 block scale per promotion warpgroup),
  // copied in ahead of use by the scale warp.
  __shared__ __align__(16) float sh_sa[SS][KG][kBM];
  __shared__ __align__(16) float sh_sb[SS][KG][B_TILE ? BN : 4];
  __shared__ __align__(8) uint64_t sh_sbar[2 * SS];   // full, empty

  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t ring = (raw + 1023u) & ~1023u;
  const uint32_t bars = ring + L::kRingBytes;
  const uint32_t full0 = bars, empty0 = bars + 8 * STAGES;
  const uint32_t pf0 = bars + 8 * (2 * STAGES);   // MMA commits: buffer b complete
  const uint32_t drain = pf0 + 32;
  const uint32_t sfull0 = smem_u32(&sh_sbar[0]), sempty0 = sfull0 + 8 * SS;
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
    }
    for (int s = 0; s < SS; ++s) {
      mbar_init(sfull0 + 8 * s, 32);      // one cp.async arrival per lane of the scale warp
      mbar_init(sempty0 + 8 * s, NPW);
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
  // K blocks this CTA runs (every role walks the same sequence)
  const uint32_t my_tiles =
      (int)blockIdx.x < total ? (uint32_t)((total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1) : 0u;
  const uint32_t T = my_tiles * (uint32_t)nkb;
  // Named barriers of the MMA -> promotion handoff (id 0 is __syncthreads):
  //   FULL[b]  the relay arrives, the promotion warps wait: buffer b holds K block it
  //   RELM[b]  the promotion warps arrive, the MMA warp waits: buffer b may be reused
  //   ISS[b]   the MMA warp arrives, the relay waits: K block it has been issued
  constexpr uint32_t kBarFull = 1, kBarRelM = 3, kBarIss = 5;
  constexpr uint32_t kFullCount = 32u * (1u + NPW), kRelCount = 32u * (NPW + 1u), kIssCount = 64u;

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(Cfg::kLowRegs));
    if (warp == 0) {
      if (lane == 0) producer_loop<BN, STAGES>(&ta, &tb, p, ring, bars, abort_flag);
      __syncwarp();
    } else if (warp == 1) {
      // MMA issuer.  Before K block it + 2 may overwrite a partial-sum buffer
      // the promotion warps must have read K block it (RELM); after issuing
      // K block it it tells the relay warp (ISS).  A failed wait marks the
      // warp dead: it issues nothing more but keeps every barrier operation,
      // so the named barriers stay balanced and nothing waits forever.
      bool dead = false;
      for (uint32_t it = 0; it < T; ++it) {
        const uint32_t pb = it & 1u;
        if (it >= 2) {
          nbar_sync(kBarRelM + pb, kRelCount);
          tc_fence_after();
        }
        if (!dead) {
          int ok = 1;
          if (lane == 0) {
            const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
            ok = wait_bounded(full0 + 8 * s, ph, abort_flag, p.err) ? 1 : 0;
            if (ok) {
              tc_fence_after();
              issue_kblock<BN, STAGES>(ring, s, tmem_base + pb * BN, p.idesc, false);
              mma_commit(empty0 + 8 * s);
              mma_commit(pf0 + 8 * pb);
            }
          }
          dead = __shfl_sync(0xFFFFFFFFu, ok, 0) == 0;
        }
        __syncwarp();
        nbar_arrive(kBarIss + pb, kIssCount);
      }
      // the releases of the last two K blocks complete their generations
      for (uint32_t k = T >= 2 ? T - 2 : 0; k < T; ++k) nbar_sync(kBarRelM + (k & 1u), kRelCount);
      if (lane == 0) drain_mma(drain, abort_flag);
      __syncwarp();
    } else if (warp == 2) {
      // Scale warp: every lane copies its share of each K block's scales into
      // the ring with cp.async (rows / columns past the matrix are
      // zero-filled without a read), KG consecutive K blocks of the CTA's
      // sequence per slot, and arrives once its copies for the slot have
      // landed (or when its sequence ends inside a slot); the promotion warps
      // release a slot after the FMAs of its last K block.
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        int mt, nt;
        tile_coords(tile, p.num_m_tiles, p.num_n_tiles, mt, nt, kBlockGroupM, 0);
        const int64_t m0 = (int64_t)mt * kBM, n0 = (int64_t)nt * BN;
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const uint32_t grp = it / KG, ss = grp % SS, sph = (grp / SS) & 1u, j = it % KG;
          if (j == 0 && !wait_bounded_warp(sempty0 + 8 * ss, sph ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          const uint32_t da = smem_u32(&sh_sa[ss][j][0]), db = smem_u32(&sh_sb[ss][j][0]);
#pragma unroll
          for (int u = 0; u < kBM / 32; ++u) {
            const int r = lane + 32 * u;
            const bool v = m0 + r < p.M;
            const float *src = v ? p.scale_a + (kb * p.a_stride_k + (m0 + r) * p.a_stride_row)
                                 : p.scale_a;
            cp_async_4(da + 4 * r, src, v ? 4u : 0u);
          }
          if (B_TILE) {
#pragma unroll
            for (int u = 0; u < BN / 32; ++u) {
              const int c = lane + 32 * u;
              const bool v = n0 + c < p.N;
              const float *src = v ? p.scale_b + (kb * p.b_stride_k + (n0 + c) * p.b_stride_row)
                                   : p.scale_b;
              cp_async_4(db + 4 * c, src, v ? 4u : 0u);
            }
          } else if (lane < NWG) {
            // warpgroup `lane` covers columns [n0 + lane C, n0 + (lane + 1) C),
            // all inside one 128-column block
            const int64_t nc = n0 + lane * C;
            const bool v = nc < p.N;
            const float *src = v ? p.scale_b + ((nc / 128) * p.b_stride_row + kb * p.b_stride_k)
                                 : p.scale_b;
            cp_async_4(db + 4 * lane, src, v ? 4u : 0u);
          }
          if (j == KG - 1) cp_async_mbar_arrive(sfull0 + 8 * ss);
        }
      }
      if (ok && it % KG != 0) cp_async_mbar_arrive(sfull0 + 8 * ((it / KG) % SS));
      cp_async_wait_all();
    } else {
      // Relay (warp 3): once K block it is issued (ISS), wait for its MMAs to
      // complete and wake the promotion warps (FULL) with a named barrier, so
      // that they never poll a shared-memory barrier on this path.  After an
      // abort the wait returns at once and the arrivals continue.
      for (uint32_t it = 0; it < T; ++it) {
        const uint32_t pb = it & 1u;
        nbar_sync(kBarIss + pb, kIssCount);
        if (lane == 0) (void)wait_bounded(pf0 + 8 * pb, (it >> 1) & 1u, abort_flag, p.err);
        __syncwarp();
        nbar_arrive(kBarFull + pb, kFullCount);
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(Cfg::kHighRegs));
    const int pw = warp - 4;              // promotion warp 0 .. NPW-1
    const int wg = pw >> 2;
    const int quarter = warp & 3;         // TMEM lane quarter of this warp
    uint32_t it = 0, run_max = 0;
    // Look-ahead carried from one K block to the next: the next K block's A
    // scale when it sits in the same ring slot (read while this K block's FMAs
    // run; per-column B scales only).
    float sa_pre = 0.0f;
    bool have_pre = false;
    // Every tile and K block is walked even after an abort, so that the named
    // barriers stay balanced; nothing is stored then.
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      int mt, nt;
      tile_coords(tile, p.num_m_tiles, p.num_n_tiles, mt, nt, kBlockGroupM, 0);
      const int64_t m = (int64_t)mt * kBM + quarter * 32 + lane;
      const int64_t ncol0 = (int64_t)nt * BN + wg * C;   // first column of this warpgroup
      float2 acc2[C / 2];   // columns (2 j, 2 j + 1)
#pragma unroll
      for (int j = 0; j < C / 2; ++j) acc2[j] = make_float2(0.0f, 0.0f);
      for (int kb = 0; kb < nkb; ++kb, ++it) {
        const uint32_t grp = it / KG, ss = grp % SS, sph = (grp / SS) & 1u, j = it % KG;
        const uint32_t pb = it & 1u;
        nbar_sync(kBarFull + pb, kFullCount);   // buffer pb holds K block it
        if (j == 0) (void)wait_bounded_all(sfull0 + 8 * ss, sph, abort_flag, p.err);
        tc_fence_after();
        const float sa = have_pre ? sa_pre : sh_sa[ss][j][quarter * 32 + lane];
        const float sbk = B_TILE ? 0.0f : sh_sb[ss][j][wg];
        const float sab = B_TILE ? 0.0f : __fmul_rn(sa, sbk);
        const float2 sa2 = make_float2(sa, sa);
        const float *bs = &sh_sb[ss][j][B_TILE ? wg * C : 0];
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
            nbar_arrive(kBarRelM + pb, kRelCount);   // buffer pb may be overwritten
            if (B_TILE) {
              have_pre = j + 1 < (uint32_t)KG;
              if (have_pre) sa_pre = sh_sa[ss][j + 1][quarter * 32 + lane];
            }
          }
          // acc += P * scale.  With per-column B scales, two columns per
          // packed fmul2 / ffma2 (each lane rounds like the scalar
          // instruction): that path has a multiply per element on top of the
          // FMA, and its promotion is issue-bound.
          if (B_TILE) {
#pragma unroll
            for (int j = 0; j < 64; j += 4) {
              const float4 b4 = *reinterpret_cast<const float4 *>(&bs[h * 64 + j]);
              const float2 s01 = __fmul2_rn(sa2, make_float2(b4.x, b4.y));
              const float2 s23 = __fmul2_rn(sa2, make_float2(b4.z, b4.w));
              const uint32_t *rr = j < 32 ? &r0[j] : &r1[j - 32];
              acc2[h * 32 + j / 2] = __ffma2_rn(
                  make_float2(__uint_as_float(rr[0]), __uint_as_float(rr[1])), s01,
                  acc2[h * 32 + j / 2]);
              acc2[h * 32 + j / 2 + 1] = __ffma2_rn(
                  make_float2(__uint_as_float(rr[2]), __uint_as_float(rr[3])), s23,
                  acc2[h * 32 + j / 2 + 1]);
            }
          } else {
            // one scale for the whole row segment: scalar FFMAs (the packed
            // form spills here and measured slower)
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              acc2[h * 32 + j].x = __fmaf_rn(__uint_as_float(r0[2 * j]), sab, acc2[h * 32 + j].x);
              acc2[h * 32 + j].y =
                  __fmaf_rn(__uint_as_float(r0[2 * j + 1]), sab, acc2[h * 32 + j].y);
              acc2[h * 32 + 16 + j].x =
                  __fmaf_rn(__uint_as_float(r1[2 * j]), sab, acc2[h * 32 + 16 + j].x);
              acc2[h * 32 + 16 + j].y =
                  __fmaf_rn(__uint_as_float(r1[2 * j + 1]), sab, acc2[h * 32 + 16 + j].y);
            }
          }
        }
        // the slot's last K block has been read: hand the slot back
        if (j == KG - 1) {
          __syncwarp();
          if (lane == 0) mbar_arrive(sempty0 + 8 * ss);
        }
      }
      if (m < p.M && *abort_flag == 0) {
#pragma unroll
        for (int c = 0; c < C / 32; ++c) {
          const int64_t n0 = ncol0 + c * 32;
          if (n0 < p.N) {
            float v[32];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              v[2 * j] = acc2[c * 16 + j].x;
              v[2 * j + 1] = acc2[c * 16 + j].y;
            }
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

template <int BN, int NWG, bool B_TILE, bool OUT_BF16>
int run_blockscaled(const CUtensorMap &ta, const CUtensorMap &tb, const GemmArgs &a, int grid,
                    cudaStream_t stream) {
  using Cfg = BSConfig<BN, NWG>;
  using L = Layout<BN, Cfg::kStages>;
  auto kernel = gemm_blockscaled_kernel<BN, NWG, B_TILE, OUT_BF16>;
  static PerDeviceOnce setup;  // per instantiation
  const int ready = setup.get([&] {
    // The setmaxnreg split is only safe if the kernel launches with at least
    // kLaunchRegs registers per thread; refuse to launch otherwise.
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kernel) != cudaSuccess) return 0;
    if (fa.numRegs < Cfg::kLaunchRegs) return 0;
    return set_smem(kernel, L::kSmemBytes) == cudaSuccess ? 1 : 0;
  });
  if (ready != 1) return FP8Q_ERR_CUDA;
  kernel<<<grid, Cfg::kThreads, L::kSmemBytes, stream>>>(ta, tb, a);
  return cudaGetLastError() == cudaSuccess ? FP8Q_OK : FP8Q_ERR_CUDA;
}

}  // namespace

int run_blockscaled_family(const CUtensorMap &ta, const CUtensorMap &tb, const GemmArgs &a,
                           int grid, bool bf16, bool b_tile, cudaStream_t stream) {
  constexpr int BBN = kBlockScaledBN, BWG = kBlockScaledWG;
  if (b_tile)
    return bf16 ? run_blockscaled<BBN, BWG, true, true>(ta, tb, a, grid, stream)
                : run_blockscaled<BBN, BWG, true, false>(ta, tb, a, grid, stream);
  return bf16 ? run_blockscaled<BBN, BWG, false, true>(ta, tb, a, grid, stream)
              : run_blockscaled<BBN, BWG, false, false>(ta, tb, a, grid, stream);
}

}  // namespace gemm
}  // namespace fp8q
