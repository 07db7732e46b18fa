// Two-SM (CTA-pair) block-scaled NVFP4 GEMM, sm_103a.
//
// A cluster of two CTAs computes one 256 x 256 output tile with
// tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X (K = 64
// per instruction).  Per 128-byte K slice (256 E2M1 elements) each CTA
// stages its 128 rows of A, its 128 rows of B, the 4 scale tiles of its A
// rows (2 KB, one TMA box) and the 4 scale tiles of each of the two
// 128-row blocks of B (2 x 2 KB): the B scales of all 256 columns, because
// each CTA's tensor core produces its 128 rows for every column.  The leader
// copies the stage's scale tiles into per-stage TMEM columns of both CTAs
// (tcgen05.cp.cta_group::2) ahead of the MMAs that read them.
//
// TMEM per CTA: one 256-column fp32 accumulator plus STAGES x 48 scale
// columns.  With no room for a second accumulator, eight epilogue warps drain
// it into registers and release it before doing the epilogue math and the
// stores (epilogue_loop_regdrain), so the next tile's MMAs start at once.
#pragma once

#include "gemm_epilogue.cuh"
#include "gemm_kernel_common.cuh"

namespace spg {

template <int EPI, int STAGES, bool HAS_BIAS = false>
struct Nvfp4PairCfg {
  static constexpr int kBN = 256;
  static constexpr int kBKBytes = 128;  // 256 E2M1 elements
  static constexpr int kKSteps = 4;     // MMAs per stage (K = 64 each)
  static constexpr int kABytes = 128 * kBKBytes;
  static constexpr int kBBytes = 128 * kBKBytes;
  static constexpr int kSfaBytes = 4 * 512;
  static constexpr int kSfbBytes = 2 * 4 * 512;
  static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
  static constexpr int kSfColsPerKStep = 4 + 8;  // A scales, then B scales (two 128-row tiles)
  static constexpr int kSfColsPerStage = kKSteps * kSfColsPerKStep;
  static constexpr int kTmemUsed = kBN + STAGES * kSfColsPerStage;
  static constexpr int kTmemCols = 512;
  static constexpr int kEpiWarps = 8;
  static constexpr int kEpiBytes = kEpiWarps * 2 * 32 * 64;
  static constexpr int kBarBytes = 512;
  static constexpr int kSmemBytes = 1024 + STAGES * kStageBytes + kEpiBytes + kBarBytes;
  static constexpr int kThreads = 64 + 32 * kEpiWarps;

  static_assert(kTmemUsed <= kTmemCols, "TMEM budget exceeded");
  static_assert(kStageBytes % 1024 == 0, "stage bases must stay 1024-byte aligned");
  static_assert(kSmemBytes <= 232448, "shared memory budget exceeded");
  // barriers, tmem slot + abort flag, stall barrier, PairExit
  static_assert((2 * STAGES + 5) * 8 + sizeof(PairExit) <= kBarBytes, "barrier area too small");

  // Block-scaled descriptor: A, B = E2M1 (1), UE4M3 scales, M = 256, N = 256, K = 64.
  __host__ __device__ static constexpr uint32_t idesc() {
    return (1u << 7) | (1u << 10) | (uint32_t(kBN >> 3) << 17) | (uint32_t(256 >> 4) << 24);
  }
};

template <int EPI, int STAGES, bool HAS_BIAS>
// 10 warps: the 4 SM sub-partitions hold 3, 3, 2, 2 of them, so a thread may
// use at most 16384 / (3 * 32) -> 168 registers.
__global__ void __launch_bounds__(Nvfp4PairCfg<EPI, STAGES>::kThreads, 1)
    gemm_kernel_nvfp4_2sm(const __grid_constant__ CUtensorMap tmA,
                          const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ CUtensorMap tmY,
                          const __grid_constant__ CUtensorMap tmSFA,
                          const __grid_constant__ CUtensorMap tmSFB, const GemmParams p) {
  using Cfg = Nvfp4PairCfg<EPI, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint8_t* epi = smem + STAGES * Cfg::kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(epi + Cfg::kEpiBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* acc_full = bars + 2 * STAGES;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* drain = acc_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  uint64_t* stall = drain + 2;  // test hook: nothing arrives on it
  PairExit* pexit = reinterpret_cast<PairExit*>(stall + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int pair = blockIdx.x >> 1;
  const int num_pairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 2 * Cfg::kEpiWarps);
    mbar_init(drain, 1);
    mbar_init(stall, 1);
    mbar_init(&pexit->bar, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmY);
    prefetch_tmap(&tmSFA);
    prefetch_tmap(&tmSFB);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, Cfg::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtl ctl{p.timeout_ns, p.err, abort_flag};

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      uint32_t issued = 0;
      uint32_t tx[STAGES] = {};  // this CTA's copy bytes per ring slot (last use)
      bool ok = true;
      const int64_t tpr = p.sf_tiles_per_row_block;
      const int a_row_blocks = (p.M + 127) / 128;
      const int b_row_blocks = (p.N + 127) / 128;
      for (int item = pair; ok && item < p.total_items; item += num_pairs) {
        const WorkItem tc = work_item(item, p, Cfg::kBN);
        const int a_rb = tc.mb * 2 + int(rank);
        const int m0 = a_rb * 128;
        const int n0 = tc.nb * 256 + int(rank) * 128;
        // Scale tiles of row blocks past the operand are never multiplied by
        // a non-zero code (TMA zero-fills those rows): read the last real
        // block instead of running past the buffer.
        const int a_rb_sf = a_rb < a_row_blocks ? a_rb : a_row_blocks - 1;
        const int b_rb0 = tc.nb * 2 < b_row_blocks ? tc.nb * 2 : b_row_blocks - 1;
        const int b_rb1 = tc.nb * 2 + 1 < b_row_blocks ? tc.nb * 2 + 1 : b_row_blocks - 1;
        for (int kb = tc.kb_begin; kb < tc.kb_end; ++kb) {
          if (!mbar_wait(&empty[s], ph ^ 1u, ctl, kErrWaitEmpty)) {
            ok = false;
            break;
          }
          uint8_t* sa = ring + s * Cfg::kStageBytes;
          uint8_t* sb = sa + Cfg::kABytes;
          uint8_t* ssfa = sb + Cfg::kBBytes;
          uint8_t* ssfb = ssfa + Cfg::kSfaBytes;
          if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * Cfg::kStageBytes);
          const uint32_t bar = mapa_shared(smem_u32(&full[s]), 0);
          const int kx = kb * Cfg::kBKBytes;
          tma_load_3d_pair(sa, &tmA, bar, kx, m0, 0);
          tma_load_3d_pair(sb, &tmB, bar, kx, n0, 0);
          // Scale tiles: 4 consecutive 512-byte tiles (one row of 128 uint32
          // per tile in the 2-D view) = one 2 KB TMA box per 128-row block.
          const int k_tile = kb * 4;
          tma_load_3d_pair(ssfa, &tmSFA, bar, 0, a_rb_sf * int(tpr) + k_tile, 0);
          tma_load_3d_pair(ssfb, &tmSFB, bar, 0, b_rb0 * int(tpr) + k_tile, 0);
          tma_load_3d_pair(ssfb + 2048, &tmSFB, bar, 0, b_rb1 * int(tpr) + k_tile, 0);
          tx[s] = Cfg::kStageBytes;
          ++issued;
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      // Both CTAs' copies complete on the leader's barriers: settle the two
      // producers' accounts, then wait for the last stages.
      if (rank == 0)
        pair_exit_drain<STAGES>(pexit, full, issued, tx, p);
      else
        pair_exit_publish<STAGES>(pexit, issued, tx);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------- MMA issuer (leader)
    if (lane == 0 && rank == 0) {
      constexpr uint32_t kIdesc = Cfg::idesc();
      int s = 0;
      uint32_t ph = 0;
      int it = 0;
      bool ok = true;
      for (int item = pair; ok && item < p.total_items; item += num_pairs, ++it) {
        const WorkItem w = work_item(item, p, Cfg::kBN);
        // The peer CTA's epilogue warps release this barrier across the pair.
        if (!mbar_wait_cluster(acc_empty, (it & 1) ^ 1u, ctl, kErrWaitAccEmpty)) break;
        tc_fence_after();
        for (int kb = w.kb_begin; kb < w.kb_end; ++kb) {
          if (!mbar_wait(&full[s], ph, ctl, kErrWaitFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(ring + s * Cfg::kStageBytes);
          const uint32_t sb = sa + Cfg::kABytes;
          const uint32_t ssfa = sb + Cfg::kBBytes;
          const uint32_t ssfb = ssfa + Cfg::kSfaBytes;
          const uint32_t sf_col0 = tmem_base + uint32_t(Cfg::kBN + s * Cfg::kSfColsPerStage);
#pragma unroll
          for (int j = 0; j < Cfg::kKSteps; ++j) {
            const uint32_t col = sf_col0 + uint32_t(j * Cfg::kSfColsPerKStep);
            tc_cp_32x128b_warpx4_pair(col, smem_desc(ssfa + j * 512, 0, 128, kSwizzleNone));
            tc_cp_32x128b_warpx4_pair(col + 4, smem_desc(ssfb + j * 512, 0, 128, kSwizzleNone));
            tc_cp_32x128b_warpx4_pair(col + 8,
                                      smem_desc(ssfb + 2048 + j * 512, 0, 128, kSwizzleNone));
          }
#pragma unroll
          for (int j = 0; j < Cfg::kKSteps; ++j) {
            const uint32_t col = sf_col0 + uint32_t(j * Cfg::kSfColsPerKStep);
            mma_nvf4_pair(tmem_base, smem_desc(sa + j * 32, 16, 1024, kSwizzle128B),
                          smem_desc(sb + j * 32, 16, 1024, kSwizzle128B), kIdesc, col, col + 4,
                          (kb != w.kb_begin) || j != 0);
          }
          tc_commit_pair_multicast(&empty[s], 0x3);
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_pair_multicast(acc_full, 0x3);
      }
      tc_commit_pair(drain);
      mbar_wait_drain(drain, 0, p.drain_ns, p.err);
    }
  } else if (p.debug_stall && !mbar_wait(stall, 0, ctl, kErrInjectedStall)) {
    // Test hook: the epilogue waited on a barrier nothing arrives on; the CTA
    // has aborted and its other roles drain and return.
  } else {
    // -------------------------------------------------------------- epilogue
    epilogue_loop_regdrain<EPI, kScaleScalar, HAS_BIAS>(
        p, &tmY, tmem_base, acc_full,
        [&](int) { mbar_arrive_cluster(mapa_shared(smem_u32(acc_empty), 0)); }, epi, pair,
        num_pairs,
        [&](int item) {
          WorkItem w = work_item(item, p, Cfg::kBN);
          w.mb = w.mb * 2 + int(rank);
          return w;
        },
        ctl, int(rank));
  }

  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
}

}  // namespace spg
