// Block-scaled NVFP4 GEMM on CTA clusters of two that share the weight tile
// by TMA multicast, each CTA running its own one-CTA MMAs, sm_103a.
//
// A cluster computes one 256 x 256 output tile, like the pair kernels: CTA r
// owns rows 128r .. 128r + 127.  Unlike them, each CTA issues its own
// tcgen05.mma.cta_group::1 (M = 128, N = 256, one per 64-element k-step)
// into its own TMEM, so every operand and every scale an MMA reads
// lives in its own CTA.  The 256 weight rows of a stage are fetched once
// from L2: CTA r loads rows 128r .. 128r + 127 of B and their scale tiles
// with a multicast copy that lands in both CTAs' shared memory.
//
// Why: in the pair kernels the peer CTA's scale factors reach TMEM either
// through 12 tcgen05.cp per stage, which occupy the tensor pipe about 35-45
// cycles each next to 4 MMAs of 128 cycles (measured on GB300), or through
// tcgen05.st by the peer's warps followed by a cluster-scope release to the
// leader's MMA issuer, which takes 1.3 us or more under load (measured with
// a per-stage trace) and puts the MMAs on that latency every stage; the
// pair's accumulator hand-back crosses the cluster the same way.  Here the
// scale stores, their signal and the accumulator hand-back stay inside one
// CTA; what crosses the cluster is the multicast data itself and each CTA's
// MMA commit, which frees a ring slot in both CTAs (the peer's multicast
// writes into this CTA's slot too).
//
// Per stage (256 K elements) a CTA stages 16 KB of A codes, 32 KB of B codes,
// 2 KB of A scale tiles and 4 KB of B scale tiles: 54 KB, three stages deep.
// TMEM: one 256-column accumulator drained by eight epilogue warps into
// registers (epilogue_loop_regdrain) plus 3 x 48 scale columns, stored by
// the same warps with tcgen05.st between their epilogue chunks.
//
// Barriers (per ring slot s, in each CTA): full[s] (codes: own A, both B
// halves), sf_full[s] (scale tiles: own A, both B halves), sf_ready[s] (the
// 4 scale writers of this stage), empty[s] (two arrivals: the MMA commits of
// both CTAs, each multicast to both).  Every wait is bounded.
#pragma once

#include "gemm_epilogue.cuh"
#include "gemm_kernel_common.cuh"
#include "gemm_kernel_nvfp4_2sm_st.cuh"

namespace spg {

template <int EPI, int STAGES>
struct Nvfp4McCfg {
  static constexpr int kBN = 256;
  static constexpr int kBKBytes = 128;  // 256 E2M1 elements per row and stage
  static constexpr int kKSteps = 4;     // K = 64 per MMA
  static constexpr int kABytes = 128 * kBKBytes;
  static constexpr int kBHalfBytes = 128 * kBKBytes;  // one CTA's multicast share of B
  static constexpr int kBBytes = 2 * kBHalfBytes;
  static constexpr int kSfaBytes = 4 * 512;
  static constexpr int kSfbHalfBytes = 4 * 512;
  static constexpr int kSfbBytes = 2 * kSfbHalfBytes;
  static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
  static constexpr int kSfColsPerKStep = 4 + 8;  // A scales, then the two B halves
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
  // full, empty, sf_full, sf_ready per slot; acc_full, acc_empty, drain,
  // stall; residual barriers; tmem slot + abort flag; slot-use counters;
  // the exit record.
  static_assert((4 * STAGES + 4 + 2 * kEpiWarps) * 8 + 8 + 4 * STAGES + 8 + sizeof(PairExit) <=
                    kBarBytes,
                "barrier area too small");

  // Block-scaled descriptor: A, B = E2M1 (1), UE4M3 scales, M = 128, N = 256, K = 64.
  // One instruction covers both 128-row halves of B (its scales: the two
  // 4-column groups after A's), so each k-step reads A from shared memory
  // once.
  __host__ __device__ static constexpr uint32_t idesc() {
    return (1u << 7) | (1u << 10) | (uint32_t(kBN >> 3) << 17) | (uint32_t(128 >> 4) << 24);
  }
};

// Exit of a multicast cluster: each CTA's full / sf_full barriers count the
// copies of both producers (its own and the peer's multicast share).  The
// two producers exchange how many stages they issued; every stage of the
// last ring's worth that only one of them issued is settled on this CTA's
// barriers (the arrival and bytes of peer copies this CTA never announced,
// or the announced bytes of a peer share that was never sent), and every
// outstanding stage is waited for, so no copy into this CTA's memory is in
// flight when the cluster passes its final barrier.
template <int STAGES>
__device__ __forceinline__ void mc_exit_settle(PairExit* mine, uint64_t* full, uint64_t* sf_full,
                                               uint32_t issued, uint32_t peer_code_bytes,
                                               uint32_t peer_sf_bytes, uint32_t rank,
                                               const GemmParams& p) {
  const uint32_t peer_px = mapa_shared(smem_u32(mine), rank ^ 1u);
  st_cluster_u32(peer_px + uint32_t(offsetof(PairExit, issued)), issued);
  mbar_arrive_cluster(peer_px + uint32_t(offsetof(PairExit, bar)));
  uint32_t peer = issued;
  if (mbar_wait_drain_cluster(&mine->bar, 0, p.drain_ns, p.err))
    peer = *reinterpret_cast<volatile uint32_t*>(&mine->issued);
  const uint32_t hi = issued > peer ? issued : peer;
  const uint32_t lo = hi > uint32_t(STAGES) ? hi - uint32_t(STAGES) : 0u;
  for (uint32_t idx = lo; idx < hi; ++idx) {
    const uint32_t s = idx % uint32_t(STAGES);
    if (idx >= issued) {
      mbar_arrive_expect_tx(&full[s], peer_code_bytes);
      mbar_arrive_expect_tx(&sf_full[s], peer_sf_bytes);
    } else if (idx >= peer) {
      mbar_complete_tx(&full[s], peer_code_bytes);
      mbar_complete_tx(&sf_full[s], peer_sf_bytes);
    }
    const uint32_t par = (idx / uint32_t(STAGES)) & 1u;
    mbar_wait_drain(&full[s], par, p.drain_ns, p.err);
    mbar_wait_drain(&sf_full[s], par, p.drain_ns, p.err);
  }
}

template <int EPI, int STAGES, bool HAS_BIAS>
__global__ void __launch_bounds__(Nvfp4McCfg<EPI, STAGES>::kThreads, 1)
    gemm_kernel_nvfp4_mc(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmY,
                         const __grid_constant__ CUtensorMap tmSFA,
                         const __grid_constant__ CUtensorMap tmSFB,
                         const __grid_constant__ CUtensorMap tmR, const GemmParams p) {
  using Cfg = Nvfp4McCfg<EPI, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint8_t* epi = smem + STAGES * Cfg::kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(epi + Cfg::kEpiBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* sf_full = bars + 2 * STAGES;
  uint64_t* sf_ready = bars + 3 * STAGES;
  uint64_t* acc_full = bars + 4 * STAGES;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* drain = acc_empty + 1;
  uint64_t* stall = drain + 1;     // test hook: nothing arrives on it
  uint64_t* res_bars = stall + 1;  // linear_add residual: 2 per epilogue warp
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(res_bars + 2 * Cfg::kEpiWarps);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int* landed = abort_flag + 1;  // STAGES counters (ScaleService)
  PairExit* cexit = reinterpret_cast<PairExit*>(
      (reinterpret_cast<uintptr_t>(landed + STAGES) + 7) & ~uintptr_t(7));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cluster = blockIdx.x >> 1;
  const int num_clusters = gridDim.x >> 1;
  constexpr uint16_t kBoth = 0x3;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 2);
      mbar_init(&sf_full[s], 1);
      mbar_init(&sf_ready[s], 4);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, Cfg::kEpiWarps);
    mbar_init(drain, 1);
    mbar_init(stall, 1);
    for (int w = 0; w < 2 * Cfg::kEpiWarps; ++w) mbar_init(&res_bars[w], 1);
    *abort_flag = 0;
    for (int s = 0; s < STAGES; ++s) landed[s] = 0;
    mbar_init(&cexit->bar, 1);
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmY);
    prefetch_tmap(&tmSFA);
    prefetch_tmap(&tmSFB);
    if (EPI == SPG_EPI_ADD) prefetch_tmap(&tmR);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Cfg::kTmemCols);
    tmem_relinquish();
  }
  // Both CTAs' barriers must be initialised before either multicasts into
  // the other.
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
      bool ok = true;
      const int64_t tpr = p.sf_tiles_per_row_block;
      const int a_row_blocks = (p.M + 127) / 128;
      const int b_row_blocks = (p.N + 127) / 128;
      for (int item = cluster; ok && item < p.total_items; item += num_clusters) {
        const WorkItem tc = work_item(item, p, Cfg::kBN);
        const int a_rb = tc.mb * 2 + int(rank);
        const int b_rb = tc.nb * 2 + int(rank);  // this CTA's multicast share of B
        // Scale tiles of row blocks past the operand are never multiplied by
        // a non-zero code (TMA zero-fills those rows): read the last real
        // block instead of running past the buffer.
        const int a_rb_sf = a_rb < a_row_blocks ? a_rb : a_row_blocks - 1;
        const int b_rb_sf = b_rb < b_row_blocks ? b_rb : b_row_blocks - 1;
        for (int kb = tc.kb_begin; kb < tc.kb_end; ++kb) {
          // Both CTAs' MMAs must be done with this slot: the peer's multicast
          // writes into it too.
          if (!mbar_wait_cluster(&empty[s], ph ^ 1u, ctl, kErrWaitEmpty)) {
            ok = false;
            break;
          }
          uint8_t* sa = ring + s * Cfg::kStageBytes;
          uint8_t* sb = sa + Cfg::kABytes;
          uint8_t* ssfa = sb + Cfg::kBBytes;
          uint8_t* ssfb = ssfa + Cfg::kSfaBytes;
          // Scale tiles first (6 KB against 48 KB of codes), so their stores
          // into TMEM overlap the codes' arrival.
          mbar_arrive_expect_tx(&sf_full[s], Cfg::kSfaBytes + Cfg::kSfbBytes);
          const int k_tile = kb * 4;
          tma_load_3d(ssfa, &tmSFA, &sf_full[s], 0, a_rb_sf * int(tpr) + k_tile, 0);
          tma_load_3d_multicast(ssfb + int(rank) * Cfg::kSfbHalfBytes, &tmSFB, &sf_full[s], 0,
                                b_rb_sf * int(tpr) + k_tile, 0, kBoth);
          mbar_arrive_expect_tx(&full[s], Cfg::kABytes + Cfg::kBBytes);
          const int kx = kb * Cfg::kBKBytes;
          tma_load_3d(sa, &tmA, &full[s], kx, a_rb * 128, 0);
          tma_load_3d_multicast(sb + int(rank) * Cfg::kBHalfBytes, &tmB, &full[s], kx, b_rb * 128,
                                0, kBoth);
          ++issued;
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      mc_exit_settle<STAGES>(cexit, full, sf_full, issued, Cfg::kBHalfBytes, Cfg::kSfbHalfBytes,
                             rank, p);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdesc = Cfg::idesc();
      int s = 0;
      uint32_t ph = 0;
      int it = 0;
      bool ok = true;
      for (int item = cluster; ok && item < p.total_items; item += num_clusters, ++it) {
        const WorkItem w = work_item(item, p, Cfg::kBN);
        if (!mbar_wait(acc_empty, (it & 1) ^ 1u, ctl, kErrWaitAccEmpty)) break;
        tc_fence_after();
        for (int kb = w.kb_begin; kb < w.kb_end; ++kb) {
          if (!mbar_wait(&full[s], ph, ctl, kErrWaitFull) ||
              !mbar_wait(&sf_ready[s], ph, ctl, kErrWaitFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(ring + s * Cfg::kStageBytes);
          const uint32_t sb = sa + Cfg::kABytes;
          const uint32_t sf_col0 = tmem_base + uint32_t(Cfg::kBN + s * Cfg::kSfColsPerStage);
#pragma unroll
          for (int j = 0; j < Cfg::kKSteps; ++j) {
            const uint32_t col = sf_col0 + uint32_t(j * Cfg::kSfColsPerKStep);
            mma_nvf4(tmem_base, smem_desc(sa + j * 32, 16, 1024, kSwizzle128B),
                     smem_desc(sb + j * 32, 16, 1024, kSwizzle128B), kIdesc, col, col + 4,
                     (kb != w.kb_begin) || j != 0);
          }
          tc_commit_multicast(&empty[s], kBoth);
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(acc_full);
      }
      tc_commit(drain);
      mbar_wait_drain(drain, 0, p.drain_ns, p.err);
    }
  } else if (p.debug_stall && !mbar_wait(stall, 0, ctl, kErrInjectedStall)) {
    // Test hook: the epilogue (and with it the scale service) waited on a
    // barrier nothing arrives on; the CTA has aborted and its other roles
    // drain and return.
  } else {
    // ------------------------------------- epilogue + scale-factor stores
    int my_stages = 0;
    for (int item = cluster; item < p.total_items; item += num_clusters) {
      const WorkItem w = work_item(item, p, Cfg::kBN);
      my_stages += w.kb_end - w.kb_begin;
    }
    ScaleService<STAGES> svc;
    svc.next = (warp - 2) >> 2;
    svc.end = my_stages;
    svc.sf_full = sf_full;
    svc.landed = landed;
    svc.sf_ready = sf_ready;
    svc.sf_ready_leader = 0;
    svc.leader = true;  // every CTA signals its own MMA issuer
    svc.ring = ring;
    svc.stage_bytes = Cfg::kStageBytes;
    svc.sf_offset = Cfg::kABytes + Cfg::kBBytes;
    svc.tmem_base = tmem_base;
    svc.sf_col_base = uint32_t(Cfg::kBN);
    svc.sf_cols_per_stage = uint32_t(Cfg::kSfColsPerStage);
    svc.q = warp & 3;
    svc.lane = lane;
    auto arrive_fn = [&](int) { mbar_arrive(acc_empty); };
    auto item_fn = [&](int item) {
      WorkItem w = work_item(item, p, Cfg::kBN);
      w.mb = w.mb * 2 + int(rank);
      return w;
    };
    epilogue_loop_regdrain<EPI, kScaleScalar, HAS_BIAS, decltype(item_fn), decltype(arrive_fn),
                           ScaleService<STAGES>, true>(
        p, &tmY, tmem_base, acc_full, arrive_fn, epi, cluster, num_clusters, item_fn, ctl,
        int(rank), svc, &tmR, res_bars);
  }

  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, Cfg::kTmemCols);
}

}  // namespace spg
