// Two-SM block-scaled NVFP4 GEMM with the scale factors written into TMEM by
// warps (tcgen05.st) instead of copied by the tensor core (tcgen05.cp),
// sm_103a.
//
// The tile, the operand ring, the producer, the MMAs and the register-drain
// epilogue are those of gemm_kernel_nvfp4_2sm.  What changes is how each
// stage's scales reach TMEM.  A block-scaled MMA computing the rows of one
// TMEM lane quarter reads its scales from that quarter's 32 lanes: lane i of
// every quarter must hold, in the 4 columns of a scale group, the words (four
// E4M3 scales each) of rows i, 32 + i, 64 + i and 96 + i of the 128-row
// block -- the layout a tcgen05.cp 32x128b.warpx4 produces by broadcasting a
// 512-byte scale tile to the four quarters (measured on GB300: with the B
// scales of one quarter only, the other quarters' rows come out wrong).  That
// copy runs in the tensor pipe, where the 12 copies of a stage cost about as
// much time as its 4 MMAs.  Here the eight epilogue warps store the same 12
// groups with tcgen05.st, each into its own lane quarter, outside the tensor
// pipe: the warps with (warp - 2) / 4 == h serve the stages k with
// k % 2 == h, one warp per quarter, whenever they wait for the accumulator
// and between their output chunks.  The scale tiles land on a barrier of
// their own CTA (sf_full), so they can be written up to STAGES stages ahead
// of the MMAs.
//
// Barriers (per stage s): full[s] (leader; both CTAs' A/B codes), sf_full[s]
// (each CTA; its scale tiles), sf_ready[s] (leader; 5 arrivals: the 4 scale
// writers of the leader and one forwarded for the peer's 4; the MMA issuer
// waits with a cluster-scope acquire), peer_ready[s] (peer; its 4 writers),
// empty[s] (both CTAs; multicast commit after the stage's MMAs).  Every wait
// is bounded.
//
// The peer's scale writers do not signal the leader themselves: a
// cluster-scope release arrival holds the issuing warp about 0.8 us (median;
// 1.3 us at the 90th percentile, measured in this kernel on GB300), and a
// writer warp serves every other stage, so the MMAs waited for it.  They
// arrive on a barrier of their own CTA (cheap), and three otherwise idle
// warps of the peer (its MMA warp and two forwarder warps) take turns
// forwarding one cluster-scope arrival per stage, so three of those slow
// releases are in flight at once.
#pragma once

#include "gemm_epilogue.cuh"
#include "gemm_kernel_common.cuh"
#include "gemm_kernel_nvfp4_2sm.cuh"

namespace spg {

template <int EPI, int STAGES>
struct Nvfp4StCfg {
  using Base = Nvfp4PairCfg<EPI, STAGES>;
  static constexpr int kBN = Base::kBN;
  static constexpr int kBKBytes = Base::kBKBytes;
  static constexpr int kKSteps = Base::kKSteps;
  static constexpr int kABytes = Base::kABytes;
  static constexpr int kBBytes = Base::kBBytes;
  static constexpr int kSfaBytes = Base::kSfaBytes;
  static constexpr int kSfbBytes = Base::kSfbBytes;
  static constexpr int kStageBytes = Base::kStageBytes;
  static constexpr int kSfColsPerKStep = Base::kSfColsPerKStep;
  static constexpr int kSfColsPerStage = Base::kSfColsPerStage;
  static constexpr int kTmemCols = Base::kTmemCols;
  static constexpr int kEpiWarps = 8;
  static constexpr int kEpiBytes = kEpiWarps * 2 * 32 * 64;
  static constexpr int kBarBytes = 512;
  static constexpr int kSmemBytes = 1024 + STAGES * kStageBytes + kEpiBytes + kBarBytes;
  static constexpr int kFwdWarps = 2;  // forwarder warps after the epilogue warps
  static constexpr int kThreads = 64 + 32 * kEpiWarps + 32 * kFwdWarps;

  static_assert(kSmemBytes <= 232448, "shared memory budget exceeded");
  // barriers, residual barriers, tmem slot + abort flag, slot-use counters
  // (writers and forwarders), stall barrier, PairExit
  static_assert((5 * STAGES + 3 + 2 * kEpiWarps) * 8 + 8 + 8 * STAGES + 8 + 8 +
                        sizeof(PairExit) <= kBarBytes,
                "barrier area too small");
  __host__ __device__ static constexpr uint32_t idesc() { return Base::idesc(); }
};

// Issue the stores of one stage's scales into lane quarter q: its 12 scale
// groups (4 k-steps x {A, B rows 0-127, B rows 128-255}) at sf_col0, 4
// columns each.  Scale tile layout in shared memory: 512 bytes per (128-row
// block, k-step), row r's four scales at (r % 32) * 16 + (r / 32) * 4, so
// lane i's 16 bytes are exactly the 4 columns it holds.  The caller waits
// for the stores (tcgen05.wait::st) before it signals them.
__device__ __forceinline__ void store_stage_scales(uint32_t tmem_base, uint32_t sf_col0,
                                                   const uint8_t* ssfa, const uint8_t* ssfb,
                                                   int q, int lane) {
  const uint32_t col0 = tmem_base + (uint32_t(q * 32) << 16) + sf_col0;
  const int off = lane * 16;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint4 a = *reinterpret_cast<const uint4*>(ssfa + j * 512 + off);
    const uint4 b0 = *reinterpret_cast<const uint4*>(ssfb + j * 512 + off);
    const uint4 b1 = *reinterpret_cast<const uint4*>(ssfb + 2048 + j * 512 + off);
    const uint32_t col = col0 + uint32_t(j * 12);
    tmem_st_32x32b_x4(col, a);
    tmem_st_32x32b_x4(col + 4, b0);
    tmem_st_32x32b_x4(col + 8, b1);
  }
}

// The epilogue warps' side duty: store the scales of every stage of this
// warp's parity whose scale tiles have landed, for its lane quarter, and
// signal each one as soon as its stores are done (non-blocking).
//
// Stage uses alternate between the two halves of the warps while the ring
// has an odd number of stages, so the previous use of a ring slot belongs to
// the other half.  A parity test alone cannot tell "use n has landed" from
// "use n - STAGES has not landed yet" (both phases have the same parity
// distance), so a use is tested only once landed[slot] -- the count of uses
// of that slot seen complete, raised by whichever warp saw them -- shows the
// previous use complete.  Without this guard a warp that ran ahead at the
// start of a launch stored scales for a later use into a slot whose current
// use the MMAs had not yet read (measured on GB300: whole lane quarters of a
// kernel's first tiles wrong in a few of 40 launches).  The guard costs about
// 2.5% of the kernel's throughput (measured; 0 of 100 launches differ).
template <int STAGES>
struct ScaleService {
  static constexpr bool kActive = true;
  int next;           // next stage to serve (this warp's parity)
  int end;            // stages of this CTA pair
  uint64_t* sf_full;         // this CTA's scale-tile barriers
  int* landed;               // per ring slot: uses seen complete (shared)
  uint64_t* sf_ready;        // stage barriers the writers arrive on (this CTA)
  uint32_t sf_ready_leader;  // unused (0)
  bool leader;
  uint8_t* ring;
  int stage_bytes, sf_offset;  // ring stride; scale tiles' offset in a stage
  uint32_t tmem_base, sf_col_base, sf_cols_per_stage;
  int q, lane;

  __device__ __forceinline__ void operator()() {
    while (next < end) {
      const int s = next % STAGES;
      const int u = next / STAGES;  // use of slot s
      const uint32_t par = uint32_t(u) & 1u;
      int ready = 0;
      if (lane == 0) {
        // Both reads issued before either result is used.
        const int seen = *reinterpret_cast<volatile int*>(&landed[s]);
        const bool done = mbar_test_wait(smem_u32(&sf_full[s]), par);
        ready = done & (seen >= u);
      }
      ready = __shfl_sync(0xffffffffu, ready, 0);
      if (!ready) return;
      // Every lane acquires the completed phase before it reads the tiles.
      (void)mbar_test_wait(smem_u32(&sf_full[s]), par);
      __syncwarp();
      const uint8_t* ssfa = ring + s * stage_bytes + sf_offset;
      store_stage_scales(tmem_base, sf_col_base + uint32_t(s) * sf_cols_per_stage, ssfa,
                         ssfa + 2048, q, lane);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      // Release at CTA scope on a barrier of this CTA: the MMA issuer's own
      // stage barrier in the leader; in the peer, the barrier its forwarders
      // wait on, whose cluster-scope release then orders these TMEM stores
      // before the leader's cluster-scope acquire and its MMAs (causality
      // is transitive).  A relaxed arrival is not enough: the MMAs could
      // read the scales before the stores land.
      if (lane == 0) {
        mbar_arrive(&sf_ready[s]);
        // Off the path to the MMAs: the other half tests use u + 1 of this
        // slot only after it has landed, long after this.
        atomicMax(&landed[s], u + 1);
      }
      next += 2;
    }
  }
};

template <int EPI, int STAGES, bool HAS_BIAS>
__global__ void __launch_bounds__(Nvfp4StCfg<EPI, STAGES>::kThreads, 1)
    gemm_kernel_nvfp4_2sm_st(const __grid_constant__ CUtensorMap tmA,
                             const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmY,
                             const __grid_constant__ CUtensorMap tmSFA,
                             const __grid_constant__ CUtensorMap tmSFB,
                             const __grid_constant__ CUtensorMap tmR, const GemmParams p) {
  using Cfg = Nvfp4StCfg<EPI, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint8_t* epi = smem + STAGES * Cfg::kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(epi + Cfg::kEpiBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* sf_full = bars + 2 * STAGES;
  uint64_t* sf_ready = bars + 3 * STAGES;    // leader: writers + forwarded peer arrivals
  uint64_t* peer_ready = bars + 4 * STAGES;  // peer: its 4 writers, read by the forwarders
  uint64_t* acc_full = bars + 5 * STAGES;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* drain = acc_empty + 1;
  uint64_t* res_bars = drain + 1;  // linear_add residual: 2 per epilogue warp
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(res_bars + 2 * Cfg::kEpiWarps);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int* landed = abort_flag + 1;       // STAGES counters (ScaleService)
  int* forwarded = landed + STAGES;  // STAGES counters: uses forwarded per slot
  // test hook barrier (nothing arrives on it), then the pair's exit record
  uint64_t* stall = reinterpret_cast<uint64_t*>(
      (reinterpret_cast<uintptr_t>(forwarded + STAGES) + 7) & ~uintptr_t(7));
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
      mbar_init(&sf_full[s], 1);
      mbar_init(&sf_ready[s], 5);
      mbar_init(&peer_ready[s], 4);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 2 * Cfg::kEpiWarps);
    mbar_init(drain, 1);
    for (int w = 0; w < 2 * Cfg::kEpiWarps; ++w) mbar_init(&res_bars[w], 1);
    *abort_flag = 0;
    for (int s = 0; s < STAGES; ++s) landed[s] = forwarded[s] = 0;
    mbar_init(stall, 1);
    mbar_init(&pexit->bar, 1);
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
      uint32_t tx[STAGES] = {};  // this CTA's code-copy bytes per ring slot (last use)
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
          // Scale tiles first (4 consecutive 512-byte tiles per 128-row block,
          // on this CTA's own barrier): they are 6 KB against 64 KB of codes,
          // so their stores into TMEM overlap the codes' arrival instead of
          // following it.
          mbar_arrive_expect_tx(&sf_full[s], Cfg::kSfaBytes + Cfg::kSfbBytes);
          const int k_tile = kb * 4;
          tma_load_3d(ssfa, &tmSFA, &sf_full[s], 0, a_rb_sf * int(tpr) + k_tile, 0);
          tma_load_3d(ssfb, &tmSFB, &sf_full[s], 0, b_rb0 * int(tpr) + k_tile, 0);
          tma_load_3d(ssfb + 2048, &tmSFB, &sf_full[s], 0, b_rb1 * int(tpr) + k_tile, 0);
          if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * (Cfg::kABytes + Cfg::kBBytes));
          const uint32_t bar = mapa_shared(smem_u32(&full[s]), 0);
          const int kx = kb * Cfg::kBKBytes;
          tma_load_3d_pair(sa, &tmA, bar, kx, m0, 0);
          tma_load_3d_pair(sb, &tmB, bar, kx, n0, 0);
          tx[s] = Cfg::kABytes + Cfg::kBBytes;
          ++issued;
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      // No copy may still be writing this CTA's memory (or signalling the
      // leader's barriers) at exit: the scale tiles land on this CTA's own
      // barriers; both CTAs' code copies land on the leader's, whose
      // accounts the two producers settle.
      const uint32_t outstanding = issued < uint32_t(STAGES) ? issued : uint32_t(STAGES);
      for (uint32_t i = 0; i < outstanding; ++i) {
        const uint32_t idx = issued - 1 - i;
        mbar_wait_drain(&sf_full[idx % STAGES], (idx / STAGES) & 1u, p.drain_ns, p.err);
      }
      if (rank == 0)
        pair_exit_drain<STAGES>(pexit, full, issued, tx, p);
      else
        pair_exit_publish<STAGES>(pexit, issued, tx);
    }
  } else if ((warp == 1 && rank == 1) || warp >= 2 + Cfg::kEpiWarps) {
    // ------------------------------------------- forwarders (peer CTA only)
    // Forwarder f (the peer's MMA warp, then the forwarder warps) takes the
    // stages n with n % 3 == f: it waits until the peer's 4 writers have
    // stored stage n's scales (peer_ready), then releases one arrival at
    // cluster scope on the leader's sf_ready.  Uses of a ring slot come 5
    // stages apart and rotate over the forwarders; a parity test cannot tell
    // use u complete from use u - 2, so use u is tested only once
    // forwarded[slot] shows use u - 1 passed on.
    if (rank == 1 && lane == 0) {
      const int f = warp == 1 ? 0 : warp - (2 + Cfg::kEpiWarps) + 1;
      int my_stages = 0;
      for (int item = pair; item < p.total_items; item += num_pairs) {
        const WorkItem w = work_item(item, p, Cfg::kBN);
        my_stages += w.kb_end - w.kb_begin;
      }
      const uint32_t leader_ready = mapa_shared(smem_u32(sf_ready), 0);
      for (int n = f; n < my_stages; n += 1 + Cfg::kFwdWarps) {
        const int s = n % STAGES;
        const int u = n / STAGES;
        const uint64_t t0 = globaltimer_ns();
        bool ok = false;
        for (uint32_t i = 1;; ++i) {
          if (*reinterpret_cast<volatile int*>(&forwarded[s]) >= u) {
            ok = true;
            break;
          }
          if ((i & 15u) == 0 && (*ctl.abort_flag || globaltimer_ns() - t0 > ctl.timeout_ns)) {
            *ctl.abort_flag = 1;
            atomicCAS(ctl.err, 0u, kErrWaitFull);
            break;
          }
        }
        if (!ok || !mbar_wait(&peer_ready[s], uint32_t(u) & 1u, ctl, kErrWaitFull)) break;
        atomicMax(&forwarded[s], u + 1);
        mbar_arrive_cluster(leader_ready + uint32_t(s * 8));
      }
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
          if (!mbar_wait(&full[s], ph, ctl, kErrWaitFull) ||
              !mbar_wait_cluster(&sf_ready[s], ph, ctl, kErrWaitFull)) {
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
    // Test hook: the epilogue (and with it the scale service) waited on a
    // barrier nothing arrives on; the CTA has aborted and its other roles
    // drain and return.
  } else {
    // ------------------------------------- epilogue + scale-factor stores
    int my_stages = 0;
    for (int item = pair; item < p.total_items; item += num_pairs) {
      const WorkItem w = work_item(item, p, Cfg::kBN);
      my_stages += w.kb_end - w.kb_begin;
    }
    ScaleService<STAGES> svc;
    svc.next = (warp - 2) >> 2;
    svc.end = my_stages;
    svc.sf_full = sf_full;
    svc.landed = landed;
    svc.sf_ready = rank == 0 ? sf_ready : peer_ready;
    svc.sf_ready_leader = 0;
    svc.leader = rank == 0;
    svc.ring = ring;
    svc.stage_bytes = Cfg::kStageBytes;
    svc.sf_offset = Cfg::kABytes + Cfg::kBBytes;
    svc.tmem_base = tmem_base;
    svc.sf_col_base = uint32_t(Cfg::kBN);
    svc.sf_cols_per_stage = uint32_t(Cfg::kSfColsPerStage);
    svc.q = warp & 3;
    svc.lane = lane;
    auto arrive_fn = [&](int) { mbar_arrive_cluster(mapa_shared(smem_u32(acc_empty), 0)); };
    auto item_fn = [&](int item) {
      WorkItem w = work_item(item, p, Cfg::kBN);
      w.mb = w.mb * 2 + int(rank);
      return w;
    };
    epilogue_loop_regdrain<EPI, kScaleScalar, HAS_BIAS, decltype(item_fn), decltype(arrive_fn),
                           ScaleService<STAGES>, true>(
        p, &tmY, tmem_base, acc_full, arrive_fn, epi, pair, num_pairs, item_fn, ctl, int(rank),
        svc, &tmR, res_bars);
  }

  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
}

}  // namespace spg
