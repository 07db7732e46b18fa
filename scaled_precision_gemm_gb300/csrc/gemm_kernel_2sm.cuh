// Two-SM (CTA-pair) tcgen05 GEMM for FP8 operands, sm_103a.
//
// A cluster of two CTAs computes one 256 x BN output tile with
// tcgen05.mma.cta_group::2: each CTA stages its own 128 rows of A and its
// half (BN/2 rows) of B in shared memory, the leader CTA issues the MMA for
// the pair, and each CTA's TMEM receives its own 128 x BN accumulator.  Per
// SM this halves the B bytes staged per MMA compared with a one-CTA
// 128 x BN tile, which is what lets the ring run six stages deep and keeps
// the operand feed below the shared-memory and L2 limits.
//
// Synchronisation of the pair:
//   full[s]      leader only; the leader's producer posts the byte count of
//                both CTAs' loads, both CTAs' TMA loads complete on it.
//   empty[s]     in both CTAs; released by one multicast tcgen05.commit.
//   acc_full[b]  in both CTAs; released by one multicast tcgen05.commit.
//   acc_empty[b] leader only; the 4 epilogue warps of each CTA arrive on it.
// Every wait is bounded in time, as in the one-CTA kernel.
//
// Schedule: pair p processes work items p, p + pairs, ...; the last partial
// wave of tiles is split along N into narrower items, whose MMAs carry the
// narrower N in the instruction descriptor, or along K into pieces whose
// partial sums meet in a workspace (work_item, split_piece_finish).
// CSPLIT (swapped tile): every tile is split along K into split_k pieces run
// by the split_k pairs of one cluster of 2 x split_k CTAs, one piece per
// pair, and reduced through distributed shared memory (cluster_piece_finish):
// a CTA pair is two CTAs whose cluster ranks differ in bit 0, the even one
// leading it.
#pragma once

#include "gemm_epilogue.cuh"
#include "gemm_kernel_common.cuh"

namespace spg {

// SWAP: the operands' roles exchanged for narrow T -- A is the weight matrix
// (256 weight rows per pair tile, the MMA's M), B the activations (BN
// tokens, the MMA's N), and the epilogue writes the transposed accumulator
// (epilogue_loop_swap).  The swapped tile never splits along N, so its
// fourth tensor map (tmBnarrow) carries the residual of linear_add.
template <int EPI, int BN, int STAGES, bool A_MN, bool B_MN, int SCALE, bool SWAP = false,
          bool CSPLIT = false>
struct Gemm2smCfg {
  static constexpr int kBM = 128;  // rows per CTA (the pair covers 256)
  static constexpr int kBKBytes = 128;
  static constexpr int kKSteps = 4;
  static constexpr int kBHalf = BN / 2;
  static constexpr int kABytes = kBM * kBKBytes;
  static constexpr int kBBytes = kBHalf * kBKBytes;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTmemCols = 2 * BN <= 256 ? 256 : 512;
  static constexpr int kEpiWarps = 4;
  static constexpr int kEpiBytes = kEpiWarps * 2 * 32 * 64;
  // Swapped linear_add: one 32 x 32 bf16 residual block per epilogue warp
  // and 32-token chunk.
  static constexpr int kResBytes =
      (SWAP && EPI == SPG_EPI_ADD) ? kEpiWarps * (BN / 32) * 32 * 64 : 0;
  static constexpr int kBarBytes = 512;
  static constexpr int kSmemBytes =
      1024 + STAGES * kStageBytes + kEpiBytes + kResBytes + kBarBytes;
  static constexpr int kThreads = 192;

  static_assert(SWAP ? (BN == 32 || BN == 64 || BN == 128)
                     : (BN == 128 || BN == 160 || BN == 192 || BN == 256),
                "pair tiles are 256 x {128, 160, 192, 256} (256 x {32, 64, 128} swapped)");
  static_assert(!SWAP || (EPI != SPG_EPI_SWIGLU && !A_MN && !B_MN &&
                          (SCALE == kScaleRow || EPI == SPG_EPI_LINEAR)),
                "the swapped tile serves row-scaled linear / linear_add and per-tensor linear, "
                "with K-major operands");
  static_assert(EPI != SPG_EPI_SWIGLU || BN % 64 == 0, "SwiGLU tiles hold whole 64-column chunks");
  static_assert(!B_MN || BN == 256, "an N-major B half must be one 128-byte swizzle row");
  static_assert(kStageBytes % 1024 == 0, "stage bases must stay 1024-byte aligned");
  static_assert(kSmemBytes <= 232448, "shared memory budget exceeded");
  // linear_add residual by TMA into the epilogue staging buffers (the last
  // item's whole into the idle operand ring)
  static constexpr bool kResTma = !SWAP && EPI == SPG_EPI_ADD;
  static_assert(!kResTma || kEpiWarps * (BN / 32) * 32 * 64 <= STAGES * kStageBytes,
                "the last item's residual blocks must fit the operand ring");
  // barriers, tmem slot + abort flag, residual barriers (two per epilogue
  // warp), stall barrier, the cluster reduction's two barriers, PairExit
  static_assert((2 * STAGES + 9 + 2 * kEpiWarps) * 8 + sizeof(PairExit) <= kBarBytes,
                "barrier area too small");
  static_assert(!CSPLIT || SWAP, "the cluster K split serves the swapped tile");

  // kind::f8f6f4, E4M3 x E4M3 -> f32, M = 256 (pair), N = BN.
  __host__ __device__ static constexpr uint32_t idesc() {
    return (1u << 4) | (uint32_t(A_MN) << 15) | (uint32_t(B_MN) << 16) |
           (uint32_t(BN >> 3) << 17) | (uint32_t(256 >> 4) << 24);
  }
};

template <int EPI, int BN, int STAGES, bool A_MN, bool B_MN, int SCALE, bool SWAP = false,
          bool CSPLIT = false>
__global__ void __launch_bounds__(192, 1)
    gemm_kernel_2sm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmY,
                    const __grid_constant__ CUtensorMap tmBnarrow,
                    const __grid_constant__ CUtensorMap tmR, const GemmParams p) {
  using Cfg = Gemm2smCfg<EPI, BN, STAGES, A_MN, B_MN, SCALE, SWAP, CSPLIT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint8_t* epi = smem + STAGES * Cfg::kStageBytes;
  uint8_t* res_smem = epi + Cfg::kEpiBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(res_smem + Cfg::kResBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* acc_full = bars + 2 * STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  // linear_add residual copies: one per epilogue warp (swapped tile) or two
  // (one per staging buffer)
  uint64_t* res_bars = drain + 2;
  uint64_t* stall = res_bars + 2 * Cfg::kEpiWarps;  // test hook: nothing arrives on it
  uint64_t* cs_free = stall + 1;  // CSPLIT: cluster reduction barriers
  uint64_t* cs_ready = stall + 2;
  PairExit* pexit = reinterpret_cast<PairExit*>(stall + 3);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();
  const uint32_t rank = crank & 1u;      // this CTA's side of its pair
  const uint32_t leader = crank & ~1u;   // cluster rank of the pair's leader
  const uint16_t pair_mask = uint16_t(0x3u << leader);
  const int pair = blockIdx.x >> 1;
  const int num_pairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 2 * Cfg::kEpiWarps);
    }
    mbar_init(drain, 1);
    if constexpr (Cfg::kResBytes != 0 || Cfg::kResTma)
      for (int w = 0; w < 2 * Cfg::kEpiWarps; ++w) mbar_init(&res_bars[w], 1);
    mbar_init(stall, 1);
    if constexpr (CSPLIT) {
      mbar_init(cs_free, uint32_t(Cfg::kEpiWarps * p.split_k));
      mbar_init(cs_ready, uint32_t(Cfg::kEpiWarps * p.split_k));
    }
    mbar_init(&pexit->bar, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmY);
    if (p.split_ways > 1 || Cfg::kResBytes != 0) prefetch_tmap(&tmBnarrow);
    if constexpr (Cfg::kResTma) prefetch_tmap(&tmR);
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
      for (int item = pair; ok && item < p.total_items; item += num_pairs) {
        const WorkItem tc = work_item(item, p, BN);
        const int m0 = tc.mb * 256 + int(rank) * 128;
        // Each CTA stages its half of the item's columns.
        const int nb0 = tc.nb * BN + tc.n_off + int(rank) * (tc.width / 2);
        const int za = tc.b * p.a_batch_mul;
        const int zb = tc.b * p.b_batch_mul;
        for (int kb = tc.kb_begin; kb < tc.kb_end; ++kb) {
          if (!mbar_wait(&empty[s], ph ^ 1u, ctl, kErrWaitEmpty)) {
            ok = false;
            break;
          }
          uint8_t* sa = ring + s * Cfg::kStageBytes;
          uint8_t* sb = sa + Cfg::kABytes;
          // A narrower item stages only its B rows (the narrow box map).
          const bool narrow = tc.width < BN;
          const uint32_t b_bytes = narrow ? uint32_t(tc.width / 2) * Cfg::kBKBytes : Cfg::kBBytes;
          if (rank == 0) mbar_arrive_expect_tx(&full[s], 2 * (Cfg::kABytes + b_bytes));
          const uint32_t bar = mapa_shared(smem_u32(&full[s]), leader);
          const int kx = kb * Cfg::kBKBytes;
          if constexpr (A_MN)
            tma_load_3d_pair(sa, &tmA, bar, m0, kx, za);
          else
            tma_load_3d_pair(sa, &tmA, bar, kx, m0, za);
          if constexpr (B_MN)
            tma_load_3d_pair(sb, &tmB, bar, nb0, kx, zb);
          else
            tma_load_3d_pair(sb, narrow ? &tmBnarrow : &tmB, bar, kx, nb0, zb);
          tx[s] = Cfg::kABytes + b_bytes;
          ++issued;
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      // The leader's full barriers count both CTAs' bytes: once the two
      // producers' accounts are settled and the last stages have landed, no
      // TMA write of the pair is in flight.
      if (rank == 0)
        pair_exit_drain<STAGES>(pexit, full, issued, tx, p);
      else
        pair_exit_publish<STAGES>(pexit, issued, tx, leader);
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
        const int buf = it & 1;
        const uint32_t acc_ph = (it >> 1) & 1;
        const WorkItem w = work_item(item, p, BN);
        const int width = w.width;
        // The instruction descriptor's N field carries the item's width.
        const uint32_t idesc = (kIdesc & ~(0x3Fu << 17)) | (uint32_t(width >> 3) << 17);
        // The peer CTA's epilogue warps release this barrier across the pair.
        if (!mbar_wait_cluster(&acc_empty[buf], acc_ph ^ 1u, ctl, kErrWaitAccEmpty)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + uint32_t(buf * BN);
        for (int kb = w.kb_begin; kb < w.kb_end; ++kb) {
          if (!mbar_wait(&full[s], ph, ctl, kErrWaitFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(ring + s * Cfg::kStageBytes);
          const uint32_t sb = sa + Cfg::kABytes;
#pragma unroll
          for (int j = 0; j < Cfg::kKSteps; ++j) {
            uint64_t adesc, bdesc;
            if constexpr (A_MN)
              adesc = smem_desc(sa + j * 32 * 128, 16384, 1024, kSwizzle128B);
            else
              adesc = smem_desc(sa + j * 32, 16, 1024, kSwizzle128B);
            if constexpr (B_MN)
              bdesc = smem_desc(sb + j * 32 * 128, 16384, 1024, kSwizzle128B);
            else
              bdesc = smem_desc(sb + j * 32, 16, 1024, kSwizzle128B);
            mma_f8f6f4_pair(d_tmem, adesc, bdesc, idesc, (kb != w.kb_begin) || j != 0);
          }
          tc_commit_pair_multicast(&empty[s], pair_mask);
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_pair_multicast(&acc_full[buf], pair_mask);
      }
      tc_commit_pair(drain);
      mbar_wait_drain(drain, 0, p.drain_ns, p.err);
    }
  } else if (p.debug_stall && !mbar_wait(stall, 0, ctl, kErrInjectedStall)) {
    // Test hook: the epilogue waited on a barrier nothing arrives on; the CTA
    // has aborted and its other roles drain and return.
  } else {
    // -------------------------------------------------------------- epilogue
    auto arrive_fn = [&](int b) {
      mbar_arrive_cluster(mapa_shared(smem_u32(&acc_empty[b]), leader));
    };
    auto item_fn = [&](int item) {
      WorkItem w = work_item(item, p, BN);
      w.mb = w.mb * 2 + int(rank);
      return w;
    };
    if constexpr (SWAP) {
      ClusterSplit cs{cs_free, cs_ready, ring, false, 2u, rank};
      epilogue_loop_swap<EPI, BN, decltype(item_fn), decltype(arrive_fn), SCALE, CSPLIT>(
          p, &tmY, tmem_base, acc_full, arrive_fn, epi, pair, p.total_items, num_pairs, item_fn,
          ctl, int(rank), &tmBnarrow, res_bars, res_smem, &cs);
      // Leave only once every epilogue warp of the cluster has finished
      // writing into this CTA.
      if constexpr (CSPLIT) cluster_split_exit(p, cs);
    } else
      epilogue_loop<EPI, SCALE, BN, decltype(item_fn), decltype(arrive_fn), Cfg::kResTma>(
          p, &tmY, tmem_base, acc_full, arrive_fn, epi, pair, p.total_items, num_pairs, item_fn,
          ctl, int(rank), &tmR, res_bars, ring);
  }

  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
}

}  // namespace spg
