// Persistent, warp-specialised tcgen05 GEMM for sm_103a.
//
//   warp 0      TMA producer: fills a STAGES-deep shared-memory ring with
//               128-byte-wide K slices of A and B (and, for NVFP4, the
//               matching 128x4 scale tiles as single bulk copies).
//   warp 1      TMEM owner and MMA issuer: one elected lane issues
//               tcgen05.mma (kind::f8f6f4 for E4M3, kind::mxf4nvf4 block-scaled
//               for NVFP4) into a double-buffered fp32 TMEM accumulator and
//               releases ring slots with tcgen05.commit.
//   warps 2..5  epilogue: tcgen05.ld the accumulator (one TMEM lane = one
//               output row per thread), apply the scales and the fused
//               epilogue (linear / linear_add / linear_swiglu), stage the bf16
//               tile in 64-byte-swizzled shared memory and write it with TMA
//               stores, overlapping the next tile's main loop.
//
// The arithmetic is the same on every route and tile shape: per output
// element one fp32 accumulation of the K products in the tensor core, then
// y = acc * scale (row scales sa[t]*sw[n], or the scalar product of two
// device scalars), then the epilogue and one bf16 rounding (ninfer PR #167,
// opening paragraph: same accumulator, same scale application, same
// epilogue and output policies on both routes).
//
// Every mbarrier wait is bounded in time; on time-out the kernel records a
// code in the device error word and every role drains and returns.
#pragma once

#include "gemm_epilogue.cuh"
#include "gemm_kernel_common.cuh"

namespace spg {

// ACC_BUFS: TMEM accumulator buffers (2: the epilogue of one tile overlaps
// the next tile's main loop; 1 when every CTA runs one work item).
template <int KIND, int EPI, int BN, int STAGES, bool A_MN, bool B_MN, int SCALE, int ACC_BUFS = 2>
struct GemmCfg {
  static constexpr int kBM = 128;
  static constexpr int kBKBytes = 128;  // K bytes per stage (one 128-byte swizzle row)
  static constexpr int kKSteps = 4;     // MMAs per stage, 32 bytes of K each
  static constexpr int kABytes = kBM * kBKBytes;
  static constexpr int kBBytes = BN * kBKBytes;
  static constexpr int kNHalves = BN / 128;  // 128-row blocks of B (NVFP4 scale tiles)
  static constexpr int kSfaBytes = KIND == kKindNvfp4 ? 4 * 512 : 0;
  static constexpr int kSfbBytes = KIND == kKindNvfp4 ? kNHalves * 4 * 512 : 0;
  static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
  static constexpr int kMmaN = KIND == kKindNvfp4 ? 128 : BN;
  static constexpr int kAccBufs = ACC_BUFS;
  static constexpr int kSfColsPerKStep = KIND == kKindNvfp4 ? 4 + 4 * kNHalves : 0;
  static constexpr int kSfColsPerStage = kKSteps * kSfColsPerKStep;
  static constexpr int kTmemUsed = kAccBufs * BN + STAGES * kSfColsPerStage;
  static constexpr int kTmemCols =
      kTmemUsed <= 32 ? 32 : kTmemUsed <= 64 ? 64 : kTmemUsed <= 128 ? 128 : kTmemUsed <= 256 ? 256 : 512;
  static constexpr int kEpiWarps = 4;
  static constexpr int kEpiBufBytes = 32 * 64;  // 32 rows x 32 bf16
  static constexpr int kEpiBytes = kEpiWarps * 2 * kEpiBufBytes;
  static constexpr int kBarBytes = 256;
  static constexpr int kSmemBytes = 1024 + STAGES * kStageBytes + kEpiBytes + kBarBytes;
  static constexpr int kThreads = 192;
  static constexpr int kOutColsPerChunk = 32;
  static constexpr int kAccColsPerChunk = EPI == SPG_EPI_SWIGLU ? 64 : 32;
  static constexpr int kChunks = BN / kAccColsPerChunk;

  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN must be 64..256, a multiple of 64");
  static_assert(KIND != kKindNvfp4 || BN % 128 == 0, "NVFP4 tiles are whole 128-row scale blocks");
  static_assert(kTmemUsed <= 512, "TMEM budget exceeded");
  static_assert(kStageBytes % 1024 == 0, "stage bases must stay 1024-byte aligned (128B swizzle)");
  static_assert(kSmemBytes <= 232448, "shared memory budget exceeded");
  static_assert(2 * STAGES + 8 <= kBarBytes / 8 - 2, "barrier area too small");
  static_assert(!(KIND == kKindNvfp4 && (A_MN || B_MN)), "NVFP4 operands are K-major");

  // Instruction descriptor.
  __host__ __device__ static constexpr uint32_t idesc() {
    if constexpr (KIND == kKindFp8) {
      // [4,6) D = f32; [7,10) A = E4M3 (0); [10,13) B = E4M3 (0);
      // [15] A major; [16] B major; [17,23) N >> 3; [24,29) M >> 4.
      return (1u << 4) | (uint32_t(A_MN) << 15) | (uint32_t(B_MN) << 16) |
             (uint32_t(kMmaN >> 3) << 17) | (uint32_t(kBM >> 4) << 24);
    } else {
      // Block-scaled: [4,6) B scale id 0; [7,10) A = E2M1 (1); [10,13) B = E2M1 (1);
      // [17,23) N >> 3; [23] scale type UE4M3 (0); [24,29) M >> 4;
      // [29,31) A scale id 0; [31] K = 64 (0).
      return (1u << 7) | (1u << 10) | (uint32_t(kMmaN >> 3) << 17) | (uint32_t(kBM >> 4) << 24);
    }
  }
};

// CSPLIT: launched in clusters of p.split_k CTAs, one work item per CTA:
// the K-split pieces of a tile (cluster rank = piece) reduced through
// distributed shared memory into the idle operand rings
// (cluster_piece_finish); no workspace.
template <int KIND, int EPI, int BN, int STAGES, bool A_MN, bool B_MN, int SCALE,
          bool CSPLIT = false>
__global__ void __launch_bounds__(192, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmY, const GemmParams p) {
  using Cfg = GemmCfg<KIND, EPI, BN, STAGES, A_MN, B_MN, SCALE, CSPLIT ? 1 : 2>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint8_t* epi = smem + STAGES * Cfg::kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(epi + Cfg::kEpiBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* acc_full = bars + 2 * STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint64_t* stall = drain + 1;  // test hook: never arrived on
  uint64_t* cs_free = stall + 1;  // CSPLIT: cluster reduction barriers
  uint64_t* cs_ready = stall + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(stall + 3);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], Cfg::kEpiWarps);
    }
    mbar_init(drain, 1);
    mbar_init(stall, 1);
    if constexpr (CSPLIT) {
      mbar_init(cs_free, uint32_t(Cfg::kEpiWarps * p.split_k));
      mbar_init(cs_ready, uint32_t(Cfg::kEpiWarps * p.split_k));
    }
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmY);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  // The peers arrive on this CTA's reduction barriers: their initialisation
  // must be visible across the cluster first.
  if constexpr (CSPLIT)
    cluster_sync();
  else
    __syncthreads();
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
      for (int item = blockIdx.x; ok && item < p.total_items; item += gridDim.x) {
        const WorkItem tc = work_item(item, p, BN);
        const int m0 = tc.mb * Cfg::kBM;
        const int n0 = tc.nb * BN;
        const int za = tc.b * p.a_batch_mul;
        const int zb = tc.b * p.b_batch_mul;
        for (int kb = tc.kb_begin; kb < tc.kb_end; ++kb) {
          if (!mbar_wait(&empty[s], ph ^ 1u, ctl, kErrWaitEmpty)) {
            ok = false;
            break;
          }
          uint8_t* sa = ring + s * Cfg::kStageBytes;
          uint8_t* sb = sa + Cfg::kABytes;
          mbar_arrive_expect_tx(&full[s], Cfg::kStageBytes);
          const int kx = kb * Cfg::kBKBytes;
          if constexpr (A_MN) {
            tma_load_3d(sa, &tmA, &full[s], m0, kx, za);
          } else {
            tma_load_3d(sa, &tmA, &full[s], kx, m0, za);
          }
          if constexpr (B_MN) {
#pragma unroll
            for (int h = 0; h < BN / 128; ++h)
              tma_load_3d(sb + h * 128 * Cfg::kBKBytes, &tmB, &full[s], n0 + h * 128, kx, zb);
          } else {
            tma_load_3d(sb, &tmB, &full[s], kx, n0, zb);
          }
          if constexpr (KIND == kKindNvfp4) {
            uint8_t* ssfa = sb + Cfg::kBBytes;
            uint8_t* ssfb = ssfa + Cfg::kSfaBytes;
            const int64_t tpr = p.sf_tiles_per_row_block;
            bulk_load(ssfa, p.sfa + (int64_t(tc.mb) * tpr + int64_t(kb) * 4) * 512, 2048, &full[s]);
#pragma unroll
            for (int h = 0; h < Cfg::kNHalves; ++h)
              bulk_load(ssfb + h * 2048,
                        p.sfb + ((int64_t(tc.nb) * Cfg::kNHalves + h) * tpr + int64_t(kb) * 4) * 512,
                        2048, &full[s]);
          }
          ++issued;
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      // Wait (bounded) until every copy issued into the ring has landed, so
      // no TMA write is in flight when the CTA leaves.
      const uint32_t outstanding = issued < uint32_t(STAGES) ? issued : uint32_t(STAGES);
      for (uint32_t i = 0; i < outstanding; ++i) {
        const uint32_t idx = issued - 1 - i;
        mbar_wait_drain(&full[idx % STAGES], (idx / STAGES) & 1u, p.drain_ns, p.err);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdesc = Cfg::idesc();
      int s = 0;
      uint32_t ph = 0;
      int it = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < p.total_items; item += gridDim.x, ++it) {
        const WorkItem w = work_item(item, p, BN);
        const int buf = it & 1;
        const uint32_t acc_ph = (it >> 1) & 1;
        if (!mbar_wait(&acc_empty[buf], acc_ph ^ 1u, ctl, kErrWaitAccEmpty)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + uint32_t(buf * BN);
        for (int kb = w.kb_begin; kb < w.kb_end; ++kb) {
          const bool acc = kb != w.kb_begin;
          if (!mbar_wait(&full[s], ph, ctl, kErrWaitFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(ring + s * Cfg::kStageBytes);
          const uint32_t sb = sa + Cfg::kABytes;
          if constexpr (KIND == kKindNvfp4) {
            const uint32_t ssfa = sb + Cfg::kBBytes;
            const uint32_t ssfb = ssfa + Cfg::kSfaBytes;
            const uint32_t sf_col0 =
                tmem_base + uint32_t(Cfg::kAccBufs * BN + s * Cfg::kSfColsPerStage);
#pragma unroll
            for (int j = 0; j < Cfg::kKSteps; ++j) {
              const uint32_t col = sf_col0 + uint32_t(j * Cfg::kSfColsPerKStep);
              tc_cp_32x128b_warpx4(col, smem_desc(ssfa + j * 512, 0, 128, kSwizzleNone));
#pragma unroll
              for (int h = 0; h < Cfg::kNHalves; ++h)
                tc_cp_32x128b_warpx4(col + 4 + 4 * h,
                                     smem_desc(ssfb + h * 2048 + j * 512, 0, 128, kSwizzleNone));
            }
#pragma unroll
            for (int j = 0; j < Cfg::kKSteps; ++j) {
              const uint32_t col = sf_col0 + uint32_t(j * Cfg::kSfColsPerKStep);
              const uint64_t adesc = smem_desc(sa + j * 32, 16, 1024, kSwizzle128B);
#pragma unroll
              for (int h = 0; h < Cfg::kNHalves; ++h) {
                const uint64_t bdesc =
                    smem_desc(sb + h * 128 * Cfg::kBKBytes + j * 32, 16, 1024, kSwizzle128B);
                mma_nvf4(d_tmem + h * 128, adesc, bdesc, kIdesc, col, col + 4 + 4 * h,
                         acc || j != 0);
              }
            }
          } else {
#pragma unroll
            for (int j = 0; j < Cfg::kKSteps; ++j) {
              uint64_t adesc, bdesc;
              if constexpr (A_MN)
                adesc = smem_desc(sa + j * 32 * 128, 128 * Cfg::kBKBytes, 1024, kSwizzle128B);
              else
                adesc = smem_desc(sa + j * 32, 16, 1024, kSwizzle128B);
              if constexpr (B_MN)
                bdesc = smem_desc(sb + j * 32 * 128, 128 * Cfg::kBKBytes, 1024, kSwizzle128B);
              else
                bdesc = smem_desc(sb + j * 32, 16, 1024, kSwizzle128B);
              mma_f8f6f4(d_tmem, adesc, bdesc, kIdesc, acc || j != 0);
            }
          }
          tc_commit(&empty[s]);
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&acc_full[buf]);
      }
      // All MMAs (and scale copies) must be complete before TMEM is freed.
      tc_commit(drain);
      mbar_wait_drain(drain, 0, p.drain_ns, p.err);
    }
  } else {
    // -------------------------------------------------------------- epilogue
    ClusterSplit cs{cs_free, cs_ready, ring, false, 1u, 0u};
    auto arrive_fn = [&](int b) { mbar_arrive(&acc_empty[b]); };
    auto item_fn = [&](int item) { return work_item(item, p, BN); };
    // Test hook: wait on a barrier nothing arrives on, so the bounded wait
    // runs out, the CTA aborts and every role drains and returns.
    if (p.debug_stall && !mbar_wait(stall, 0, ctl, kErrInjectedStall)) {
      // aborted: skip the tiles; the other roles see the abort flag
    } else {
      epilogue_loop<EPI, SCALE, BN, decltype(item_fn), decltype(arrive_fn), false, CSPLIT>(
          p, &tmY, tmem_base, acc_full, arrive_fn, epi, blockIdx.x, p.total_items, gridDim.x,
          item_fn, ctl, 0, nullptr, nullptr, nullptr, &cs);
    }
    // Leave only once every epilogue warp of the cluster has finished
    // writing into this CTA.
    if constexpr (CSPLIT) cluster_split_exit(p, cs);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, Cfg::kTmemCols);
}

}  // namespace spg
