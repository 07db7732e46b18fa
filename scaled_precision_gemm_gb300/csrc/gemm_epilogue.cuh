// Epilogue warps of the tcgen05 GEMMs: drain the fp32 accumulator from TMEM,
// apply the scales and the fused epilogue, and write bf16 through
// 64-byte-swizzled shared memory with TMA stores.
//
// Per output tile each epilogue warp owns 32 rows (one TMEM lane quarter);
// each thread owns one row.  The global operands of the epilogue (row scale,
// column scales, the first residual chunk) are requested before the
// accumulator is ready so their latency overlaps the main loop; the residual
// of chunk c+1 is requested while chunk c is being processed.
#pragma once

#include "gemm_kernel_common.cuh"

namespace spg {

template <int EPI, int SCALE, int BN>
struct EpilogueCfg {
  static constexpr int kAccColsPerChunk = EPI == SPG_EPI_SWIGLU ? 64 : 32;
  static constexpr int kChunks = BN / kAccColsPerChunk;
  static constexpr int kBufBytes = 32 * 64;  // 32 rows x 32 bf16
  static constexpr int kSwRegs = BN / 32;    // column scales held per lane
};

// Residual of one 32-column chunk of this thread's row (zeros outside).
__device__ __forceinline__ void load_residual_chunk(const GemmParams& p, int m, int n_c0,
                                                    bool row_ok, uint4 (&r)[4]) {
#pragma unroll
  for (int g = 0; g < 4; ++g) r[g] = make_uint4(0u, 0u, 0u, 0u);
  if (row_ok) {
    const uint4* rp = reinterpret_cast<const uint4*>(p.residual + int64_t(m) * p.N + n_c0);
#pragma unroll
    for (int g = 0; g < 4; ++g)
      if (n_c0 + g * 8 < p.N) r[g] = __ldg(rp + g);
  }
}

// Per-warp resources of the K-split reduction: a scratch area in the
// shared-memory operand ring (idle by then: a K-split piece is always the
// last item of its CTA pair, so every stage has been consumed once its
// accumulator is full) and one mbarrier for the bulk copies into it.
struct SplitScratch {
  uint8_t* buf;        // 1024-byte aligned
  int bytes;           // at least 4096
  uint64_t* bar;       // this warp's copy barrier (arrival count 1)
  uint32_t* phase;     // its parity, kept by the caller across items
};

// K-split piece of a tile (two-SM kernels).  The calling warp owns TMEM
// lane quarter q = row / 32 (t_row addresses column 0 of the tile's
// accumulator in that quarter) and accumulator columns [c0, c0 + ncols), a
// multiple of 32.  rows_live: some row of the quarter is inside the output.
//  1. The piece's partial sums go to its workspace slice.
//  2. Every epilogue warp arrives on split_bars[0] once its writes are
//     fenced; the first epilogue thread then counts the CTA's arrival on the
//     tile's counter and posts the outcome through split_bars[1].
//  3. In the CTA of the last piece to arrive, every warp bulk-copies the
//     other pieces' 4 KB blocks of its rows into its scratch, adds all
//     pieces in split order (its own from TMEM, so the total does not depend
//     on the arrival order) and writes the total back to TMEM, where the
//     ordinary epilogue picks it up.
// Returns 1 if this CTA holds the total, 0 if not, -1 if a wait ran out.
// Nothing waits for another CTA, so pieces never rely on running at the same
// time; the waits inside the CTA are bounded like every other.  `phase`
// counts the K-split pieces this CTA has processed (mod 2).  At most 4
// pieces per tile.
template <int BN>
__device__ __forceinline__ int split_piece_reduce(const GemmParams& p, uint32_t t_row,
                                                  const WorkItem& tc, int rank, int row, int c0,
                                                  int ncols, bool rows_live, uint64_t* split_bars,
                                                  int* flag, uint32_t phase,
                                                  const SplitScratch& scr, const WaitCtl& ctl) {
  const int lane = threadIdx.x & 31;
  const int q = row >> 5;
  const bool have_k = tc.kb_end > tc.kb_begin;
  if (rows_live) {
    float4* own = split_slice(p, tc.tail, tc.split, rank, BN);
#pragma unroll 1
    for (int c = c0; c < c0 + ncols; c += 32) {
      uint32_t r[32];
      if (have_k) {
        tmem_ld_32x32b_x32(t_row + c, r);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = 0u;
      }
      float4* blk = own + split_block_index(c >> 5, q) + lane;
#pragma unroll
      for (int g = 0; g < 8; ++g)
        __stcg(blk + g * 32,
               make_float4(__uint_as_float(r[4 * g]), __uint_as_float(r[4 * g + 1]),
                           __uint_as_float(r[4 * g + 2]), __uint_as_float(r[4 * g + 3])));
    }
  }
  __threadfence();
  __syncwarp();
  if (lane == 0) mbar_arrive(&split_bars[0]);
  if (threadIdx.x == 64) {  // first epilogue thread
    int outcome = -1;
    if (mbar_wait(&split_bars[0], phase, ctl, kErrWaitSplit)) {
      const int before = split_arrive(p, tc.tail, rank);
      __threadfence();
      outcome = before == p.split_k - 1 ? 1 : 0;
    }
    *reinterpret_cast<volatile int*>(flag) = outcome;
    mbar_arrive(&split_bars[1]);
  }
  if (!mbar_wait(&split_bars[1], phase, ctl, kErrWaitSplit)) return -1;
  const int outcome = *reinterpret_cast<volatile int*>(flag);
  if (outcome <= 0 || !rows_live) return outcome;
  __threadfence();

  const int own_s = tc.split;
  const int others = p.split_k - 1;
  const int nbuf = scr.bytes >> 12;
  int per_round = nbuf / others;  // chunks whose other blocks fit the scratch at once
  if (per_round < 1) per_round = 1;
  const int nchunks = ncols >> 5;
#pragma unroll 1
  for (int ch0 = 0; ch0 < nchunks; ch0 += per_round) {
    const int nch = nchunks - ch0 < per_round ? nchunks - ch0 : per_round;
    if (lane == 0) {
      fence_proxy_async_global();
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(scr.bar, uint32_t(nch * others) * 4096u);
      for (int i = 0; i < nch; ++i) {
        const int chunk = (c0 >> 5) + ch0 + i;
        for (int k = 0; k < others; ++k) {
          const int s2 = k + (k >= own_s ? 1 : 0);
          const float4* src =
              split_slice(p, tc.tail, s2, rank, BN) + split_block_index(chunk, q);
          bulk_load(scr.buf + (i * others + k) * 4096, src, 4096u, scr.bar);
        }
      }
    }
    __syncwarp();
    if (!mbar_wait(scr.bar, *scr.phase, ctl, kErrWaitSplit)) return -1;
    *scr.phase ^= 1u;
#pragma unroll 1
    for (int i = 0; i < nch; ++i) {
      const int c = c0 + (ch0 + i) * 32;
      uint32_t r[32];
      if (have_k) {
        tmem_ld_32x32b_x32(t_row + c, r);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = 0u;
      }
      const float4* blk = reinterpret_cast<const float4*>(scr.buf + i * others * 4096) + lane;
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 mine = make_float4(__uint_as_float(r[4 * g]), __uint_as_float(r[4 * g + 1]),
                                        __uint_as_float(r[4 * g + 2]),
                                        __uint_as_float(r[4 * g + 3]));
        for (int s2 = 0; s2 < p.split_k; ++s2) {
          const float4 x =
              s2 == own_s ? mine : blk[(s2 - (s2 > own_s ? 1 : 0)) * 256 + g * 32];
          t.x += x.x;
          t.y += x.y;
          t.z += x.z;
          t.w += x.w;
        }
        r[4 * g] = __float_as_uint(t.x);
        r[4 * g + 1] = __float_as_uint(t.y);
        r[4 * g + 2] = __float_as_uint(t.z);
        r[4 * g + 3] = __float_as_uint(t.w);
      }
      tmem_st_32x32b_x32(t_row + c, r);
    }
    __syncwarp();
  }
  tmem_wait_st();
  return 1;
}

// ItemFn(item) -> WorkItem with mb already offset for this CTA's rows (a
// whole tile has n_off = 0, width = BN); the loop runs over items
// [item_begin, item_end) with stride item_step.  ArriveEmpty(buf) releases
// accumulator buffer `buf` to the MMA issuer.  K-split pieces (two-SM
// kernels only) go through split_piece_reduce first; cta_rank, split_bars
// (two mbarriers: arrival count 4 and 1), split_flag (one shared int),
// copy_bars (one mbarrier of count 1 per epilogue warp) and the operand ring
// (ring, ring_bytes: the warps' scratch) serve them.
template <int EPI, int SCALE, int BN, typename ItemFn, typename ArriveEmpty>
__device__ __forceinline__ void epilogue_loop(const GemmParams& p, const CUtensorMap* tmY,
                                              uint32_t tmem_base, uint64_t* acc_full,
                                              ArriveEmpty arrive_empty, uint8_t* epi_smem,
                                              int item_begin, int item_end, int item_step,
                                              ItemFn item_fn, const WaitCtl& ctl, int cta_rank,
                                              uint64_t* split_bars, int* split_flag,
                                              uint64_t* copy_bars, uint8_t* ring,
                                              int ring_bytes) {
  using E = EpilogueCfg<EPI, SCALE, BN>;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int e = warp - 2;
  const int q = warp & 3;  // TMEM lane quarter this warp may access
  uint8_t* stage0 = epi_smem + (e * 2) * E::kBufBytes;
  int it = 0;
  int chunk_ctr = 0;
  uint32_t split_phase = 0, copy_phase = 0;
  const int scr_bytes = (ring_bytes / 4) & ~4095;
  const SplitScratch scr{ring + e * scr_bytes, scr_bytes, copy_bars + e, &copy_phase};
  float scalar = 1.f;
  if constexpr (SCALE == kScaleScalar) scalar = __ldg(p.scalar_a) * __ldg(p.scalar_b);

  for (int item = item_begin; item < item_end; item += item_step, ++it) {
    const int buf = it & 1;
    const uint32_t acc_ph = (it >> 1) & 1;
    const WorkItem tc = item_fn(item);
    const uint32_t t_row = tmem_base + (uint32_t(q * 32) << 16) + uint32_t(buf * BN);
    if (tc.split >= 0) {
      if (!mbar_wait(&acc_full[buf], acc_ph, ctl, kErrWaitAccFull)) break;
      tc_fence_after();
      const int outcome = split_piece_reduce<BN>(
          p, t_row, tc, cta_rank, q * 32 + lane, 0, tc.width, tc.mb * 128 + q * 32 < p.M,
          split_bars, split_flag, split_phase, scr, ctl);
      split_phase ^= 1u;
      if (outcome < 0) break;
      if (outcome == 0) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_empty(buf);
        continue;
      }
    }
    // After a K-split reduction TMEM holds the total of all pieces.
    const bool have_k = tc.split >= 0 || tc.kb_end > tc.kb_begin;
    const int m0 = tc.mb * 128;
    const int n0 = tc.nb * BN + tc.n_off;  // first accumulator column of the item (global)
    const int nch = tc.width / E::kAccColsPerChunk;
    const int m = m0 + q * 32 + lane;
    const bool row_ok = m < p.M;

    // Epilogue operands, requested before the accumulator is ready.
    float row_s = scalar;
    if constexpr (SCALE == kScaleRow) row_s = row_ok ? __ldg(p.row_scale + m) : 0.f;
    float swr[E::kSwRegs];
    if constexpr (SCALE == kScaleRow) {
#pragma unroll
      for (int j = 0; j < E::kSwRegs; ++j) {
        const int n = n0 + 32 * j + lane;
        swr[j] = (32 * j < tc.width && n < p.N) ? __ldg(p.col_scale + n) : 0.f;
      }
    }
    float biasr[E::kSwRegs];
    const bool has_bias = p.bias_kind != 0;
    if (has_bias) {
#pragma unroll
      for (int j = 0; j < E::kSwRegs; ++j)
        biasr[j] = 32 * j < tc.width ? load_bias(p, n0 + 32 * j + lane) : 0.f;
    }
    uint4 res_cur[4];
    if constexpr (EPI == SPG_EPI_ADD) load_residual_chunk(p, m, n0, row_ok, res_cur);

    if (tc.split < 0) {
      if (!mbar_wait(&acc_full[buf], acc_ph, ctl, kErrWaitAccFull)) break;
      tc_fence_after();
    }

#pragma unroll
    for (int c = 0; c < E::kChunks; ++c) {
      if (c >= nch) break;
      const int acc_c0 = c * E::kAccColsPerChunk;
      uint32_t raw[E::kAccColsPerChunk];
      if (have_k) {
        tmem_ld_32x32b_x32(t_row + acc_c0, *reinterpret_cast<uint32_t(*)[32]>(&raw[0]));
        if constexpr (E::kAccColsPerChunk == 64)
          tmem_ld_32x32b_x32(t_row + acc_c0 + 32, *reinterpret_cast<uint32_t(*)[32]>(&raw[32]));
      } else {
#pragma unroll
        for (int i = 0; i < E::kAccColsPerChunk; ++i) raw[i] = 0u;
      }
      uint4 res_next[4];
      if constexpr (EPI == SPG_EPI_ADD) {
        if (c + 1 < nch) load_residual_chunk(p, m, n0 + acc_c0 + 32, row_ok, res_next);
      }
      if (have_k) tmem_wait_ld();
      if (c == nch - 1) {
        // Every column of this accumulator buffer has been read: hand it back.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_empty(buf);
      }
      float v[E::kAccColsPerChunk];
#pragma unroll
      for (int i = 0; i < E::kAccColsPerChunk; ++i) {
        float s = row_s;
        if constexpr (SCALE == kScaleRow) {
          const int col = acc_c0 + i;  // column inside the tile
          s = row_s * __shfl_sync(0xffffffffu, swr[col >> 5], col & 31);
        }
        v[i] = __uint_as_float(raw[i]) * s;
      }
      if (has_bias) {
#pragma unroll
        for (int i = 0; i < E::kAccColsPerChunk; ++i) {
          const int col = acc_c0 + i;
          v[i] += __shfl_sync(0xffffffffu, biasr[col >> 5], col & 31);
        }
      }
      float o[32];
      if constexpr (EPI == SPG_EPI_SWIGLU) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float gate = v[2 * j], up = v[2 * j + 1];
          o[j] = __fdividef(gate, 1.f + __expf(-gate)) * up;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) o[j] = v[j];
        if constexpr (EPI == SPG_EPI_ADD) {
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const uint32_t w[4] = {res_cur[g].x, res_cur[g].y, res_cur[g].z, res_cur[g].w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              o[g * 8 + 2 * h] += __uint_as_float(w[h] << 16);
              o[g * 8 + 2 * h + 1] += __uint_as_float(w[h] & 0xFFFF0000u);
            }
          }
#pragma unroll
          for (int g = 0; g < 4; ++g) res_cur[g] = res_next[g];
        }
      }
      // Stage the 32 x 32 bf16 block (64-byte swizzle) and TMA-store it.
      uint8_t* sbuf = stage0 + (chunk_ctr & 1) * E::kBufBytes;
      ++chunk_ctr;
      if (lane == 0) bulk_wait_read<1>();
      __syncwarp();
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        uint4 pk;
        pk.x = pack_bf16x2(o[jj * 8 + 0], o[jj * 8 + 1]);
        pk.y = pack_bf16x2(o[jj * 8 + 2], o[jj * 8 + 3]);
        pk.z = pack_bf16x2(o[jj * 8 + 4], o[jj * 8 + 5]);
        pk.w = pack_bf16x2(o[jj * 8 + 6], o[jj * 8 + 7]);
        const int phys = jj ^ ((lane >> 1) & 3);
        *reinterpret_cast<uint4*>(sbuf + lane * 64 + phys * 16) = pk;
      }
      fence_proxy_async_smem();
      __syncwarp();
      const int out_x = (EPI == SPG_EPI_SWIGLU ? n0 / 2 : n0) + c * 32;
      const int out_y = m0 + q * 32;
      if (lane == 0) {
        if (out_y < p.M && out_x < p.n_out) tma_store_3d(tmY, sbuf, out_x, out_y, tc.b);
        bulk_commit();
      }
    }
  }
  if (lane == 0) bulk_wait<0>();
  __syncwarp();
}

}  // namespace spg

namespace spg {

// Side duty of the register-drain epilogue warps: a functor called while
// they wait for the accumulator and between output chunks, which must not
// block.  NoService: none.
struct NoService {
  static constexpr bool kActive = false;
  __device__ __forceinline__ void operator()() {}
};

// Bounded wait for phase `parity` of `bar` that keeps calling svc() while it
// waits.  The warp polls through lane 0, so every decision is warp-uniform;
// once the phase is complete every lane acquires it.
template <typename Svc>
__device__ __forceinline__ bool wait_serving(uint64_t* bar, uint32_t parity, const WaitCtl& ctl,
                                             unsigned int code, Svc& svc) {
  if constexpr (!Svc::kActive) {
    return mbar_wait(bar, parity, ctl, code);
  } else {
    const int lane = threadIdx.x & 31;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
      int st = 0;
      if (lane == 0) {
        if (mbar_test_wait(smem_u32(bar), parity)) {
          st = 1;
        } else if ((i & 15u) == 0) {
          if (*ctl.abort_flag) {
            st = 2;
          } else if (globaltimer_ns() - t0 > ctl.timeout_ns) {
            *ctl.abort_flag = 1;
            atomicCAS(ctl.err, 0u, code);
            st = 2;
          }
        }
      }
      st = __shfl_sync(0xffffffffu, st, 0);
      if (st == 1) {
        // Lane 0's test was the acquire; the shuffle orders nothing, so every
        // lane acquires the completed phase itself before it reads what the
        // phase guards.
        (void)mbar_test_wait(smem_u32(bar), parity);
        __syncwarp();
        return true;
      }
      if (st == 2) return false;
      svc();
    }
  }
}

// Register-drain epilogue for a single TMEM accumulator of 256 columns:
// eight epilogue warps, two per TMEM lane quarter, each owning 128 columns.
// A warp copies its 128 fp32 columns into registers, hands the accumulator
// back to the MMA issuer at once, and only then scales, applies the
// epilogue and stores -- so the next tile's main loop overlaps the math and
// the stores although TMEM holds one accumulator (the rest of TMEM holds the
// block scales of the NVFP4 pipeline).
// ItemFn(item) -> WorkItem (mb offset for this CTA); K-split pieces are
// reduced first as in epilogue_loop.
// Residual by TMA (RES_TMA, linear_add): each 32 x 32 bf16 residual block
// is loaded by a TMA copy into the warp's staging buffer one chunk ahead
// (res_bars: two mbarriers per epilogue warp, one per buffer), the output is
// computed in place and TMA-stored from the same buffer, and the wait for a
// block is one the warp can serve svc() in.
template <int EPI, int SCALE, bool HAS_BIAS, typename ItemFn, typename ArriveEmpty,
          typename Svc = NoService, bool RES_TMA = false>
__device__ __forceinline__ void epilogue_loop_regdrain(const GemmParams& p, const CUtensorMap* tmY,
                                                       uint32_t tmem_base, uint64_t* acc_full,
                                                       ArriveEmpty arrive_empty, uint8_t* epi_smem,
                                                       int item_begin, int item_step, ItemFn item_fn,
                                                       const WaitCtl& ctl, int cta_rank,
                                                       uint64_t* split_bars, int* split_flag,
                                                       uint64_t* copy_bars, uint8_t* ring,
                                                       int ring_bytes, Svc svc = Svc(),
                                                       const CUtensorMap* tmR = nullptr,
                                                       uint64_t* res_bars = nullptr) {
  constexpr int kCols = 128;                 // accumulator columns per warp
  constexpr bool kResTma = RES_TMA && EPI == SPG_EPI_ADD;
  constexpr int kBufBytes = 32 * 64;
  constexpr int kOutChunks = EPI == SPG_EPI_SWIGLU ? 2 : 4;  // 32-wide output chunks
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int e = warp - 2;
  const int q = warp & 3;
  const int half = e >> 2;
  uint8_t* stage0 = epi_smem + (e * 2) * kBufBytes;
  int it = 0;
  int chunk_ctr = 0;
  uint32_t split_phase = 0, copy_phase = 0;
  const int scr_bytes = (ring_bytes / 8) & ~4095;
  const SplitScratch scr{ring + e * scr_bytes, scr_bytes, copy_bars + e, &copy_phase};
  float scalar = 1.f;
  if constexpr (SCALE == kScaleScalar) scalar = __ldg(p.scalar_a) * __ldg(p.scalar_b);
  bool aborted = false;
  int res_inflight = -1;  // chunk index of a residual copy not yet waited for

  for (int item = item_begin; item < p.total_items && !aborted; item += item_step, ++it) {
    const WorkItem tc = item_fn(item);
    // First residual block of the item, into the buffer of its first chunk
    // (whose previous store, two chunks back, must have been read).  For a
    // K-split piece only once it is known to hold the tile's total.
    auto first_residual = [&]() {
      if constexpr (kResTma) {
        if (lane == 0) {
          bulk_wait_read<1>();
          uint64_t* bar = &res_bars[e * 2 + (chunk_ctr & 1)];
          mbar_arrive_expect_tx(bar, kBufBytes);
          tma_load_3d(stage0 + (chunk_ctr & 1) * kBufBytes, tmR, bar, tc.nb * 256 + half * kCols,
                      tc.mb * 128 + q * 32, tc.b);
        }
        res_inflight = chunk_ctr;
        __syncwarp();
      }
    };
    if (tc.split < 0) first_residual();
    if (tc.split >= 0) {
      if (!wait_serving(&acc_full[0], it & 1, ctl, kErrWaitAccFull, svc)) break;
      tc_fence_after();
      const int outcome = split_piece_reduce<256>(
          p, tmem_base + (uint32_t(q * 32) << 16), tc, cta_rank, q * 32 + lane, half * kCols,
          kCols, tc.mb * 128 + q * 32 < p.M, split_bars, split_flag, split_phase, scr, ctl);
      split_phase ^= 1u;
      if (outcome < 0) break;
      if (outcome == 0) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_empty(0);
        continue;
      }
      first_residual();
    }
    const bool have_k = tc.split >= 0 || tc.kb_end > tc.kb_begin;
    const int m0 = tc.mb * 128;
    const int n_acc0 = tc.nb * 256 + half * kCols;  // first accumulator column of this warp
    const int m = m0 + q * 32 + lane;
    const bool row_ok = m < p.M;
    float row_s = scalar;
    if constexpr (SCALE == kScaleRow) row_s = row_ok ? __ldg(p.row_scale + m) : 0.f;
    float swr[kCols / 32];
    if constexpr (SCALE == kScaleRow) {
#pragma unroll
      for (int j = 0; j < kCols / 32; ++j) {
        const int n = n_acc0 + 32 * j + lane;
        swr[j] = n < p.N ? __ldg(p.col_scale + n) : 0.f;
      }
    }
    // The bias is loaded per chunk (one or two registers) to leave room for
    // the 128 accumulator registers; its code exists only in the HAS_BIAS
    // instantiation.
    constexpr bool has_bias = HAS_BIAS;
    uint4 res_cur[4];
    if constexpr (EPI == SPG_EPI_ADD && !kResTma) load_residual_chunk(p, m, n_acc0, row_ok, res_cur);

    if (tc.split < 0) {
      if (!wait_serving(&acc_full[0], it & 1, ctl, kErrWaitAccFull, svc)) break;
      tc_fence_after();
    }
    uint32_t acc[kCols];
    const uint32_t t_row = tmem_base + (uint32_t(q * 32) << 16) + uint32_t(half * kCols);
    if (have_k) {
#pragma unroll
      for (int j = 0; j < kCols / 32; ++j)
        tmem_ld_32x32b_x32(t_row + 32 * j, *reinterpret_cast<uint32_t(*)[32]>(&acc[32 * j]));
      tmem_wait_ld();
    } else {
#pragma unroll
      for (int i = 0; i < kCols; ++i) acc[i] = 0u;
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) arrive_empty(0);

#pragma unroll
    for (int c = 0; c < kOutChunks; ++c, ++chunk_ctr) {
      svc();
      float o[32];
      if constexpr (EPI == SPG_EPI_SWIGLU) {
        float biasr[2] = {0.f, 0.f};
        if (has_bias) {
          biasr[0] = load_bias(p, n_acc0 + c * 64 + lane);
          biasr[1] = load_bias(p, n_acc0 + c * 64 + 32 + lane);
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int cg = c * 64 + 2 * j;  // gate column inside this warp's 128
          float sg = row_s, su = row_s;
          if constexpr (SCALE == kScaleRow) {
            sg *= __shfl_sync(0xffffffffu, swr[cg >> 5], cg & 31);
            su *= __shfl_sync(0xffffffffu, swr[(cg + 1) >> 5], (cg + 1) & 31);
          }
          float gate = __uint_as_float(acc[cg]) * sg;
          float up = __uint_as_float(acc[cg + 1]) * su;
          if (has_bias) {
            gate += __shfl_sync(0xffffffffu, biasr[(2 * j) >> 5], (2 * j) & 31);
            up += __shfl_sync(0xffffffffu, biasr[(2 * j + 1) >> 5], (2 * j + 1) & 31);
          }
          o[j] = __fdividef(gate, 1.f + __expf(-gate)) * up;
        }
      } else {
        const float bias_c = has_bias ? load_bias(p, n_acc0 + 32 * c + lane) : 0.f;
        uint4 res_next[4];
        if constexpr (kResTma) {
          // This chunk's residual block (serving svc() while it lands), then
          // the next one into the other buffer once that buffer's store has
          // been read.
          if (!wait_serving(&res_bars[e * 2 + (chunk_ctr & 1)], uint32_t(chunk_ctr >> 1) & 1u,
                            ctl, kErrWaitFull, svc)) {
            aborted = true;
            break;
          }
          res_inflight = -1;
          if (c + 1 < kOutChunks) {
            if (lane == 0) {
              bulk_wait_read<0>();
              uint64_t* bar = &res_bars[e * 2 + ((chunk_ctr + 1) & 1)];
              mbar_arrive_expect_tx(bar, kBufBytes);
              tma_load_3d(stage0 + ((chunk_ctr + 1) & 1) * kBufBytes, tmR, bar,
                          n_acc0 + 32 * (c + 1), m0 + q * 32, tc.b);
            }
            res_inflight = chunk_ctr + 1;
            __syncwarp();
          }
          const uint8_t* rbuf = stage0 + (chunk_ctr & 1) * kBufBytes + lane * 64;
#pragma unroll
          for (int g = 0; g < 4; ++g)
            res_cur[g] = *reinterpret_cast<const uint4*>(rbuf + ((g ^ ((lane >> 1) & 3)) * 16));
        } else if constexpr (EPI == SPG_EPI_ADD) {
          if (c + 1 < kOutChunks) load_residual_chunk(p, m, n_acc0 + 32 * (c + 1), row_ok, res_next);
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          float s = row_s;
          if constexpr (SCALE == kScaleRow) s *= __shfl_sync(0xffffffffu, swr[c], j);
          o[j] = __uint_as_float(acc[c * 32 + j]) * s;
          if (has_bias) o[j] += __shfl_sync(0xffffffffu, bias_c, j);
        }
        if constexpr (EPI == SPG_EPI_ADD) {
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const uint32_t w[4] = {res_cur[g].x, res_cur[g].y, res_cur[g].z, res_cur[g].w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              o[g * 8 + 2 * h] += __uint_as_float(w[h] << 16);
              o[g * 8 + 2 * h + 1] += __uint_as_float(w[h] & 0xFFFF0000u);
            }
          }
          if constexpr (!kResTma) {
#pragma unroll
            for (int g = 0; g < 4; ++g) res_cur[g] = res_next[g];
          }
        }
      }
      uint8_t* sbuf = stage0 + (chunk_ctr & 1) * kBufBytes;
      if constexpr (!kResTma) {
        if (lane == 0) bulk_wait_read<1>();
      }
      __syncwarp();
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        uint4 pk;
        pk.x = pack_bf16x2(o[jj * 8 + 0], o[jj * 8 + 1]);
        pk.y = pack_bf16x2(o[jj * 8 + 2], o[jj * 8 + 3]);
        pk.z = pack_bf16x2(o[jj * 8 + 4], o[jj * 8 + 5]);
        pk.w = pack_bf16x2(o[jj * 8 + 6], o[jj * 8 + 7]);
        const int phys = jj ^ ((lane >> 1) & 3);
        *reinterpret_cast<uint4*>(sbuf + lane * 64 + phys * 16) = pk;
      }
      fence_proxy_async_smem();
      __syncwarp();
      const int out_x = (EPI == SPG_EPI_SWIGLU ? n_acc0 / 2 : n_acc0) + c * 32;
      const int out_y = m0 + q * 32;
      if (lane == 0) {
        if (out_y < p.M && out_x < p.n_out) tma_store_3d(tmY, sbuf, out_x, out_y, tc.b);
        bulk_commit();
      }
    }
  }
  if constexpr (kResTma) {
    // No residual copy may still be writing the staging buffers at exit.
    if (res_inflight >= 0 && lane == 0)
      mbar_wait_drain(&res_bars[e * 2 + (res_inflight & 1)], uint32_t(res_inflight >> 1) & 1u,
                      p.drain_ns, p.err);
  }
  if constexpr (kResTma) {
    // No residual copy may still be writing the staging buffers at exit.
    if (res_inflight >= 0 && lane == 0)
      mbar_wait_drain(&res_bars[e * 2 + (res_inflight & 1)], uint32_t(res_inflight >> 1) & 1u,
                      p.drain_ns, p.err);
  }
  if (lane == 0) bulk_wait<0>();
  __syncwarp();
}

}  // namespace spg
