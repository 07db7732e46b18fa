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

// K-split piece of a tile (two-SM kernels), one epilogue warp's share.  The
// warp owns TMEM lane quarter q (rows q*32 .. q*32+31 of the CTA's 128; t_row
// addresses column 0 of the tile's accumulator in that quarter) and
// accumulator columns [c0, c0 + ncols), which its epilogue processes in
// chunks of CW columns.
//  1. It writes its partial sums of those columns to the piece's slice.
//  2. After one fence, lane i counts the piece's arrival on the counter of
//     chunk i (all chunks at once, one round trip).
//  3. For every chunk where this piece arrived last, it adds all pieces in
//     split order (its own from TMEM, so the total does not depend on the
//     arrival order) and writes the total back to TMEM.
// Returns the mask of chunks whose total this warp now holds (bit i: chunk
// i); the caller runs the epilogue on exactly those.  The chunks of a tile
// finish in whichever pieces arrive last for them, so the reduction and the
// epilogue spread over the pieces; nothing waits for another CTA or warp.
// rows_live == false (every row of the quarter past the output): only the
// arrivals, so the counters still return to zero.  G: float4 groups of a
// 32-column block loaded at once per other piece (8 or 4, trading registers
// against round trips).  At most 4 pieces per tile.
template <int BN, int CW, int G>
__device__ __forceinline__ uint32_t split_piece_finish(const GemmParams& p, uint32_t t_row,
                                                       const WorkItem& tc, int rank, int q,
                                                       int c0, int ncols, bool rows_live) {
  static_assert(CW == 32 || CW == 64, "epilogue chunks are 32 or 64 columns");
  static_assert(G == 4 || G == 8, "a 32-column block is 8 float4 groups");
  const int lane = threadIdx.x & 31;
  const bool have_k = tc.kb_end > tc.kb_begin;
  float4* own = split_slice(p, tc.tail, tc.split, rank, BN);
#pragma unroll 1
  for (int c = c0; rows_live && c < c0 + ncols; c += 32) {
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
  __threadfence();
  __syncwarp();
  const int nch = ncols / CW;
  int last = 0;
  if (lane < nch) {
    const int before =
        split_arrive(p, split_counter_index(tc.tail, rank, q, (c0 + lane * CW) / CW, BN, CW));
    last = before == p.split_k - 1 ? 1 : 0;
    __threadfence();
  }
  // Warps with no live row still count their arrivals (so every counter
  // returns to zero) but finish nothing.
  const uint32_t mask = rows_live ? __ballot_sync(0xffffffffu, last) : 0u;
  if (mask == 0u) return 0u;
  __syncwarp();
  __threadfence();
  const int own_s = tc.split;
#pragma unroll 1
  for (int i = 0; i < nch; ++i) {
    if (!((mask >> i) & 1u)) continue;
#pragma unroll 1
    for (int sb = 0; sb < CW; sb += 32) {
      const int c = c0 + i * CW + sb;
      uint32_t r[32];
      if (have_k) {
        tmem_ld_32x32b_x32(t_row + c, r);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = 0u;
      }
#pragma unroll
      for (int g0 = 0; g0 < 8; g0 += G) {
        // The other pieces: slot k holds piece k, or k + 1 past this one.
        float4 part[3][G];
#pragma unroll
        for (int k = 0; k < 3; ++k) {
          const int s2 = k + (k >= own_s ? 1 : 0);
          if (s2 < p.split_k) {
            const float4* src =
                split_slice(p, tc.tail, s2, rank, BN) + split_block_index(c >> 5, q) + lane;
#pragma unroll
            for (int g = 0; g < G; ++g) part[k][g] = __ldcg(src + (g0 + g) * 32);
          } else {
#pragma unroll
            for (int g = 0; g < G; ++g) part[k][g] = make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const int j = 4 * (g0 + g);
          const float4 mine = make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                                          __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
          float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int k = 0; k < 3; ++k) {
            if (k == own_s) {
              t.x += mine.x; t.y += mine.y; t.z += mine.z; t.w += mine.w;
            }
            if (k + (k >= own_s ? 1 : 0) < p.split_k) {
              t.x += part[k][g].x; t.y += part[k][g].y; t.z += part[k][g].z; t.w += part[k][g].w;
            }
          }
          if (own_s == 3) {
            t.x += mine.x; t.y += mine.y; t.z += mine.z; t.w += mine.w;
          }
          r[j] = __float_as_uint(t.x);
          r[j + 1] = __float_as_uint(t.y);
          r[j + 2] = __float_as_uint(t.z);
          r[j + 3] = __float_as_uint(t.w);
        }
      }
      tmem_st_32x32b_x32(t_row + c, r);
    }
  }
  tmem_wait_st();
  return mask;
}

// K split inside a thread-block cluster (one-CTA kernel): the split_k
// pieces of a tile run as the CTAs of one cluster, cluster rank = piece, and
// are reduced through distributed shared memory instead of a global
// workspace.  Each CTA runs exactly one piece, so once its accumulator is
// full its operand ring is idle; chunk i of the tile is finished by the CTA
// of rank i mod split_k, whose ring receives every piece's partial sums of
// that chunk.
//   free:  one arrival per epilogue warp of the cluster once its CTA's
//          accumulator is full (its ring is idle and may receive)
//   ready: one arrival per epilogue warp of the cluster once its partial
//          sums are written to their owners (or it gave up); a CTA leaves
//          only after its ready phase completed, so no write into it is
//          still in flight
// Every warp gives both arrivals exactly once (cluster_piece_finish, or the
// kernel's exit path for a warp that never got there), so neither phase
// waits on a warp that has left.
struct ClusterSplit {
  uint64_t* free_bar;
  uint64_t* ready;
  uint8_t* ring;     // this CTA's operand ring (receive area)
  bool arrived;      // this warp has given its free and ready arrivals
  // Cluster rank of the CTA holding piece s of this CTA's rows:
  // s * rank_stride + rank_offset (one-CTA tiles 1, 0; CTA pairs 2 and the
  // CTA's side of its pair).
  uint32_t rank_stride, rank_offset;
  __device__ __forceinline__ uint32_t peer(int s) const {
    return uint32_t(s) * rank_stride + rank_offset;
  }
};

// Exit path of an epilogue warp under a cluster K split: give the free and
// ready arrivals if the reduction never ran (a time-out), then wait (drain
// bound) until every warp of the cluster has finished writing into this CTA.
__device__ __forceinline__ void cluster_split_exit(const GemmParams& p, ClusterSplit& cs) {
  const int lane = threadIdx.x & 31;
  if (!cs.arrived) {
    __syncwarp();
    if (lane == 0) {
      for (int s = 0; s < p.split_k; ++s)
        mbar_arrive_cluster(mapa_shared(smem_u32(cs.free_bar), cs.peer(s)));
      for (int s = 0; s < p.split_k; ++s)
        mbar_arrive_cluster(mapa_shared(smem_u32(cs.ready), cs.peer(s)));
    }
    cs.arrived = true;
  }
  if (lane == 0) mbar_wait_drain_cluster(cs.ready, 0, p.drain_ns, p.err);
  __syncwarp();
}

// One epilogue warp's share of the cluster reduction of a K-split piece.
// The warp owns TMEM lane quarter q (t_row: column 0 of the accumulator in
// that quarter).  Once every CTA of the cluster has a full accumulator
// (free), it writes its rows' partial sums of every chunk into the chunk's
// owner (st.shared::cluster, its own CTA included; two TMEM blocks loaded
// per wait), arrives on every CTA's ready barrier and waits for its own;
// then, for each chunk this CTA owns, it adds the pieces in split order
// (piece 0 first) and writes the total back to TMEM.
// Returns the mask of chunks whose total this warp now holds (bit i: chunk
// i), 0 after a time-out.  An empty K range (have_k false) contributes
// zeros.
template <int BN, int CW>
__device__ __forceinline__ uint32_t cluster_piece_finish(const GemmParams& p, uint32_t t_row,
                                                         const WorkItem& tc, int q,
                                                         ClusterSplit& cs, const WaitCtl& ctl) {
  static_assert(CW == 32 || CW == 64, "epilogue chunks are 32 or 64 columns");
  constexpr int kSub = CW / 32;
  constexpr int kChunks = BN / CW;
  constexpr int kBlocks = BN / 32;
  const int lane = threadIdx.x & 31;
  const int S = p.split_k;
  const int rank = tc.split;
  const bool have_k = tc.kb_end > tc.kb_begin;
  // Receive area (cluster_recv_bytes): per owned chunk (li: its index among
  // the owner's chunks), 32-column sub-block sb, source piece src and lane
  // quarter q one 4 KB block of 32 rows x 32 fp32, stored group-major: the
  // 16-byte group g (columns 4g .. 4g+3) of the warp's 32 rows is one
  // contiguous 512-byte run, so each warp-wide store to another CTA moves
  // whole 128-byte lines and each local load is conflict-free.  Byte offset
  // of group g of this lane's row:
  auto slot = [&](int li, int sb, int src, int g) {
    return uint32_t((((li * kSub + sb) * S + src) * 4 + q) * 4096 + g * 512 + lane * 16);
  };
  auto load_block = [&](int b, uint32_t (&r)[32]) {
    if (have_k) {
      tmem_ld_32x32b_x32(t_row + b * 32, r);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) r[j] = 0u;
    }
  };
  const uint32_t ring_base = smem_u32(cs.ring);
  auto send_block = [&](int b, const uint32_t (&r)[32]) {
    const int i = b / kSub;
    const uint32_t dst = mapa_shared(ring_base, cs.peer(i % S));
#pragma unroll
    for (int g = 0; g < 8; ++g)
      st_cluster_v4(dst + slot(i / S, b % kSub, rank, g), r[4 * g], r[4 * g + 1], r[4 * g + 2],
                    r[4 * g + 3]);
  };
  __syncwarp();
  if (lane == 0)
    for (int s = 0; s < S; ++s) mbar_arrive_cluster(mapa_shared(smem_u32(cs.free_bar), cs.peer(s)));
  const bool can_send =
      __all_sync(0xffffffffu, mbar_wait_cluster(cs.free_bar, 0, ctl, kErrWaitFull));
  if (can_send) {
    static_assert(kBlocks % 2 == 0, "blocks go out in pairs");
#pragma unroll 1
    for (int b = 0; b < kBlocks; b += 2) {
      uint32_t r0[32], r1[32];
      load_block(b, r0);
      load_block(b + 1, r1);
      if (have_k) tmem_wait_ld();
      send_block(b, r0);
      send_block(b + 1, r1);
    }
  }
  fence_acq_rel_cluster();
  __syncwarp();
  if (lane == 0)
    for (int s = 0; s < S; ++s) mbar_arrive_cluster(mapa_shared(smem_u32(cs.ready), cs.peer(s)));
  cs.arrived = true;
  const bool ok = can_send &&
                  __all_sync(0xffffffffu, mbar_wait_cluster(cs.ready, 0, ctl, kErrWaitFull));
  if (!ok) return 0u;
  uint32_t mask = 0u;
#pragma unroll 1
  for (int i = rank; i < kChunks; i += S) {
    mask |= 1u << i;
#pragma unroll 1
    for (int sb = 0; sb < kSub; ++sb) {
      float t[32];
#pragma unroll 1
      for (int src = 0; src < S; ++src) {
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const float4 v = *reinterpret_cast<const float4*>(cs.ring + slot(i / S, sb, src, g));
          if (src == 0) {
            t[4 * g] = v.x; t[4 * g + 1] = v.y; t[4 * g + 2] = v.z; t[4 * g + 3] = v.w;
          } else {
            t[4 * g] += v.x; t[4 * g + 1] += v.y; t[4 * g + 2] += v.z; t[4 * g + 3] += v.w;
          }
        }
      }
      uint32_t r[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(t[j]);
      tmem_st_32x32b_x32(t_row + (i * kSub + sb) * 32, r);
    }
  }
  tmem_wait_st();
  return mask;
}

// ItemFn(item) -> WorkItem with mb already offset for this CTA's rows (a
// whole tile has n_off = 0, width = BN); the loop runs over items
// [item_begin, item_end) with stride item_step.  ArriveEmpty(buf) releases
// accumulator buffer `buf` to the MMA issuer.  K-split pieces go through
// split_piece_finish (two-SM kernels, global workspace; cta_rank: this CTA's
// rank in the pair) or, with CLUSTER_SPLIT (one-CTA kernel, one piece per
// CTA of a cluster), cluster_piece_finish with *csplit, and then run the
// epilogue on the chunks whose total they hold.
// RES_TMA (linear_add): the residual of each 32 x 32 output block comes by a
// TMA copy (tmR, 32 x 32 boxes, the output's swizzle) into the warp's
// staging buffer, one chunk ahead -- the first chunk's before the
// accumulator is ready -- and the output is computed in place and stored
// from the same buffer (res_bars: two mbarriers per epilogue warp, one per
// buffer).  Without it each thread loads its row's residual with 16-byte
// loads, 32 rows apart across the warp.  On the CTA's last item nothing
// follows to hide the chunk-by-chunk copies behind, so once that item's
// accumulator is full (every MMA, hence every read of the operand ring, is
// done, and no load into the ring remains) all of its residual blocks are
// requested at once into the idle ring (idle_ring: BN/32 x 2 KB per warp)
// and waited for together: one memory round trip instead of one per chunk.
template <int EPI, int SCALE, int BN, typename ItemFn, typename ArriveEmpty, bool RES_TMA = false,
          bool CLUSTER_SPLIT = false>
__device__ __forceinline__ void epilogue_loop(const GemmParams& p, const CUtensorMap* tmY,
                                              uint32_t tmem_base, uint64_t* acc_full,
                                              ArriveEmpty arrive_empty, uint8_t* epi_smem,
                                              int item_begin, int item_end, int item_step,
                                              ItemFn item_fn, const WaitCtl& ctl, int cta_rank,
                                              const CUtensorMap* tmR = nullptr,
                                              uint64_t* res_bars = nullptr,
                                              uint8_t* idle_ring = nullptr,
                                              ClusterSplit* csplit = nullptr) {
  using E = EpilogueCfg<EPI, SCALE, BN>;
  constexpr bool kResTma = RES_TMA && EPI == SPG_EPI_ADD;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int e = warp - 2;
  const int q = warp & 3;  // TMEM lane quarter this warp may access
  uint8_t* stage0 = epi_smem + (e * 2) * E::kBufBytes;
  int it = 0;
  int chunk_ctr = 0;
  float scalar = 1.f;
  if constexpr (SCALE == kScaleScalar) scalar = __ldg(p.scalar_a) * __ldg(p.scalar_b);
  // TMA residual: buffer of the copy in flight (-1: none) and the parity
  // each buffer's barrier completes next.
  int res_inflight = -1;
  uint32_t res_ph = 0;
  auto res_load = [&](int buf, int x, int y, int b) {
    if (lane == 0) {
      uint64_t* bar = &res_bars[e * 2 + buf];
      mbar_arrive_expect_tx(bar, E::kBufBytes);
      tma_load_3d(stage0 + buf * E::kBufBytes, tmR, bar, x, y, b);
    }
    res_inflight = buf;
    __syncwarp();
  };
  bool aborted = false;

  for (int item = item_begin; item < item_end && !aborted; item += item_step, ++it) {
    const int buf = it & 1;
    const uint32_t acc_ph = (it >> 1) & 1;
    const WorkItem tc = item_fn(item);
    const uint32_t t_row = tmem_base + (uint32_t(q * 32) << 16) + uint32_t(buf * BN);
    // Chunks this warp finishes: all of them, or those whose K-split total
    // it holds.
    uint32_t own_mask = 0xffffffffu;
    if (tc.split >= 0 && CLUSTER_SPLIT) {
      // The chunks of rank tc.split: known before the reduction, which runs
      // below, after this item's epilogue operands have been requested.
      own_mask = 0u;
      for (int i = tc.split; i < 32; i += p.split_k) own_mask |= 1u << i;
    } else if (tc.split >= 0) {
      if (!mbar_wait(&acc_full[buf], acc_ph, ctl, kErrWaitAccFull)) break;
      tc_fence_after();
      own_mask = split_piece_finish<BN, E::kAccColsPerChunk, 8>(
          p, t_row, tc, cta_rank, q, 0, tc.width, tc.mb * 128 + q * 32 < p.M);
      if (own_mask == 0u) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_empty(buf);
        continue;
      }
    }
    const bool split_item = tc.split >= 0;
    // A chunk's residual is loaded one chunk ahead (the first before the
    // accumulator is ready) unless a global-workspace K split decides the
    // chunks only after its reduction.
    const bool res_ahead = !split_item || CLUSTER_SPLIT;
    // After a K-split reduction TMEM holds the total of all pieces.
    const bool have_k = tc.split >= 0 || tc.kb_end > tc.kb_begin;
    const int m0 = tc.mb * 128;
    const int n0 = tc.nb * BN + tc.n_off;  // first accumulator column of the item (global)
    const int nch = tc.width / E::kAccColsPerChunk;
    const int m = m0 + q * 32 + lane;
    const bool row_ok = m < p.M;
    own_mask &= nch >= 32 ? 0xffffffffu : ((1u << nch) - 1u);
    const int last_c = 31 - __clz(own_mask);  // the accumulator goes back after this chunk

    // Epilogue operands, requested before the accumulator is ready.
    float row_s = scalar;
    if constexpr (SCALE == kScaleRow) row_s = row_ok ? __ldg(p.row_scale + m) : 0.f;
    // Column scales and bias of one chunk per lane (lane j: column 32 i + j
    // of the chunk's i-th 32 columns), the next chunk's requested while the
    // current one is processed.  The chunk loop stays rolled: unrolled over
    // all chunks its code outgrew the instruction cache, and with every CTA
    // of a wave in the same chunk at once the refetches serialized.
    constexpr int kCw = E::kAccColsPerChunk / 32;
    const bool has_bias = p.bias_kind != 0;
    auto chunk_cols = [&](int c, float (&sw)[kCw], float (&bi)[kCw]) {
#pragma unroll
      for (int j = 0; j < kCw; ++j) {
        const int col = c * E::kAccColsPerChunk + 32 * j;  // inside the item
        const int n = n0 + col + lane;
        sw[j] = 1.f;
        if constexpr (SCALE == kScaleRow) sw[j] = (col < tc.width && n < p.N) ? __ldg(p.col_scale + n) : 0.f;
        bi[j] = (has_bias && col < tc.width) ? load_bias(p, n) : 0.f;
      }
    };
    float swc[kCw], biasc[kCw];
    const int c_first = own_mask == 0xffffffffu ? 0 : __ffs(own_mask) - 1;
    if (c_first >= 0 && c_first < nch) chunk_cols(c_first, swc, biasc);
    uint4 res_cur[4];
    // The last item's residual comes whole into the idle operand ring.
    const bool res_bulk = kResTma && !split_item && idle_ring != nullptr &&
                          item + item_step >= item_end;
    uint8_t* ring_w = idle_ring + e * (E::kChunks * E::kBufBytes);
    if constexpr (kResTma) {
      // The first chunk's block, into the buffer whose store of two chunks
      // back must have been read.
      if (!split_item && !res_bulk) {
        if (lane == 0) bulk_wait_read<1>();
        res_load(chunk_ctr & 1, n0, m0 + q * 32, tc.b);
      }
    } else if constexpr (EPI == SPG_EPI_ADD) {
      if (res_ahead && c_first >= 0 && c_first < nch)
        load_residual_chunk(p, m, n0 + c_first * 32, row_ok, res_cur);
    }

    if (tc.split < 0 || CLUSTER_SPLIT) {
      if (!mbar_wait(&acc_full[buf], acc_ph, ctl, kErrWaitAccFull)) break;
      tc_fence_after();
    }
    if constexpr (CLUSTER_SPLIT) {
      // Every CTA of the cluster takes part, including one that finishes no
      // chunk; 0 back means the reduction timed out.
      if (split_item &&
          cluster_piece_finish<BN, E::kAccColsPerChunk>(p, t_row, tc, q, *csplit, ctl) == 0u &&
          own_mask != 0u)
        break;
    }
    if constexpr (kResTma) {
      if (res_bulk) {
        if (lane == 0) {
          uint64_t* bar = &res_bars[e * 2];
          mbar_arrive_expect_tx(bar, uint32_t(nch * E::kBufBytes));
          for (int c = 0; c < nch; ++c)
            tma_load_3d(ring_w + c * E::kBufBytes, tmR, bar, n0 + 32 * c, m0 + q * 32, tc.b);
        }
        res_inflight = 0;
        __syncwarp();
        if (!mbar_wait(&res_bars[e * 2], res_ph & 1u, ctl, kErrWaitFull)) break;
        res_ph ^= 1u;
        res_inflight = -1;
      }
    }

#pragma unroll 1
    for (int c = 0; c < E::kChunks; ++c) {
      if (c >= nch) break;
      if (!((own_mask >> c) & 1u)) continue;
      const int acc_c0 = c * E::kAccColsPerChunk;
      // The next chunk this warp finishes: its column scales and bias now.
      float swn[kCw], biasn[kCw];
      const uint32_t later = (c + 1 < 32) ? (own_mask >> (c + 1)) : 0u;
      const int c_next = later ? c + __ffs(later) : -1;
      if (c_next >= 0 && c_next < nch) chunk_cols(c_next, swn, biasn);
      if constexpr (EPI == SPG_EPI_ADD) {
        // A global-workspace K-split piece finishes scattered chunks: load
        // each one's residual.
        if (!res_ahead) load_residual_chunk(p, m, n0 + acc_c0, row_ok, res_cur);
      }
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
      if constexpr (kResTma) {
        if (res_bulk) {
          const uint8_t* rbuf = ring_w + c * E::kBufBytes + lane * 64;
#pragma unroll
          for (int g = 0; g < 4; ++g)
            res_cur[g] = *reinterpret_cast<const uint4*>(rbuf + ((g ^ ((lane >> 1) & 3)) * 16));
        } else if (!split_item) {
          // This chunk's block, then the next one into the other buffer once
          // that buffer's store has been read.
          const int rb = chunk_ctr & 1;
          if (!mbar_wait(&res_bars[e * 2 + rb], (res_ph >> rb) & 1u, ctl, kErrWaitFull)) {
            aborted = true;
            break;
          }
          res_ph ^= 1u << rb;
          res_inflight = -1;
          if (c + 1 < nch) {
            if (lane == 0) bulk_wait_read<0>();
            res_load(rb ^ 1, n0 + acc_c0 + 32, m0 + q * 32, tc.b);
          }
          const uint8_t* rbuf = stage0 + rb * E::kBufBytes + lane * 64;
#pragma unroll
          for (int g = 0; g < 4; ++g)
            res_cur[g] = *reinterpret_cast<const uint4*>(rbuf + ((g ^ ((lane >> 1) & 3)) * 16));
        }
      } else if constexpr (EPI == SPG_EPI_ADD) {
        if (res_ahead && c_next >= 0 && c_next < nch)
          load_residual_chunk(p, m, n0 + c_next * 32, row_ok, res_next);
      }
      if (have_k) tmem_wait_ld();
      if (c == last_c && item + item_step < item_end) {
        // Every column of this accumulator buffer has been read: hand it back
        // (after the CTA's last item no MMA waits for it, and the cluster-
        // scope arrival would only delay the last stores).
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
          s = row_s * __shfl_sync(0xffffffffu, swc[(col - acc_c0) >> 5], col & 31);
        }
        v[i] = __uint_as_float(raw[i]) * s;
      }
      if (has_bias) {
#pragma unroll
        for (int i = 0; i < E::kAccColsPerChunk; ++i) {
          const int col = acc_c0 + i;
          v[i] += __shfl_sync(0xffffffffu, biasc[(col - acc_c0) >> 5], col & 31);
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
          if constexpr (!kResTma) {
#pragma unroll
            for (int g = 0; g < 4; ++g) res_cur[g] = res_next[g];
          }
        }
      }
      // Stage the 32 x 32 bf16 block (64-byte swizzle) and TMA-store it.
      // The buffer's store of two chunks back must have been read (the TMA
      // residual path waited for that before loading this chunk's block).
      uint8_t* sbuf = stage0 + (chunk_ctr & 1) * E::kBufBytes;
      ++chunk_ctr;
      if (!kResTma || split_item || res_bulk) {
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
      const int out_x = (EPI == SPG_EPI_SWIGLU ? n0 / 2 : n0) + c * 32;
      const int out_y = m0 + q * 32;
      if (lane == 0) {
        if (out_y < p.M && out_x < p.n_out) tma_store_3d(tmY, sbuf, out_x, out_y, tc.b);
        bulk_commit();
      }
      if (c_next >= 0 && c_next < nch) {
#pragma unroll
        for (int j = 0; j < kCw; ++j) {
          swc[j] = swn[j];
          biasc[j] = biasn[j];
        }
      }
    }
  }
  if constexpr (kResTma) {
    // No residual copy may still be writing the staging buffers at exit.
    if (res_inflight >= 0 && lane == 0)
      mbar_wait_drain(&res_bars[e * 2 + res_inflight], (res_ph >> res_inflight) & 1u, p.drain_ns,
                      p.err);
  }
  if (lane == 0) bulk_wait<0>();
  __syncwarp();
}

}  // namespace spg

namespace spg {

// Epilogue of the swapped pair tile (narrow T): TMEM lane = weight row n
// (the output column), TMEM column = token t (the output row).  Each thread
// owns one weight row; a 32-token chunk of its accumulator row becomes a
// column of a 32 x 32 bf16 output block, staged through 64-byte-swizzled
// shared memory (row t of the block = 64 bytes; each warp writes one row per
// token with conflict-free 2-byte stores) and TMA-stored.  Scales: p.row_scale
// holds the weight scales (per lane), p.col_scale the token scales (per
// column); bias per weight row.  The residual [T, N] arrives by TMA (tmR:
// the same 32 x 32 box and swizzle as the output) into this warp's blocks
// of res_smem (one 2 KB block per chunk), requested before the accumulator
// is ready and completing on res_bars[warp].  p.M = weight rows (N of the
// layer), p.N = tokens (T).  K-split pieces go through split_piece_finish
// like the unswapped tile.
template <int EPI, int BN, typename ItemFn, typename ArriveEmpty, int SCALE = kScaleRow,
          bool CLUSTER_SPLIT = false>
__device__ __forceinline__ void epilogue_loop_swap(const GemmParams& p, const CUtensorMap* tmY,
                                                   uint32_t tmem_base, uint64_t* acc_full,
                                                   ArriveEmpty arrive_empty, uint8_t* epi_smem,
                                                   int item_begin, int item_end, int item_step,
                                                   ItemFn item_fn, const WaitCtl& ctl,
                                                   int cta_rank, const CUtensorMap* tmR,
                                                   uint64_t* res_bars, uint8_t* res_smem,
                                                   ClusterSplit* csplit = nullptr) {
  static_assert(EPI != SPG_EPI_SWIGLU, "the swapped tile has no SwiGLU epilogue");
  constexpr int kBufBytes = 32 * 64;
  constexpr int kChunks = BN / 32;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int e = warp - 2;
  const int q = warp & 3;  // TMEM lane quarter this warp may access
  uint8_t* stage0 = epi_smem + (e * 2) * kBufBytes;
  uint8_t* res0 = res_smem + e * kChunks * kBufBytes;
  uint64_t* res_bar = res_bars + e;
  uint32_t res_phase = 0;
  bool res_inflight = false;
  int it = 0;
  int chunk_ctr = 0;
  const int n_w = p.M;  // weight rows = output columns
  const int n_t = p.N;  // tokens = output rows
  // Per-tensor scales (kScaleScalar): the product sA * sB stands in for the
  // weight row's scale and every token scale is 1.
  float scalar = 1.f;
  if constexpr (SCALE == kScaleScalar) scalar = __ldg(p.scalar_a) * __ldg(p.scalar_b);

  for (int item = item_begin; item < item_end; item += item_step, ++it) {
    const int buf = it & 1;
    const uint32_t acc_ph = (it >> 1) & 1;
    const WorkItem tc = item_fn(item);
    const uint32_t t_row = tmem_base + (uint32_t(q * 32) << 16) + uint32_t(buf * BN);
    const int n0 = tc.mb * 128 + q * 32;  // this warp's first weight row
    const int n = n0 + lane;
    const bool live = n0 < n_w;
    const bool n_ok = n < n_w;
    const int t0 = tc.nb * BN;  // first token of the tile

    // Epilogue operands, requested before the accumulator is ready: the
    // weight scale and bias of this thread's row, the token scales (token
    // t0 + 32 c + lane in sar[c]) and the residual of the first chunk.
    float sw = 0.f;
    if (n_ok) sw = SCALE == kScaleRow ? __ldg(p.row_scale + n) : scalar;
    float bias = 0.f;
    if (p.bias_kind != 0 && n_ok) {
      if (p.bias_kind == 1) {
        bias = __uint_as_float(uint32_t(__ldg(static_cast<const unsigned short*>(p.bias) + n))
                               << 16);
      } else {
        const uint16_t code = __ldg(static_cast<const uint8_t*>(p.bias) + n);
        bias = __fmul_rn(e4m3x2_to_float2(uint16_t(code | (code << 8))).x, __ldg(p.bias_scale));
      }
    }
    float sar[kChunks];
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
      const int t = t0 + c * 32 + lane;
      sar[c] = t < n_t ? (SCALE == kScaleRow ? __ldg(p.col_scale + t) : 1.f) : 0.f;
    }
    if constexpr (EPI == SPG_EPI_ADD) {
      if (live) {
        // The blocks were last read by this warp's generic loads (previous
        // item): order those before the asynchronous writes.
        __syncwarp();
        if (lane == 0) {
          fence_proxy_async_smem();
          mbar_arrive_expect_tx(res_bar, kChunks * kBufBytes);
#pragma unroll
          for (int c = 0; c < kChunks; ++c)
            tma_load_3d(res0 + c * kBufBytes, tmR, res_bar, n0, t0 + c * 32, 0);
        }
        res_inflight = true;
      }
    }

    if (!mbar_wait(&acc_full[buf], acc_ph, ctl, kErrWaitAccFull)) break;
    tc_fence_after();
    uint32_t own_mask = live ? 0xffffffffu : 0u;
    if (tc.split >= 0) {
      if constexpr (CLUSTER_SPLIT)
        own_mask &= cluster_piece_finish<BN, 32>(p, t_row, tc, q, *csplit, ctl);
      else
        own_mask = split_piece_finish<BN, 32, 8>(p, t_row, tc, cta_rank, q, 0, BN, live);
    }
    own_mask &= (1u << kChunks) - 1u;
    if constexpr (EPI == SPG_EPI_ADD) {
      // Every lane observes the completed copies itself.
      if (res_inflight) {
        if (!mbar_wait(res_bar, res_phase, ctl, kErrWaitFull)) break;
        res_inflight = false;
        res_phase ^= 1u;
      }
    }
    // After a K-split reduction TMEM holds the total of all pieces.
    const bool have_k = tc.split >= 0 || tc.kb_end > tc.kb_begin;
    if (own_mask == 0u) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_empty(buf);
      continue;
    }
    const int last_c = 31 - __clz(own_mask);
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
      if (!((own_mask >> c) & 1u)) continue;
      const int tc0 = t0 + c * 32;  // first token of the chunk
      uint32_t raw[32];
      if (have_k) {
        tmem_ld_32x32b_x32(t_row + c * 32, raw);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) raw[j] = 0u;
      }
      unsigned short resv[32];
      if constexpr (EPI == SPG_EPI_ADD) {
        // Row j of the block = token tc0 + j; this lane's weight row sits in
        // 16-byte unit lane / 8 of it, swizzled like the output.
        const uint8_t* rb = res0 + c * kBufBytes + (lane & 7) * 2;
#pragma unroll
        for (int j = 0; j < 32; ++j)
          resv[j] = *reinterpret_cast<const unsigned short*>(
              rb + j * 64 + (((lane >> 3) ^ ((j >> 1) & 3)) * 16));
      }
      if (have_k) tmem_wait_ld();
      if (c == last_c && item + item_step < item_end) {
        // Every column of this accumulator buffer has been read: hand it back
        // (after the CTA's last item no MMA waits for it, and the cluster-
        // scope arrival would only delay the last stores).
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_empty(buf);
      }
      uint8_t* sbuf = stage0 + (chunk_ctr & 1) * kBufBytes;
      ++chunk_ctr;
      if (lane == 0) bulk_wait_read<1>();
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        float v = __uint_as_float(raw[j]) * (sw * __shfl_sync(0xffffffffu, sar[c], j));
        v += bias;
        if constexpr (EPI == SPG_EPI_ADD) v += __uint_as_float(uint32_t(resv[j]) << 16);
        // Row j of the block (token tc0 + j), column `lane` (weight row n),
        // 16-byte unit swizzled as in the unswapped epilogue.
        const int unit = (lane >> 3) ^ ((j >> 1) & 3);
        *reinterpret_cast<__nv_bfloat16*>(sbuf + j * 64 + unit * 16 + (lane & 7) * 2) =
            __float2bfloat16_rn(v);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        if (n0 < n_w && tc0 < n_t) tma_store_3d(tmY, sbuf, n0, tc0, 0);
        bulk_commit();
      }
    }
  }
  // After an abort no residual copy may still be writing shared memory.
  if (EPI == SPG_EPI_ADD && res_inflight && lane == 0)
    mbar_wait_drain(res_bar, res_phase, p.drain_ns, p.err);
  if (lane == 0) bulk_wait<0>();
  __syncwarp();
}

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
                                                       Svc svc = Svc(),
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
  float scalar = 1.f;
  if constexpr (SCALE == kScaleScalar) scalar = __ldg(p.scalar_a) * __ldg(p.scalar_b);
  bool aborted = false;
  int res_inflight = -1;  // chunk index of a residual copy not yet waited for

  for (int item = item_begin; item < p.total_items && !aborted; item += item_step, ++it) {
    const WorkItem tc = item_fn(item);
    // First residual block of the item, into the buffer of its first chunk
    // (whose previous store, two chunks back, must have been read).  A
    // K-split piece finishes scattered chunks and loads their residual
    // directly instead.
    const bool split_item = tc.split >= 0;
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
    uint32_t own_mask = 0xffffffffu;  // chunks this warp finishes
    if (!split_item) first_residual();
    if (split_item) {
      if (!wait_serving(&acc_full[0], it & 1, ctl, kErrWaitAccFull, svc)) break;
      tc_fence_after();
      own_mask = split_piece_finish<256, EPI == SPG_EPI_SWIGLU ? 64 : 32, 4>(
          p, tmem_base + (uint32_t(q * 32) << 16), tc, cta_rank, q, half * kCols, kCols,
          tc.mb * 128 + q * 32 < p.M);
      if (own_mask == 0u) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_empty(0);
        continue;
      }
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
    if constexpr (EPI == SPG_EPI_ADD && !kResTma) {
      if (!split_item) load_residual_chunk(p, m, n_acc0, row_ok, res_cur);
    }

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
    if (item + item_step < p.total_items) {
      // Released at once (the next item's main loop overlaps the math and
      // stores below); after the CTA's last item no MMA waits for it.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_empty(0);
    }

#pragma unroll
    for (int c = 0; c < kOutChunks; ++c) {
      if (!((own_mask >> c) & 1u)) continue;
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
        if (EPI == SPG_EPI_ADD && split_item) {
          load_residual_chunk(p, m, n_acc0 + 32 * c, row_ok, res_cur);
        } else if constexpr (kResTma) {
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
      // The buffer's store of two chunks back must have been read (the TMA
      // residual path has waited for it before loading the residual here).
      if (!kResTma || split_item) {
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
      ++chunk_ctr;
    }
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
