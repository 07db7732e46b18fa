// Shared definitions of the tcgen05 GEMM kernels: parameters, error codes,
// tile rasterization and small device helpers.
#pragma once

#include <cuda_bf16.h>

#include <cstddef>

#include "common.h"
#include "ptx.cuh"

namespace spg {
enum GemmKind : int { kKindFp8 = 0, kKindNvfp4 = 1 };
enum ScaleMode : int { kScaleRow = 0, kScaleScalar = 1 };

// Error codes written to the device error word (first one wins).
enum : unsigned int {
  kErrWaitEmpty = 0x101,
  kErrWaitFull = 0x102,
  kErrWaitAccEmpty = 0x103,
  kErrWaitAccFull = 0x104,
  kErrDrain = 0x105,
  kErrInjectedStall = 0x106,
  kErrSplitCounter = 0x107,
};

struct GemmParams {
  int M;             // output rows (T)
  int N;             // accumulator columns
  int K;             // reduction length in elements
  int n_out;         // output columns (N, or N/2 for SwiGLU)
  int num_m_blocks;  // ceil(M / 128)
  int num_n_blocks;  // ceil(N / BN)
  int num_k_blocks;  // ceil(K_bytes / 128)
  int tiles_per_batch;
  int total_tiles;
  int group_m;      // m-blocks per rasterization group
  int a_batch_mul;  // 0 broadcasts A matrix 0 over the batch, else 1
  int b_batch_mul;
  const float* row_scale;  // kScaleRow: sa [M]
  const float* col_scale;  // kScaleRow: sw [N]
  const float* scalar_a;   // kScaleScalar: device scalars
  const float* scalar_b;
  const __nv_bfloat16* residual;  // SPG_EPI_ADD: [M, N] row-major
  const void* bias;               // fused bias per output column, or nullptr
  const float* bias_scale;        // bias_kind 2: device scalar
  int bias_kind;                  // 0 none, 1 bf16 [N], 2 E4M3 codes [N] x bias_scale
  const uint8_t* sfa;             // NVFP4 scales, blocked layout
  const uint8_t* sfb;
  int sf_tiles_per_row_block;  // K / 64
  // Tail split (two-SM kernels): work items [0, split_full) are whole tiles;
  // the remaining tiles are each split along N into split_ways pieces, or
  // along K into split_k pieces of kb_per_split K blocks, so the last,
  // partial wave is shorter.  total_items counts both kinds of item.
  int split_full;
  int split_ways;
  int split_k;
  int kb_per_split;
  int total_items;
  // K-split workspace: per (tail tile, split, CTA of the pair) one 128 x BN
  // fp32 slice of partial sums, then one 64-bit arrival counter per (tail
  // tile, CTA, lane quarter, epilogue chunk).  A counter holds
  // (epoch << 32) | arrivals; a value tagged with another epoch counts as
  // zero arrivals.
  float* ws_partial;
  unsigned long long* ws_counter;
  uint32_t epoch;
  uint64_t timeout_ns;  // bound of every pipeline wait
  uint64_t drain_ns;    // bound of the exit waits for copies / MMAs in flight
  unsigned int* err;
  int debug_stall;      // test hook: the epilogue first waits on a barrier nothing arrives on
};

// One unit of work of the persistent schedule: a tile, or a piece of one.
struct WorkItem {
  int b, mb, nb;         // batch, m-block, n-block of the tile
  int n_off;             // first accumulator column of the piece inside the tile
  int width;             // accumulator columns of the piece
  int kb_begin, kb_end;  // K blocks the piece reduces over
  int split;             // K-split index of the piece, -1 for an unsplit K range
  int tail;              // tile index relative to split_full (K-split pieces)
};

struct TileCoord {
  int b, mb, nb;
};

__device__ __forceinline__ TileCoord tile_coord(int tile, const GemmParams& p) {
  TileCoord c;
  c.b = tile / p.tiles_per_batch;
  const int t = tile - c.b * p.tiles_per_batch;
  const int span = p.group_m * p.num_n_blocks;
  const int g = t / span;
  const int first_m = g * p.group_m;
  const int rem = p.num_m_blocks - first_m;
  const int gsize = rem < p.group_m ? rem : p.group_m;
  const int local = t - g * span;
  c.mb = first_m + local % gsize;
  c.nb = local / gsize;
  return c;
}

__device__ __forceinline__ WorkItem work_item(int item, const GemmParams& p, int bn) {
  WorkItem w;
  int tile = item, piece = 0, ways = 1;
  w.split = -1;
  w.tail = 0;
  w.kb_begin = 0;
  w.kb_end = p.num_k_blocks;
  if (item >= p.split_full) {
    const int rel = item - p.split_full;
    if (p.split_k > 1) {
      w.tail = rel / p.split_k;
      w.split = rel - w.tail * p.split_k;
      tile = p.split_full + w.tail;
      w.kb_begin = w.split * p.kb_per_split;
      const int e = w.kb_begin + p.kb_per_split;
      w.kb_end = e < p.num_k_blocks ? e : p.num_k_blocks;
      if (w.kb_begin > w.kb_end) w.kb_begin = w.kb_end;
    } else {
      ways = p.split_ways;
      tile = p.split_full + rel / ways;
      piece = rel % ways;
    }
  }
  const TileCoord tc = tile_coord(tile, p);
  w.b = tc.b;
  w.mb = tc.mb;
  w.nb = tc.nb;
  w.width = bn / ways;
  w.n_off = piece * w.width;
  return w;
}

// ---------------------------------------------------------------- K split
// Slice of partial sums of (tail tile, split, CTA rank): 128 rows x bn fp32,
// stored as float4 groups ordered (32-column chunk, 32-row quarter, 4-column
// group, row in the quarter): the lanes of an epilogue warp (32 consecutive
// rows) write 512 contiguous bytes per access, and the 32 x 32 block of one
// warp and chunk is one contiguous 4 KB run that a bulk copy moves whole.
__device__ __forceinline__ float4* split_slice(const GemmParams& p, int tail, int split, int rank,
                                               int bn) {
  const int64_t idx = (int64_t(tail) * p.split_k + split) * 2 + rank;
  return reinterpret_cast<float4*>(p.ws_partial + idx * 128 * bn);
}

// float4 index of (column col, row) inside a slice.
__device__ __forceinline__ int split_f4_index(int col, int row) {
  return (((col >> 5) * 4 + (row >> 5)) * 8 + ((col >> 2) & 7)) * 32 + (row & 31);
}

// float4 index of the 4 KB block of (chunk, quarter) inside a slice.
__device__ __forceinline__ int split_block_index(int chunk, int quarter) {
  return (chunk * 4 + quarter) * 256;
}

// Arrival counter of (tail tile, CTA rank, lane quarter, epilogue chunk of
// cw columns).
__device__ __forceinline__ int split_counter_index(int tail, int rank, int quarter, int chunk,
                                                   int bn, int cw) {
  return ((tail * 2 + rank) * 4 + quarter) * (bn / cw) + chunk;
}

// Record one arrival on counter `idx` and return how many pieces arrived
// before (0 .. split_k - 1).  Called after this thread's piece of the
// partial sums is written and fenced.  The last arrival puts the counter
// back to zero so the workspace stays clean for the next call.
__device__ __forceinline__ int split_arrive(const GemmParams& p, int idx) {
  unsigned long long* c = p.ws_counter + idx;
  unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(c);
  int before = -1;
  for (int i = 0; i < (1 << 20); ++i) {
    const bool mine = uint32_t(old >> 32) == p.epoch;
    const unsigned long long nv = mine ? old + 1ull : ((unsigned long long)p.epoch << 32) | 1ull;
    const unsigned long long prev = atomicCAS(c, old, nv);
    if (prev == old) {
      before = mine ? int(uint32_t(old)) : 0;
      break;
    }
    old = prev;
  }
  if (before < 0) {
    atomicCAS(p.err, 0u, kErrSplitCounter);
    return 0;
  }
  if (before == p.split_k - 1) *reinterpret_cast<volatile unsigned long long*>(c) = 0ull;
  return before;
}

// Bias of accumulator column n (0 when there is none or n is out of range).
__device__ __forceinline__ float load_bias(const GemmParams& p, int n) {
  if (n >= p.N) return 0.f;
  if (p.bias_kind == 1)
    return __uint_as_float(uint32_t(__ldg(static_cast<const unsigned short*>(p.bias) + n)) << 16);
  const uint16_t c = __ldg(static_cast<const uint8_t*>(p.bias) + n);
  return __fmul_rn(e4m3x2_to_float2(uint16_t(c | (c << 8))).x, __ldg(p.bias_scale));
}

// Drain-mode wait: bounded, but not cut short by the abort flag.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity,
                                                uint64_t timeout_ns, unsigned int* err) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(a, parity)) return true;
    if ((i & 15u) == 15u && (globaltimer_ns() - t0 > timeout_ns || i > (1u << 30))) {
      atomicCAS(err, 0u, kErrDrain);
      return false;
    }
  }
}

// Drain-mode wait with a cluster-scope acquire (the phase is completed by a
// release from the other CTA of the pair).
__device__ __forceinline__ bool mbar_wait_drain_cluster(uint64_t* bar, uint32_t parity,
                                                        uint64_t timeout_ns, unsigned int* err) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait_cluster(a, parity)) return true;
    if ((i & 15u) == 15u && (globaltimer_ns() - t0 > timeout_ns || i > (1u << 30))) {
      atomicCAS(err, 0u, kErrDrain);
      return false;
    }
  }
}

// ------------------------------------------------------------- pair exit
// In the two-SM kernels both CTAs' operand copies complete on the leader's
// full[] barriers, and the leader's producer posts the expected bytes of both
// halves.  Normally both producers issue the same stages; after a time-out
// they may stop after different numbers of stages, and then the leader alone
// cannot tell which copies are still landing.  So at exit the peer's producer
// publishes, in the leader's PairExit, how many stages it issued and the
// bytes of its copies into each ring slot (its last use of each), and the
// leader's producer (pair_exit_drain) settles every stage of the last ring's
// worth that only one side issued -- the arrival and bytes of peer copies
// the leader never announced, or the announced bytes of a peer half that was
// never issued -- and waits (bounded) for every one of them.  After that no
// copy of either CTA is in flight, and both CTAs pass the final cluster
// barrier only after it.
constexpr int kPairExitMaxStages = 12;
struct PairExit {
  uint64_t bar;        // leader: one arrival, released by the peer's producer
  uint32_t issued;     // the peer's count of issued stages
  uint32_t pad;
  uint32_t bytes[kPairExitMaxStages];  // the peer's copy bytes per ring slot
};

// Peer CTA's producer: publish its issued count and per-slot bytes in the
// leader's PairExit (leader: the leader's cluster rank).
template <int STAGES>
__device__ __forceinline__ void pair_exit_publish(PairExit* px, uint32_t issued,
                                                  const uint32_t (&bytes)[STAGES],
                                                  uint32_t leader = 0) {
  static_assert(STAGES <= kPairExitMaxStages, "PairExit holds at most 12 ring slots");
  const uint32_t base = mapa_shared(smem_u32(px), leader);
  st_cluster_u32(base + uint32_t(offsetof(PairExit, issued)), issued);
#pragma unroll
  for (int s = 0; s < STAGES; ++s)
    st_cluster_u32(base + uint32_t(offsetof(PairExit, bytes)) + 4u * s, bytes[s]);
  mbar_arrive_cluster(base + uint32_t(offsetof(PairExit, bar)));
}

// Leader CTA's producer: wait for the peer's account, settle the stages only
// one side issued and wait for every stage still outstanding.  `bytes` are
// the leader's own copy bytes per ring slot (the same as the peer's for a
// stage both issue).
template <int STAGES>
__device__ __forceinline__ void pair_exit_drain(PairExit* px, uint64_t* full, uint32_t issued,
                                                const uint32_t (&bytes)[STAGES],
                                                const GemmParams& p) {
  uint32_t peer = issued;
  if (mbar_wait_drain_cluster(&px->bar, 0, p.drain_ns, p.err))
    peer = *reinterpret_cast<volatile uint32_t*>(&px->issued);
  const uint32_t hi = issued > peer ? issued : peer;
  const uint32_t lo = hi > uint32_t(STAGES) ? hi - uint32_t(STAGES) : 0u;
  for (uint32_t idx = lo; idx < hi; ++idx) {
    const uint32_t s = idx % uint32_t(STAGES);
    if (idx >= issued)
      mbar_arrive_expect_tx(&full[s], reinterpret_cast<volatile uint32_t*>(px->bytes)[s]);
    else if (idx >= peer)
      mbar_complete_tx(&full[s], bytes[s]);
    mbar_wait_drain(&full[s], (idx / uint32_t(STAGES)) & 1u, p.drain_ns, p.err);
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

}  // namespace spg
