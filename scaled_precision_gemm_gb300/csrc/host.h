// Host-side helpers shared by the GEMM launchers.
#pragma once

#include <cuda.h>

#include <cstdint>

#include "common.h"
#include "spg.h"

namespace spg {

// Encode a 3-D tiled TMA descriptor (uint8 or bf16 elements).  d0 is the
// contiguous dimension; strides are in bytes; the box is box0 x box1 x 1.
bool make_tmap_3d(CUtensorMap* out, const void* base, bool bf16, uint64_t d0, uint64_t d1,
                  uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0,
                  uint32_t box1, int swizzle_bytes);

// TMA descriptor of a 2-D array of 32-bit elements (no swizzle): d0
// contiguous elements per row, d1 rows of stride1_bytes; box box0 x box1.
// Encoded as rank 3 with a unit third dimension.
bool make_tmap_2d_u32(CUtensorMap* out, const void* base, uint64_t d0, uint64_t d1,
                      uint64_t stride1_bytes, uint32_t box0, uint32_t box1);

// Hits and misses of the tensor-map cache behind the two functions above;
// switching the cache off (A/B timing of the host path) also empties it.
void tmap_cache_stats(uint64_t* hits, uint64_t* misses);
void set_tmap_cache(bool on);

// Make the route selector read SPG_FORCE_VARIANT / SPG_FORCE_TAIL again on
// its next call.
void reload_forced_route();

// Whether SPG_FORCE_VARIANT (as last read) names this variant.
bool forced_variant_is(const char* name);

// Tail split of a two-SM schedule along N (see plan_items): with `units` CTA
// pairs and `tiles` tiles of width bn, the tiles of the last partial wave
// are split into `ways` (1, 2 or 4) narrower items, each a whole number of
// epilogue chunks wide (32 columns, 64 for SwiGLU).
inline int tail_split_ways(int64_t tiles, int64_t units, int bn, int epilogue) {
  if (units <= 0) return 1;
  const int64_t rem = tiles % units;
  const int chunk = epilogue == SPG_EPI_SWIGLU ? 64 : 32;
  for (int ways : {4, 2}) {
    if (rem > 0 && rem * ways <= units && bn % (ways * chunk) == 0) return ways;
  }
  return 1;
}

// Relative duration of a tail item split `ways` ways: its MMAs shrink with
// the width but the A operand it stages does not (measured on GB300).
inline double tail_item_time(int ways) { return ways <= 1 ? 1.0 : 0.45 + 0.55 / ways; }

// K split of a two-SM schedule's last partial wave: the tiles of that wave
// (tiles mod units; all tiles when there are fewer than units) are each
// reduced by split_k pieces of kb_per_split K blocks, as many pieces as still
// fit the wave, at most kMaxSplitK, each at least 4 K blocks deep.
constexpr int kMaxSplitK = 4;
struct KSplit {
  int split_k = 1;
  int kb_per_split = 0;
  int64_t tail_tiles = 0;
};

inline KSplit ksplit_plan(int64_t tiles, int64_t units, int64_t nkb) {
  KSplit k;
  if (units <= 0 || nkb <= 0) return k;
  const int64_t rem = tiles % units;
  if (rem == 0) return k;
  int64_t s = units / rem;
  if (s > kMaxSplitK) s = kMaxSplitK;
  while (s > 1 && (nkb + s - 1) / s < 4) --s;
  if (s < 2) return k;
  const int64_t kbps = (nkb + s - 1) / s;
  s = (nkb + kbps - 1) / kbps;  // no empty piece
  if (s < 2) return k;
  k.split_k = static_cast<int>(s);
  k.kb_per_split = static_cast<int>(kbps);
  k.tail_tiles = rem;
  return k;
}

// K split of one-CTA tiles inside thread-block clusters: with fewer tiles
// than SMs every tile is reduced by split_k CTAs of one cluster, as many as
// the SMs allow (one wave, one piece per CTA), at most kMaxClusterSplit,
// each piece at least min_kb K blocks deep and none empty, and the partial
// sums each CTA receives (cluster_recv_bytes for tiles bn wide with
// epilogue chunks of cw columns) within its ring_bytes of operand ring.
// The pieces are summed through distributed shared memory: no workspace.
constexpr int kMaxClusterSplit = 4;
inline KSplit csplit_plan(int64_t tiles, int64_t sms, int64_t nkb, int64_t min_kb, int bn,
                          int cw, int ring_bytes) {
  KSplit k;
  if (tiles <= 0 || nkb <= 0 || sms <= 0) return k;
  int64_t s = sms / tiles;
  if (s > kMaxClusterSplit) s = kMaxClusterSplit;
  while (s > 1 && ((nkb + s - 1) / s < min_kb ||
                   cluster_recv_bytes(bn, cw, static_cast<int>(s)) > ring_bytes))
    --s;
  if (s < 2) return k;
  const int64_t kbps = (nkb + s - 1) / s;
  s = (nkb + kbps - 1) / kbps;  // no empty piece
  if (s < 2) return k;
  k.split_k = static_cast<int>(s);
  k.kb_per_split = static_cast<int>(kbps);
  k.tail_tiles = tiles;
  return k;
}

// Workspace of a K split with tiles bn columns wide: one 128 x bn fp32 slice
// per (tail tile, piece, CTA of the pair), then one 64-bit arrival counter
// per (tail tile, CTA, lane quarter, epilogue chunk: 32 columns, 64 for
// SwiGLU).
inline int64_t ksplit_workspace_bytes(const KSplit& k, int bn, int epilogue) {
  if (k.split_k < 2) return 0;
  const int cw = epilogue == SPG_EPI_SWIGLU ? 64 : 32;
  return k.tail_tiles * k.split_k * 2 * 128 * int64_t(bn) * 4 +
         k.tail_tiles * 2 * 4 * (bn / cw) * 8;
}

// Duration of a K-split tail piece in K blocks of the tile: its own K
// blocks, the partial sums written by every piece and read back where each
// chunk finishes (about 2.5 K blocks per 128 x 256 fp32 slice), and the
// finish itself (partial store, fence, arrival, reduction, epilogue: about
// 6 us on GB300, some 20 K blocks, measured), which makes the split lose
// at short K.
inline double ksplit_piece_time(const KSplit& k, int bn) {
  return k.kb_per_split + 20.0 + 2.5 * k.split_k * (bn / 256.0);
}

// The selector behind spg_select_route (no validation).
// b_mn_major: the B operand is N-major (per-tensor GEMM with layout_b 'N').
// allow_ksplit: the caller provides a workspace, so the last partial wave may
// be split along K.  allow_swap: the swapped narrow-T tile may be taken (the
// per-tensor GEMM clears it for an M-major A, which that tile cannot read).
spg_route select_route_internal(int kind, int64_t T, int64_t N, int64_t K, int epilogue,
                                int64_t batch, bool b_mn_major, bool allow_ksplit,
                                bool allow_swap = true);

}  // namespace spg
