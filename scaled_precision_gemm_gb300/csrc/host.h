// Host-side helpers shared by the GEMM launchers.
#pragma once

#include <cuda.h>

#include <cstdint>

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

// Tail split of a two-SM schedule (see plan_tail_split): with `units` CTA
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

// The selector behind spg_select_route (no validation).
// b_mn_major: the B operand is N-major (per-tensor GEMM with layout_b 'N').
spg_route select_route_internal(int kind, int64_t T, int64_t N, int64_t K, int epilogue,
                                int64_t batch, bool b_mn_major);

}  // namespace spg
