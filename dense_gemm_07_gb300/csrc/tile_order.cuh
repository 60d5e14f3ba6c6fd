// tile_order.cuh -- block-order swizzle shared by the host planner and the
// kernels.
//
// "GEMM Optimization" (infra.bea.ai), section "L2 Cache and Wave Analysis":
// blocks that run at the same time should read the same rows of A and
// columns of B so that the second read hits L2.  A linear tile index is
// mapped to (tile_m, tile_n) in bands of `group` tile-rows; inside a band the
// index walks down a column of tiles first, so a run of consecutive indices
// covers a compact group x (run / group) patch of C.
#pragma once

#include <cstdint>

namespace g07 {

struct TileCoord {
  int32_t m;
  int32_t n;
};

__host__ __device__ __forceinline__ TileCoord tile_order(int64_t linear,
                                                         int32_t tiles_m,
                                                         int32_t tiles_n,
                                                         int32_t group) {
  const int64_t per_band = static_cast<int64_t>(group) * tiles_n;
  const int64_t band = linear / per_band;
  const int32_t first_m = static_cast<int32_t>(band) * group;
  const int32_t rows =
      (tiles_m - first_m) < group ? (tiles_m - first_m) : group;
  const int64_t in_band = linear - band * per_band;
  TileCoord t;
  t.m = first_m + static_cast<int32_t>(in_band % rows);
  t.n = static_cast<int32_t>(in_band / rows);
  return t;
}

}  // namespace g07
