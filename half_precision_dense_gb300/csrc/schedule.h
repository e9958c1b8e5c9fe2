// schedule.h - the persistent tile schedule, shared by the host planner and
// every CTA role (producer, MMA issuer, epilogue), so all of them walk the
// same tiles in the same order.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define HG_HD __host__ __device__ __forceinline__
#else
#define HG_HD inline
#endif

namespace hg {

// Tile t -> (tile row tm, tile column tn). Tiles are taken in groups of
// `group_m` tile rows; inside a group the row index varies fastest, then the
// column. CTAs that run at the same time therefore work on a band of at most
// group_m tile rows and a few tile columns, so the A row panels and B column
// panels they read are shared in L2 (the grid swizzling of
// "[CUDA 优化实战] hgemm - 超越 cuBLAS", section 1, with SWIZZLE_W playing the
// part of group_m).
HG_HD void tile_coord(int32_t t, int32_t tiles_m, int32_t tiles_n, int32_t group_m,
                      int32_t& tm, int32_t& tn) {
    const int32_t per_group = group_m * tiles_n;
    const int32_t g = t / per_group;
    const int32_t first_m = g * group_m;
    const int32_t rows = (tiles_m - first_m) < group_m ? (tiles_m - first_m) : group_m;
    const int32_t r = t - g * per_group;
    tm = first_m + r % rows;
    tn = r / rows;
}

}  // namespace hg
