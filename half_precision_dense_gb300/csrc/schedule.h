// schedule.h - the persistent work schedule, shared by the host planner and
// every CTA role (producer, MMA issuer, epilogue), so all of them walk the
// same work units in the same order.
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

// One unit of work: K blocks [kb0, kb1) of tile `tile`.
//
// Units [0, dp_units) are whole tiles (tile = unit). The tiles after them are
// split along K into `split` parts each, so that a last, partial wave of
// tiles becomes split x as many shorter units and keeps every cluster busy:
// unit dp_units + split * s + part is part `part` of tile dp_units + s, and
// `split_idx` = s numbers the split tiles. The last part owns the tile: it
// adds the other parts' fp32 partial sums to its own and writes C. Every part
// it waits for has a lower unit index; clusters take units in increasing
// order, so these waits never form a cycle, however many parts one cluster
// holds.
struct WorkUnit {
    int32_t tile;
    int32_t kb0, kb1;
    int32_t part;       // 0 for whole tiles
    int32_t split_idx;  // -1 for whole tiles
};

HG_HD WorkUnit work_unit(int32_t u, int32_t dp_units, int32_t split, int32_t num_kb) {
    WorkUnit w;
    if (u < dp_units || split <= 1) {
        w.tile = u;
        w.kb0 = 0;
        w.kb1 = num_kb;
        w.part = 0;
        w.split_idx = -1;
    } else {
        const int32_t v = u - dp_units;
        const int32_t s = v / split;
        w.part = v - s * split;
        w.tile = dp_units + s;
        w.split_idx = s;
        w.kb0 = static_cast<int32_t>(static_cast<int64_t>(w.part) * num_kb / split);
        w.kb1 = static_cast<int32_t>(static_cast<int64_t>(w.part + 1) * num_kb / split);
    }
    return w;
}

// Number of work units for `num_tiles` tiles of which the first `dp_units`
// are whole.
HG_HD int32_t work_units(int32_t num_tiles, int32_t dp_units, int32_t split) {
    return split <= 1 ? num_tiles : dp_units + (num_tiles - dp_units) * split;
}

}  // namespace hg
