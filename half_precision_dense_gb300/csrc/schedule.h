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

// The K blocks [lo, hi) of a unit's range [kb0, kb1) that rank `rank` of a
// K-split cluster of `parts` CTAs multiplies: contiguous shares in rank
// order, equal to within one block.
HG_HD void split_share(int32_t kb0, int32_t kb1, uint32_t rank, int parts, int32_t& lo, int32_t& hi) {
    const int32_t n = kb1 - kb0;
    lo = kb0 + static_cast<int32_t>((static_cast<int64_t>(n) * rank) / parts);
    hi = kb0 + static_cast<int32_t>((static_cast<int64_t>(n) * (rank + 1)) / parts);
}

// The schedule: tiles [0, dp_tiles) are data-parallel (cluster c takes tiles
// c, c + C, c + 2C, ... whole); the remaining tiles [dp_tiles, num_tiles) are
// stream-K: their K blocks, numbered g = (t - dp_tiles) * num_kb + kb, are cut
// into C contiguous ranges of sk_base or sk_base + 1 blocks (the first
// sk_extra clusters take one more), and cluster c walks its range after its
// data-parallel tiles, one unit per tile it touches.
struct Schedule {
    int32_t num_tiles, dp_tiles, num_kb, clusters;
    int32_t sk_base, sk_extra;  // total stream-K blocks = sk_base * clusters + sk_extra
};

// A unit: K blocks [kb0, kb1) of tile `tile`. `kind` 0 = the whole tile;
// 1 = the stream-K part holding K block 0 of a tile split across clusters (the
// owner: it adds the other parts' fp32 partial sums and writes C); 2 = any
// other stream-K part (it publishes its partial sums). An owner part is the
// last unit of its cluster's range and the other parts of its tile are the
// first units of the following clusters' ranges, which never wait: waits
// cannot form a cycle.
struct WorkUnit {
    int32_t tile;
    int32_t kb0, kb1;
    int32_t kind;
};

HG_HD int64_t sk_range_start(const Schedule& s, int32_t c) {
    return static_cast<int64_t>(c) * s.sk_base + (c < s.sk_extra ? c : s.sk_extra);
}

// Cluster whose stream-K range holds block g.
HG_HD int32_t sk_cluster_of(const Schedule& s, int64_t g) {
    const int64_t big = static_cast<int64_t>(s.sk_extra) * (s.sk_base + 1);
    if (g < big) return static_cast<int32_t>(g / (s.sk_base + 1));
    return static_cast<int32_t>(s.sk_extra + (g - big) / s.sk_base);
}

HG_HD int32_t dp_tiles_of(const Schedule& s, int32_t c) {
    return c < s.dp_tiles ? (s.dp_tiles - c + s.clusters - 1) / s.clusters : 0;
}

// The i-th unit of cluster c; false once its work is done.
HG_HD bool next_unit(const Schedule& s, int32_t c, int32_t i, WorkUnit& w) {
    const int32_t ndp = dp_tiles_of(s, c);
    if (i < ndp) {
        w.tile = c + i * s.clusters;
        w.kb0 = 0;
        w.kb1 = s.num_kb;
        w.kind = 0;
        return true;
    }
    const int64_t start = sk_range_start(s, c);
    const int64_t end = start + s.sk_base + (c < s.sk_extra ? 1 : 0);
    const int32_t j = i - ndp;
    const int64_t t_first = start / s.num_kb;
    const int64_t t = t_first + j;
    const int64_t t_begin = t * s.num_kb;
    if (end <= start || t_begin >= end) return false;
    const int64_t lo = j == 0 ? start : t_begin;
    const int64_t hi = end < t_begin + s.num_kb ? end : t_begin + s.num_kb;
    w.tile = s.dp_tiles + static_cast<int32_t>(t);
    w.kb0 = static_cast<int32_t>(lo - t_begin);
    w.kb1 = static_cast<int32_t>(hi - t_begin);
    w.kind = (w.kb0 == 0 && w.kb1 == s.num_kb) ? 0 : (w.kb0 == 0 ? 1 : 2);
    return true;
}

// For an owner unit of stream-K tile `tile`, the last cluster holding part of
// it (the contributors are the owner's cluster + 1 .. that cluster).
HG_HD int32_t sk_last_contributor(const Schedule& s, int32_t tile) {
    const int64_t g_last = static_cast<int64_t>(tile - s.dp_tiles) * s.num_kb + s.num_kb - 1;
    return sk_cluster_of(s, g_last);
}

}  // namespace hg
