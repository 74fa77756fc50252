// Grouped rasterisation of output tiles, shared by the GEMM kernels.
//
// Consecutive CTAs take tiles column by column inside a group of `group_m`
// tile rows, so the CTAs resident at the same time read the same few A row
// panels and B column panels, which then stay in L2 (the grouped block order
// of blog.lightlisten.com "gemm优化", section "Swizzle 增强L2缓存命中", which
// moves on to the next row after a group of 8 tiles instead of finishing the
// row).
#pragma once

namespace sgemm_gb300 {

// Maps a linear CTA index onto (tile row, tile column): tiles are taken
// column by column inside groups of `group_m` tile rows.
__device__ __forceinline__ void raster_tile(int tile, int tiles_m, int tiles_n, int group_m, int &tm,
                                            int &tn) {
    const int per_group = group_m * tiles_n;
    const int group = tile / per_group;
    const int first_m = group * group_m;
    const int rows = min(tiles_m - first_m, group_m);
    const int in_group = tile - group * per_group;
    tm = first_m + in_group % rows;
    tn = in_group / rows;
}

}  // namespace sgemm_gb300
