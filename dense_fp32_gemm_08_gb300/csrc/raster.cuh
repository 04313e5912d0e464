// raster.cuh: the order in which output tiles are handed to CTAs.
#pragma once

namespace sg {

// Grouped raster order: `group_m` consecutive tile rows are swept column by column, so CTAs
// that run at the same time share A row panels and B column panels in L2.
__device__ __forceinline__ void tile_coords(int pid, int tiles_m, int tiles_n, int group_m,
                                            int &tm, int &tn) {
    const int width = group_m * tiles_n;
    const int group = pid / width;
    const int first_m = group * group_m;
    const int gsize = min(tiles_m - first_m, group_m);
    const int in = pid - group * width;
    tm = first_m + in % gsize;
    tn = in / gsize;
}

}  // namespace sg
