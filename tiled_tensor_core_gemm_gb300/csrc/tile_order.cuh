// Order in which output tiles are visited, shared by the tensor-core kernel
// and the split-tail reduction so both agree on where tile t lies.
//
// Grouped raster: tiles are taken in groups of `group_m` tile-rows; within a
// group, down the rows first, then across the columns.  Tiles that run at the
// same time then share A row-panels and B column-panels in L2 (the persistent
// schedule of "Learn CuTeDSL" section 8.1, with a raster swizzle).
#pragma once

namespace tcgemm {

__host__ __device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int group_m, int &tm, int &tn) {
    const int per_group = group_m * tiles_n;
    const int g = t / per_group;
    const int first = g * group_m;
    const int rest = tiles_m - first;
    const int gm = rest < group_m ? rest : group_m;
    const int r = t - g * per_group;
    tm = first + r % gm;
    tn = r / gm;
}

}  // namespace tcgemm
