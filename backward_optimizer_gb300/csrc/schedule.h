// schedule.h -- the persistent tile order shared by the tile kernel (device) and the host code that
// chooses it.  Plain C++ with no CUDA dependency besides the __host__ __device__ qualifiers, so that
// host-only builds (the library's tests) can compile and check it.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define FORGE_HD __host__ __device__ __forceinline__
#else
#define FORGE_HD inline
#endif

namespace forge {

// Tiles are visited in groups of `group` consecutive tile rows (raster_cols == 0) or tile columns
// (raster_cols == 1); within a group the short side runs fastest.  With rows grouped, the group's
// dY row blocks are read by every tile column in turn and the X column blocks stream past; with
// columns grouped, the roles swap.  The host picks the grouping that keeps the smaller operand
// resident in L2 (schedule_for).
struct TileOrder {
    int tiles_m, tiles_n;  // tile rows (output rows) and tile columns
    int group;             // tile rows (or columns) per group, >= 1
    int raster_cols;       // 0: group tile rows; 1: group tile columns
};

// Tile number `tile` (0 .. tiles_m * tiles_n - 1) -> its tile row mb and tile column nb.
FORGE_HD void tile_coords(int tile, const TileOrder& o, int& mb, int& nb) {
    const int tg = o.raster_cols ? o.tiles_n : o.tiles_m;  // the grouped dimension
    const int to = o.raster_cols ? o.tiles_m : o.tiles_n;  // the other one
    const int per_group = o.group * to;
    const int g = tile / per_group;
    const int first = g * o.group;
    const int gm = tg - first < o.group ? tg - first : o.group;
    const int in_group = tile - g * per_group;
    const int p = first + in_group % gm;
    const int q = in_group / gm;
    mb = o.raster_cols ? q : p;
    nb = o.raster_cols ? p : q;
}

// The order for an output of tiles_m x tiles_n tiles whose row blocks read a_block bytes of the A
// operand each and whose column blocks read b_block bytes of B each (over the whole reduction):
// the operand with fewer bytes in total is the resident one, and a group holds as many of its
// blocks as fit in `budget` bytes (at least one).
FORGE_HD TileOrder schedule_for(int tiles_m, int tiles_n, int64_t a_block, int64_t b_block, int64_t budget) {
    TileOrder o;
    o.tiles_m = tiles_m;
    o.tiles_n = tiles_n;
    const bool a_resident = a_block * tiles_m <= b_block * tiles_n;
    const int64_t blk = a_resident ? a_block : b_block;
    const int dim = a_resident ? tiles_m : tiles_n;
    int64_t fit = blk > 0 ? budget / blk : dim;
    if (fit < 1) fit = 1;
    o.group = fit < dim ? static_cast<int>(fit) : dim;
    if (o.group < 1) o.group = 1;
    o.raster_cols = a_resident ? 0 : 1;
    return o;
}

}  // namespace forge
