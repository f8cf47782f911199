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
// columns grouped, the roles swap.  The library groups 8 tile rows (forge_api.cu, tile_order).
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

// First tile of a pair launch's split tail.  The persistent grid runs `units` pairs; when the last
// wave of 256 x 256 tiles would occupy at most half of them, its tiles run as two 256 x 128 halves
// each (the kernel numbers them after the whole tiles), so that the wave occupies up to all of the
// pairs.  Returns `tiles` when nothing is split: a single wave, a full last wave, or one more than
// half full (two rounds of halves would take longer than one of whole tiles).
FORGE_HD int split_tail_from(int tiles, int units) {
    if (units <= 0 || tiles <= units) return tiles;
    const int rest = tiles % units;
    return (rest > 0 && 2 * rest <= units) ? tiles - rest : tiles;
}

// Launch tile t -> the tile of the layers' order it covers (returned) and its part: -1 the whole
// tile, 0 or 1 the left or right 128 columns of it.  Tiles from `split_from` on are halves.
FORGE_HD int tail_tile(int t, int split_from, int& part) {
    if (t < split_from) {
        part = -1;
        return t;
    }
    part = (t - split_from) & 1;
    return split_from + ((t - split_from) >> 1);
}

}  // namespace forge
