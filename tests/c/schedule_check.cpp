// Host build of the tile kernel's schedule (backward_optimizer_gb300/csrc/schedule.h), checked on
// the CPU: every tile order is a bijection onto the tile grid; the first tiles of a 20 x 4 grid
// grouped by 8 rows, and of the same grid grouped by 3 columns, are printed for the Python test;
// the split tail covers every tile and shortens the busiest pair's work.
#include <cstdio>
#include <vector>

#include "schedule.h"

int main() {
    int bad = 0;
    for (int tm = 1; tm <= 37; ++tm)
        for (int tn = 1; tn <= 37; tn += (tn < 9 ? 1 : 4))
            for (int rc = 0; rc < 2; ++rc)
                for (int g = 1; g <= (rc ? tn : tm) + 1; ++g) {
                    forge::TileOrder o{tm, tn, g, rc};
                    std::vector<int> seen(tm * tn, 0);
                    for (int t = 0; t < tm * tn; ++t) {
                        int mb = -1, nb = -1;
                        forge::tile_coords(t, o, mb, nb);
                        if (mb < 0 || mb >= tm || nb < 0 || nb >= tn || seen[mb * tn + nb]++) ++bad;
                    }
                }
    std::printf("bijection_failures %d\n", bad);
    for (int rc = 0; rc < 2; ++rc) {
        forge::TileOrder o{20, 4, rc ? 3 : 8, rc};
        std::printf("%s", rc ? "cols3" : "rows8");
        for (int t : {0, 1, 7, 8, 31, 32, 33, 79}) {
            int mb, nb;
            forge::tile_coords(t, o, mb, nb);
            std::printf(" %d:%d", mb, nb);
        }
        std::printf("\n");
    }
    // split tail: every tile of the layers' order is covered once whole or by its two halves, and
    // a pair's work (whole tile 2, half tile 1) never exceeds the unsplit schedule's, and is less
    // whenever a tail was split
    int split_bad = 0;
    for (int tiles = 1; tiles <= 400; ++tiles)
        for (int units = 1; units <= 100; ++units) {
            const int from = forge::split_tail_from(tiles, units);
            if (from > tiles || from < 0) ++split_bad;
            const int launch = tiles + (tiles - from);
            std::vector<int> cover(tiles, 0);
            std::vector<int> work(units, 0);
            for (int t = 0; t < launch; ++t) {
                int part = -2;
                const int o = forge::tail_tile(t, from, part);
                if (o < 0 || o >= tiles || part < -1 || part > 1) { ++split_bad; continue; }
                cover[o] += part < 0 ? 2 : 1 + 2 * part;  // whole: 2; halves: 1 and 3 -> 4
                work[t % units] += part < 0 ? 2 : 1;
            }
            for (int o = 0; o < tiles; ++o)
                if (cover[o] != (o < from ? 2 : 4)) ++split_bad;
            int span = 0;
            for (int w : work) span = w > span ? w : span;
            const int unsplit = 2 * ((tiles + units - 1) / units);
            if (span > unsplit || (from < tiles && span >= unsplit)) ++split_bad;
        }
    std::printf("split_failures %d\n", split_bad);
    std::printf("split_from");
    for (int tiles : {256, 80, 896, 400, 76, 40, 1360, 152}) std::printf(" %d", forge::split_tail_from(tiles, 76));
    std::printf("\n");
    return bad != 0 || split_bad != 0;
}
