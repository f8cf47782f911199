// Host build of the tile kernel's schedule (backward_optimizer_gb300/csrc/schedule.h), checked on
// the CPU: every tile order is a bijection onto the tile grid; the first tiles of a 20 x 4 grid
// grouped by 8 rows, and of the same grid grouped by 3 columns, are printed for the Python test.
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
    return bad != 0;
}
