// Host build of the tile kernel's schedule (backward_optimizer_gb300/csrc/schedule.h), checked on
// the CPU: every tile order is a bijection onto the tile grid, and schedule_for picks the grouping
// named on the command line for a few layer shapes (printed for the Python test to compare).
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
    // (tiles_m, tiles_n, a_block, b_block): pair tiles of the Llama-3.1-8B MLP at T = 4096 and of
    // Qwen3-14B at T = 8192 (bf16 operands: 256 rows x T tokens x 2 bytes per block)
    const long long MiB = 1 << 20;
    struct Case { const char* name; int tm, tn; long long a, b; } cases[] = {
        {"llama_gate", 56, 16, 2 * MiB, 2 * MiB}, {"llama_down", 16, 56, 2 * MiB, 2 * MiB},
        {"qwen_q", 20, 20, 4 * MiB, 4 * MiB}, {"qwen_k", 4, 20, 4 * MiB, 4 * MiB},
        {"qwen_gate", 68, 20, 4 * MiB, 4 * MiB}, {"qwen_down", 20, 68, 4 * MiB, 4 * MiB}};
    for (const Case& c : cases) {
        forge::TileOrder o = forge::schedule_for(c.tm, c.tn, c.a, c.b, 48 * MiB);
        std::printf("%s raster_cols %d group %d\n", c.name, o.raster_cols, o.group);
    }
    return bad != 0;
}
