// launch.h -- host-side launchers of the library's kernels (internal; not part of the C ABI).
// Each kernel instantiation lives in its own translation unit so the build compiles in parallel.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "opt_math.cuh"

namespace forge {

struct TileArgs;
struct OptArgs;

struct TileLaunch {
    CUtensorMap tmap_dy;
    CUtensorMap tmap_x;
    const TileArgs* args;
    int grid;
    cudaStream_t stream;
};

// EPI: 0 = store FP32 dW, 1 = fused optimizer with FP32 states, 2 = fused optimizer with INT8 states.
template <int OPT, int EPI> cudaError_t launch_tile(const TileLaunch& l);
template <int OPT, bool INT8> cudaError_t launch_opt(const OptArgs& a, int grid, cudaStream_t stream);

// Shared-memory bytes the tile kernel needs (for the host's capacity check).
int tile_smem_bytes();

}  // namespace forge
