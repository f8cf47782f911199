// launch.h -- host-side launchers of the library's kernels (internal; not part of the C ABI).
// Each kernel instantiation lives in its own translation unit so the build compiles in parallel.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "opt_math.cuh"

namespace forge {

struct TileArgs;
struct OptArgs;
template <int G> struct TileGroup;

// Group sizes the tile kernels are built for: one layer per launch, or up to kMaxGroup independent
// layers on CTA pairs (forge_fused_dw_step_layers).
constexpr int kMaxGroup = 16;

struct TileLaunch {
    const void* group;  // the TileGroup<G> of the launch (host memory, copied into the kernel's parameters)
    int num_tiles;      // tiles of all the group's layers (per CTA or CTA pair)
    int num_sms;
    cudaStream_t stream;
};

// EPI: 0 = store FP32 dW, 1 = fused optimizer with FP32 states, 2 = fused optimizer with INT8 states,
// 3 = input gradient dX = dY W stored as bf16 (tile rows are tokens, columns d_in), 4 = fused optimizer
// with bfloat16 states.
// BN: tile columns (128, or 256 = two 128 x 128 tiles side by side).
// CL: CTAs per cluster (1: a 128 x BN tile per CTA; 2: a 256 x BN tile per CTA pair).
// OPS: operand format of dY and X, 0 = bf16, 1 = E4M3 (the gradient tile is scaled by s_dY * s_X).
// G: the group size the kernel is built for (1, or kMaxGroup).
template <int OPT, int EPI, int BN, int CL, int OPS, int G> cudaError_t launch_tile(const TileLaunch& l);

// CTAs a tile launch of the given shape would run (persistent grid size).
cudaError_t tile_ctas(int bn, int cl, int num_tiles, int num_sms, int* ctas);
// STATE: 0 = binary32 moments, 1 = INT8 with per-64 scales, 2 = bfloat16.
template <int OPT, int STATE> cudaError_t launch_opt(const OptArgs& a, int grid, cudaStream_t stream);


}  // namespace forge
