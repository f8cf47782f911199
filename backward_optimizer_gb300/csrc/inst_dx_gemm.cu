// Kernel instantiations of the input-gradient GEMM dX = dY W (bfloat16 dX to device memory).
#include "instantiate.cuh"

FORGE_INSTANTIATE_TILES(0, forge::kEpiDX)
FORGE_INSTANTIATE_NARROW(0, forge::kEpiDX)
