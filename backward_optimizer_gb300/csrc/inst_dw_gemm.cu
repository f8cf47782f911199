// Kernel instantiations of the unfused weight-gradient GEMM (FP32 dW to device memory).
#include "instantiate.cuh"

FORGE_INSTANTIATE_TILES(0, forge::kEpiStoreGrad)
