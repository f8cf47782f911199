// Kernel instantiation of the unfused weight-gradient GEMM (FP32 dW to device memory).
#include "instantiate.cuh"

template cudaError_t forge::launch_tile<0, forge::kEpiStoreGrad>(const forge::TileLaunch&);

int forge::tile_smem_bytes() { return forge::TileCfg<forge::kTileBN>::kSmemBytes; }
