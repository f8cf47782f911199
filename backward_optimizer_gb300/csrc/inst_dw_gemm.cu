// Kernel instantiations of the unfused weight-gradient GEMM (FP32 dW to device memory).
#include "instantiate.cuh"

template cudaError_t forge::launch_tile<0, forge::kEpiStoreGrad, 128>(const forge::TileLaunch&);
template cudaError_t forge::launch_tile<0, forge::kEpiStoreGrad, 256>(const forge::TileLaunch&);
