// Kernel instantiations with E4M3 operands for one optimizer (sgd, which has no states), and the
// E4M3 weight-gradient GEMM (FP32 dW to device memory).
#include "instantiate.cuh"
FORGE_INSTANTIATE_TILES_OPS(forge::kSGD, forge::kEpiOptFP32, forge::kOpsE4M3)
FORGE_INSTANTIATE_TILES_OPS(0, forge::kEpiStoreGrad, forge::kOpsE4M3)
