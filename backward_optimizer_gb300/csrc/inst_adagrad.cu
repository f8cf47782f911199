// Kernel instantiations for one optimizer (adagrad).
#include "instantiate.cuh"
FORGE_INSTANTIATE_OPT(forge::kAdaGrad)
FORGE_INSTANTIATE_OPT_INT8(forge::kAdaGrad)
FORGE_INSTANTIATE_OPT_BF16(forge::kAdaGrad)
