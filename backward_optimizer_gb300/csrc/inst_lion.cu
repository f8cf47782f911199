// Kernel instantiations for one optimizer (lion).
#include "instantiate.cuh"
FORGE_INSTANTIATE_OPT(forge::kLion)
FORGE_INSTANTIATE_OPT_INT8(forge::kLion)
FORGE_INSTANTIATE_OPT_BF16(forge::kLion)
