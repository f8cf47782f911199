// Kernel instantiations for one optimizer (nadam).
#include "instantiate.cuh"
FORGE_INSTANTIATE_OPT(forge::kNAdam)
FORGE_INSTANTIATE_OPT_INT8(forge::kNAdam)
FORGE_INSTANTIATE_OPT_BF16(forge::kNAdam)
