// Kernel instantiations for one optimizer (radam).
#include "instantiate.cuh"
FORGE_INSTANTIATE_OPT(forge::kRAdam)
FORGE_INSTANTIATE_OPT_INT8(forge::kRAdam)
FORGE_INSTANTIATE_OPT_BF16(forge::kRAdam)
