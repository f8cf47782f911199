// Kernel instantiations for one optimizer (adamw).
#include "instantiate.cuh"
FORGE_INSTANTIATE_OPT(forge::kAdamW)
FORGE_INSTANTIATE_OPT_INT8(forge::kAdamW)
FORGE_INSTANTIATE_OPT_BF16(forge::kAdamW)
