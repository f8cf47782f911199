// Kernel instantiations for one optimizer (sgd_momentum).
#include "instantiate.cuh"
FORGE_INSTANTIATE_OPT(forge::kSGDMomentum)
FORGE_INSTANTIATE_OPT_INT8(forge::kSGDMomentum)
FORGE_INSTANTIATE_OPT_BF16(forge::kSGDMomentum)
