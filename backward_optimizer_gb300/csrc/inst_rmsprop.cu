// Kernel instantiations for one optimizer (rmsprop).
#include "instantiate.cuh"
FORGE_INSTANTIATE_OPT(forge::kRMSprop)
FORGE_INSTANTIATE_OPT_INT8(forge::kRMSprop)
FORGE_INSTANTIATE_OPT_BF16(forge::kRMSprop)
