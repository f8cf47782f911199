// Kernel instantiations with E4M3 operands for one optimizer (rmsprop).
#include "instantiate.cuh"
FORGE_INSTANTIATE_OPT_E4M3(forge::kRMSprop)
