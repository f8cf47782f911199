// Kernel instantiations for one optimizer (sgd).
#include "instantiate.cuh"
FORGE_INSTANTIATE_OPT(forge::kSGD)
