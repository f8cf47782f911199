// Kernel instantiations with E4M3 operands for one optimizer (lion).
#include "instantiate.cuh"
FORGE_INSTANTIATE_OPT_E4M3(forge::kLion)
