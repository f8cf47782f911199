// Kernel instantiations of the unfused weight-gradient GEMM (FP32 dW to device memory), and the
// launch-shape query (every tile kernel runs one CTA per SM, so the GEMM's occupancy stands for all).
#include "instantiate.cuh"

FORGE_INSTANTIATE_TILES(0, forge::kEpiStoreGrad)
FORGE_INSTANTIATE_NARROW(0, forge::kEpiStoreGrad)

cudaError_t forge::tile_ctas(int bn, int cl, int num_tiles, int num_sms, int* ctas) {
    if (cl == 2) return tile_grid<0, kEpiStoreGrad, 256, 2>(num_tiles, num_sms, ctas);
    if (bn == 256) return tile_grid<0, kEpiStoreGrad, 256, 1>(num_tiles, num_sms, ctas);
    if (bn == 64) return tile_grid<0, kEpiStoreGrad, 64, 1>(num_tiles, num_sms, ctas);
    return tile_grid<0, kEpiStoreGrad, 128, 1>(num_tiles, num_sms, ctas);
}
