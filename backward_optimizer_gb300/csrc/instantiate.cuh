// instantiate.cuh -- defines the launchers declared in launch.h for one optimizer.
#pragma once

#include <atomic>

#include "launch.h"
#include "opt_step_kernel.cuh"
#include "tile_kernel.cuh"

namespace forge {

template <int OPT, int EPI, int BN>
cudaError_t launch_tile(const TileLaunch& l) {
    using C = TileCfg<BN>;
    auto kernel = forge_tile_kernel<BN, EPI, OPT>;
    static std::atomic<uint64_t> configured{0};  // one bit per device ordinal
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(configured.load() & bit)) {
        err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (err != cudaSuccess) return err;
        configured.fetch_or(bit);
    }
    kernel<<<l.grid, kThreads, C::kSmemBytes, l.stream>>>(l.tmap_dy, l.tmap_x, *l.args);
    return cudaGetLastError();
}

template <int OPT, bool INT8>
cudaError_t launch_opt(const OptArgs& a, int grid, cudaStream_t stream) {
    forge_opt_kernel<OPT, INT8><<<grid, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace forge

#define FORGE_INSTANTIATE_OPT(OPT)                                                             \
    template cudaError_t forge::launch_tile<OPT, forge::kEpiOptFP32, 128>(const forge::TileLaunch&); \
    template cudaError_t forge::launch_tile<OPT, forge::kEpiOptFP32, 256>(const forge::TileLaunch&); \
    template cudaError_t forge::launch_opt<OPT, false>(const forge::OptArgs&, int, cudaStream_t);

#define FORGE_INSTANTIATE_OPT_INT8(OPT)                                                        \
    template cudaError_t forge::launch_tile<OPT, forge::kEpiOptINT8, 128>(const forge::TileLaunch&); \
    template cudaError_t forge::launch_tile<OPT, forge::kEpiOptINT8, 256>(const forge::TileLaunch&); \
    template cudaError_t forge::launch_opt<OPT, true>(const forge::OptArgs&, int, cudaStream_t);
