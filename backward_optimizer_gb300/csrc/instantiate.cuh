// instantiate.cuh -- defines the launchers declared in launch.h for one optimizer.
#pragma once

#include <atomic>

#include "launch.h"
#include "opt_step_kernel.cuh"
#include "tile_kernel.cuh"

namespace forge {

// a launch copies its whole group into the kernel's parameter space, whose limit is 32764 bytes
static_assert(sizeof(TileGroup<kMaxGroup>) <= 32764, "group of layers too large for the kernel parameters");

template <int OPT, int EPI, int BN, int CL, int OPS, int G>
cudaError_t launch_tile(const TileLaunch& l) {
    constexpr int CG = CL == 1 ? 1 : 2;
    using C = TileCfg<BN, CG, EPI, OPS>;
    auto kernel = forge_tile_kernel<BN, CL, EPI, OPT, OPS, G>;
    static std::atomic<uint64_t> configured{0};  // one bit per device ordinal
    static std::atomic<int> max_clusters[64];    // co-resident clusters per device
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    dev &= 63;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = CL;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(C::kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = l.stream;
    cfg.attrs = CL > 1 ? &attr : nullptr;
    cfg.numAttrs = CL > 1 ? 1 : 0;
    const uint64_t bit = 1ull << dev;
    if (!(configured.load() & bit)) {
        err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (err != cudaSuccess) return err;
        if (CL > 1) {
            int n = 0;
            cfg.gridDim = dim3(CL * l.num_sms, 1, 1);
            err = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
            if (err != cudaSuccess) return err;
            max_clusters[dev].store(n > 0 ? n : 1);
        }
        configured.fetch_or(bit);
    }
    // persistent grid: one CTA per SM (or one cluster per CL SMs), never more units than tiles.
    // Pair kernels with bf16 operands split a short last wave into half tiles (schedule.h).
    const int cap = CL == 1 ? l.num_sms : max_clusters[dev].load();
    constexpr bool kSplitTail = CG == 2 && BN == 256 && OPS == kOpsBF16;
    const int split_from = kSplitTail ? split_tail_from(l.num_tiles, cap) : l.num_tiles;
    const int launch_tiles = l.num_tiles + (l.num_tiles - split_from);
    const int units = launch_tiles < cap ? launch_tiles : cap;
    cfg.gridDim = dim3(units * CL, 1, 1);
    return cudaLaunchKernelEx(&cfg, kernel, *static_cast<const TileGroup<G>*>(l.group), split_from);
}

// CTA count and cluster size a launch_tile<..., BN, CL> call with `num_tiles` tiles would use.
template <int OPT, int EPI, int BN, int CL>
cudaError_t tile_grid(int num_tiles, int num_sms, int* ctas) {
    constexpr int CG = CL == 1 ? 1 : 2;
    using C = TileCfg<BN, CG, EPI>;
    auto kernel = forge_tile_kernel<BN, CL, EPI, OPT, kOpsBF16, 1>;
    int cap = num_sms;
    if (CL > 1) {
        cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (err != cudaSuccess) return err;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = CL;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.blockDim = dim3(C::kThreads, 1, 1);
        cfg.dynamicSmemBytes = C::kSmemBytes;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        cfg.gridDim = dim3(CL * num_sms, 1, 1);
        err = cudaOccupancyMaxActiveClusters(&cap, kernel, &cfg);
        if (err != cudaSuccess) return err;
    }
    *ctas = (num_tiles < cap ? num_tiles : cap) * CL;
    return cudaSuccess;
}

template <int OPT, int STATE>
cudaError_t launch_opt(const OptArgs& a, int grid, cudaStream_t stream) {
    forge_opt_kernel<OPT, STATE><<<grid, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace forge

#define FORGE_INSTANTIATE_TILES_OPS(OPT, EPI, OPS)                                               \
    template cudaError_t forge::launch_tile<OPT, EPI, 128, 1, OPS, 1>(const forge::TileLaunch&);    \
    template cudaError_t forge::launch_tile<OPT, EPI, 256, 1, OPS, 1>(const forge::TileLaunch&);    \
    template cudaError_t forge::launch_tile<OPT, EPI, 256, 2, OPS, 1>(const forge::TileLaunch&);

// Groups of up to kMaxGroup layers: CTA pairs, bf16 operands.
#define FORGE_INSTANTIATE_GROUP(OPT, EPI) \
    template cudaError_t forge::launch_tile<OPT, EPI, 256, 2, forge::kOpsBF16, forge::kMaxGroup>(const forge::TileLaunch&);

// 128 x 64 tiles for small layers: bf16 operands, every epilogue but the INT8 one.
#define FORGE_INSTANTIATE_NARROW(OPT, EPI) \
    template cudaError_t forge::launch_tile<OPT, EPI, 64, 1, forge::kOpsBF16, 1>(const forge::TileLaunch&);

#define FORGE_INSTANTIATE_TILES(OPT, EPI) FORGE_INSTANTIATE_TILES_OPS(OPT, EPI, forge::kOpsBF16)

// E4M3 operands, every state format.
#define FORGE_INSTANTIATE_OPT_E4M3(OPT)                                    \
    FORGE_INSTANTIATE_TILES_OPS(OPT, forge::kEpiOptFP32, forge::kOpsE4M3) \
    FORGE_INSTANTIATE_TILES_OPS(OPT, forge::kEpiOptINT8, forge::kOpsE4M3) \
    FORGE_INSTANTIATE_TILES_OPS(OPT, forge::kEpiOptBF16, forge::kOpsE4M3)

#define FORGE_INSTANTIATE_OPT(OPT)                    \
    FORGE_INSTANTIATE_TILES(OPT, forge::kEpiOptFP32) \
    FORGE_INSTANTIATE_NARROW(OPT, forge::kEpiOptFP32) \
    FORGE_INSTANTIATE_GROUP(OPT, forge::kEpiOptFP32) \
    template cudaError_t forge::launch_opt<OPT, 0>(const forge::OptArgs&, int, cudaStream_t);

#define FORGE_INSTANTIATE_OPT_INT8(OPT)               \
    FORGE_INSTANTIATE_TILES(OPT, forge::kEpiOptINT8) \
    FORGE_INSTANTIATE_GROUP(OPT, forge::kEpiOptINT8) \
    template cudaError_t forge::launch_opt<OPT, 1>(const forge::OptArgs&, int, cudaStream_t);

#define FORGE_INSTANTIATE_OPT_BF16(OPT)               \
    FORGE_INSTANTIATE_TILES(OPT, forge::kEpiOptBF16) \
    FORGE_INSTANTIATE_NARROW(OPT, forge::kEpiOptBF16) \
    FORGE_INSTANTIATE_GROUP(OPT, forge::kEpiOptBF16) \
    template cudaError_t forge::launch_opt<OPT, 2>(const forge::OptArgs&, int, cudaStream_t);
