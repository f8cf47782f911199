// forge_api.cu -- the C ABI (include/forge.h): argument checks, step-dependent scalars,
// TMA descriptors, grid sizing and kernel dispatch.  Host code only, apart from the device
// status word.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "forge.h"
#include "launch.h"
#include "opt_step_kernel.cuh"
#include "tile_kernel.cuh"

// Device status word: 0, or the forge_status of the first bounded wait that ran out.
__device__ int g_forge_status_word;

namespace {

using forge::OptScalars;

constexpr int kMaxDevices = 64;
std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};
std::atomic<uint64_t> g_launches{0};
std::atomic<int> g_withhold_next{0};  // test switch, consumed by the next tile-kernel launch

struct DeviceInfo {
    bool ready = false;
    bool sm103 = false;
    int num_sms = 0;
    int* status = nullptr;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mutex;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

forge_status device_info(DeviceInfo** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FORGE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return FORGE_ERR_CUDA;
        d.sm103 = (major == 10 && minor == 3);
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_forge_status_word) != cudaSuccess) return FORGE_ERR_CUDA;
        d.status = static_cast<int*>(p);
        if (g_encode == nullptr) {
            cudaDriverEntryPointQueryResult q;
            void* fn = nullptr;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess || fn == nullptr)
                return FORGE_ERR_CUDA;
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        d.ready = true;
    }
    if (!d.sm103) return FORGE_ERR_NOT_SM103;
    *out = &d;
    return FORGE_OK;
}

bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

bool uses_m(forge_opt_kind k) {
    return k == FORGE_ADAMW || k == FORGE_NADAM || k == FORGE_RADAM || k == FORGE_LION || k == FORGE_SGD_MOMENTUM;
}
bool uses_v(forge_opt_kind k) {
    return k == FORGE_ADAMW || k == FORGE_NADAM || k == FORGE_RADAM || k == FORGE_RMSPROP || k == FORGE_ADAGRAD;
}

// NAdam's product of mu_1 .. mu_t, multiplied in order from i = 1.  Training calls this with the
// same (beta1, psi) and a step that grows by one, so each thread keeps its last product and
// extends it (the same sequence of multiplications, so the same bits); a step that goes
// backwards, or other hyperparameters, start again from 1.
double nadam_mu_product(double b1, double psi, int64_t step) {
    thread_local double c_b1 = -1.0, c_psi = -1.0, c_prod = 1.0;
    thread_local int64_t c_step = 0;
    if (b1 != c_b1 || psi != c_psi || step < c_step) {
        c_b1 = b1;
        c_psi = psi;
        c_step = 0;
        c_prod = 1.0;
    }
    for (int64_t i = c_step + 1; i <= step; ++i)
        c_prod *= b1 * (1.0 - 0.5 * std::pow(0.96, static_cast<double>(i) * psi));
    c_step = step;
    return c_prod;
}

// Step-dependent factors in binary64, rounded once to binary32 (optimizer definitions as cited
// in opt_math.cuh).
OptScalars derive_scalars(forge_opt_kind k, const forge_hparams& hp, int64_t step) {
    const double t = static_cast<double>(step);
    const double lr = hp.lr, b1 = hp.beta1, b2 = hp.beta2, eps = hp.eps, wd = hp.weight_decay;
    OptScalars s;
    std::memset(&s, 0, sizeof(s));
    s.lr = static_cast<float>(lr);
    s.eps = static_cast<float>(eps);
    s.wd = static_cast<float>(wd);
    s.decay = static_cast<float>(1.0 - lr * wd);
    s.b1 = static_cast<float>(b1);
    s.omb1 = static_cast<float>(1.0 - b1);
    s.b2 = static_cast<float>(b2);
    s.omb2 = static_cast<float>(1.0 - b2);
    const double bc1 = 1.0 - std::pow(b1, t), bc2 = 1.0 - std::pow(b2, t);
    switch (k) {
        case FORGE_ADAMW:
            s.step_size = static_cast<float>(lr / bc1);
            s.inv_sqrt_bc2 = static_cast<float>(1.0 / std::sqrt(bc2));
            break;
        case FORGE_NADAM: {
            const double psi = hp.momentum_decay;
            auto mu = [&](double i) { return b1 * (1.0 - 0.5 * std::pow(0.96, i * psi)); };
            const double prod = nadam_mu_product(b1, psi, step);
            const double mu_t = mu(t), mu_next = mu(t + 1.0);
            s.c_g = static_cast<float>(lr * (1.0 - mu_t) / (1.0 - prod));
            s.c_m = static_cast<float>(lr * mu_next / (1.0 - prod * mu_next));
            s.inv_sqrt_bc2 = static_cast<float>(1.0 / std::sqrt(bc2));
            break;
        }
        case FORGE_RADAM: {
            const double rho_inf = 2.0 / (1.0 - b2) - 1.0;
            const double rho_t = rho_inf - 2.0 * t * std::pow(b2, t) / bc2;
            if (rho_t > 5.0) {
                const double r = std::sqrt((rho_t - 4.0) * (rho_t - 2.0) * rho_inf /
                                           ((rho_inf - 4.0) * (rho_inf - 2.0) * rho_t));
                s.rectified = 1;
                s.step_size = static_cast<float>(lr * r * std::sqrt(bc2) / bc1);
            } else {
                s.rectified = 0;
                s.step_size = static_cast<float>(lr / bc1);
            }
            break;
        }
        case FORGE_LION:
            break;
        case FORGE_RMSPROP:
            s.b2 = hp.alpha;
            s.omb2 = static_cast<float>(1.0 - static_cast<double>(hp.alpha));
            break;
        case FORGE_ADAGRAD:
            s.lr = static_cast<float>(lr / (1.0 + (t - 1.0) * static_cast<double>(hp.lr_decay)));
            break;
        case FORGE_SGD:
            break;
        case FORGE_SGD_MOMENTUM:
            s.mu = hp.momentum;
            break;
    }
    return s;
}

forge_status encode_operand_map(CUtensorMap* map, const void* base, int64_t cols, int64_t rows, bool e4m3) {
    // A [rows, cols] row-major operand, bf16 or E4M3, read in boxes of 64 rows whose rows are
    // exactly one 128-byte swizzle span (64 bf16 or 128 E4M3 columns).
    const int64_t esize = e4m3 ? 1 : 2;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * esize)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / esize), 64};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, e4m3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                          const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FORGE_OK : FORGE_ERR_CUDA;
}

// Encoded tensor maps of recent calls, per host thread.  A training loop passes the same buffers
// with the same shapes every step, and encoding a map costs host time comparable to a small layer's
// whole kernel.  A map is plain host data determined by (base, cols, rows, element type), handed to
// the kernel by value, so a cached one is exactly the one a new encoding would give, whatever
// happened to the buffer in between.
struct MapKey {
    const void* base;
    int64_t cols, rows;
    bool e4m3;
    bool operator==(const MapKey& o) const {
        return base == o.base && cols == o.cols && rows == o.rows && e4m3 == o.e4m3;
    }
};
struct MapSlot {
    MapKey key;
    CUtensorMap map;
    bool used;
};
constexpr int kMapSlots = 64;
thread_local MapSlot t_maps[kMapSlots];

forge_status make_operand_map(CUtensorMap* map, const void* base, int64_t cols, int64_t rows, bool e4m3 = false) {
    const MapKey key{base, cols, rows, e4m3};
    uint64_t h = reinterpret_cast<uintptr_t>(base) * 0x9E3779B97F4A7C15ull;
    h ^= static_cast<uint64_t>(cols) * 0xC2B2AE3D27D4EB4Full ^ static_cast<uint64_t>(rows) * 0x165667B19E3779F9ull;
    h ^= e4m3 ? 0x27D4EB2F165667C5ull : 0;
    MapSlot& slot = t_maps[(h >> 32) % kMapSlots];
    if (slot.used && slot.key == key) {
        *map = slot.map;
        return FORGE_OK;
    }
    forge_status st = encode_operand_map(map, base, cols, rows, e4m3);
    if (st == FORGE_OK) {
        slot.key = key;
        slot.map = *map;
        slot.used = true;
    }
    return st;
}

// Sizes: any T >= 0 (the last 64-token slice is zero-filled past T); d_out and d_in multiples of 8,
// which a TMA row stride (16 bytes) and the epilogue's 16- and 32-byte accesses need.  Tiles that
// reach past the last row or column compute on zero fill and store nothing there.
forge_status check_shape(const forge_shape* shape) {
    if (shape == nullptr) return FORGE_ERR_INVALID_ARGUMENT;
    if (shape->d_out < 0 || shape->d_in < 0 || shape->T < 0 || shape->reserved != 0) return FORGE_ERR_INVALID_ARGUMENT;
    if (shape->d_out % 8 != 0 || shape->d_in % 8 != 0) return FORGE_ERR_INVALID_ARGUMENT;
    // TMA coordinates are 32-bit; the tile scheduler counts tiles in int.
    if (shape->d_out > (1ll << 30) || shape->d_in > (1ll << 30) || shape->T > (1ll << 30))
        return FORGE_ERR_INVALID_ARGUMENT;
    if ((shape->d_out / 128 + 1) * (shape->d_in / 128 + 1) > (1ll << 30)) return FORGE_ERR_INVALID_ARGUMENT;
    if (shape->state != FORGE_STATE_FP32 && shape->state != FORGE_STATE_INT8_B64 && shape->state != FORGE_STATE_BF16)
        return FORGE_ERR_INVALID_ARGUMENT;
    return FORGE_OK;
}

forge_status check_opt_args(const void* W, const void* m, const void* v, const float* qscales, forge_opt_kind k,
                            const forge_hparams* hp, const forge_shape* shape, int64_t step) {
    if (static_cast<int>(k) < 0 || static_cast<int>(k) > 7 || hp == nullptr || step < 1)
        return FORGE_ERR_INVALID_ARGUMENT;
    if (W == nullptr) return FORGE_ERR_INVALID_ARGUMENT;
    if (uses_m(k) && m == nullptr) return FORGE_ERR_INVALID_ARGUMENT;
    if (uses_v(k) && v == nullptr) return FORGE_ERR_INVALID_ARGUMENT;
    const bool int8 = shape->state == FORGE_STATE_INT8_B64;
    if (shape->state != FORGE_STATE_FP32 && k == FORGE_SGD) return FORGE_ERR_UNSUPPORTED;  // no states to store
    if (int8 && qscales == nullptr) return FORGE_ERR_INVALID_ARGUMENT;
    if (int8 && shape->d_in % 64 != 0) return FORGE_ERR_INVALID_ARGUMENT;  // a 64-block never spans two rows
    if (!aligned32(W) || (uses_m(k) && !aligned32(m)) || (uses_v(k) && !aligned32(v)) ||
        (int8 && (reinterpret_cast<uintptr_t>(qscales) & 3u)))
        return FORGE_ERR_MISALIGNED;
    return FORGE_OK;
}

forge_status cuda_status(cudaError_t e) { return e == cudaSuccess ? FORGE_OK : FORGE_ERR_CUDA; }

// Tile order: groups of kGroupRows tile rows, each group swept one tile column at a time, so the
// CTAs running at once share about kGroupRows dY slices and 76 / kGroupRows X slices in L2.  Both
// operands load with an L2 evict-last hint, ahead of the epilogue's weight and moment stream, which
// passes through L2 once.  Orders that keep the smaller operand wholly resident in L2 and stream the
// other (fewer DRAM bytes) measured 3-4 % slower on every Llama-3.1-8B and Qwen3-14B layer shape.
constexpr int kGroupRows = 8;

forge::TileOrder tile_order(int tiles_m, int tiles_n) {
    return forge::TileOrder{tiles_m, tiles_n, tiles_m < kGroupRows ? tiles_m : kGroupRows, 0};
}

// The epilogue's wait for a finished accumulator spans a whole tile mainloop: the base limit plus
// 4 us per reduction slice (a slice takes well under 1 us on a GB300), saturating.
uint64_t acc_wait_limit(uint64_t base_ns, int64_t k_blocks) {
    const uint64_t per = 4000ull, extra = static_cast<uint64_t>(k_blocks) * per;
    return extra > ~0ull - base_ns ? ~0ull : base_ns + extra;
}

// Dispatch tables (filled by template instantiation in the inst_*.cu units).
using TileFn = cudaError_t (*)(const forge::TileLaunch&);
using OptFn = cudaError_t (*)(const forge::OptArgs&, int, cudaStream_t);

template <int OPT, int BN, int CL, int OPS, int G = 1>
TileFn tile_fn_state(int state) {
    using namespace forge;
    if (state == FORGE_STATE_INT8_B64) {
        if constexpr (BN == 64) return nullptr;  // INT8 blocks need 64 columns per epilogue warp
        else return launch_tile<OPT, kEpiOptINT8, BN, CL, OPS, G>;
    }
    if (state == FORGE_STATE_BF16) return launch_tile<OPT, kEpiOptBF16, BN, CL, OPS, G>;
    return launch_tile<OPT, kEpiOptFP32, BN, CL, OPS, G>;
}

template <int BN, int CL, int OPS, int G = 1>
TileFn tile_fn_v(forge_opt_kind k, int state) {
    using namespace forge;
    switch (k) {
        case FORGE_ADAMW: return tile_fn_state<kAdamW, BN, CL, OPS, G>(state);
        case FORGE_NADAM: return tile_fn_state<kNAdam, BN, CL, OPS, G>(state);
        case FORGE_RADAM: return tile_fn_state<kRAdam, BN, CL, OPS, G>(state);
        case FORGE_LION: return tile_fn_state<kLion, BN, CL, OPS, G>(state);
        case FORGE_RMSPROP: return tile_fn_state<kRMSprop, BN, CL, OPS, G>(state);
        case FORGE_ADAGRAD: return tile_fn_state<kAdaGrad, BN, CL, OPS, G>(state);
        case FORGE_SGD:
            return state == FORGE_STATE_FP32 ? launch_tile<kSGD, kEpiOptFP32, BN, CL, OPS, G> : nullptr;
        case FORGE_SGD_MOMENTUM: return tile_fn_state<kSGDMomentum, BN, CL, OPS, G>(state);
    }
    return nullptr;
}

// Tile shape per call.  The mainloop is bound by operand traffic from L2 into shared memory, so a
// wide shape is preferred: a CTA pair on 256 x 256 (each CTA stages half of X), one CTA on
// 128 x 256, one CTA on 128 x 128; each is a group of the method's 128 x 128 tiles side by side.
// A layer whose preferred shape would run on at most half the SMs takes 128 x 128 tiles instead:
// there the number of SMs sharing the epilogue matters more than the mainloop's efficiency
// (measured on 1024^2 and 1536^2 layers at T = 4096: 21-25 % faster).  If even those would run on
// at most half the SMs, calls that allow it (bf16 operands, an epilogue that works on 32-column
// runs: not INT8 states) take 128 x 64 tiles, twice as many CTAs again.
struct TileShape {
    int bn;     // columns per CTA pair (or per CTA)
    int cg;     // CTAs per MMA = CTAs per cluster
};
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// rows x cols of the output (dW: d_out x d_in; dX: T x d_in).  A ragged dimension (not a multiple
// of the tile) takes the wide shape once it is large enough that the zero-filled tail costs little
// (over 1024).
TileShape pick_tiles(int64_t rows, int64_t cols, int num_sms, bool narrow_ok) {
    const bool rows256 = rows % 256 == 0 || (rows % 128 != 0 && rows > 1024);
    const bool cols256 = cols % 256 == 0 || (cols % 128 != 0 && cols > 1024);
    auto ctas = [&](TileShape t) { return ceil_div(rows, 128 * t.cg) * ceil_div(cols, t.bn) * t.cg; };
    TileShape t{128, 1};
    if (rows256 && cols256) t = {256, 2};
    else if (cols256) t = {256, 1};
    if (2 * ctas(t) > num_sms) return t;
    t = {128, 1};
    if (narrow_ok && 2 * ctas(t) <= num_sms) return {64, 1};
    return t;
}

// narrow_ok: bf16 operands and binary32 or bfloat16 states (or the dW GEMM alone)
TileShape pick_shape(int64_t d_out, int64_t d_in, int64_t /*T*/, int num_sms, bool narrow_ok) {
    return pick_tiles(d_out, d_in, num_sms, narrow_ok);
}

// Input gradient dX = dY W: tile rows are tokens (M = T), columns d_in (N), reduction over d_out (K).
TileShape pick_dx_shape(int64_t T, int64_t /*d_out*/, int64_t d_in, int num_sms) {
    return pick_tiles(T, d_in, num_sms, true);
}

template <int OPS>
TileFn tile_fn_ops(forge_opt_kind k, int state, int epi, TileShape t) {
    using namespace forge;
    if (epi == kEpiDX) {
        if constexpr (OPS != kOpsBF16) return nullptr;
        if (t.cg == 2) return launch_tile<0, kEpiDX, 256, 2, kOpsBF16, 1>;
        if (t.bn == 64) return launch_tile<0, kEpiDX, 64, 1, kOpsBF16, 1>;
        return t.bn == 256 ? launch_tile<0, kEpiDX, 256, 1, kOpsBF16, 1> : launch_tile<0, kEpiDX, 128, 1, kOpsBF16, 1>;
    }
    if (epi == kEpiStoreGrad) {
        if (t.cg == 2) return launch_tile<0, kEpiStoreGrad, 256, 2, OPS, 1>;
        if (t.bn == 64) {
            if constexpr (OPS != kOpsBF16) return nullptr;
            else return launch_tile<0, kEpiStoreGrad, 64, 1, kOpsBF16, 1>;
        }
        return t.bn == 256 ? launch_tile<0, kEpiStoreGrad, 256, 1, OPS, 1> : launch_tile<0, kEpiStoreGrad, 128, 1, OPS, 1>;
    }
    if (t.cg == 2) return tile_fn_v<256, 2, OPS>(k, state);
    if (t.bn == 64) {
        if constexpr (OPS != kOpsBF16) return nullptr;
        else return state == FORGE_STATE_INT8_B64 ? nullptr : tile_fn_v<64, 1, OPS>(k, state);
    }
    return t.bn == 256 ? tile_fn_v<256, 1, OPS>(k, state) : tile_fn_v<128, 1, OPS>(k, state);
}

TileFn tile_fn(forge_opt_kind k, int state, int epi, TileShape t, bool e4m3) {
    return e4m3 ? tile_fn_ops<forge::kOpsE4M3>(k, state, epi, t) : tile_fn_ops<forge::kOpsBF16>(k, state, epi, t);
}

template <int OPT>
OptFn opt_fn_state(int state) {
    using namespace forge;
    if (state == FORGE_STATE_INT8_B64) return launch_opt<OPT, 1>;
    if (state == FORGE_STATE_BF16) return launch_opt<OPT, 2>;
    return launch_opt<OPT, 0>;
}

OptFn opt_fn(forge_opt_kind k, int state) {
    using namespace forge;
    switch (k) {
        case FORGE_ADAMW: return opt_fn_state<kAdamW>(state);
        case FORGE_NADAM: return opt_fn_state<kNAdam>(state);
        case FORGE_RADAM: return opt_fn_state<kRAdam>(state);
        case FORGE_LION: return opt_fn_state<kLion>(state);
        case FORGE_RMSPROP: return opt_fn_state<kRMSprop>(state);
        case FORGE_ADAGRAD: return opt_fn_state<kAdaGrad>(state);
        case FORGE_SGD: return state == FORGE_STATE_FP32 ? launch_opt<kSGD, 0> : nullptr;
        case FORGE_SGD_MOMENTUM: return opt_fn_state<kSGDMomentum>(state);
    }
    return nullptr;
}

forge_status run_opt(const float* dW, void* W, void* m, void* v, float* qscales, forge_opt_kind k,
                     const forge_hparams* hp, const forge_shape* shape, int64_t step, uint64_t seed,
                     cudaStream_t stream, const DeviceInfo& dev) {
    const bool int8 = shape->state == FORGE_STATE_INT8_B64;
    const uint64_t n = static_cast<uint64_t>(shape->d_out) * static_cast<uint64_t>(shape->d_in);
    forge::OptArgs a;
    a.dW = dW;
    a.W = static_cast<uint16_t*>(W);
    a.m = m;
    a.v = v;
    a.m_scales = int8 ? qscales : nullptr;
    a.v_scales = int8 ? qscales + n / 64 : nullptr;
    a.n8 = n / 8;
    a.s = derive_scalars(k, *hp, step);
    a.seed = seed;
    a.step = static_cast<uint64_t>(step);
    const uint64_t blocks = (a.n8 + 255) / 256;
    const uint64_t cap = static_cast<uint64_t>(dev.num_sms) * 8;
    const int grid = static_cast<int>(blocks < cap ? blocks : cap);
    OptFn fn = opt_fn(k, shape->state);
    if (fn == nullptr) return FORGE_ERR_UNSUPPORTED;
    g_launches.fetch_add(1);
    return cuda_status(fn(a, grid, stream));
}

// One layer's kernel arguments and tensor maps for tile shape ts.  e4m3: dY and X are E4M3 codes and
// the gradient tile is scaled by g_scale = s_dY * s_X (or per channel by row_scales x col_scales).
forge_status prepare_layer(forge::TileArgs& a, CUtensorMap* maps, const void* dY, const void* X, float* dW, void* W,
                           void* m, void* v, float* qscales, forge_opt_kind k, const forge_hparams* hp,
                           const forge_shape* shape, int64_t step, uint64_t seed, const DeviceInfo& dev, TileShape ts,
                           bool e4m3, float g_scale, const float* row_scales, const float* col_scales,
                           int withhold) {
    const bool int8 = shape->state == FORGE_STATE_INT8_B64;
    const uint64_t n = static_cast<uint64_t>(shape->d_out) * static_cast<uint64_t>(shape->d_in);
    std::memset(&a, 0, sizeof(a));
    a.d_out = static_cast<int>(shape->d_out);
    a.d_in = static_cast<int>(shape->d_in);
    a.T = static_cast<int>(shape->T);
    const int tiles_m = static_cast<int>(ceil_div(a.d_out, forge::kBM * ts.cg));
    const int tiles_n = static_cast<int>(ceil_div(a.d_in, ts.bn));
    a.num_tiles = tiles_m * tiles_n;
    a.k_blocks = static_cast<int>(ceil_div(a.T, e4m3 ? 128 : forge::kBK));
    a.order = tile_order(tiles_m, tiles_n);
    a.g_scale = g_scale;
    a.row_scales = row_scales;
    a.col_scales = col_scales;
    a.dW = dW;
    a.W = static_cast<uint16_t*>(W);
    a.m = m;
    a.v = v;
    a.m_scales = int8 ? qscales : nullptr;
    a.v_scales = int8 ? qscales + n / 64 : nullptr;
    if (hp != nullptr) a.s = derive_scalars(k, *hp, step);
    a.seed = seed;
    a.step = static_cast<uint64_t>(step);
    a.status = dev.status;
    a.wait_limit_ns = g_wait_limit_ns.load();
    a.acc_wait_limit_ns = acc_wait_limit(a.wait_limit_ns, a.k_blocks);
    a.withhold_first_stage = withhold;
    forge_status st = make_operand_map(&maps[0], dY, shape->d_out, shape->T, e4m3);
    if (st != FORGE_OK) return st;
    return make_operand_map(&maps[1], X, shape->d_in, shape->T, e4m3);
}

forge_status run_tile(const void* dY, const void* X, float* dW, void* W, void* m, void* v, float* qscales,
                      forge_opt_kind k, int epi, const forge_hparams* hp, const forge_shape* shape, int64_t step,
                      uint64_t seed, cudaStream_t stream, const DeviceInfo& dev, bool e4m3 = false,
                      float g_scale = 1.0f, const float* row_scales = nullptr, const float* col_scales = nullptr) {
    // 128 x 64 tiles need bf16 operands and an epilogue on 32-column runs (not INT8 states)
    const bool narrow_ok = !e4m3 && (epi == forge::kEpiStoreGrad || shape->state != FORGE_STATE_INT8_B64);
    const TileShape ts = pick_shape(shape->d_out, shape->d_in, shape->T, dev.num_sms, narrow_ok);
    forge::TileGroup<1> g;
    g.n = 1;
    forge_status st = prepare_layer(g.layer[0], g.maps, dY, X, dW, W, m, v, qscales, k, hp, shape, step, seed, dev,
                                    ts, e4m3, g_scale, row_scales, col_scales, g_withhold_next.exchange(0));
    if (st != FORGE_OK) return st;
    g.tile_start[0] = 0;
    g.tile_start[1] = g.layer[0].num_tiles;
    forge::TileLaunch l{&g, g.tile_start[1], dev.num_sms, stream};
    // epi is kEpiStoreGrad (dW to memory) or kEpiOptFP32 (the fused step, whose epilogue follows the state dtype)
    TileFn fn = tile_fn(k, shape->state, epi, ts, e4m3);
    if (fn == nullptr) return FORGE_ERR_UNSUPPORTED;
    g_launches.fetch_add(1);
    return cuda_status(fn(l));
}

forge_status run_dx(const void* dY, const void* W, void* dX, const forge_shape* shape, cudaStream_t stream,
                    const DeviceInfo& dev) {
    forge::TileGroup<1> g;
    g.n = 1;
    forge::TileArgs& a = g.layer[0];
    std::memset(&a, 0, sizeof(a));
    a.d_out = static_cast<int>(shape->d_out);
    a.d_in = static_cast<int>(shape->d_in);
    a.T = static_cast<int>(shape->T);
    const TileShape ts = pick_dx_shape(shape->T, shape->d_out, shape->d_in, dev.num_sms);
    const int rows = forge::kBM * ts.cg;
    const int tiles_m = static_cast<int>(ceil_div(a.T, rows));
    const int tiles_n = static_cast<int>(ceil_div(a.d_in, ts.bn));
    a.num_tiles = tiles_m * tiles_n;
    a.k_blocks = static_cast<int>(ceil_div(a.d_out, forge::kBK));
    a.order = tile_order(tiles_m, tiles_n);
    a.dX = static_cast<uint16_t*>(dX);
    a.status = dev.status;
    a.wait_limit_ns = g_wait_limit_ns.load();
    a.acc_wait_limit_ns = acc_wait_limit(a.wait_limit_ns, a.k_blocks);
    a.withhold_first_stage = g_withhold_next.exchange(0);
    // A = dY [T, d_out] read K-major with the same box as the weight gradient's dY^T; B = W
    // [d_out, d_in] read MN-major like X
    forge_status st = make_operand_map(&g.maps[0], dY, shape->d_out, shape->T);
    if (st != FORGE_OK) return st;
    st = make_operand_map(&g.maps[1], W, shape->d_in, shape->d_out);
    if (st != FORGE_OK) return st;
    g.tile_start[0] = 0;
    g.tile_start[1] = a.num_tiles;
    forge::TileLaunch l{&g, a.num_tiles, dev.num_sms, stream};
    TileFn fn = tile_fn(FORGE_SGD, FORGE_STATE_FP32, forge::kEpiDX, ts, false);
    if (fn == nullptr) return FORGE_ERR_UNSUPPORTED;
    g_launches.fetch_add(1);
    return cuda_status(fn(l));
}

// Argument checks of each entry point, separate from its launch so that forge_linear_backward can
// check both calls before launching either.
forge_status check_fused(const void* dY, const void* X, const void* W, const void* m, const void* v,
                         const float* qscales, forge_opt_kind k, const forge_hparams* hp, const forge_shape* shape,
                         int64_t step) {
    forge_status st = check_shape(shape);
    if (st != FORGE_OK) return st;
    if (shape->d_out == 0 || shape->d_in == 0) return FORGE_OK;  // empty layer: nothing to read or write
    st = check_opt_args(W, m, v, qscales, k, hp, shape, step);
    if (st != FORGE_OK) return st;
    if (shape->T > 0 && (dY == nullptr || X == nullptr)) return FORGE_ERR_INVALID_ARGUMENT;
    if (shape->T > 0 && (!aligned32(dY) || !aligned32(X))) return FORGE_ERR_MISALIGNED;
    return FORGE_OK;
}

forge_status launch_fused(const void* dY, const void* X, void* W, void* m, void* v, float* qscales,
                          forge_opt_kind k, const forge_hparams* hp, const forge_shape* shape, int64_t step,
                          uint64_t seed, cudaStream_t stream, bool e4m3 = false, float g_scale = 1.0f,
                          const float* row_scales = nullptr, const float* col_scales = nullptr) {
    if (shape->d_out == 0 || shape->d_in == 0) return FORGE_OK;
    DeviceInfo* dev = nullptr;
    forge_status st = device_info(&dev);
    if (st != FORGE_OK) return st;
    if (shape->T == 0)  // no tokens: the gradient is exactly zero
        return run_opt(nullptr, W, m, v, qscales, k, hp, shape, step, seed, stream, *dev);
    return run_tile(dY, X, nullptr, W, m, v, qscales, k, forge::kEpiOptFP32, hp, shape, step, seed, stream, *dev,
                    e4m3, g_scale, row_scales, col_scales);
}

// E4M3 operands: rows of dY and X are d_out and d_in bytes, a multiple of 16 for TMA; the scales are
// finite and positive.
forge_status check_e4m3(const forge_shape* shape, float dy_scale, float x_scale) {
    if (shape->d_out % 16 != 0 || shape->d_in % 16 != 0) return FORGE_ERR_INVALID_ARGUMENT;
    if (!(dy_scale > 0.0f && dy_scale < INFINITY) || !(x_scale > 0.0f && x_scale < INFINITY))
        return FORGE_ERR_INVALID_ARGUMENT;
    return FORGE_OK;
}

forge_status check_dx(const void* dY, const void* W, const void* dX, const forge_shape* shape) {
    forge_status st = check_shape(shape);
    if (st != FORGE_OK) return st;
    if (shape->T == 0 || shape->d_in == 0) return FORGE_OK;  // dX is empty
    if ((shape->T / 128 + 1) * (shape->d_in / 128) > (1ll << 30)) return FORGE_ERR_INVALID_ARGUMENT;
    if (dX == nullptr) return FORGE_ERR_INVALID_ARGUMENT;
    if (!aligned32(dX)) return FORGE_ERR_MISALIGNED;
    if (shape->d_out == 0) return FORGE_OK;  // dX is zero; dY and W are empty
    if (dY == nullptr || W == nullptr) return FORGE_ERR_INVALID_ARGUMENT;
    if (!aligned32(dY) || !aligned32(W)) return FORGE_ERR_MISALIGNED;
    return FORGE_OK;
}

forge_status launch_dx(const void* dY, const void* W, void* dX, const forge_shape* shape, cudaStream_t stream) {
    if (shape->T == 0 || shape->d_in == 0) return FORGE_OK;
    DeviceInfo* dev = nullptr;
    forge_status st = device_info(&dev);
    if (st != FORGE_OK) return st;
    if (shape->d_out == 0)
        return cuda_status(
            cudaMemsetAsync(dX, 0, static_cast<size_t>(shape->T) * static_cast<size_t>(shape->d_in) * 2, stream));
    return run_dx(dY, W, dX, shape, stream, *dev);
}

}  // namespace

extern "C" {

forge_status forge_fused_dw_step(const void* dY, const void* X, void* W, void* m, void* v, float* qscales,
                                 forge_opt_kind opt_kind, const forge_hparams* hp, const forge_shape* shape,
                                 int64_t step, uint64_t seed, struct CUstream_st* stream) {
    forge_status st = check_fused(dY, X, W, m, v, qscales, opt_kind, hp, shape, step);
    if (st != FORGE_OK) return st;
    return launch_fused(dY, X, W, m, v, qscales, opt_kind, hp, shape, step, seed, stream);
}

forge_status forge_fused_dw_step_e4m3(const void* dY, const void* X, float dy_scale, float x_scale, void* W, void* m,
                                      void* v, float* qscales, forge_opt_kind opt_kind, const forge_hparams* hp,
                                      const forge_shape* shape, int64_t step, uint64_t seed,
                                      struct CUstream_st* stream) {
    forge_status st = check_fused(dY, X, W, m, v, qscales, opt_kind, hp, shape, step);
    if (st != FORGE_OK) return st;
    st = check_e4m3(shape, dy_scale, x_scale);
    if (st != FORGE_OK) return st;
    const float g_scale = dy_scale * x_scale;  // one binary32 rounding
    return launch_fused(dY, X, W, m, v, qscales, opt_kind, hp, shape, step, seed, stream, true, g_scale);
}

// Per-channel E4M3 scales: device vectors of d_out and d_in binary32 values, 16-byte aligned.
forge_status check_channel_scales(const forge_shape* shape, const float* dy_scales, const float* x_scales) {
    if (shape->d_out == 0 || shape->d_in == 0 || shape->T == 0) return FORGE_OK;  // not read
    if (dy_scales == nullptr || x_scales == nullptr) return FORGE_ERR_INVALID_ARGUMENT;
    if ((reinterpret_cast<uintptr_t>(dy_scales) & 15u) || (reinterpret_cast<uintptr_t>(x_scales) & 15u))
        return FORGE_ERR_MISALIGNED;
    return FORGE_OK;
}

forge_status forge_fused_dw_step_e4m3_channels(const void* dY, const void* X, const float* dy_scales,
                                               const float* x_scales, void* W, void* m, void* v, float* qscales,
                                               forge_opt_kind opt_kind, const forge_hparams* hp,
                                               const forge_shape* shape, int64_t step, uint64_t seed,
                                               struct CUstream_st* stream) {
    forge_status st = check_fused(dY, X, W, m, v, qscales, opt_kind, hp, shape, step);
    if (st != FORGE_OK) return st;
    st = check_e4m3(shape, 1.0f, 1.0f);
    if (st != FORGE_OK) return st;
    st = check_channel_scales(shape, dy_scales, x_scales);
    if (st != FORGE_OK) return st;
    return launch_fused(dY, X, W, m, v, qscales, opt_kind, hp, shape, step, seed, stream, true, 1.0f, dy_scales,
                        x_scales);
}

forge_status forge_dw_gemm_e4m3_channels(const void* dY, const void* X, const float* dy_scales, const float* x_scales,
                                         float* dW, const forge_shape* shape, struct CUstream_st* stream) {
    forge_status st = check_shape(shape);
    if (st != FORGE_OK) return st;
    st = check_e4m3(shape, 1.0f, 1.0f);
    if (st != FORGE_OK) return st;
    st = check_channel_scales(shape, dy_scales, x_scales);
    if (st != FORGE_OK) return st;
    if (shape->d_out == 0 || shape->d_in == 0) return FORGE_OK;
    if (dW == nullptr || (shape->T > 0 && (dY == nullptr || X == nullptr))) return FORGE_ERR_INVALID_ARGUMENT;
    if (!aligned32(dW) || (shape->T > 0 && (!aligned32(dY) || !aligned32(X)))) return FORGE_ERR_MISALIGNED;
    DeviceInfo* dev = nullptr;
    st = device_info(&dev);
    if (st != FORGE_OK) return st;
    if (shape->T == 0)
        return cuda_status(cudaMemsetAsync(dW, 0, static_cast<size_t>(shape->d_out) * shape->d_in * sizeof(float),
                                           stream));
    return run_tile(dY, X, dW, nullptr, nullptr, nullptr, nullptr, FORGE_SGD, forge::kEpiStoreGrad, nullptr, shape,
                    1, 0, stream, *dev, true, 1.0f, dy_scales, x_scales);
}

forge_status forge_dw_gemm_e4m3(const void* dY, const void* X, float dy_scale, float x_scale, float* dW,
                                const forge_shape* shape, struct CUstream_st* stream) {
    forge_status st = check_shape(shape);
    if (st != FORGE_OK) return st;
    st = check_e4m3(shape, dy_scale, x_scale);
    if (st != FORGE_OK) return st;
    if (shape->d_out == 0 || shape->d_in == 0) return FORGE_OK;
    if (dW == nullptr || (shape->T > 0 && (dY == nullptr || X == nullptr))) return FORGE_ERR_INVALID_ARGUMENT;
    if (!aligned32(dW) || (shape->T > 0 && (!aligned32(dY) || !aligned32(X)))) return FORGE_ERR_MISALIGNED;
    DeviceInfo* dev = nullptr;
    st = device_info(&dev);
    if (st != FORGE_OK) return st;
    if (shape->T == 0)
        return cuda_status(cudaMemsetAsync(dW, 0, static_cast<size_t>(shape->d_out) * shape->d_in * sizeof(float),
                                           stream));
    return run_tile(dY, X, dW, nullptr, nullptr, nullptr, nullptr, FORGE_SGD, forge::kEpiStoreGrad, nullptr, shape,
                    1, 0, stream, *dev, true, dy_scale * x_scale);
}

forge_status forge_dx_gemm(const void* dY, const void* W, void* dX, const forge_shape* shape,
                           struct CUstream_st* stream) {
    forge_status st = check_dx(dY, W, dX, shape);
    if (st != FORGE_OK) return st;
    return launch_dx(dY, W, dX, shape, stream);
}

forge_status forge_linear_backward(const void* dY, const void* X, void* W, void* m, void* v, float* qscales,
                                   void* dX, forge_opt_kind opt_kind, const forge_hparams* hp,
                                   const forge_shape* shape, int64_t step, uint64_t seed,
                                   struct CUstream_st* stream) {
    forge_status st = check_fused(dY, X, W, m, v, qscales, opt_kind, hp, shape, step);
    if (st != FORGE_OK) return st;
    st = check_dx(dY, W, dX, shape);
    if (st != FORGE_OK) return st;
    // dX reads W before the fused step replaces it: same stream, this order
    st = launch_dx(dY, W, dX, shape, stream);
    if (st != FORGE_OK) return st;
    return launch_fused(dY, X, W, m, v, qscales, opt_kind, hp, shape, step, seed, stream);
}

forge_status forge_fused_dw_step_layers(const forge_layer* layers, int32_t n_layers, int32_t state,
                                        forge_opt_kind opt_kind, const forge_hparams* hp, int64_t step,
                                        struct CUstream_st* stream) {
    if (n_layers < 0 || (n_layers > 0 && layers == nullptr)) return FORGE_ERR_INVALID_ARGUMENT;
    auto shape_of = [&](const forge_layer& L) { return forge_shape{L.T, L.d_out, L.d_in, state, 0}; };
    for (int32_t i = 0; i < n_layers; ++i) {
        const forge_layer& L = layers[i];
        const forge_shape sh = shape_of(L);
        forge_status st = check_fused(L.dY, L.X, L.W, L.m, L.v, L.qscales, opt_kind, hp, &sh, step);
        if (st != FORGE_OK) return st;
    }
    if (n_layers == 0) return FORGE_OK;
    DeviceInfo* dev = nullptr;
    forge_status st = device_info(&dev);
    if (st != FORGE_OK) return st;
    // layers that run together: non-empty, with tokens, whose preferred tile is a CTA pair; together
    // they must still fill more than half the SMs, else each takes its own shape
    auto pair_shaped = [](const forge_layer& L) {
        const bool rows256 = L.d_out % 256 == 0 || (L.d_out % 128 != 0 && L.d_out > 1024);
        const bool cols256 = L.d_in % 256 == 0 || (L.d_in % 128 != 0 && L.d_in > 1024);
        return L.T > 0 && L.d_out > 0 && L.d_in > 0 && rows256 && cols256;
    };
    int64_t pair_ctas = 0;
    for (int32_t i = 0; i < n_layers; ++i)
        if (pair_shaped(layers[i])) pair_ctas += 2 * ceil_div(layers[i].d_out, 256) * ceil_div(layers[i].d_in, 256);
    const bool group = 2 * pair_ctas > dev->num_sms;
    TileFn fn = group ? tile_fn_v<256, 2, forge::kOpsBF16, forge::kMaxGroup>(opt_kind, state) : nullptr;
    if (group && fn == nullptr) return FORGE_ERR_UNSUPPORTED;
    constexpr TileShape kPair{256, 2};
    int32_t next = 0;  // layers [0, next) are launched
    while (next < n_layers) {
        // a layer with no pair-shaped neighbour to share a launch with runs alone, on the
        // single-layer kernel (the grouped one reads its arguments through a layer index)
        const bool alone = next + 1 >= n_layers || !pair_shaped(layers[next + 1]);
        if (!group || !pair_shaped(layers[next]) || alone) {
            const forge_layer& L = layers[next++];
            const forge_shape sh = shape_of(L);
            st = launch_fused(L.dY, L.X, L.W, L.m, L.v, L.qscales, opt_kind, hp, &sh, step, L.seed, stream);
            if (st != FORGE_OK) return st;
            continue;
        }
        // up to kMaxGroup consecutive pair-shaped layers in one launch
        static thread_local forge::TileGroup<forge::kMaxGroup> g;
        g.n = 0;
        g.tile_start[0] = 0;
        const int withhold = g_withhold_next.exchange(0);
        while (next < n_layers && g.n < forge::kMaxGroup && pair_shaped(layers[next])) {
            const forge_layer& L = layers[next++];
            const forge_shape sh = shape_of(L);
            st = prepare_layer(g.layer[g.n], &g.maps[2 * g.n], L.dY, L.X, nullptr, L.W, L.m, L.v, L.qscales, opt_kind,
                               hp, &sh, step, L.seed, *dev, kPair, false, 1.0f, nullptr, nullptr,
                               g.n == 0 ? withhold : 0);
            if (st != FORGE_OK) return st;
            g.tile_start[g.n + 1] = g.tile_start[g.n] + g.layer[g.n].num_tiles;
            ++g.n;
        }
        forge::TileLaunch l{&g, g.tile_start[g.n], dev->num_sms, stream};
        g_launches.fetch_add(1);
        st = cuda_status(fn(l));
        if (st != FORGE_OK) return st;
    }
    return FORGE_OK;
}

forge_status forge_dw_gemm(const void* dY, const void* X, float* dW, const forge_shape* shape,
                           struct CUstream_st* stream) {
    forge_status st = check_shape(shape);
    if (st != FORGE_OK) return st;
    if (shape->d_out == 0 || shape->d_in == 0) return FORGE_OK;
    if (dW == nullptr || (shape->T > 0 && (dY == nullptr || X == nullptr))) return FORGE_ERR_INVALID_ARGUMENT;
    if (!aligned32(dW) || (shape->T > 0 && (!aligned32(dY) || !aligned32(X)))) return FORGE_ERR_MISALIGNED;
    DeviceInfo* dev = nullptr;
    st = device_info(&dev);
    if (st != FORGE_OK) return st;
    if (shape->T == 0)
        return cuda_status(cudaMemsetAsync(dW, 0, static_cast<size_t>(shape->d_out) * shape->d_in * sizeof(float),
                                           stream));
    return run_tile(dY, X, dW, nullptr, nullptr, nullptr, nullptr, FORGE_SGD, forge::kEpiStoreGrad, nullptr, shape,
                    1, 0, stream, *dev);
}

forge_status forge_opt_step(const float* dW, void* W, void* m, void* v, float* qscales, forge_opt_kind opt_kind,
                            const forge_hparams* hp, const forge_shape* shape, int64_t step, uint64_t seed,
                            struct CUstream_st* stream) {
    forge_status st = check_shape(shape);
    if (st != FORGE_OK) return st;
    if (shape->d_out == 0 || shape->d_in == 0) return FORGE_OK;
    st = check_opt_args(W, m, v, qscales, opt_kind, hp, shape, step);
    if (st != FORGE_OK) return st;
    if (dW != nullptr && !aligned32(dW)) return FORGE_ERR_MISALIGNED;
    DeviceInfo* dev = nullptr;
    st = device_info(&dev);
    if (st != FORGE_OK) return st;
    return run_opt(dW, W, m, v, qscales, opt_kind, hp, shape, step, seed, stream, *dev);
}

forge_status forge_sync_status(struct CUstream_st* stream) {
    DeviceInfo* dev = nullptr;
    forge_status st = device_info(&dev);
    if (st != FORGE_OK) return st;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return FORGE_ERR_CUDA;
    int word = 0;
    if (cudaMemcpy(&word, dev->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FORGE_ERR_CUDA;
    if (word != 0) {
        const int zero = 0;
        if (cudaMemcpy(dev->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return FORGE_ERR_CUDA;
        return static_cast<forge_status>(word);
    }
    return FORGE_OK;
}

void forge_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns.store(ns < 1000000ull ? 1000000ull : ns); }

void forge_debug_withhold_next_stage(void) { g_withhold_next.store(1); }

forge_status forge_launch_shape(const forge_shape* shape, int32_t* tile_rows, int32_t* tile_cols,
                                int32_t* cluster, int32_t* ctas) {
    forge_status st = check_shape(shape);
    if (st != FORGE_OK) return st;
    if (tile_rows == nullptr || tile_cols == nullptr || cluster == nullptr || ctas == nullptr)
        return FORGE_ERR_INVALID_ARGUMENT;
    *tile_rows = *tile_cols = *cluster = *ctas = 0;
    DeviceInfo* dev = nullptr;
    st = device_info(&dev);
    if (st != FORGE_OK) return st;
    const TileShape ts = pick_shape(shape->d_out, shape->d_in, shape->T, dev->num_sms,
                                    shape->state != FORGE_STATE_INT8_B64);
    *tile_rows = forge::kBM * ts.cg;
    *tile_cols = ts.bn;
    *cluster = ts.cg;
    if (shape->d_out == 0 || shape->d_in == 0) return FORGE_OK;
    const int64_t tiles = ceil_div(shape->d_out, *tile_rows) * ceil_div(shape->d_in, *tile_cols);
    int n = 0;
    if (forge::tile_ctas(ts.bn, ts.cg, static_cast<int>(tiles), dev->num_sms, &n) != cudaSuccess) return FORGE_ERR_CUDA;
    *ctas = n;
    return FORGE_OK;
}

forge_status forge_dx_launch_shape(const forge_shape* shape, int32_t* tile_rows, int32_t* tile_cols,
                                   int32_t* cluster, int32_t* ctas) {
    forge_status st = check_shape(shape);
    if (st != FORGE_OK) return st;
    if (tile_rows == nullptr || tile_cols == nullptr || cluster == nullptr || ctas == nullptr)
        return FORGE_ERR_INVALID_ARGUMENT;
    *tile_rows = *tile_cols = *cluster = *ctas = 0;
    DeviceInfo* dev = nullptr;
    st = device_info(&dev);
    if (st != FORGE_OK) return st;
    const TileShape ts = pick_dx_shape(shape->T, shape->d_out, shape->d_in, dev->num_sms);
    *tile_rows = forge::kBM * ts.cg;
    *tile_cols = ts.bn;
    *cluster = ts.cg;
    if (shape->T == 0 || shape->d_in == 0 || shape->d_out == 0) return FORGE_OK;
    const int64_t tiles = ceil_div(shape->T, *tile_rows) * ceil_div(shape->d_in, *tile_cols);
    int n = 0;
    if (forge::tile_ctas(ts.bn, ts.cg, static_cast<int>(tiles), dev->num_sms, &n) != cudaSuccess) return FORGE_ERR_CUDA;
    *ctas = n;
    return FORGE_OK;
}

uint64_t forge_launch_count(void) { return g_launches.load(); }

const char* forge_status_string(forge_status s) {
    switch (s) {
        case FORGE_OK: return "ok";
        case FORGE_ERR_INVALID_ARGUMENT: return "invalid argument";
        case FORGE_ERR_UNSUPPORTED: return "unsupported combination";
        case FORGE_ERR_MISALIGNED: return "pointer not 32-byte aligned";
        case FORGE_ERR_CUDA: return "CUDA error";
        case FORGE_ERR_NOT_SM103: return "device is not compute capability 10.3 (sm_103a)";
        case FORGE_ERR_TIMEOUT: return "a bounded on-device wait ran out";
    }
    return "unknown status";
}

}  // extern "C"
