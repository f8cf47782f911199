// tile_kernel.cuh -- the persistent weight-gradient tile kernel for sm_103a.
//
// FORGE ("FORGE: Fused On-Register Gradient Elimination for Memory-Efficient LLM Training",
// gist.science technical summary), §2 Methodology, Core mechanism: for one weight tile,
// (1) accumulate dY^T X over all tokens in FP32 on chip, (2) apply the optimizer to the
// finished tile on chip, (3) discard the gradient tile, (4) write back only the weight and
// moment tiles.
//
// GB300 mapping of that mechanism:
//   warp 0      TMA producer: 128 x 64-token slices of dY and BN x 64-token slices of X into a
//               shared-memory ring (128-byte swizzle, both operands MN-major as stored).
//   warp 1      MMA issuer: tcgen05.mma kind::f16 (bf16 x bf16 -> f32), M = 128, N = BN, K = 16,
//               accumulating the whole tile in TMEM (step 1 happens in TMEM, not registers).
//               TMEM holds two accumulators so the next tile's mainloop overlaps this tile's
//               epilogue.
//   warps 2-9   epilogue: tcgen05.ld moves a 32-column strip of the finished tile into
//               registers (thread = weight row); the optimizer runs in registers (step 2); the
//               gradient registers are then dropped (step 3); W/m/v are read and written with
//               256-bit accesses (step 4).  The gradient never reaches device memory.
// Tiles are visited by a static persistent schedule (tile = blockIdx.x + k * gridDim.x) in the
// grouped order of schedule.h, so that concurrently running CTAs share dY and X slices in L2.
//
// The same pipeline also computes the layer's input gradient dX = dY W (EPI = kEpiDX), which the
// fused step's ordering requires before W is overwritten: there the tile rows are tokens, the
// columns d_in and the reduction runs over d_out; A = dY is K-major (d_out runs along memory),
// B = W is MN-major like X, and the epilogue rounds each row to bfloat16.
//
// Every wait is bounded in time: on expiry the kernel records FORGE_ERR_TIMEOUT in the device
// status word, raises a CTA-wide abort flag that every other wait observes, waits (bounded)
// for its own copies and MMAs in flight, frees TMEM and returns.
#pragma once

#include <cstdint>

#include "opt_math.cuh"
#include "ptx.cuh"
#include "schedule.h"

namespace forge {

constexpr int kBM = 128;         // tile rows (d_out) = TMEM lanes
constexpr int kBK = 64;          // tokens per pipeline stage = 128 bytes of one operand column
constexpr int kUmmaK = 16;       // K of one kind::f16 MMA
constexpr int kStatusTimeout = 6;  // FORGE_ERR_TIMEOUT

enum EpiKind : int { kEpiStoreGrad = 0, kEpiOptFP32 = 1, kEpiOptINT8 = 2, kEpiDX = 3, kEpiOptBF16 = 4 };

// Operand formats.  Either way a stage row is 128 bytes (the swizzle span) and a stage of one
// operand is 16 KiB per 128 MN rows: 64 tokens of bf16, or 128 tokens of E4M3, whose products the
// tensor core takes 32 tokens at a time (kind::f8f6f4) instead of 16.
enum OperandKind : int { kOpsBF16 = 0, kOpsE4M3 = 1 };

template <int OPS>
struct OperandTraits {
    static constexpr int kTok = OPS == kOpsE4M3 ? 128 : 64;          // tokens per pipeline stage
    static constexpr int kMNPerRow = OPS == kOpsE4M3 ? 128 : 64;     // MN elements per 128-byte row
    static constexpr int kBlockBytes = kTok * 128;                   // one MN block of a stage
    static constexpr int kStepBytes = OPS == kOpsE4M3 ? 4096 : 2048;  // rows one MMA consumes (K)
};

template <int BN, int CG, int EPI, int OPS = kOpsBF16>
struct TileCfg {
    // 64-column tiles (one X box per stage, N = 64 MMAs) serve small layers with bf16 operands and
    // epilogues that work on 32-column runs; E4M3 rows hold 128 elements, INT8 blocks 64 per warp
    static_assert(BN == 128 || BN == 256 || (BN == 64 && CG == 1 && OPS == kOpsBF16 && EPI != kEpiOptINT8),
                  "tile width");
    static_assert(CG == 1 || CG == 2, "CTA group");
    static constexpr int kBLoad = BN / CG;         // X columns staged by this CTA
    static constexpr int kABytes = kBM * kBK * 2;  // one stage of A: 2 boxes of 64 x 64 (dY^T, or dY for dX)
    static constexpr int kBBytes = kBLoad * kBK * 2;  // one stage of X: kBLoad/64 boxes of [64 tokens][64 cols]
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kTmemCols = 2 * BN;       // double-buffered FP32 accumulator (128 lanes x BN)
    // epilogue warps: two per TMEM lane quarter, each owning half the tile's columns.  A CTA pair
    // runs four per quarter, one 64-column block each, where the epilogue rather than the
    // operand stream sets the pace: the INT8-state epilogue, whose dependent arithmetic needs more
    // warps per scheduler to keep issuing, and the
    // bfloat16-state epilogue behind the E4M3 mainloop, which is half as long as the bf16 one.
    // Binary32 states behind the E4M3 mainloop keep two warps per quarter: their W/m/v stream
    // needs the four row groups each such warp keeps in flight more than it needs more warps
    // (Llama-8B MLP: 0.762 against 0.844 ms per step)
    static constexpr bool kWideEpi = CG == 2 && (EPI == kEpiOptINT8 || (OPS == kOpsE4M3 && EPI == kEpiOptBF16));
    static constexpr int kEpiWarps = kWideEpi ? 16 : 8;
    static constexpr int kThreads = 64 + 32 * kEpiWarps;
    // one warp's 4 KiB transpose strip: 32 x 32 binary32 values, or for the INT8 epilogue 16 rows
    // of a 64-column block; the input-gradient epilogue stores rows as they come out of TMEM and
    // needs none
    static constexpr int kStripBytes = EPI == kEpiDX ? 0 : 32 * 32 * 4;
    static constexpr int kEpiBytes = kEpiWarps * kStripBytes;
    static constexpr int kBarrierBytes = 256;
    static constexpr int kMaxSmem = 232448;
    // as many operand stages as fit beside the epilogue buffers, at most 6
    static constexpr int kFitStages = (kMaxSmem - kEpiBytes - kBarrierBytes - 1024) / kStageBytes;
    static constexpr int kStages = kFitStages < 6 ? kFitStages : 6;
    static constexpr int kSmemBytes = kStages * kStageBytes + kEpiBytes + kBarrierBytes + 1024;  // + alignment slack
    static_assert(kStages >= 3, "operand pipeline depth");
    static_assert(kSmemBytes <= kMaxSmem, "shared memory");
};

struct TileArgs {
    int d_out, d_in, T;
    TileOrder order;              // tile rows x columns and the order they are visited in
    int num_tiles;
    int k_blocks;                 // reduction slices per tile: T / 64 (dW; T / 128 for E4M3), d_out / 64 (dX)
    float g_scale;                // E4M3 operands: s_dY * s_X, applied to the FP32 gradient tile
    const float* row_scales;      // or per channel (both set): s_dY [d_out] and s_X [d_in], each
    const float* col_scales;      //   element's tile value times RN(s_dY[o] * s_X[i])
    float* dW;                    // kEpiStoreGrad: [d_out, d_in] FP32
    uint16_t* dX;                 // kEpiDX: [T, d_in] bf16; token rows >= T are not stored
    uint16_t* W;                  // bf16 [d_out, d_in]
    void* m;                      // FP32, int8 or bf16 [d_out, d_in]
    void* v;
    float* m_scales;              // INT8: [d_out, d_in/64]
    float* v_scales;
    OptScalars s;
    uint64_t seed, step;
    int* status;                  // device status word
    uint64_t wait_limit_ns;       // every wait but the epilogue's for a finished accumulator
    uint64_t acc_wait_limit_ns;   // that one: it spans a whole tile mainloop (wait_limit_ns + k_blocks * 4 us)
    int withhold_first_stage;     // test switch: the producer arms its first stage but never fills it, so a wait runs out
};

// Up to G independent layers in one launch: their tiles are numbered one layer after another
// (layer l owns tiles tile_start[l] .. tile_start[l+1]-1) and visited by one persistent schedule,
// so the pipeline fills and drains once for the group instead of once per layer, and the last
// wave of one layer overlaps the first of the next.  A single-layer call is a group of one.  The
// tensor maps live in the kernel's parameter space (64-byte aligned, as TMA requires).
template <int G>
struct TileGroup {
    int n;                        // layers, 1 .. G
    int tile_start[G + 1];        // prefix sums of the layers' tile counts
    CUtensorMap maps[2 * G];      // per layer: dY (or dY for dX), X (or W for dX)
    TileArgs layer[G];
};

// The layer owning tile `tile`, from a layer index known to be at or before it.
template <int G>
__device__ __forceinline__ int layer_of(const TileGroup<G>& grp, int tile, int l) {
    if constexpr (G == 1) return 0;  // a compile-time layer: its arguments are read at fixed offsets
    while (l + 1 < grp.n && tile >= grp.tile_start[l + 1]) ++l;
    return l;
}

// ---------------------------------------------------------------- bounded waits

struct AbortCtx {
    volatile int* flag;
    int* status;
    uint64_t limit_ns;
};

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, const AbortCtx& ab) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*ab.flag) return false;
        if ((n & 15u) == 0 && global_timer_ns() - t0 > ab.limit_ns) {
            *ab.flag = 1;
            atomicCAS(ab.status, 0, kStatusTimeout);
            return false;
        }
    }
}

// Used only after an abort, to let this thread's own asynchronous work land before exit.
__device__ __forceinline__ void drain_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > limit_ns) return;
    }
}

// ---------------------------------------------------------------- epilogues
// Each is called by one warp for one tile.  The warp owns weight rows row0 .. row0+31 (its TMEM
// lane quarter) and columns col0 .. col0+WIDTH-1; `taddr` is the TMEM address of (row0, col0);
// `strip` is the warp's private 4 KiB shared-memory transpose buffer.  A tile may reach past the
// last row or column of a ragged layer (its operands were zero-filled there): device-memory
// accesses are then skipped per 8-column run and per row, while TMEM reads and shuffles, which
// are warp-wide, still run on every lane.

__device__ __forceinline__ void st_v8_f32(float* p, const uint32_t (&r)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(r[0]), "r"(r[1]),
                 "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

// Moves a 32-row x 32-column FP32 strip of the accumulator from TMEM, where thread i holds row i,
// to the ownership used for device-memory accesses: lane l receives columns 8(l mod 4) .. +7 of
// rows (l div 4) + 8k, k = 0..3, in out[k][0..7].  Four consecutive lanes then cover one row's
// 32 columns, so every warp-wide access touches 8 rows x one contiguous span instead of 32 rows.
// The strip is written with its 16-byte chunks XOR-swizzled by (row mod 8), which makes both the
// row-wise writes and the column-wise reads free of bank conflicts.
// E4M3 dequantisation of one TMEM strip while each thread still holds its own row `row`, columns
// col .. col+31: by the per-tensor product, or by each element's channel-scale product.  Column
// scales are the same for every lane (broadcast loads); d_in is a multiple of 16 with E4M3
// operands, so each 4-column group is wholly inside or outside the layer.
template <bool SCALE>
__device__ __forceinline__ void scale_strip(uint32_t (&g)[32], const TileArgs& a, int row, int col) {
    if constexpr (SCALE) {
        if (a.row_scales == nullptr) {
#pragma unroll
            for (int i = 0; i < 32; ++i) g[i] = __float_as_uint(__fmul_rn(__uint_as_float(g[i]), a.g_scale));
        } else {
            const float rs = row < a.d_out ? a.row_scales[row] : 0.0f;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                uint32_t cs[4] = {0u, 0u, 0u, 0u};
                if (col + 4 * q < a.d_in) ld_v4(a.col_scales + col + 4 * q, cs);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float s = __fmul_rn(rs, __uint_as_float(cs[j]));
                    g[4 * q + j] = __float_as_uint(__fmul_rn(__uint_as_float(g[4 * q + j]), s));
                }
            }
        }
    }
}

template <bool SCALE = false>
__device__ __forceinline__ void strip_transpose(uint32_t taddr, uint8_t* strip, uint32_t (&out)[4][8],
                                                const TileArgs& a, int row, int col) {
    const uint32_t lane = threadIdx.x & 31u;
    uint32_t g[32];
    tmem_ld_32x32b_x32(taddr, g);
    tmem_ld_wait(g);
    scale_strip<SCALE>(g, a, row, col);
    const uint32_t base = smem_addr(strip);
#pragma unroll
    for (uint32_t j = 0; j < 8; ++j)
        st_shared_v4(base + lane * 128u + ((j ^ (lane & 7u)) << 4), g[4 * j], g[4 * j + 1], g[4 * j + 2],
                     g[4 * j + 3]);
    __syncwarp();
    const uint32_t sub_row = lane >> 2;  // < 8, so (row mod 8) of every row this lane reads
#pragma unroll
    for (uint32_t k = 0; k < 4; ++k) {
        const uint32_t r = sub_row + 8u * k;
#pragma unroll
        for (uint32_t h = 0; h < 2; ++h) {
            const uint32_t chunk = 2u * (lane & 3u) + h;
            ld_shared_v4(base + r * 128u + ((chunk ^ sub_row) << 4), &out[k][4 * h]);
        }
    }
    __syncwarp();  // the strip may be overwritten by the next call
}

// The two halves of strip_transpose, for callers that consume one row group at a time: the strip
// is written once, then lane l reads the 8 columns it owns of row (l div 4) + 8k.
template <bool SCALE = false>
__device__ __forceinline__ void strip_store(uint32_t taddr, uint8_t* strip, const TileArgs& a, int row, int col) {
    const uint32_t lane = threadIdx.x & 31u;
    uint32_t g[32];
    tmem_ld_32x32b_x32(taddr, g);
    tmem_ld_wait(g);
    scale_strip<SCALE>(g, a, row, col);
    const uint32_t base = smem_addr(strip);
    __syncwarp();  // earlier reads of the strip are complete
#pragma unroll
    for (uint32_t j = 0; j < 8; ++j)
        st_shared_v4(base + lane * 128u + ((j ^ (lane & 7u)) << 4), g[4 * j], g[4 * j + 1], g[4 * j + 2],
                     g[4 * j + 3]);
    __syncwarp();
}

__device__ __forceinline__ void strip_load_row(const uint8_t* strip, int k, uint32_t (&out)[8]) {
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t sub_row = lane >> 2;
    const uint32_t r = sub_row + 8u * static_cast<uint32_t>(k);
    const uint32_t base = smem_addr(strip);
#pragma unroll
    for (uint32_t h = 0; h < 2; ++h)
        ld_shared_v4(base + r * 128u + (((2u * (lane & 3u) + h) ^ sub_row) << 4), &out[4 * h]);
}

// width: columns of this warp's part (WIDTH, or half of it on a split tail tile)
template <int WIDTH, bool SCALE>
__device__ __forceinline__ void epi_store_grad(const TileArgs& a, int row0, int col0, uint32_t taddr, int width,
                                               uint8_t* strip) {
    const int lane = threadIdx.x & 31;
    const int row = row0 + (lane >> 2), col = col0 + 8 * (lane & 3);
    float* base = a.dW + static_cast<size_t>(row) * a.d_in + col;
#pragma unroll 1
    for (int c = 0; c < width; c += 32) {
        uint32_t t[4][8];
        strip_transpose<SCALE>(taddr + c, strip, t, a, row0 + lane, col0 + c);
        if (col + c < a.d_in) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (row + 8 * k < a.d_out) st_v8_f32(base + static_cast<size_t>(8 * k) * a.d_in + c, t[k]);
        }
    }
}

// Dense states: binary32 (BF16S = false) or bfloat16 rounded stochastically with their own Philox
// streams (BF16S = true).  The update always runs on binary32 moments; only their storage differs.
template <int OPT, int WIDTH, bool BF16S, bool SCALE, int R>
__device__ __forceinline__ void epi_opt_dense(const TileArgs& a, const OptScalars& s, int row0, int col0,
                                              uint32_t taddr, int width, uint8_t* strip, int row0n = -1,
                                              int col0n = 0) {
    using Tr = OptTraits<OPT>;
    constexpr int kSW = BF16S ? 4 : 8;  // 32-bit words holding a lane's 8 moment values
    const int lane = threadIdx.x & 31;
    const int row = row0 + (lane >> 2), col = col0 + 8 * (lane & 3);
    // first element of this lane's 8-column run in row (row0 + lane/4); rows k = 1..3 follow at +8 rows
    const size_t lane_base = static_cast<size_t>(row) * a.d_in + col;
    const size_t row_step = static_cast<size_t>(8) * a.d_in;
#pragma unroll 1
    for (int c = 0; c < width; c += 32) {
        // R of the four row groups hold their W/m/v in registers at once: all four with two
        // epilogue warps per scheduler, so that every group's loads overlap the TMEM read; one
        // with four warps per scheduler, whose 96 registers a thread leave no room for more and
        // whose other warps cover the load latency instead
#pragma unroll 1
        for (int kk = 0; kk < 4; kk += R) {
            uint32_t w[R][4], m[R][kSW], v[R][kSW];
            bool ok[R];
            // the W/m/v loads do not depend on the gradient: issue them before the TMEM read.  They
            // are read once: L2 may evict them first, ahead of the operand slices
            const uint64_t once = policy_evict_first();
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int k = kk + r;
                ok[r] = col + c < a.d_in && row + 8 * k < a.d_out;
                // a run outside the layer loads the layer's first run instead (always valid) and
                // stores nothing, so the loads stay unconditional
                const size_t el = ok[r] ? lane_base + k * row_step + c : 0;
                ld_v4_policy(a.W + el, w[r], once);
                if constexpr (BF16S) {
                    if constexpr (Tr::kM) ld_v4_policy(static_cast<uint16_t*>(a.m) + el, m[r], once);
                    if constexpr (Tr::kV) ld_v4_policy(static_cast<uint16_t*>(a.v) + el, v[r], once);
                } else {
                    if constexpr (Tr::kM) ld_v8_policy(static_cast<float*>(a.m) + el, m[r], once);
                    if constexpr (Tr::kV) ld_v8_policy(static_cast<float*>(a.v) + el, v[r], once);
                }
                // the next 32 columns' W/m/v into L2 now, so their loads wait on L2 rather than DRAM;
                // in the last step, the first 32 columns of this warp's next tile
                const bool last = c + 32 >= width;
                const int rn = last ? row0n + (lane >> 2) + 8 * k : row + 8 * k;
                const int cn = last ? col0n + 8 * (lane & 3) : col + c + 32;
                if ((!last || row0n >= 0) && cn < a.d_in && rn < a.d_out) {
                    const size_t en = static_cast<size_t>(rn) * a.d_in + cn;
                    prefetch_l2(a.W + en);
                    if constexpr (BF16S) {
                        if constexpr (Tr::kM) prefetch_l2(static_cast<uint16_t*>(a.m) + en);
                        if constexpr (Tr::kV) prefetch_l2(static_cast<uint16_t*>(a.v) + en);
                    } else {
                        if constexpr (Tr::kM) prefetch_l2(static_cast<float*>(a.m) + en);
                        if constexpr (Tr::kV) prefetch_l2(static_cast<float*>(a.v) + en);
                    }
                }
            }
            // the gradient strip goes to shared memory once; each row group then reads its 8 values
            if (kk == 0) strip_store<SCALE>(taddr + c, strip, a, row0 + lane, col0 + c);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int k = kk + r;
                const size_t e = lane_base + k * row_step + c;
                uint32_t g[8];
                strip_load_row(strip, k, g);
                const Philox4 p = sr_words(e >> 3, a.seed, a.step);
                Philox4 pm{}, pv{};
                if constexpr (BF16S && Tr::kM) pm = sr_words(e >> 3, a.seed, a.step, kStreamM);
                if constexpr (BF16S && Tr::kV) pv = sr_words(e >> 3, a.seed, a.step, kStreamV);
#pragma unroll
                for (int j = 0; j < 8; j += 2) {
                    const uint32_t wp = w[r][j >> 1];
                    float m0 = 0.f, m1 = 0.f, v0 = 0.f, v1 = 0.f;
                    if constexpr (BF16S) {
                        if constexpr (Tr::kM) { m0 = bf16_lo(m[r][j >> 1]); m1 = bf16_hi(m[r][j >> 1]); }
                        if constexpr (Tr::kV) { v0 = bf16_lo(v[r][j >> 1]); v1 = bf16_hi(v[r][j >> 1]); }
                    } else {
                        if constexpr (Tr::kM) { m0 = __uint_as_float(m[r][j]); m1 = __uint_as_float(m[r][j + 1]); }
                        if constexpr (Tr::kV) { v0 = __uint_as_float(v[r][j]); v1 = __uint_as_float(v[r][j + 1]); }
                    }
                    const float w0 = opt_update<OPT, true>(__uint_as_float(g[j]), bf16_lo(wp), m0, v0, s);
                    const float w1 = opt_update<OPT, true>(__uint_as_float(g[j + 1]), bf16_hi(wp), m1, v1, s);
                    w[r][j >> 1] = sr_bf16(w0, sr_r16(p, j)) | (sr_bf16(w1, sr_r16(p, j + 1)) << 16);
                    if constexpr (BF16S) {
                        if constexpr (Tr::kM) m[r][j >> 1] = sr_bf16(m0, sr_r16(pm, j)) | (sr_bf16(m1, sr_r16(pm, j + 1)) << 16);
                        if constexpr (Tr::kV) v[r][j >> 1] = sr_bf16(v0, sr_r16(pv, j)) | (sr_bf16(v1, sr_r16(pv, j + 1)) << 16);
                    } else {
                        if constexpr (Tr::kM) { m[r][j] = __float_as_uint(m0); m[r][j + 1] = __float_as_uint(m1); }
                        if constexpr (Tr::kV) { v[r][j] = __float_as_uint(v0); v[r][j + 1] = __float_as_uint(v1); }
                    }
                }
                if (ok[r]) {
                    st_v4(a.W + e, w[r]);
                    if constexpr (BF16S) {
                        if constexpr (Tr::kM) st_v4(static_cast<uint16_t*>(a.m) + e, m[r]);
                        if constexpr (Tr::kV) st_v4(static_cast<uint16_t*>(a.v) + e, v[r]);
                    } else {
                        if constexpr (Tr::kM) st_v8(static_cast<float*>(a.m) + e, m[r]);
                        if constexpr (Tr::kV) st_v8(static_cast<float*>(a.v) + e, v[r]);
                    }
                }
            }
        }
    }
}

// Before the first tile's accumulator is ready: bring the W/m/v of the warp's first 32-column run
// into L2, so that the epilogue's first loads wait on L2 while the mainloop runs.  Later runs are
// prefetched by epi_opt_dense itself, one run ahead.
template <int OPT, bool BF16S>
__device__ __forceinline__ void prefetch_first_run(const TileArgs& a, int row0, int col0) {
    using Tr = OptTraits<OPT>;
    const int lane = threadIdx.x & 31;
    const int col = col0 + 8 * (lane & 3);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int row = row0 + (lane >> 2) + 8 * k;
        if (row < a.d_out && col < a.d_in) {
            const size_t e = static_cast<size_t>(row) * a.d_in + col;
            prefetch_l2(a.W + e);
            if constexpr (BF16S) {
                if constexpr (Tr::kM) prefetch_l2(static_cast<uint16_t*>(a.m) + e);
                if constexpr (Tr::kV) prefetch_l2(static_cast<uint16_t*>(a.v) + e);
            } else {
                if constexpr (Tr::kM) prefetch_l2(static_cast<float*>(a.m) + e);
                if constexpr (Tr::kV) prefetch_l2(static_cast<float*>(a.v) + e);
            }
        }
    }
}

// Input gradient: TMEM lane = token row, so each thread rounds its own row's 32-column runs to
// bfloat16 and stores them as two 32-byte pieces.  Rows past the last token (the tail tile when T is
// not a multiple of the tile height) are computed on TMA's zero fill and not stored; past the last
// column (d_in a multiple of 8 only) a 16-column piece shrinks to its first 8 or is skipped.
template <int WIDTH>
__device__ __forceinline__ void epi_store_dx(const TileArgs& a, int row0, int col0, uint32_t taddr, int width) {
    const int row = row0 + static_cast<int>(threadIdx.x & 31u);
    uint16_t* out = a.dX + static_cast<size_t>(row) * a.d_in + col0;
#pragma unroll 1
    for (int c = 0; c < width; c += 32) {
        uint32_t g[32];
        tmem_ld_32x32b_x32(taddr + c, g);  // warp-wide: every lane takes part, stored or not
        tmem_ld_wait(g);
        uint32_t p[2][8];
#pragma unroll
        for (int j = 0; j < 16; ++j) p[j >> 3][j & 7] = pack_bf16x2_rn(g[2 * j], g[2 * j + 1]);
        if (row < a.T) {
            // rows start 32-byte aligned only when d_in is a multiple of 16; else 16-byte stores
            const bool wide = (a.d_in & 15) == 0;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int left = a.d_in - (col0 + c + 16 * h);  // columns of this 16-run inside the layer
                if (wide && left >= 16) {
                    st_v8(out + c + 16 * h, p[h]);
                } else {
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        if (left >= 8 * (q + 1)) {
                            const uint32_t r4[4] = {p[h][4 * q], p[h][4 * q + 1], p[h][4 * q + 2], p[h][4 * q + 3]};
                            st_v4(out + c + 16 * h + 8 * q, r4);
                        }
                    }
                }
            }
        }
    }
}

// INT8 moments.  For each group of 64 columns (one quantisation block per row) the warp stages
// both 32-column gradient strips; lane l then owns the 8 columns 8 (l mod 8) .. +7 of the block in
// rows (l div 8) + 4k, k = 0..7, so the 8 lanes 8r .. 8r+7 together hold a row's block and its
// absmax takes three shuffles.  Per row, one pass computes everything but the codes -- the new
// moments in binary32, the weight update from them and its stochastic rounding, the block
// absmax -- and keeps the new moments in registers; the codes then follow from the new scale.
template <int OPT>
struct Int8RowIn {
    uint32_t w[4];  // 8 bf16
    uint32_t mq[2];  // 8 codes, biased (c + 128 per byte, as int8_at_flipped decodes)
    uint32_t vq[2];
    float ms, vs;
};

template <int OPT>
__device__ __forceinline__ void int8_row_load(const TileArgs& a, size_t e, bool ok, Int8RowIn<OPT>& in) {
    using Tr = OptTraits<OPT>;
    if (!ok) e = 0;  // a row past the layer's last reads the first (always valid) and stores nothing
    ld_v4(a.W + e, in.w);
    if constexpr (Tr::kM) ld_v2(static_cast<int8_t*>(a.m) + e, in.mq);
    if constexpr (Tr::kV) ld_v2(static_cast<int8_t*>(a.v) + e, in.vq);
    in.ms = Tr::kM ? a.m_scales[e >> 6] : 0.f;
    in.vs = Tr::kV ? a.v_scales[e >> 6] : 0.f;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        in.mq[i] ^= 0x80808080u;
        in.vq[i] ^= 0x80808080u;
    }
}

// The INT8 epilogue's strip: 16 rows x 64 columns of the binary32 gradient, the rows 16 hh ..
// 16 hh + 15 of a warp's 32 (one 64-column block), 256 bytes a row, its 16-byte chunk c at chunk
// position c ^ (r mod 8).  Half the rows at a time keep the strip at 4 KiB a warp, so 16 epilogue
// warps leave shared memory for 5 operand stages.  The TMEM reads are warp-wide; only the lanes of
// rows 16 hh .. 16 hh + 15 store (16 lanes x 16 bytes: two wavefronts, no bank conflict).
template <bool SCALE>
__device__ __forceinline__ void int8_strip_store(uint32_t taddr, uint8_t* strip, const TileArgs& a, int row0,
                                                 int col0, int hh) {
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t r = lane & 15u;  // strip row, for the lanes that store
    const bool mine = (lane >> 4) == static_cast<uint32_t>(hh);
    const uint32_t base = smem_addr(strip) + r * 256u;
    __syncwarp();  // earlier reads of the strip are complete
    // one 32-column read in registers at a time (unrolled, the second read is hoisted above the
    // first's stores and both stay live)
#pragma unroll 1
    for (uint32_t h = 0; h < 2; ++h) {
        uint32_t g[32];
        tmem_ld_32x32b_x32(taddr + 32u * h, g);
        tmem_ld_wait(g);
        // per-channel scales here; a per-tensor scale multiplies each lane's 8 values as it reads
        // them (int8_scale_run), once per element rather than once per half
        if (SCALE && a.row_scales != nullptr)
            scale_strip<SCALE>(g, a, row0 + static_cast<int>(lane), col0 + 32 * static_cast<int>(h));
        if (mine) {
#pragma unroll
            for (uint32_t j = 0; j < 8; ++j)
                st_shared_v4(base + (((8u * h + j) ^ (r & 7u)) << 4), g[4 * j], g[4 * j + 1], g[4 * j + 2],
                             g[4 * j + 3]);
        }
    }
    __syncwarp();
}

// A per-tensor gradient scale (E4M3 operands), applied to the values a lane reads from the strip.
template <bool SCALE>
__device__ __forceinline__ void int8_scale_run(const TileArgs& a, uint32_t (&g)[8]) {
    if constexpr (SCALE) {
        if (a.row_scales == nullptr) {
#pragma unroll
            for (int j = 0; j < 8; ++j) g[j] = __float_as_uint(__fmul_rn(__uint_as_float(g[j]), a.g_scale));
        }
    }
}

// The 8 gradient values of INT8 strip row r (< 16), columns 8 q .. 8 q + 7 (q < 8).  The 32 lanes
// of a warp read rows rsub + 4k' (rsub < 4) and runs q < 8: four wavefronts, no bank conflict.
__device__ __forceinline__ void int8_strip_load_run(const uint8_t* strip, uint32_t r, uint32_t q, uint32_t (&out)[8]) {
    const uint32_t base = smem_addr(strip) + r * 256u;
#pragma unroll
    for (uint32_t h = 0; h < 2; ++h) ld_shared_v4(base + (((2u * q + h) ^ (r & 7u)) << 4), &out[4 * h]);
}

template <int OPT>
__device__ __forceinline__ void int8_row_update(const TileArgs& a, const OptScalars& s, size_t e, bool ok,
                                                const uint32_t (&g)[8],
                                                const Int8RowIn<OPT>& in) {
    using Tr = OptTraits<OPT>;
    const Philox4 p = sr_words(e >> 3, a.seed, a.step);
    float mn[8], vn[8];
    uint32_t wo[4];
    float am = 0.f, av = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float wf = (j & 1) ? bf16_hi(in.w[j >> 1]) : bf16_lo(in.w[j >> 1]);
        float mm = Tr::kM ? __fmul_rn(int8_at_flipped(in.mq[j >> 2], j & 3), in.ms) : 0.f;
        float vv = Tr::kV ? __fmul_rn(int8_at_flipped(in.vq[j >> 2], j & 3), in.vs) : 0.f;
        const float wn = opt_update<OPT, false>(__uint_as_float(g[j]), wf, mm, vv, s);
        const uint32_t b = sr_bf16(wn, sr_r16(p, j));
        wo[j >> 1] = (j & 1) ? (wo[j >> 1] | (b << 16)) : b;
        mn[j] = mm;
        vn[j] = vv;
        am = fmaxf(am, fabsf(mm));
        av = fmaxf(av, fabsf(vv));
    }
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) {
        if constexpr (Tr::kM) am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, off));
        if constexpr (Tr::kV) av = fmaxf(av, __shfl_xor_sync(0xFFFFFFFFu, av, off));
    }
    const float nms = __fdiv_rn(am, 127.0f), nvs = __fdiv_rn(av, 127.0f);
    const Int8Coder cm = int8_coder(Tr::kM ? nms : 0.f), cv = int8_coder(Tr::kV ? nvs : 0.f);
    uint32_t mo[2] = {0u, 0u}, vo[2] = {0u, 0u};
    uint32_t redo = 0u;  // bit j: m code j needs the division; bit 8 + j: v code j
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        bool exact = true;
        if constexpr (Tr::kM) {
            mo[j >> 2] = put_byte(mo[j >> 2], int8_code_fast(mn[j], cm, exact), j & 3);
            redo |= exact ? 0u : (1u << j);
        }
        if constexpr (Tr::kV) {
            vo[j >> 2] = put_byte(vo[j >> 2], int8_code_fast(vn[j], cv, exact), j & 3);
            redo |= exact ? 0u : (0x100u << j);
        }
    }
    if (redo != 0u) {
        // rare: a code next to a rounding boundary, or a scale that is not a normal number: the IEEE
        // division decides (one branch per 8 elements, not one per code)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if constexpr (Tr::kM)
                if ((redo >> j) & 1u) mo[j >> 2] = put_byte(mo[j >> 2], int8_code(mn[j], nms), j & 3);
            if constexpr (Tr::kV)
                if ((redo >> (8 + j)) & 1u) vo[j >> 2] = put_byte(vo[j >> 2], int8_code(vn[j], nvs), j & 3);
        }
    }
    if (ok) {
        st_v4(a.W + e, wo);
        if constexpr (Tr::kM) st_v2(static_cast<int8_t*>(a.m) + e, mo);
        if constexpr (Tr::kV) st_v2(static_cast<int8_t*>(a.v) + e, vo);
        if ((threadIdx.x & 7u) == 0) {
            if constexpr (Tr::kM) a.m_scales[e >> 6] = nms;
            if constexpr (Tr::kV) a.v_scales[e >> 6] = nvs;
        }
    }
}

// width: columns of this warp's part (a multiple of 64).  krange: the row iterations k (rows
// rsub + 4k) this warp updates, first | (end << 4): all eight, or on a split tail tile, where the
// 16-warp epilogue (no PREFETCH) gives each 64-column block to two warps, k < 4 or k >= 4.  Rows
// are staged in two halves (int8_strip_store): iterations 0..3, then 4..7.
template <int OPT, int WIDTH, bool SCALE, bool PREFETCH>
__device__ __forceinline__ void epi_opt_int8(const TileArgs& a, const OptScalars& s, int row0, int col0,
                                             uint32_t taddr, int width, uint8_t* strip, int krange) {
    static_assert(WIDTH % 64 == 0, "whole quantisation blocks");
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t q = lane & 7u, rsub = lane >> 3;  // column run (8 columns) and first row of this lane
    const int row = row0 + static_cast<int>(rsub);
#pragma unroll 1
    for (int c = 0; c < width; c += 64) {
        // d_in is a multiple of 64, so a 64-column block lies wholly inside or outside the layer:
        // the same for every lane of the warp
        if (col0 + c >= a.d_in) break;
        if constexpr (PREFETCH) {
            const size_t e0 = static_cast<size_t>(row) * a.d_in + col0 + c + 8 * q;
            const size_t row_step = static_cast<size_t>(4) * a.d_in;
            // the next row's inputs load while this one updates (across the two halves too)
            Int8RowIn<OPT> in[2];
            int8_row_load<OPT>(a, e0, row < a.d_out, in[0]);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                int8_strip_store<SCALE>(taddr + c, strip, a, row0, col0 + c, hh);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const int k = 4 * hh + kk;
                    if (k < 7)
                        int8_row_load<OPT>(a, e0 + (k + 1) * row_step, row + 4 * (k + 1) < a.d_out, in[(k + 1) & 1]);
                    uint32_t g[8];
                    int8_strip_load_run(strip, rsub + 4u * kk, q, g);
                    int8_scale_run<SCALE>(a, g);
                    int8_row_update<OPT>(a, s, e0 + k * row_step, row + 4 * k < a.d_out, g, in[k & 1]);
                }
            }
        } else {
            // enough warps per scheduler to cover the load latency without a second row in flight
#pragma unroll 1
            for (int hh = (krange & 15) >> 2; hh < ((krange >> 4) + 3) >> 2; ++hh) {
                int8_strip_store<SCALE>(taddr + c, strip, a, row0, col0 + c, hh);
                // this half's first row of the lane, and its element index
                const int rh = row + 16 * hh;
                const size_t eh = static_cast<size_t>(rh) * a.d_in + col0 + c + 8 * q;
#pragma unroll 1
                for (int kk = 0; kk < 4; ++kk) {
                    const size_t e = eh + static_cast<size_t>(4 * kk) * a.d_in;
                    const bool ok = rh + 4 * kk < a.d_out;
                    Int8RowIn<OPT> in;
                    int8_row_load<OPT>(a, e, ok, in);
                    uint32_t g[8];
                    int8_strip_load_run(strip, rsub + 4u * kk, q, g);
                    int8_scale_run<SCALE>(a, g);
                    int8_row_update<OPT>(a, s, e, ok, g, in);
                }
            }
        }
    }
    __syncwarp();  // every lane has read the strip before the warp's next tile overwrites it
}

// ---------------------------------------------------------------- the kernel
//
// CL = 1: one CTA owns a 128 x BN tile (M = 128 MMA).
// CL = 2: a cluster of two CTAs (a pair) owns a 256 x BN tile.  Each CTA stages its own 128 rows of
//         dY^T and its own BN/2 columns of X; the pair's even CTA issues tcgen05.mma.cta_group::2
//         (M = 256), which reads both CTAs' shared memory and writes each CTA's 128 accumulator
//         rows into that CTA's TMEM.  Both CTAs' TMA copies complete on the even CTA's stage
//         barrier; the MMA commits arrive in both CTAs; both epilogues release a TMEM buffer on
//         the even CTA's barrier.  Per SM this halves the X bytes pulled from L2.  Every TMA load
//         reads this GPU's own memory into one CTA's shared memory (no multicast).

// After an abort, before the CTA (or the pair) tears down: waits, bounded, until every TMA copy
// this CTA (and, in a pair, the odd CTA) has issued into shared memory has landed.  Copies of
// both CTAs of a pair complete on the even CTA's stage barriers, so its producer does this for
// both, from the issue counts of the two producers (`n_own`, `n_peer`: stages passed in issue
// order; stage i uses slot i mod S in phase (i div S) mod 2).  A producer passes stage i only once
// the MMA consumed stage i - S, so the two counts differ by at most S and each slot is short of
// at most one side's copies in its last phase; that side's bytes are settled on the barrier
// (armed for copies that were issued but never armed, or retired for copies that were armed but
// never issued) and the phase then completes exactly when the copies that were issued have landed.
template <int S, int CG>
__device__ __forceinline__ void drain_copies(uint64_t* full, uint64_t n_own, uint64_t n_peer, int64_t withheld,
                                             uint32_t stage_bytes, uint64_t limit_ns) {
    for (int s = 0; s < S; ++s) {
        const int64_t lo = n_own > static_cast<uint64_t>(s) ? s + S * static_cast<int64_t>((n_own - 1 - s) / S) : -1;
        const int64_t lp =
            CG == 1 ? lo : (n_peer > static_cast<uint64_t>(s) ? s + S * static_cast<int64_t>((n_peer - 1 - s) / S) : -1);
        const int64_t last = lo > lp ? lo : lp;
        if (last < 0) continue;
        if (CG == 2 && lo < last) mbar_arrive_expect_tx(&full[s], stage_bytes);  // the odd CTA's copies, unarmed
        if (CG == 2 && lp < last) mbar_complete_tx(&full[s], stage_bytes);       // armed for copies never issued
        if (last == withheld) mbar_complete_tx(&full[s], stage_bytes);           // the test switch's skipped copies
        drain_bounded(&full[s], static_cast<uint32_t>((last / S) & 1), limit_ns);
    }
}

template <int BN, int CL, int EPI, int OPT, int OPS, int G>
__global__ void __launch_bounds__(TileCfg<BN, CL, EPI, OPS>::kThreads, 1)
    forge_tile_kernel(const __grid_constant__ TileGroup<G> grp, const int split_from) {
    static_assert(CL == 1 || CL == 2, "cluster size");
    static_assert(OPS == kOpsBF16 || EPI != kEpiDX, "the input gradient takes bf16 operands");
    using O = OperandTraits<OPS>;
    constexpr bool kScale = OPS == kOpsE4M3;
    constexpr int CG = CL;                    // CTAs per MMA (cta_group)
    using C = TileCfg<BN, CG, EPI, OPS>;
    constexpr bool kAKMajor = EPI == kEpiDX;  // A = dY with d_out (= K) along memory
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);  // 128B-swizzle atoms need 1024B alignment
    uint8_t* sA = smem;
    uint8_t* sB = smem + C::kStages * C::kABytes;
    uint8_t* strips = smem + C::kStages * C::kStageBytes;  // one transpose strip (or two) per epilogue warp
    uint64_t* full = reinterpret_cast<uint64_t*>(strips + C::kEpiBytes);
    uint64_t* empty = full + C::kStages;
    uint64_t* acc_full = empty + C::kStages;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* drain = acc_empty + 2;
    uint64_t* peer_done = drain + 1;     // a pair's odd CTA: its producer has stopped issuing
    uint64_t* peer_count = peer_done + 1;  // ... after this many stages
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(peer_count + 1);
    int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = CL > 1 ? cluster_ctarank() : 0u;  // CTA within its pair; 0 issues the pair's MMAs
    const int first_tile = static_cast<int>(blockIdx.x) / CL;
    const int tile_stride = static_cast<int>(gridDim.x) / CL;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], C::kEpiWarps * CG);
        }
        mbar_init(drain, 1);
        mbar_init(peer_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
        for (int l = 0; l < grp.n; ++l) {
            tma_prefetch_desc(&grp.maps[2 * l]);
            tma_prefetch_desc(&grp.maps[2 * l + 1]);
        }
    }
    if (warp == 1) {
        tmem_alloc<CG>(tmem_slot, C::kTmemCols);
        tmem_relinquish<CG>();
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (CL > 1) cluster_sync();  // the peer's barriers exist before anything signals them
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // status word, wait limits, test switch and optimizer scalars (one optimizer, hyperparameter set and
    // step per launch): the same for every layer, read at a fixed offset of the parameter bank
    const TileArgs& a0 = grp.layer[0];
    const AbortCtx ab{abort_flag, a0.status, a0.wait_limit_ns};
    // pair kernels with bf16 operands run the tiles from split_from on as two 256 x 128 halves
    // (schedule.h, split_tail_from); the others take split_from = the tile count
    constexpr bool kSplitTail = CG == 2 && BN == 256 && OPS == kOpsBF16;
    const int layer_tiles = grp.tile_start[grp.n];
    const int num_tiles = kSplitTail ? layer_tiles + (layer_tiles - split_from) : layer_tiles;
    uint64_t n_issued = 0;   // producer: stages passed (armed and copied, but for the withheld one)
    int64_t withheld = -1;   // producer: the stage the test switch left without this CTA's copies

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer (every CTA)
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            const uint64_t keep = policy_evict_last();
            int l = 0;
            for (int tile = first_tile; ok && tile < num_tiles; tile += tile_stride) {
                int part = -1;
                const int ot = kSplitTail ? tail_tile(tile, split_from, part) : tile;
                l = layer_of(grp, ot, l);
                const TileArgs& a = grp.layer[l];
                const CUtensorMap* tmap_dy = &grp.maps[2 * l];
                const CUtensorMap* tmap_x = &grp.maps[2 * l + 1];
                int mb, nb;
                tile_coords(ot - grp.tile_start[l], a.order, mb, nb);
                const int row_a = mb * kBM * CG + static_cast<int>(rank) * kBM;
                // a half tile's 128 columns: each CTA of the pair stages 64 of them in its first box
                // (its second box, still copied so that every stage carries the same bytes, holds
                // the next 64 columns, which the N = 128 MMA does not read)
                const int col_b = part < 0 ? nb * BN + static_cast<int>(rank) * C::kBLoad
                                           : nb * BN + part * (BN / 2) + static_cast<int>(rank) * (C::kBLoad / 2);
                const int kblocks = a.k_blocks;
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!wait_bounded(&empty[stage], phase ^ 1u, ab)) { ok = false; break; }
                    uint32_t bar = smem_addr(&full[stage]);
                    if constexpr (CG == 2) bar = map_to_rank(bar, 0);
                    if (rank == 0) mbar_arrive_expect_tx(&full[stage], CG * C::kStageBytes);
                    if (a0.withhold_first_stage && rank == 0 && tile == first_tile && kb == 0) {
                        // test switch: arm this stage but never copy into it, so the MMA thread's wait
                        // for it runs out
                        withheld = static_cast<int64_t>(n_issued);
                    } else {
                        uint8_t* a_dst = sA + stage * C::kABytes;
                        uint8_t* b_dst = sB + stage * C::kBBytes;
                        const int k0 = kb * O::kTok;
                        // A box j holds rows row_a + 64j .. +63 of this CTA's 128 A rows; dY's tensor
                        // map has d_out innermost, so its coordinates are (row, token) for dY^T and
                        // (d_out slice, token row) for the K-major dY of dX
                        if constexpr (OPS == kOpsE4M3) {
                            // E4M3: 128 rows of dY^T fill one 128-byte row; box j is token half j of
                            // the stage (64 token rows at j * 8 KiB)
#pragma unroll
                            for (int j = 0; j < 2; ++j)
                                tma_load_2d_cg<CG>(a_dst + j * 8192, tmap_dy, bar, row_a, k0 + 64 * j, keep);
#pragma unroll
                            for (int j = 0; j < C::kBLoad / 128; ++j)
#pragma unroll
                                for (int h = 0; h < 2; ++h)
                                    tma_load_2d_cg<CG>(b_dst + j * O::kBlockBytes + h * 8192, tmap_x, bar,
                                                       col_b + 128 * j, k0 + 64 * h, keep);
                        } else {
#pragma unroll
                            for (int j = 0; j < 2; ++j) {
                                const int r = row_a + 64 * j;
                                tma_load_2d_cg<CG>(a_dst + j * kBK * 128, tmap_dy, bar, kAKMajor ? k0 : r,
                                                   kAKMajor ? r : k0, keep);
                            }
#pragma unroll
                            for (int j = 0; j < C::kBLoad / 64; ++j)
                                tma_load_2d_cg<CG>(b_dst + j * kBK * 128, tmap_x, bar, col_b + 64 * j, k0, keep);
                        }
                    }
                    ++n_issued;
                    if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
                }
            }
            if constexpr (CG == 2) {
                if (rank == 1) {
                    // tell the even CTA how far this producer got: it settles the accounts of the
                    // stage barriers if the pair aborts
                    st_shared_cluster_u64(map_to_rank(smem_addr(peer_count), 0), n_issued);
                    mbar_arrive_remote(map_to_rank(smem_addr(peer_done), 0));
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ------------------------------------------------ MMA issuer (the even CTA of a pair)
            constexpr uint32_t idesc = OPS == kOpsE4M3 ? idesc_e4m3_f32(kBM * CG, BN, true, true)
                                                       : idesc_bf16_f32(kBM * CG, BN, !kAKMajor, true);
            constexpr uint32_t idesc_half = idesc_bf16_f32(kBM * CG, BN / 2, !kAKMajor, true);  // split tail
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true, issued_any = false;
            int l = 0;
            for (int tile = first_tile; ok && tile < num_tiles; tile += tile_stride) {
                int part = -1;
                const int ot = kSplitTail ? tail_tile(tile, split_from, part) : tile;
                l = layer_of(grp, ot, l);
                const int kblocks = grp.layer[l].k_blocks;
                const uint32_t id = part < 0 ? idesc : idesc_half;
                if (!wait_bounded(&acc_empty[acc], acc_phase ^ 1u, ab)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!wait_bounded(&full[stage], phase, ab)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_base = smem_addr(sA + stage * C::kABytes);
                    const uint32_t b_base = smem_addr(sB + stage * C::kBBytes);
#pragma unroll
                    for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
                        // MN-major: 16 K = 16 rows of 128 bytes, so advance 2048 bytes per MMA.
                        // Within a stage, the MN-direction 64-element column blocks are kBK*128
                        // bytes apart (leading byte offset) and 8-row groups 1024 bytes apart
                        // (stride).  K-major (dY for dX): 16 K = 32 bytes within each 128-byte
                        // swizzled row, 8-row groups 1024 bytes apart; the leading offset is unused.
                        // E4M3: 32 tokens per MMA, 4096 bytes; MN blocks of 128 elements 16 KiB apart
                        const uint64_t ad = kAKMajor ? smem_desc_sw128(a_base + kk * 32, 16, 1024)
                                                     : smem_desc_sw128(a_base + kk * O::kStepBytes, O::kBlockBytes, 1024);
                        const uint64_t bd = smem_desc_sw128(b_base + kk * O::kStepBytes, O::kBlockBytes, 1024);
                        if constexpr (OPS == kOpsE4M3) tc_mma_e4m3<CG>(d_tmem, ad, bd, id, (kb | kk) != 0 ? 1u : 0u);
                        else tc_mma_bf16<CG>(d_tmem, ad, bd, id, (kb | kk) != 0 ? 1u : 0u);
                    }
                    issued_any = true;
                    // the slot is free once read: tell both CTAs of the pair, whose copies fill it
                    tc_commit_mask<CG>(&empty[stage], 0x3u);
                    if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                tc_commit_mask<CG>(&acc_full[acc], 0x3u);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            if (!ok && issued_any) {
                tc_commit_local<CG>(drain);
                drain_bounded(drain, 0, a0.wait_limit_ns);
            }
        }
    } else {
        // ---------------------------------------------------- epilogue warps (every CTA)
        const int e = warp - 2;
        const int quarter = warp & 3;   // a warp may only touch TMEM lanes 32*(warp%4) .. +31
        const int half = e >> 2;                // column part owned by this warp
        constexpr int kWidth = BN / (C::kEpiWarps / 4);
        // this warp's columns within the tile's accumulator (offset, width) and, for the 16-warp
        // INT8 epilogue, its row iterations (epi_opt_int8's krange): a half tile's 128 columns are
        // split between the column parts (parts of 128 columns take 64), or, with 64-column parts,
        // two parts share a block and split its rows
        auto cols_of = [&](int part, int& off, int& width, int& krange) {
            off = half * kWidth;
            width = kWidth;
            krange = 8 << 4;
            if (kSplitTail && part >= 0) {
                if constexpr (kWidth >= 128) {
                    width = kWidth / 2;
                    off = half * width;
                } else {
                    off = (half & 1) * kWidth;
                    krange = (half >> 1) ? (4 | (8 << 4)) : (4 << 4);
                }
            }
        };
        if constexpr (EPI == kEpiOptFP32 || EPI == kEpiOptBF16) {
            if (first_tile < num_tiles) {
                int part = -1;
                const int ot = kSplitTail ? tail_tile(first_tile, split_from, part) : first_tile;
                const int l0 = layer_of(grp, ot, 0);
                int mb, nb, off, width, krange;
                tile_coords(ot - grp.tile_start[l0], grp.layer[l0].order, mb, nb);
                cols_of(part, off, width, krange);
                prefetch_first_run<OPT, EPI == kEpiOptBF16>(grp.layer[l0],
                                                            mb * kBM * CG + static_cast<int>(rank) * kBM + quarter * 32,
                                                            nb * BN + (part > 0 ? BN / 2 : 0) + off);
            }
        }
        int acc = 0;
        uint32_t acc_phase = 0;
        int l = 0;
        for (int tile = first_tile; tile < num_tiles; tile += tile_stride) {
            int part = -1;
            const int ot = kSplitTail ? tail_tile(tile, split_from, part) : tile;
            l = layer_of(grp, ot, l);
            const TileArgs& a = grp.layer[l];
            // the wait for a finished accumulator spans a whole tile mainloop, which grows with T
            const AbortCtx ab_acc{abort_flag, a0.status, a.acc_wait_limit_ns};
            int mb, nb;
            tile_coords(ot - grp.tile_start[l], a.order, mb, nb);
            int ok = 1;
            if (lane == 0) ok = wait_bounded(&acc_full[acc], acc_phase, ab_acc) ? 1 : 0;
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            int off, width, krange;
            cols_of(part, off, width, krange);
            const int row0 = mb * kBM * CG + static_cast<int>(rank) * kBM + quarter * 32;
            const int col0 = nb * BN + (part > 0 ? BN / 2 : 0) + off;
            const uint32_t taddr =
                tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * BN + off);
            uint8_t* strip = strips + e * C::kStripBytes;
            if constexpr (EPI == kEpiDX) epi_store_dx<kWidth>(a, row0, col0, taddr, width);
            else if constexpr (EPI == kEpiStoreGrad) epi_store_grad<kWidth, kScale>(a, row0, col0, taddr, width, strip);
            else if constexpr (EPI == kEpiOptFP32 || EPI == kEpiOptBF16) {
                // the next tile's first run is prefetched only within the same layer
                int row0n = -1, col0n = 0;
                if (tile + tile_stride < num_tiles) {
                    int pn = -1;
                    const int otn = kSplitTail ? tail_tile(tile + tile_stride, split_from, pn) : tile + tile_stride;
                    if (layer_of(grp, otn, l) == l) {
                        int mbn, nbn, offn, widthn, kn;
                        tile_coords(otn - grp.tile_start[l], a.order, mbn, nbn);
                        cols_of(pn, offn, widthn, kn);
                        row0n = mbn * kBM * CG + static_cast<int>(rank) * kBM + quarter * 32;
                        col0n = nbn * BN + (pn > 0 ? BN / 2 : 0) + offn;
                    }
                }
                epi_opt_dense<OPT, kWidth, EPI == kEpiOptBF16, kScale, (C::kEpiWarps == 8 ? 4 : 1)>(
                    a, a0.s, row0, col0, taddr, width, strip, row0n, col0n);
            }
            else epi_opt_int8<OPT, kWidth, kScale, C::kEpiWarps == 8>(a, a0.s, row0, col0, taddr, width, strip, krange);
            // the buffer's TMEM columns may be overwritten once every lane's reads of them have
            // completed (tcgen05.wait::ld) and been ordered before the arrive (tcgen05 fence); the
            // arrive publishes no memory, so it is relaxed
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_relaxed(map_to_rank(smem_addr(&acc_empty[acc]), 0));
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0 && lane == 0 && rank == 0 && *abort_flag) {
        // an aborted CTA (pair) exits only once no copy into its shared memory is still in flight
        uint64_t n_peer = n_issued;
        bool counted = true;
        if constexpr (CG == 2) {
            counted = false;
            const uint64_t t0 = global_timer_ns();
            while (!counted && global_timer_ns() - t0 <= 4 * a0.wait_limit_ns) counted = mbar_try_wait_cluster(peer_done, 0);
            if (counted) n_peer = ld_shared_volatile_u64(peer_count);
        }
        if (counted) {
            drain_copies<C::kStages, CG>(full, n_issued, n_peer, withheld, C::kStageBytes, a0.wait_limit_ns);
        } else {
            // the odd CTA never reported (it is itself stuck past every limit): wait for the last
            // phase this CTA armed on each slot, bounded
            drain_copies<C::kStages, 1>(full, n_issued, n_issued, withheld, C::kStageBytes, a0.wait_limit_ns);
        }
    }
    // a pair tears down together: its MMAs read both CTAs' shared memory and write both TMEMs, and
    // both CTAs' copies and commits land in the even CTA
    if constexpr (CL > 1) cluster_sync();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc<CG>(tmem_base, C::kTmemCols);
    }
}

}  // namespace forge
