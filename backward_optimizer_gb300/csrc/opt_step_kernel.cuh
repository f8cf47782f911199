// opt_step_kernel.cuh -- the optimizer half of the two-phase schedule: read a materialised FP32
// gradient and apply the same per-element update as the fused tile kernel.
//
// FORGE ("FORGE: Fused On-Register Gradient Elimination for Memory-Efficient LLM Training",
// gist.science technical summary), §1 The problem: backward writes the full gradient to device
// memory and the optimizer reads it back.  This kernel is that second read, kept as the
// ablation baseline and for T == 0 (zero gradient, dW == nullptr).
//
// Each thread owns 8 consecutive elements (one Philox call).  With INT8 states, the 8 lanes
// l = 8k .. 8k+7 of a warp hold one 64-element block and reduce its absmax with shuffles.  Whole
// warps iterate together (a lane past the last element only skips its loads and stores), so the
// shuffles always see all 32 lanes; the element count is a multiple of 64 with INT8 states, so
// each 8-lane block group is wholly in or out of range.  With BF16 states the moments are
// rounded stochastically with their own Philox streams, exactly as in the fused kernel.
#pragma once

#include <cstdint>

#include "opt_math.cuh"
#include "ptx.cuh"

namespace forge {

struct OptArgs {
    const float* dW;      // nullptr: zero gradient
    uint16_t* W;
    void* m;
    void* v;
    float* m_scales;
    float* v_scales;
    uint64_t n8;          // elements / 8
    OptScalars s;
    uint64_t seed, step;
};

// STATE: 0 = binary32 moments, 1 = INT8 with per-64 scales, 2 = bfloat16 (the forge_state_dtype values).
template <int OPT, int STATE>
__global__ void __launch_bounds__(256) forge_opt_kernel(const OptArgs a) {
    using Tr = OptTraits<OPT>;
    constexpr bool INT8 = STATE == 1;
    constexpr bool BF16S = STATE == 2;
    const uint64_t stride = static_cast<uint64_t>(gridDim.x) * blockDim.x;
    const uint64_t lane = threadIdx.x & 31u;
    for (uint64_t gi = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x; gi - lane < a.n8; gi += stride) {
        const bool valid = gi < a.n8;
        const uint64_t e0 = (valid ? gi : 0) * 8;  // lanes past the end read (and store) nothing
        uint32_t g[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        uint32_t w[4] = {0, 0, 0, 0};
        if (valid) {
            if (a.dW != nullptr) ld_v8(a.dW + e0, g);
            ld_v4(a.W + e0, w);
        }
        float mf[8], vf[8];
        float ms = 0.f, vs = 0.f;
        uint32_t mq[2] = {0, 0}, vq[2] = {0, 0};
        if constexpr (INT8) {
            if constexpr (Tr::kM) {
                if (valid) {
                    ld_v2(static_cast<int8_t*>(a.m) + e0, mq);
                    ms = a.m_scales[e0 >> 6];
                }
            }
            if constexpr (Tr::kV) {
                if (valid) {
                    ld_v2(static_cast<int8_t*>(a.v) + e0, vq);
                    vs = a.v_scales[e0 >> 6];
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                mf[j] = Tr::kM ? __fmul_rn(int8_at(mq[j >> 2], j & 3), ms) : 0.f;
                vf[j] = Tr::kV ? __fmul_rn(int8_at(vq[j >> 2], j & 3), vs) : 0.f;
            }
        } else if constexpr (BF16S) {
            uint32_t t[4] = {0, 0, 0, 0};
            if constexpr (Tr::kM) {
                if (valid) ld_v4(static_cast<uint16_t*>(a.m) + e0, t);
#pragma unroll
                for (int j = 0; j < 8; ++j) mf[j] = (j & 1) ? bf16_hi(t[j >> 1]) : bf16_lo(t[j >> 1]);
            }
            if constexpr (Tr::kV) {
                if (valid) ld_v4(static_cast<uint16_t*>(a.v) + e0, t);
#pragma unroll
                for (int j = 0; j < 8; ++j) vf[j] = (j & 1) ? bf16_hi(t[j >> 1]) : bf16_lo(t[j >> 1]);
            }
            if constexpr (!Tr::kM) {
#pragma unroll
                for (int j = 0; j < 8; ++j) mf[j] = 0.f;
            }
            if constexpr (!Tr::kV) {
#pragma unroll
                for (int j = 0; j < 8; ++j) vf[j] = 0.f;
            }
        } else {
            uint32_t t[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            if constexpr (Tr::kM) {
                if (valid) ld_v8(static_cast<float*>(a.m) + e0, t);
#pragma unroll
                for (int j = 0; j < 8; ++j) mf[j] = __uint_as_float(t[j]);
            }
            if constexpr (Tr::kV) {
                if (valid) ld_v8(static_cast<float*>(a.v) + e0, t);
#pragma unroll
                for (int j = 0; j < 8; ++j) vf[j] = __uint_as_float(t[j]);
            }
            if constexpr (!Tr::kM) {
#pragma unroll
                for (int j = 0; j < 8; ++j) mf[j] = 0.f;
            }
            if constexpr (!Tr::kV) {
#pragma unroll
                for (int j = 0; j < 8; ++j) vf[j] = 0.f;
            }
        }
        const Philox4 p = sr_words(gi, a.seed, a.step);
        float wn[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float wf = (j & 1) ? bf16_hi(w[j >> 1]) : bf16_lo(w[j >> 1]);
            wn[j] = opt_update<OPT, !INT8>(__uint_as_float(g[j]), wf, mf[j], vf[j], a.s);  // the fused kernel's forms
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
            w[k] = sr_bf16(wn[2 * k], sr_r16(p, 2 * k)) | (sr_bf16(wn[2 * k + 1], sr_r16(p, 2 * k + 1)) << 16);
        if (valid) st_v4(a.W + e0, w);
        if constexpr (INT8) {
            float am = 0.f, av = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                am = fmaxf(am, fabsf(mf[j]));
                av = fmaxf(av, fabsf(vf[j]));
            }
#pragma unroll
            for (int off = 1; off < 8; off <<= 1) {
                am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, off));
                av = fmaxf(av, __shfl_xor_sync(0xFFFFFFFFu, av, off));
            }
            const float nms = __fdiv_rn(am, 127.0f), nvs = __fdiv_rn(av, 127.0f);
            uint32_t mo[2] = {0, 0}, vo[2] = {0, 0};
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if constexpr (Tr::kM) mo[j >> 2] |= int8_code(mf[j], nms) << (8 * (j & 3));
                if constexpr (Tr::kV) vo[j >> 2] |= int8_code(vf[j], nvs) << (8 * (j & 3));
            }
            const bool leader = (threadIdx.x & 7) == 0;
            if (valid) {
                if constexpr (Tr::kM) {
                    st_v2(static_cast<int8_t*>(a.m) + e0, mo);
                    if (leader) a.m_scales[e0 >> 6] = nms;
                }
                if constexpr (Tr::kV) {
                    st_v2(static_cast<int8_t*>(a.v) + e0, vo);
                    if (leader) a.v_scales[e0 >> 6] = nvs;
                }
            }
        } else if constexpr (BF16S) {
            uint32_t t[4];
            if constexpr (Tr::kM) {
                const Philox4 pm = sr_words(gi, a.seed, a.step, kStreamM);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    t[k] = sr_bf16(mf[2 * k], sr_r16(pm, 2 * k)) | (sr_bf16(mf[2 * k + 1], sr_r16(pm, 2 * k + 1)) << 16);
                if (valid) st_v4(static_cast<uint16_t*>(a.m) + e0, t);
            }
            if constexpr (Tr::kV) {
                const Philox4 pv = sr_words(gi, a.seed, a.step, kStreamV);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    t[k] = sr_bf16(vf[2 * k], sr_r16(pv, 2 * k)) | (sr_bf16(vf[2 * k + 1], sr_r16(pv, 2 * k + 1)) << 16);
                if (valid) st_v4(static_cast<uint16_t*>(a.v) + e0, t);
            }
        } else {
            uint32_t t[8];
            if constexpr (Tr::kM) {
#pragma unroll
                for (int j = 0; j < 8; ++j) t[j] = __float_as_uint(mf[j]);
                if (valid) st_v8(static_cast<float*>(a.m) + e0, t);
            }
            if constexpr (Tr::kV) {
#pragma unroll
                for (int j = 0; j < 8; ++j) t[j] = __float_as_uint(vf[j]);
                if (valid) st_v8(static_cast<float*>(a.v) + e0, t);
            }
        }
    }
}

}  // namespace forge
