// opt_math.cuh -- per-element epilogue arithmetic of the fused step, in binary32:
// the eight optimizer updates, Philox4x32-10, stochastic rounding to bfloat16 and the
// INT8 block-64 codec.  Used by the fused tile kernel and by the unfused optimizer kernel,
// so that both apply bit-identical arithmetic to the same gradient value.
//
// Source of each piece ("FORGE: Fused On-Register Gradient Elimination for Memory-Efficient
// LLM Training", gist.science technical summary, unless stated):
//  * optimizer set: §3 Key contributions, "Generality"; the formulas are each optimizer's
//    published definition (the summary gives none): AdamW (Loshchilov & Hutter, ICLR'19),
//    NAdam (Dozat, ICLR'16 workshop), RAdam (Liu et al., ICLR'20), Lion (Chen et al.,
//    NeurIPS'23), RMSprop (Tieleman & Hinton, lecture 6.5), AdaGrad (Duchi et al., JMLR'11),
//    SGD and heavy-ball momentum.  Decoupled weight decay for AdamW and Lion, coupled L2
//    (g + wd w) for the others.
//  * gradient consumed in FP32, never rounded to BF16 first: §2 Precision and fidelity.
//  * stochastic rounding of the weight write-back: §2 Precision and fidelity, second
//    low-precision point.  Generator: Philox4x32-10 (Salmon et al., SC'11).
//  * INT8 states with 64-element absmax blocks: §2 Precision and fidelity, third point.
#pragma once

#include <cstdint>

namespace forge {

enum OptKind : int {
    kAdamW = 0, kNAdam = 1, kRAdam = 2, kLion = 3, kRMSprop = 4, kAdaGrad = 5, kSGD = 6, kSGDMomentum = 7
};

template <int OPT> struct OptTraits {
    static constexpr bool kM = (OPT == kAdamW || OPT == kNAdam || OPT == kRAdam || OPT == kLion ||
                                OPT == kSGDMomentum);
    static constexpr bool kV = (OPT == kAdamW || OPT == kNAdam || OPT == kRAdam || OPT == kRMSprop ||
                                OPT == kAdaGrad);
};

// Step-dependent scalars, derived on the host in binary64 and rounded to binary32.
struct OptScalars {
    float lr;            // learning rate (AdaGrad: lr / (1 + (t-1) lr_decay))
    float b1, omb1;      // beta1, 1 - beta1 (Lion: c coefficient)
    float b2, omb2;      // beta2, 1 - beta2 (Lion: moment coefficient); RMSprop: alpha, 1 - alpha
    float eps;
    float wd;            // coupled weight decay
    float decay;         // decoupled weight decay factor 1 - lr wd
    float step_size;     // AdamW: lr / (1 - beta1^t); RAdam: see host
    float inv_sqrt_bc2;  // 1 / sqrt(1 - beta2^t)
    float c_g, c_m;      // NAdam gradient and momentum coefficients
    float mu;            // SGD momentum
    int rectified;       // RAdam: rho_t > 5
};

// ---------------------------------------------------------------- bfloat16

__device__ __forceinline__ float bf16_lo(uint32_t pair) { return __uint_as_float(pair << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t pair) { return __uint_as_float(pair & 0xFFFF0000u); }

// binary32 -> bfloat16 bits: add 16 random bits to the pattern and truncate.  The magnitude
// rounds up with probability equal to its fractional position between the two neighbours,
// so the expectation is exact.  NaN -> canonical quiet NaN; +-Inf unchanged.
__device__ __forceinline__ uint32_t sr_bf16(float x, uint32_t r16) {
    const uint32_t u = __float_as_uint(x);
    if ((u & 0x7F800000u) == 0x7F800000u) return (u & 0x007FFFFFu) ? 0x7FC0u : (u >> 16);
    return (u + r16) >> 16;
}

// ---------------------------------------------------------------- Philox4x32-10

struct Philox4 { uint32_t x0, x1, x2, x3; };

// Ten rounds of the Philox-4x32 bijection (Salmon et al., SC'11): multiply words 0 and 2 by
// the two round multipliers, xor the high halves into words 1 and 3 with the key, swap;
// bump the key by the two Weyl increments between rounds.
__device__ __forceinline__ Philox4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0,
                                                 uint32_t k1) {
    constexpr uint32_t kM0 = 0xD2511F53u, kM1 = 0xCD9E8D57u;
    constexpr uint32_t kW0 = 0x9E3779B9u, kW1 = 0xBB67AE85u;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r) { k0 += kW0; k1 += kW1; }
        const uint32_t hi0 = __umulhi(kM0, c0), lo0 = kM0 * c0;
        const uint32_t hi1 = __umulhi(kM1, c2), lo1 = kM1 * c2;
        const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
    }
    return Philox4{c0, c1, c2, c3};
}

// Stochastic-rounding streams: the weight, and the first and second moments when they are stored
// as BF16.  The stream index goes into the top two bits of the high counter word, which the
// element index never reaches (at most 2^41 groups of 8 elements per layer).
enum SrStream : uint32_t { kStreamW = 0, kStreamM = 1, kStreamV = 2 };

// 16-bit random values for the 8 elements e8*8 .. e8*8+7 of tensor `stream` at step `step`:
// element 2k takes the low half of word k, element 2k+1 its high half.
__device__ __forceinline__ Philox4 sr_words(uint64_t e8, uint64_t seed, uint64_t step, uint32_t stream = kStreamW) {
    return philox4x32_10(static_cast<uint32_t>(e8), static_cast<uint32_t>(e8 >> 32) + (stream << 30),
                         static_cast<uint32_t>(step), static_cast<uint32_t>(step >> 32),
                         static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
}

__device__ __forceinline__ uint32_t sr_r16(const Philox4& p, int j) {
    const uint32_t w = (j >> 1) == 0 ? p.x0 : (j >> 1) == 1 ? p.x1 : (j >> 1) == 2 ? p.x2 : p.x3;
    return (j & 1) ? (w >> 16) : (w & 0xFFFFu);
}

// ---------------------------------------------------------------- INT8 block codec

__device__ __forceinline__ float int8_at(uint32_t word, int k) {
    return static_cast<float>(static_cast<int8_t>((word >> (8 * k)) & 0xFFu));
}

// code = clamp(round_half_even(x / s), -127, 127); s == 0 gives 0.  IEEE division.
__device__ __forceinline__ uint32_t int8_code(float x, float s) {
    if (!(s > 0.0f)) return 0u;
    int q = __float2int_rn(__fdiv_rn(x, s));
    q = q > 127 ? 127 : (q < -127 ? -127 : q);
    return static_cast<uint32_t>(q) & 0xFFu;
}

// The same codes without a division or a float-to-int conversion per element, for epilogues that
// code many values against one block scale.  Words of codes are first XORed with 0x80808080, which
// turns each signed code c into the byte c + 128.
//
// Decoding: that byte as the low mantissa bits of 2^23 is the binary32 value 2^23 + c + 128, and
// subtracting 2^23 + 128 leaves c exactly.
__device__ __forceinline__ float int8_at_flipped(uint32_t flipped, int k) {
    return __fsub_rn(__uint_as_float(__byte_perm(flipped, 0x4B000000u, 0x7650u | static_cast<uint32_t>(k))),
                     8388736.0f);
}

// Encoding against one scale s: r = rcp.approx(s), the hardware reciprocal (at most 2^-23 absolute
// error for s in [1, 2), so |r s - 1| <= 2^-22 at any normal s), and q = RN(x r).  Then
// |q - x/s| <= |x/s| (2^-22 + 2^-24 + 2^-46) < 3.8e-5 (|x| <= absmax, so |x/s| <= 127.00001), and
// RN(x/s) lies within 2^-18 of x/s, so the two differ by less than 4.2e-5 < 2^-14.  Where q is
// farther than 2^-14 from every half-integer both round to the same integer, which
// RN(q + 1.5 * 2^23) holds in its low mantissa bits (|q| < 2^22); the clamp cannot act
// (|q| < 127.5).  Elsewhere -- near or at a tie, s subnormal, 0 or not finite, x NaN -- the code
// comes from the IEEE division of int8_code.  The reciprocal only chooses between the two paths:
// every code equals clamp(rne(RN(x/s))) either way.
struct Int8Coder {
    float s, r;
    bool fast;  // s normal and 1/s normal
};

__device__ __forceinline__ float rcp_approx(float s) {
    float r;
    asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(s));
    return r;
}

__device__ __forceinline__ Int8Coder int8_coder(float s) {
    Int8Coder c;
    c.s = s;
    c.fast = s >= 0x1p-126f && s <= 0x1p125f;
    c.r = c.fast ? rcp_approx(s) : 0.0f;
    return c;
}

// The code in the low byte (higher bytes unspecified), without a branch; `exact` is false where
// the code must come from int8_code instead.
__device__ __forceinline__ uint32_t int8_code_fast(float x, const Int8Coder& c, bool& exact) {
    const float q = __fmul_rn(x, c.r);
    const float t = __fadd_rn(q, 12582912.0f);
    const float d = __fsub_rn(q, __fsub_rn(t, 12582912.0f));  // q - rne(q), exact
    exact = c.fast && fabsf(d) < 0.49993896484375f;           // 0.5 - 2^-14
    return __float_as_uint(t);
}

// word with its byte k (0..3) replaced by the low byte of c
__device__ __forceinline__ uint32_t put_byte(uint32_t word, uint32_t c, int k) {
    return __byte_perm(word, c, k == 0 ? 0x3214u : k == 1 ? 0x3240u : k == 2 ? 0x3410u : 0x4210u);
}

// ---------------------------------------------------------------- the eight updates
// g: binary32 gradient; w: binary32 weight (from bfloat16); m, v: binary32 moments, updated
// in place.  Returns the new binary32 weight.  Intrinsics fix each rounding so that the
// kernel's result does not depend on the compiler's contraction choices.
//
// APPROX selects how the weight step divides and takes square roots: the IEEE-rounded
// operations, or the hardware approximations (sqrt.approx.f32, div.approx.f32: a few units in
// the last place, no slow-path branches).  The moments never depend on it.  Epilogues bound by
// the memory system (binary32 and bfloat16 states) take the approximations, which measured
// 1-7 % faster there; the INT8-state epilogue, bound by its own instruction issue, measured
// faster with the IEEE forms.  The fused and the two-phase kernel of one state format always
// take the same forms, so they agree bit for bit.

__device__ __forceinline__ float sqrt_approx(float x) {
    float r;
    asm("sqrt.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ float div_approx(float a, float b) {
    float r;
    asm("div.approx.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

template <bool APPROX>
__device__ __forceinline__ float step_sqrt(float x) {
    if constexpr (APPROX) return sqrt_approx(x);
    else return __fsqrt_rn(x);
}

// a / b for the weight step; b >= eps > 0 and below 2^126 there (b = sqrt(v) c + eps, v finite)
template <bool APPROX>
__device__ __forceinline__ float step_div(float a, float b) {
    if constexpr (APPROX) return div_approx(a, b);
    else return __fdiv_rn(a, b);
}

template <int OPT, bool APPROX = false>
__device__ __forceinline__ float opt_update(float g, float w, float& m, float& v, const OptScalars& s) {
    if constexpr (OPT == kAdamW) {
        m = __fmaf_rn(s.b1, m, __fmul_rn(s.omb1, g));
        v = __fmaf_rn(s.b2, v, __fmul_rn(s.omb2, __fmul_rn(g, g)));
        const float denom = __fmaf_rn(step_sqrt<APPROX>(v), s.inv_sqrt_bc2, s.eps);
        return __fmaf_rn(-s.step_size, step_div<APPROX>(m, denom), __fmul_rn(w, s.decay));
    } else if constexpr (OPT == kNAdam) {
        const float gc = __fmaf_rn(s.wd, w, g);
        m = __fmaf_rn(s.b1, m, __fmul_rn(s.omb1, gc));
        v = __fmaf_rn(s.b2, v, __fmul_rn(s.omb2, __fmul_rn(gc, gc)));
        const float denom = __fmaf_rn(step_sqrt<APPROX>(v), s.inv_sqrt_bc2, s.eps);
        return __fsub_rn(w, step_div<APPROX>(__fmaf_rn(s.c_g, gc, __fmul_rn(s.c_m, m)), denom));
    } else if constexpr (OPT == kRAdam) {
        const float gc = __fmaf_rn(s.wd, w, g);
        m = __fmaf_rn(s.b1, m, __fmul_rn(s.omb1, gc));
        v = __fmaf_rn(s.b2, v, __fmul_rn(s.omb2, __fmul_rn(gc, gc)));
        if (s.rectified) return __fmaf_rn(-s.step_size, step_div<APPROX>(m, __fadd_rn(step_sqrt<APPROX>(v), s.eps)), w);
        return __fmaf_rn(-s.step_size, m, w);
    } else if constexpr (OPT == kLion) {
        const float c = __fmaf_rn(s.b1, m, __fmul_rn(s.omb1, g));
        const float sgn = c > 0.0f ? 1.0f : (c < 0.0f ? -1.0f : 0.0f);
        m = __fmaf_rn(s.b2, m, __fmul_rn(s.omb2, g));
        return __fmaf_rn(-s.lr, sgn, __fmul_rn(w, s.decay));
    } else if constexpr (OPT == kRMSprop) {
        const float gc = __fmaf_rn(s.wd, w, g);
        v = __fmaf_rn(s.b2, v, __fmul_rn(s.omb2, __fmul_rn(gc, gc)));
        return __fmaf_rn(-s.lr, step_div<APPROX>(gc, __fadd_rn(step_sqrt<APPROX>(v), s.eps)), w);
    } else if constexpr (OPT == kAdaGrad) {
        const float gc = __fmaf_rn(s.wd, w, g);
        v = __fmaf_rn(gc, gc, v);
        return __fmaf_rn(-s.lr, step_div<APPROX>(gc, __fadd_rn(step_sqrt<APPROX>(v), s.eps)), w);
    } else if constexpr (OPT == kSGD) {
        return __fmaf_rn(-s.lr, __fmaf_rn(s.wd, w, g), w);
    } else {  // kSGDMomentum
        m = __fmaf_rn(s.mu, m, __fmaf_rn(s.wd, w, g));
        return __fmaf_rn(-s.lr, m, w);
    }
}

// Moments only (no weight): the first pass of an INT8 block, which needs the new moments'
// absmax before any code can be written.  Same arithmetic as opt_update.
template <int OPT>
__device__ __forceinline__ void opt_moments(float g, float w, float& m, float& v, const OptScalars& s) {
    if constexpr (OPT == kAdamW) {
        m = __fmaf_rn(s.b1, m, __fmul_rn(s.omb1, g));
        v = __fmaf_rn(s.b2, v, __fmul_rn(s.omb2, __fmul_rn(g, g)));
    } else if constexpr (OPT == kNAdam || OPT == kRAdam) {
        const float gc = __fmaf_rn(s.wd, w, g);
        m = __fmaf_rn(s.b1, m, __fmul_rn(s.omb1, gc));
        v = __fmaf_rn(s.b2, v, __fmul_rn(s.omb2, __fmul_rn(gc, gc)));
    } else if constexpr (OPT == kLion) {
        m = __fmaf_rn(s.b2, m, __fmul_rn(s.omb2, g));
    } else if constexpr (OPT == kRMSprop) {
        const float gc = __fmaf_rn(s.wd, w, g);
        v = __fmaf_rn(s.b2, v, __fmul_rn(s.omb2, __fmul_rn(gc, gc)));
    } else if constexpr (OPT == kAdaGrad) {
        const float gc = __fmaf_rn(s.wd, w, g);
        v = __fmaf_rn(gc, gc, v);
    } else if constexpr (OPT == kSGDMomentum) {
        m = __fmaf_rn(s.mu, m, __fmaf_rn(s.wd, w, g));
    }
}

}  // namespace forge
