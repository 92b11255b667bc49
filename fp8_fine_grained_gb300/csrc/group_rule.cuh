// The fine-grained quantisation rule shared by the quantise kernels and the
// GEMM epilogue that emits E4M3 output.
//
// Group rule (innerforce.co.kr, fine-grained quantization paragraph, Figure
// 7(a); tonho.wtf DeepSeek-V3 entry, "como funciona"): amax = max |x| over
// the group; s = amax/448 and inv = 448/amax as IEEE FP32 divisions (s = inv
// = 1 when amax is 0 or 448/amax overflows); code = E4M3(x*inv) with one FP32
// product and one round-to-nearest-even, saturating conversion.
#pragma once

#include "ptx.cuh"

namespace fp8fg {

struct ScalePair {
    float s, inv;
};

__device__ __forceinline__ ScalePair group_scale(float amax)
{
    ScalePair r{1.0f, 1.0f};
    if (amax != 0.0f) {
        float inv = __fdiv_rn(448.0f, amax);
        if (!isinf(inv)) {
            r.inv = inv;
            r.s = __fdiv_rn(amax, 448.0f);
        }
    }
    return r;
}

// Power-of-two variant (microscaling: innerforce.co.kr relates the groups to
// microscaling formats and the Blackwell tensor cores that support them;
// tonho.wtf "o que isso custou" lists MMA with group scaling): s = 2^e, the
// smallest power of two with amax <= 448 * 2^e, e >= -127 (the UE8M0 range);
// inv = 2^-e; amax = 0 gives s = inv = 1. With amax = 1.m * 2^(E-127) and
// 448 = 1.75 * 2^8, e = E - 135, plus one when the mantissa exceeds 0.75.
// x * inv is exact, so a code is one rounding of x / s.
__device__ __forceinline__ ScalePair group_scale_pow2(float amax)
{
    ScalePair r{1.0f, 1.0f};
    if (amax != 0.0f) {
        const uint32_t b = __float_as_uint(amax);
        const int E = (int)(b >> 23);
        int e = E - 135 + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0);
        if (E == 0 || e < -127)
            e = -127;  // amax below 2^-119: 448 * 2^-127 covers it
        r.s = e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(0x00400000u);
        r.inv = __uint_as_float((uint32_t)(127 - e) << 23);
    }
    return r;
}

template <bool P2>
__device__ __forceinline__ ScalePair group_scale_rule(float amax)
{
    if constexpr (P2)
        return group_scale_pow2(amax);
    else
        return group_scale(amax);
}

}  // namespace fp8fg
