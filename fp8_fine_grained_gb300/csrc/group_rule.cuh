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

// two bf16 values (the low and high half of w) -> two E4M3 bytes
__device__ __forceinline__ uint32_t quant2(uint32_t w, float inv)
{
    return cvt_e4m3x2(__fmul_rn(bf16_lo(w), inv), __fmul_rn(bf16_hi(w), inv));
}

}  // namespace fp8fg
