// MoE combine: the gate-weighted sum of each token's k expert output rows.
//
// After the expert GEMMs, every token has k output rows (one per routed
// expert; yunhecapital.com 2.2.2 and tonho.wtf "como funciona": 8 of 256
// routed experts per token), returned in bf16 after the FP8 dispatch
// (innerforce.co.kr, the mixed-precision framework paragraph: activations
// are cached and dispatched in FP8). The layer's output for the token is
//     out[t][n] = sum_{j < k} w[t][j] * y[dest[t][j]][n],
// each product and each partial sum an FP32 operation in slot order (no
// fused multiply-add), then rounded to bf16 (nearest even) or kept in FP32.
//
// A memory stream (k bf16 rows read, one row written per token): each thread
// owns 8 consecutive columns of one token and takes its slots in batches of
// 8, issuing a batch's 16-byte loads before it folds any; the batch bounds
// the registers so that four 256-thread CTAs fit on an SM (1024 threads with
// 128 bytes each in flight). Each thread writes 16 (bf16) or 32 (FP32)
// bytes. The slot indices and gate weights of the token are read through the
// read-only cache (every thread of the token reads the same k pairs).
#include <cuda_bf16.h>

#include "host_common.h"
#include "ptx.cuh"

namespace fp8fg {
namespace {

constexpr int COMBINE_MAX_K = 16;
constexpr int COMBINE_BATCH = 8;
constexpr int COMBINE_THREADS = 256;
constexpr int COMBINE_CTAS_PER_SM = 4;

template <bool F32>
__global__ void __launch_bounds__(COMBINE_THREADS, COMBINE_CTAS_PER_SM)
    moe_combine_kernel(const uint16_t *__restrict__ y, int64_t ldy, int64_t y_rows, const int32_t *__restrict__ dest,
                       const float *__restrict__ w, int64_t T, int k, int64_t chunks, void *__restrict__ out,
                       int64_t ldo, int *status)
{
    const int64_t total = T * chunks;
    const int64_t ldy16 = ldy / 8;  // row pitch in 16-byte chunks
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = idx / chunks;
        const uint4 *yc = reinterpret_cast<const uint4 *>(y) + (idx - t * chunks);
        const int32_t *dt = dest + t * k;
        const float *wt = w + t * k;
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
            acc[e] = 0.0f;
        for (int j0 = 0; j0 < k; j0 += COMBINE_BATCH) {
            uint4 v[COMBINE_BATCH];
            unsigned live = 0;  // slots of the batch with a row; the others add nothing
#pragma unroll
            for (int b = 0; b < COMBINE_BATCH; ++b) {
                v[b] = make_uint4(0, 0, 0, 0);
                if (j0 + b < k) {
                    const int64_t d = __ldg(dt + j0 + b);
                    if (d >= y_rows) {
                        atomicCAS(status, 0, FP8FG_EDEVICE);
                    } else if (d >= 0) {
                        v[b] = __ldg(yc + d * ldy16);
                        live |= 1u << b;
                    }
                }
            }
#pragma unroll
            for (int b = 0; b < COMBINE_BATCH; ++b) {
                if (live & (1u << b)) {
                    const float g = __ldg(wt + j0 + b);
                    const uint32_t u[4] = {v[b].x, v[b].y, v[b].z, v[b].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        acc[2 * e] = __fadd_rn(acc[2 * e], __fmul_rn(g, bf16_lo(u[e])));
                        acc[2 * e + 1] = __fadd_rn(acc[2 * e + 1], __fmul_rn(g, bf16_hi(u[e])));
                    }
                }
            }
        }
        if constexpr (F32) {
            float4 *o = reinterpret_cast<float4 *>(static_cast<float *>(out) + t * ldo) + 2 * (idx - t * chunks);
            o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        } else {
            uint4 o;
            uint32_t *ow = reinterpret_cast<uint32_t *>(&o);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * e], acc[2 * e + 1]);
                ow[e] = *reinterpret_cast<const uint32_t *>(&h);
            }
            reinterpret_cast<uint4 *>(static_cast<uint16_t *>(out) + t * ldo)[idx - t * chunks] = o;
        }
    }
}

}  // namespace
}  // namespace fp8fg

using namespace fp8fg;

extern "C" int fp8_moe_combine(const void *y, int64_t ldy, int64_t y_rows, const int32_t *dest, const float *w,
                               int64_t T, int k, int64_t N, void *out, int out_kind, int64_t ldo, void *stream)
{
    if (out_kind != FP8FG_OUT_F32 && out_kind != FP8FG_OUT_BF16)
        return FP8FG_EINVAL;
    if (T < 0 || N < 0 || y_rows < 0 || k < 1 || k > COMBINE_MAX_K || N % 8 != 0 || ldy < N || ldo < N)
        return FP8FG_EINVAL;
    if (T == 0 || N == 0)
        return FP8FG_OK;
    if (!y || !dest || !w || !out)
        return FP8FG_EINVAL;
    const int64_t esz = out_kind == FP8FG_OUT_F32 ? 4 : 2;
    if (!aligned16(y) || !aligned16(out) || ldy % 8 != 0 || (ldo * esz) % 16 != 0)
        return FP8FG_EALIGN;
    if (T >= (1ll << 40) || N >= (1ll << 31))
        return FP8FG_EINVAL;
    if (!device_supported())
        return FP8FG_EUNSUPPORTED;
    int *status = status_word_ptr();
    if (!status)
        return FP8FG_ECUDA;
    const int64_t chunks = N / 8, total = T * chunks;
    const int64_t want = (total + COMBINE_THREADS - 1) / COMBINE_THREADS;
    const int64_t cap = (int64_t)sm_count() * COMBINE_CTAS_PER_SM * 4;  // four waves; the loop strides past the rest
    const unsigned grid = (unsigned)(want < cap ? want : (cap > 0 ? cap : 1));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (out_kind == FP8FG_OUT_F32)
        moe_combine_kernel<true><<<grid, COMBINE_THREADS, 0, s>>>(static_cast<const uint16_t *>(y), ldy, y_rows, dest,
                                                                  w, T, k, chunks, out, ldo, status);
    else
        moe_combine_kernel<false><<<grid, COMBINE_THREADS, 0, s>>>(static_cast<const uint16_t *>(y), ldy, y_rows,
                                                                   dest, w, T, k, chunks, out, ldo, status);
    return launch_status();
}
