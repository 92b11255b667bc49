// Fine-grained E4M3 quantisation kernels: 1x128 tiles (per row, also for
// rows gathered through a row index or scattered to several destinations), 128x1 tiles with transposed output
// (per column, for the weight-gradient operands), both of those from one
// read, and 128x128 blocks (weights).
//
// The group rule (amax, s = amax/448, inv = 448/amax, one RNE saturating
// conversion of x*inv) is in group_rule.cuh, with its power-of-two variant
// (s = the smallest 2^e with amax <= 448 * 2^e) that the *_pow2 entry points
// select through the P2 template parameter.
//
// The kernels are streams bound by HBM and instruction issue (2 bytes read,
// 1 byte + 4/128 or 4/16384 bytes written per element). They read with
// 16-byte vector loads issued back to back (several in flight per thread),
// reduce the amax with warp shuffles, and write codes and scales with full
// 32-byte sectors.
#include <cuda_bf16.h>

#include "group_rule.cuh"
#include "host_common.h"
#include "ptx.cuh"
#include "tensor_map.h"

namespace fp8fg {
namespace {

constexpr int GROUP = 128;

// max |x| over 8 bf16 values packed in a uint4 (bit patterns of magnitudes
// order like the magnitudes themselves).
__device__ __forceinline__ uint32_t absmax_bits8(const uint4 &v)
{
    uint32_t m = __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                          __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
    return max(m & 0xFFFFu, m >> 16);
}

// two bf16 values (the halves of w) times inv as one packed pair of FP32
// products (each an IEEE round-to-nearest product, as __fmul_rn) -> two
// E4M3 bytes
__device__ __forceinline__ uint32_t quant2x(uint32_t w, float2 inv2)
{
    const float2 p = __fmul2_rn(make_float2(bf16_lo(w), bf16_hi(w)), inv2);
    return cvt_e4m3x2(p.x, p.y);
}

// 8 bf16 -> 8 E4M3 bytes
__device__ __forceinline__ uint2 quant8(const uint4 &v, float inv)
{
    const float2 inv2 = make_float2(inv, inv);
    uint2 o;
    o.x = quant2x(v.x, inv2) | (quant2x(v.y, inv2) << 16);
    o.y = quant2x(v.z, inv2) | (quant2x(v.w, inv2) << 16);
    return o;
}

// Group scales of N groups per half-warp (N <= 16) with one division
// sequence per warp: on entry every lane of half-warp h holds the amax bit
// patterns m[0..N) of its N groups (shuffle-reduced over the half-warp);
// lane (16h + j) computes the scale pair of group j and the pairs are
// broadcast back. Bit-identical to calling group_scale per group.
template <int N, bool P2>
__device__ __forceinline__ void group_scales_batched(const uint32_t (&m)[N], float (&s)[N], float (&inv)[N])
{
    static_assert(N <= 16, "one group per lane of a half-warp");
    const int lane = threadIdx.x & 31;
    const int j = lane & 15;
    uint32_t mine = m[0];
#pragma unroll
    for (int i = 1; i < N; ++i)
        mine = j == i ? m[i] : mine;
    const ScalePair sp = group_scale_rule<P2>(__uint_as_float(mine << 16));
#pragma unroll
    for (int i = 0; i < N; ++i) {
        s[i] = __shfl_sync(0xffffffffu, sp.s, (lane & 16) + i);
        inv[i] = __shfl_sync(0xffffffffu, sp.inv, (lane & 16) + i);
    }
}

__device__ __forceinline__ uint4 ld_stream_v4(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// ------------------------------------------------------ 1x128, per row ----
// CTA tile: 4 rows x gt groups (gt <= 16; 16 gt threads = gt half-warps).
// Half-warp h owns group h of the tile and quantises it in each of the 4
// rows, loading all four 256-byte segments before reducing any. The grid
// walks the tiles in memory order (group blocks fastest). Small CTAs with
// few registers keep eight or more per SM resident, which keeps enough
// loads in flight to stream at HBM rate; a sweep of tile shapes on GB300
// put 4 rows ahead of taller tiles with more loads per thread. The host
// picks gt so that it divides the row's group count where it can (14 for
// 56 groups): a partly empty last tile in every row would leave its
// half-warps idle.
constexpr int QR_ROWS = 4;
constexpr int QR_GROUPS = 16;  // largest group tile
constexpr int QR_ITEMS = QR_ROWS;

// Groups per tile for a row of ngroups groups: the largest even width from 8
// to 16 that divides ngroups, else 16; short rows take one tile of ngroups
// rounded up to even. The width is even so that every warp of the CTA is
// whole (the reductions shuffle across full warps).
inline int row_group_tile(int64_t ngroups)
{
    if (ngroups <= QR_GROUPS)
        return (int)((ngroups + 1) & ~int64_t(1));
    for (int g = QR_GROUPS; g >= 8; g -= 2)
        if (ngroups % g == 0)
            return g;
    return QR_GROUPS;
}

// GATHER: output row r quantises source row row_index[r] (rows listed in
// MoE expert order); an index outside [0, n_src) is reported as
// FP8FG_EDEVICE in the status word and reads source row 0. Quantisation is
// per row, so the result equals gathering the rows of the plain output.
template <bool GATHER, bool P2>
__global__ void __launch_bounds__(256, 8) quant_rows_kernel(const uint16_t *__restrict__ x, int64_t rows,
                                                            int64_t ngroups, int64_t ldx, uint8_t *__restrict__ q,
                                                            int64_t ldq, float *__restrict__ scales, int64_t ld_s,
                                                            int64_t tiles_g, int gt, const int32_t *__restrict__ row_index,
                                                            int64_t n_src, int *status)
{
    griddep_launch_dependents();  // a dependent GEMM may set itself up under this grid's tail
    __shared__ float s_scale[QR_GROUPS][QR_ROWS];
    const int hw = threadIdx.x >> 4;
    const int l = threadIdx.x & 15;
    const int64_t gb = blockIdx.x % tiles_g, rb = blockIdx.x / tiles_g;
    const int64_t r0 = rb * QR_ROWS;
    const int64_t g = gb * gt + hw;
    const bool g_ok = g < ngroups;
    const uint16_t *src = x + r0 * ldx + g * GROUP + l * 8;
    uint8_t *dst = q + r0 * ldq + g * GROUP + l * 8;

    uint4 v[QR_ITEMS];
#pragma unroll
    for (int i = 0; i < QR_ITEMS; ++i) {
        if (g_ok && r0 + i < rows) {
            if constexpr (GATHER) {
                int64_t sr = row_index[r0 + i];
                if (sr < 0 || sr >= n_src) {
                    atomicCAS(status, 0, FP8FG_EDEVICE);
                    sr = 0;
                }
                v[i] = ld_stream_v4(x + sr * ldx + g * GROUP + l * 8);
            } else {
                v[i] = ld_stream_v4(src + (int64_t)i * ldx);
            }
        } else {
            v[i] = make_uint4(0, 0, 0, 0);
        }
    }
    uint32_t m[QR_ITEMS];
#pragma unroll
    for (int i = 0; i < QR_ITEMS; ++i) {
        m[i] = absmax_bits8(v[i]);
#pragma unroll
        for (int off = 8; off >= 1; off >>= 1)
            m[i] = max(m[i], __shfl_xor_sync(0xffffffffu, m[i], off));
    }
    float sc[QR_ITEMS], inv[QR_ITEMS];
    group_scales_batched<QR_ITEMS, P2>(m, sc, inv);
#pragma unroll
    for (int i = 0; i < QR_ITEMS; ++i) {
        if (g_ok && r0 + i < rows) {
            *reinterpret_cast<uint2 *>(dst + (int64_t)i * ldq) = quant8(v[i], inv[i]);
            if (l == 0)
                s_scale[hw][i] = sc[i];
        }
    }
    __syncthreads();
    if (threadIdx.x < QR_ROWS * gt) {
        const int gg = threadIdx.x / QR_ROWS, rr = threadIdx.x % QR_ROWS;
        const int64_t row = r0 + rr, gs = gb * gt + gg;
        if (row < rows && gs < ngroups)
            scales[gs * ld_s + row] = s_scale[gg][rr];
    }
}

// ------------------------------------- 1x128 per row, scattered copies ----
// The MoE dispatch in token order: every source row is read and quantised
// once (the tile and group rule of quant_rows_kernel) and its codes and
// scales are written to each of its k destination rows dest_index[r*k + j]
// (rows grouped by expert). A negative destination is not written; one at or
// beyond n_out is reported as FP8FG_EDEVICE and not written. The output
// equals gathering rows of the plain 1x128 quantisation.
constexpr int SCATTER_MAX_K = 16;

template <bool P2>
__global__ void __launch_bounds__(256, 8) quant_rows_scatter_kernel(const uint16_t *__restrict__ x, int64_t rows,
                                                                    int64_t ngroups, int64_t ldx,
                                                                    uint8_t *__restrict__ q, int64_t ldq,
                                                                    float *__restrict__ scales, int64_t ld_s,
                                                                    int64_t tiles_g, int gt, const int32_t *__restrict__ dest,
                                                                    int k, int64_t n_out, int *status)
{
    griddep_launch_dependents();  // a dependent GEMM may set itself up under this grid's tail
    __shared__ float s_scale[QR_GROUPS][QR_ROWS];
    __shared__ int32_t s_dst[QR_ROWS][SCATTER_MAX_K];
    const int hw = threadIdx.x >> 4;
    const int l = threadIdx.x & 15;
    const int64_t gb = blockIdx.x % tiles_g, rb = blockIdx.x / tiles_g;
    const int64_t r0 = rb * QR_ROWS;
    const int64_t g = gb * gt + hw;
    const bool g_ok = g < ngroups;
    if (threadIdx.x < QR_ROWS * k) {
        const int rr = threadIdx.x / k, j = threadIdx.x % k;
        int32_t d = -1;
        if (r0 + rr < rows) {
            d = dest[(r0 + rr) * k + j];
            if (d >= n_out) {
                atomicCAS(status, 0, FP8FG_EDEVICE);
                d = -1;
            }
        }
        s_dst[rr][j] = d;
    }
    const uint16_t *src = x + r0 * ldx + g * GROUP + l * 8;
    uint4 v[QR_ITEMS];
#pragma unroll
    for (int i = 0; i < QR_ITEMS; ++i)
        v[i] = (g_ok && r0 + i < rows) ? ld_stream_v4(src + (int64_t)i * ldx) : make_uint4(0, 0, 0, 0);
    uint32_t m[QR_ITEMS];
#pragma unroll
    for (int i = 0; i < QR_ITEMS; ++i) {
        m[i] = absmax_bits8(v[i]);
#pragma unroll
        for (int off = 8; off >= 1; off >>= 1)
            m[i] = max(m[i], __shfl_xor_sync(0xffffffffu, m[i], off));
    }
    float sc[QR_ITEMS], inv[QR_ITEMS];
    group_scales_batched<QR_ITEMS, P2>(m, sc, inv);
    __syncthreads();  // destinations
#pragma unroll
    for (int i = 0; i < QR_ITEMS; ++i) {
        if (g_ok && r0 + i < rows) {
            const uint2 code = quant8(v[i], inv[i]);
            for (int j = 0; j < k; ++j) {
                const int32_t d = s_dst[i][j];
                if (d >= 0)
                    *reinterpret_cast<uint2 *>(q + (int64_t)d * ldq + g * GROUP + l * 8) = code;
            }
            if (l == 0)
                s_scale[hw][i] = sc[i];
        }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < gt * QR_ROWS * k; idx += blockDim.x) {
        const int gg = idx / (QR_ROWS * k), rem = idx % (QR_ROWS * k);
        const int rr = rem / k, j = rem % k;
        const int64_t gs = gb * gt + gg;
        const int32_t d = s_dst[rr][j];
        if (r0 + rr < rows && gs < ngroups && d >= 0)
            scales[gs * ld_s + d] = s_scale[gg][rr];
    }
}

// ---------------------------------------- 128x1 along rows, transposed ----
// CTA tile: 128 rows (one group) x 64 columns, staged in shared memory.
// Thread (c = tid % 64, part = tid / 64) reduces rows part*32..+31 of
// column c, then writes those 32 codes as 32 contiguous bytes of row c of
// the transposed output.
constexpr int QT_COLS = 64;

template <bool P2>
__global__ void __launch_bounds__(256, 8) quant_cols_t_kernel(const uint16_t *__restrict__ x, int64_t rows,
                                                           int64_t cols, int64_t ldx, uint8_t *__restrict__ qT,
                                                           int64_t ldq, float *__restrict__ scales, int64_t ld_s)
{
    griddep_launch_dependents();  // a dependent GEMM may set itself up under this grid's tail
    __shared__ __align__(16) uint16_t tile[GROUP][QT_COLS];
    __shared__ uint32_t s_cmax[8][QT_COLS / 2];  // column-pair maxima of each 16-row part
    __shared__ float s_inv[QT_COLS];
    const int tid = threadIdx.x;
    const int64_t c0 = (int64_t)blockIdx.x * QT_COLS;
    const int64_t r0 = (int64_t)blockIdx.y * GROUP;

    uint4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int chunk = i * 256 + tid;
        const int rr = chunk >> 3, cc = (chunk & 7) * 8;
        if (c0 + cc < cols)
            v[i] = ld_stream_v4(x + (r0 + rr) * ldx + c0 + cc);
        else
            v[i] = make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int chunk = i * 256 + tid;
        *reinterpret_cast<uint4 *>(&tile[chunk >> 3][(chunk & 7) * 8]) = v[i];
    }
    __syncthreads();

    // thread (cp, part): the column pair 2cp, 2cp+1 over rows part*16 ..
    // +15, both columns read as one 32-bit word (a warp reads one 128-byte
    // row) and reduced with packed 16-bit maxima
    const int cp = tid & (QT_COLS / 2 - 1), part = tid >> 5;
    const uint32_t *t32 = reinterpret_cast<const uint32_t *>(&tile[0][0]);
    uint32_t m2 = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i)
        m2 = __vmaxu2(m2, t32[(part * 16 + i) * (QT_COLS / 2) + cp] & 0x7FFF7FFFu);
    s_cmax[part][cp] = m2;
    __syncthreads();
    if (tid < QT_COLS) {
        // column tid: the group's scale pair, once per column
        uint32_t m = 0;
#pragma unroll
        for (int pq = 0; pq < 8; ++pq) {
            const uint32_t w = s_cmax[pq][tid >> 1];
            m = max(m, (tid & 1) ? (w >> 16) : (w & 0xFFFFu));
        }
        const ScalePair sp = group_scale_rule<P2>(__uint_as_float(m << 16));
        s_inv[tid] = sp.inv;
        if (c0 + tid < cols)
            scales[(r0 / GROUP) * ld_s + c0 + tid] = sp.s;
    }
    __syncthreads();
    // codes: rows r, r+1 of one column form one packed product and one
    // E4M3 pair; each column's 16 codes go out as one 16-byte piece of its
    // transposed row
    const int64_t col = c0 + 2 * cp;
    if (col < cols) {
        const float2 inva = make_float2(s_inv[2 * cp], s_inv[2 * cp]);
        const float2 invb = make_float2(s_inv[2 * cp + 1], s_inv[2 * cp + 1]);
        uint32_t pa[4], pb[4];
#pragma unroll
        for (int rp = 0; rp < 8; ++rp) {
            const uint32_t w0 = t32[(part * 16 + 2 * rp) * (QT_COLS / 2) + cp];
            const uint32_t w1 = t32[(part * 16 + 2 * rp + 1) * (QT_COLS / 2) + cp];
            const float2 xa = __fmul2_rn(make_float2(bf16_lo(w0), bf16_lo(w1)), inva);
            const float2 xb = __fmul2_rn(make_float2(bf16_hi(w0), bf16_hi(w1)), invb);
            const uint32_t ca = cvt_e4m3x2(xa.x, xa.y), cb = cvt_e4m3x2(xb.x, xb.y);
            if (rp & 1) {
                pa[rp >> 1] |= ca << 16;
                pb[rp >> 1] |= cb << 16;
            } else {
                pa[rp >> 1] = ca;
                pb[rp >> 1] = cb;
            }
        }
        *reinterpret_cast<uint4 *>(qT + col * ldq + r0 + part * 16) = make_uint4(pa[0], pa[1], pa[2], pa[3]);
        if (col + 1 < cols)
            *reinterpret_cast<uint4 *>(qT + (col + 1) * ldq + r0 + part * 16) = make_uint4(pb[0], pb[1], pb[2], pb[3]);
    }
}

// --------------------------------------- 1x128 and 128x1 from one read ----
// Both activation layouts a training step needs (row groups for fprop and
// dgrad, column groups transposed for wgrad) from a single read of x: the
// CTA quantises a 128x128 tile's rows and its columns from one
// shared-memory copy. The outputs are bit-identical to fp8_quant_1x128
// with transpose 0 and 1 (same group rule, same products). 4.06 bytes of
// traffic per element instead of 2 x 3.03.
//
// Persistent, three CTAs per SM: each CTA walks its tiles with a stride of
// the grid and has the next tile's 32 KB brought in by TMA (into the other
// of two buffers) while it quantises the current one, so every SM keeps
// loads in flight through the compute phases. The wait on a tile is bounded
// (FP8FG_ETIMEOUT in the status word, then the CTA drains and leaves).
constexpr int DUAL_CTAS_PER_SM = 3;
constexpr uint32_t DUAL_TILE_BYTES = GROUP * GROUP * 2;

struct DualSmem {
    uint16_t tile[2][GROUP][GROUP];  // two bf16 tiles, rows of 256 bytes (the TMA box as it lands)
    uint64_t bar[2];                 // "tile landed", one per buffer
    uint32_t s_cmax[4][GROUP / 2];   // column-pair maxima (two 16-bit magnitudes) of each row quarter
    float s_cinv[GROUP];             // the columns' 448/amax
    float s_row[GROUP];
    int abort;
};

template <bool P2>
__global__ void __launch_bounds__(256, DUAL_CTAS_PER_SM)
    quant_dual_kernel(const __grid_constant__ CUtensorMap tmx, int64_t tiles_c, int64_t n_tiles,
                      uint8_t *__restrict__ q, int64_t ldq, float *__restrict__ scales, int64_t ld_s,
                      uint8_t *__restrict__ qT, int64_t ldqT, float *__restrict__ scalesT, int64_t ld_sT, int *status,
                      uint64_t wait_limit_ns, int skip_first_load)
{
    griddep_launch_dependents();  // a dependent GEMM may set itself up under this grid's tail
    extern __shared__ __align__(128) uint8_t dual_raw[];
    DualSmem &S = *reinterpret_cast<DualSmem *>(dual_raw);
    const int tid = threadIdx.x;
    const int l = tid & 15;
    const uint32_t bar0 = smem_u32(&S.bar[0]);
    if (tid == 0) {
        mbar_init(bar0, 1);
        mbar_init(bar0 + 8, 1);
        S.abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmx);
    }
    __syncthreads();
    const WaitCtl wc{&S.abort, status, wait_limit_ns};
    auto fetch = [&](int64_t t, uint32_t b) {
        mbar_arrive_expect_tx(bar0 + 8 * b, DUAL_TILE_BYTES);
        tma_load_2d(smem_u32(&S.tile[b][0][0]), &tmx, (int32_t)((t % tiles_c) * GROUP),
                    (int32_t)((t / tiles_c) * GROUP), bar0 + 8 * b);
    };
    // (test hook: CTA 0 withholds its first copy, so that its bounded wait
    // runs out and the launch reports FP8FG_ETIMEOUT)
    if (tid == 0 && (int64_t)blockIdx.x < n_tiles && !(skip_first_load && blockIdx.x == 0))
        fetch(blockIdx.x, 0);
    uint32_t it = 0;
    for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x, ++it) {
        const uint32_t b = it & 1;
        // the other buffer was last read in the previous iteration, which
        // ended at a barrier: it may be refilled
        const bool ahead = t + gridDim.x < n_tiles;
        if (tid == 0 && ahead)
            fetch(t + gridDim.x, b ^ 1);
        const bool got = mbar_wait(bar0 + 8 * b, (it >> 1) & 1, wc, FP8FG_ETIMEOUT);
        if (!__syncthreads_and(got)) {
            // drain the copies this CTA still has in flight before leaving
            if (tid == 0) {
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(bar0 + 8 * b, (it >> 1) & 1) && global_timer_ns() - t0 < wait_limit_ns) {
                }
                while (ahead && !mbar_try_wait(bar0 + 8 * (b ^ 1), ((it + 1) >> 1) & 1) &&
                       global_timer_ns() - t0 < 2 * wait_limit_ns) {
                }
            }
            return;
        }
        uint16_t(*tile)[GROUP] = S.tile[b];
        const int64_t c0 = (t % tiles_c) * GROUP, r0 = (t / tiles_c) * GROUP;

        // row groups: chunk i*256 + tid = row (i*16 + tid/16), columns
        // (tid%16)*8 .. +7; one half-warp per row, the eight rows' scales
        // in one batch
        uint4 v[8];
        uint32_t mr[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[i] = *reinterpret_cast<const uint4 *>(&tile[i * 16 + (tid >> 4)][l * 8]);
            mr[i] = absmax_bits8(v[i]);
        }
        // half-warp maxima, two rows' 16-bit magnitudes per shuffle
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
            uint32_t m2 = mr[i] | (mr[i + 1] << 16);
#pragma unroll
            for (int off = 8; off >= 1; off >>= 1)
                m2 = __vmaxu2(m2, __shfl_xor_sync(0xffffffffu, m2, off));
            mr[i] = m2 & 0xFFFFu;
            mr[i + 1] = m2 >> 16;
        }
        float sr[8], ir[8];
        group_scales_batched<8, P2>(mr, sr, ir);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int rr = i * 16 + (tid >> 4);
            *reinterpret_cast<uint2 *>(q + (r0 + rr) * ldq + c0 + l * 8) = quant8(v[i], ir[i]);
            if (l == 0)
                S.s_row[rr] = sr[i];
        }

        // column groups: thread (cp, part) covers the column pair 2cp, 2cp+1
        // over rows part*32 .. +31, reading both columns as one 32-bit word
        // (a warp reads 128 contiguous bytes of a row)
        const int cp = tid & (GROUP / 2 - 1), part = tid >> 6;
        const uint32_t *t32 = reinterpret_cast<const uint32_t *>(&tile[0][0]);
        uint32_t m2 = 0;
#pragma unroll 8
        for (int i = 0; i < 32; ++i)
            m2 = __vmaxu2(m2, t32[(part * 32 + i) * (GROUP / 2) + cp] & 0x7FFF7FFFu);
        S.s_cmax[part][cp] = m2;
        __syncthreads();
        if (tid < GROUP) {
            // column tid: its group's scale pair, once per column
            scales[(c0 / GROUP) * ld_s + r0 + tid] = S.s_row[tid];
            uint32_t m = 0;
#pragma unroll
            for (int pq = 0; pq < 4; ++pq) {
                const uint32_t w = S.s_cmax[pq][tid >> 1];
                m = max(m, (tid & 1) ? (w >> 16) : (w & 0xFFFFu));
            }
            const ScalePair sp = group_scale_rule<P2>(__uint_as_float(m << 16));
            S.s_cinv[tid] = sp.inv;
            scalesT[(r0 / GROUP) * ld_sT + c0 + tid] = sp.s;
        }
        __syncthreads();
        // codes: rows r, r+1 of one column form one packed product and one
        // E4M3 pair; each column's 32 codes go out as one 32-byte run
        const float2 inva = make_float2(S.s_cinv[2 * cp], S.s_cinv[2 * cp]);
        const float2 invb = make_float2(S.s_cinv[2 * cp + 1], S.s_cinv[2 * cp + 1]);
        uint32_t pa[8], pb[8];
#pragma unroll
        for (int rp = 0; rp < 16; ++rp) {
            const uint32_t w0 = t32[(part * 32 + 2 * rp) * (GROUP / 2) + cp];
            const uint32_t w1 = t32[(part * 32 + 2 * rp + 1) * (GROUP / 2) + cp];
            const float2 xa = __fmul2_rn(make_float2(bf16_lo(w0), bf16_lo(w1)), inva);
            const float2 xb = __fmul2_rn(make_float2(bf16_hi(w0), bf16_hi(w1)), invb);
            const uint32_t ca = cvt_e4m3x2(xa.x, xa.y), cb = cvt_e4m3x2(xb.x, xb.y);
            if (rp & 1) {
                pa[rp >> 1] |= ca << 16;
                pb[rp >> 1] |= cb << 16;
            } else {
                pa[rp >> 1] = ca;
                pb[rp >> 1] = cb;
            }
        }
        uint4 *da = reinterpret_cast<uint4 *>(qT + (c0 + 2 * cp) * ldqT + r0 + part * 32);
        uint4 *db = reinterpret_cast<uint4 *>(qT + (c0 + 2 * cp + 1) * ldqT + r0 + part * 32);
        da[0] = make_uint4(pa[0], pa[1], pa[2], pa[3]);
        da[1] = make_uint4(pa[4], pa[5], pa[6], pa[7]);
        db[0] = make_uint4(pb[0], pb[1], pb[2], pb[3]);
        db[1] = make_uint4(pb[4], pb[5], pb[6], pb[7]);
        // every read of this buffer and of s_row / s_cmax / s_cinv is done
        // before the next iteration refills the other buffer and rewrites them
        __syncthreads();
    }
}

// ------------------------------------------------------- 128x128 blocks ----
// One CTA per block: 256 threads x 8 chunks of 8 bf16 held in registers.
// DUAL: the transposed codes too (the block of W^T is the transposed block
// with the same scale): the codes go through a shared-memory tile and each
// thread writes 64 codes of one column of the block as a piece of the
// transposed row.
constexpr int QB_PITCH = GROUP + 8;  // bytes per row of the code tile (8-byte aligned rows)

template <bool P2, bool DUAL>
__global__ void __launch_bounds__(256) quant_blocks_kernel(const uint16_t *__restrict__ w, int64_t N, int64_t K,
                                                           int64_t ldw, uint8_t *__restrict__ q, int64_t ldq,
                                                           float *__restrict__ scales, uint8_t *__restrict__ qT,
                                                           int64_t ldqT, float *__restrict__ scalesT)
{
    griddep_launch_dependents();  // a dependent GEMM may set itself up under this grid's tail
    __shared__ uint32_t s_warp[8];
    __shared__ __align__(16) uint8_t s_codes[DUAL ? GROUP * QB_PITCH : 8];
    const int tid = threadIdx.x;
    const int64_t bj = blockIdx.x, bi = blockIdx.y;
    const uint16_t *src = w + bi * GROUP * ldw + bj * GROUP;

    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int chunk = i * 256 + tid;  // 16 chunks of 8 per row
        v[i] = ld_stream_v4(src + (chunk >> 4) * ldw + (chunk & 15) * 8);
    }
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        m = max(m, absmax_bits8(v[i]));
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
        m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
    if ((tid & 31) == 0)
        s_warp[tid >> 5] = m;
    __syncthreads();
    m = s_warp[0];
#pragma unroll
    for (int i = 1; i < 8; ++i)
        m = max(m, s_warp[i]);
    const ScalePair sp = group_scale_rule<P2>(__uint_as_float(m << 16));
    uint8_t *dst = q + bi * GROUP * ldq + bj * GROUP;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int chunk = i * 256 + tid;
        const uint2 c8 = quant8(v[i], sp.inv);
        *reinterpret_cast<uint2 *>(dst + (chunk >> 4) * ldq + (chunk & 15) * 8) = c8;
        if constexpr (DUAL)
            *reinterpret_cast<uint2 *>(s_codes + (chunk >> 4) * QB_PITCH + (chunk & 15) * 8) = c8;
    }
    if (tid == 0) {
        scales[bi * (K / GROUP) + bj] = sp.s;
        if constexpr (DUAL)
            scalesT[bj * (N / GROUP) + bi] = sp.s;
    }
    if constexpr (DUAL) {
        __syncthreads();
        // thread: column c of the block (a warp reads 32 consecutive bytes
        // of a row), rows h*64 .. +63 -> qT row (block column c), 64 codes
        const int c = tid & (GROUP - 1), h = tid >> 7;
        uint32_t wv[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const uint8_t *col = s_codes + (h * 64 + 4 * j) * QB_PITCH + c;
            wv[j] = (uint32_t)col[0] | ((uint32_t)col[QB_PITCH] << 8) | ((uint32_t)col[2 * QB_PITCH] << 16) |
                    ((uint32_t)col[3 * QB_PITCH] << 24);
        }
        uint4 *out = reinterpret_cast<uint4 *>(qT + (bj * GROUP + c) * ldqT + bi * GROUP + h * 64);
#pragma unroll
        for (int j = 0; j < 4; ++j)
            out[j] = make_uint4(wv[4 * j], wv[4 * j + 1], wv[4 * j + 2], wv[4 * j + 3]);
    }
}

// ----------------------------------------------------------- entry points ----
// Argument checks and launches, shared by the pages' rule (P2 = false) and
// the power-of-two variant.

template <bool P2>
int quant_1x128(const void *x, int64_t rows, int64_t cols, int64_t ldx, uint8_t *q, int64_t ldq,
                               float *scales, int64_t ld_s, int transpose, void *stream)
{
    if (rows < 0 || cols < 0 || (transpose != 0 && transpose != 1))
        return FP8FG_EINVAL;
    if (transpose == 0) {
        if (cols % GROUP != 0 || ldx < cols || ldq < cols || ld_s < rows)
            return FP8FG_EINVAL;
    } else {
        if (rows % GROUP != 0 || ldx < cols || ldq < rows || ld_s < cols)
            return FP8FG_EINVAL;
    }
    if (rows == 0 || cols == 0)
        return FP8FG_OK;
    if (!x || !q || !scales)
        return FP8FG_EINVAL;
    if (!aligned16(x) || !aligned16(q) || !aligned16(scales) || ldx % 8 != 0 || ldq % 16 != 0 || ld_s % 4 != 0)
        return FP8FG_EALIGN;
    if (!device_supported())
        return FP8FG_EUNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (transpose == 0) {
        const int64_t ngroups = cols / GROUP;
        const int gt = row_group_tile(ngroups);
        const int64_t tiles_g = (ngroups + gt - 1) / gt;
        const int64_t tiles = tiles_g * ((rows + QR_ROWS - 1) / QR_ROWS);
        if (tiles > 0x7FFFFFFF)
            return FP8FG_EINVAL;
        quant_rows_kernel<false, P2><<<(unsigned)tiles, 16 * gt, 0, s>>>(static_cast<const uint16_t *>(x), rows,
                                                                      ngroups, ldx, q, ldq, scales, ld_s, tiles_g,
                                                                      gt, nullptr, 0, nullptr);
    } else {
        const int64_t gx = (cols + QT_COLS - 1) / QT_COLS, gy = rows / GROUP;
        if (gx > 0x7FFFFFFF || gy > 65535)
            return FP8FG_EINVAL;
        quant_cols_t_kernel<P2><<<dim3((unsigned)gx, (unsigned)gy), 256, 0, s>>>(
            static_cast<const uint16_t *>(x), rows, cols, ldx, q, ldq, scales, ld_s);
    }
    return launch_status();
}

template <bool P2>
int quant_1x128_gather(const void *x, int64_t n_src, int64_t cols, int64_t ldx,
                                      const int32_t *row_index, int64_t rows, uint8_t *q, int64_t ldq, float *scales,
                                      int64_t ld_s, void *stream)
{
    if (n_src < 0 || rows < 0 || cols < 0 || cols % GROUP != 0 || ldx < cols || ldq < cols || ld_s < rows)
        return FP8FG_EINVAL;
    if (rows == 0 || cols == 0)
        return FP8FG_OK;
    if (!x || !row_index || !q || !scales || n_src == 0)
        return FP8FG_EINVAL;
    if (!aligned16(x) || !aligned16(q) || !aligned16(scales) || ldx % 8 != 0 || ldq % 16 != 0 || ld_s % 4 != 0)
        return FP8FG_EALIGN;
    if (!device_supported())
        return FP8FG_EUNSUPPORTED;
    int *status = status_word_ptr();
    if (!status)
        return FP8FG_ECUDA;
    const int64_t ngroups = cols / GROUP;
    const int gt = row_group_tile(ngroups);
    const int64_t tiles_g = (ngroups + gt - 1) / gt;
    const int64_t tiles = tiles_g * ((rows + QR_ROWS - 1) / QR_ROWS);
    if (tiles > 0x7FFFFFFF)
        return FP8FG_EINVAL;
    quant_rows_kernel<true, P2><<<(unsigned)tiles, 16 * gt, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t *>(x), rows, ngroups, ldx, q, ldq, scales, ld_s, tiles_g, gt, row_index, n_src,
        status);
    return launch_status();
}

template <bool P2>
int quant_1x128_scatter(const void *x, int64_t n_src, int64_t cols, int64_t ldx, const int32_t *dest_index, int k,
                        int64_t n_out, uint8_t *q, int64_t ldq, float *scales, int64_t ld_s, void *stream)
{
    if (n_src < 0 || n_out < 0 || cols < 0 || cols % GROUP != 0 || k < 1 || k > SCATTER_MAX_K || ldx < cols ||
        ldq < cols || ld_s < n_out)
        return FP8FG_EINVAL;
    if (n_src == 0 || n_out == 0 || cols == 0)
        return FP8FG_OK;
    if (!x || !dest_index || !q || !scales)
        return FP8FG_EINVAL;
    if (!aligned16(x) || !aligned16(q) || !aligned16(scales) || ldx % 8 != 0 || ldq % 16 != 0 || ld_s % 4 != 0)
        return FP8FG_EALIGN;
    if (!device_supported())
        return FP8FG_EUNSUPPORTED;
    int *status = status_word_ptr();
    if (!status)
        return FP8FG_ECUDA;
    const int64_t ngroups = cols / GROUP;
    const int gt = row_group_tile(ngroups);
    const int64_t tiles_g = (ngroups + gt - 1) / gt;
    const int64_t tiles = tiles_g * ((n_src + QR_ROWS - 1) / QR_ROWS);
    if (tiles > 0x7FFFFFFF)
        return FP8FG_EINVAL;
    quant_rows_scatter_kernel<P2><<<(unsigned)tiles, 16 * gt, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t *>(x), n_src, ngroups, ldx, q, ldq, scales, ld_s, tiles_g, gt, dest_index, k,
        n_out, status);
    return launch_status();
}

template <bool P2>
int quant_1x128_dual(const void *x, int64_t rows, int64_t cols, int64_t ldx, uint8_t *q,
                                    int64_t ldq, float *scales, int64_t ld_s, uint8_t *qT, int64_t ldqT,
                                    float *scalesT, int64_t ld_sT, void *stream)
{
    if (rows < 0 || cols < 0 || rows % GROUP != 0 || cols % GROUP != 0 || ldx < cols || ldq < cols || ld_s < rows ||
        ldqT < rows || ld_sT < cols)
        return FP8FG_EINVAL;
    if (rows == 0 || cols == 0)
        return FP8FG_OK;
    if (!x || !q || !scales || !qT || !scalesT)
        return FP8FG_EINVAL;
    if (!aligned16(x) || !aligned16(q) || !aligned16(scales) || !aligned16(qT) || !aligned16(scalesT) ||
        ldx % 8 != 0 || ldq % 16 != 0 || ldqT % 16 != 0 || ld_s % 4 != 0 || ld_sT % 4 != 0)
        return FP8FG_EALIGN;
    if (!device_supported())
        return FP8FG_EUNSUPPORTED;
    const int64_t tiles_c = cols / GROUP, n_tiles = tiles_c * (rows / GROUP);
    if (n_tiles > 0x7FFFFFFF)
        return FP8FG_EINVAL;
    int *status = status_word_ptr();
    CUtensorMap tmx;
    if (!status || !make_map_bf16_tile(&tmx, x, (uint64_t)cols, (uint64_t)rows, (uint64_t)ldx, GROUP, GROUP))
        return FP8FG_ECUDA;
    auto k = quant_dual_kernel<P2>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(DualSmem)) != cudaSuccess) {
        cudaGetLastError();
        return FP8FG_ECUDA;
    }
    const int64_t cap = (int64_t)sm_count() * DUAL_CTAS_PER_SM;
    const unsigned grid = (unsigned)(n_tiles < cap ? n_tiles : (cap > 0 ? cap : 1));
    k<<<grid, 256, sizeof(DualSmem), static_cast<cudaStream_t>(stream)>>>(
        tmx, tiles_c, n_tiles, q, ldq, scales, ld_s, qT, ldqT, scalesT, ld_sT, status, wait_limit_ns(),
        take_skip_first_load() ? 1 : 0);
    return launch_status();
}

template <bool P2>
int quant_128x128(const void *w, int64_t N, int64_t K, int64_t ldw, uint8_t *q, int64_t ldq,
                                 float *scales, void *stream)
{
    if (N < 0 || K < 0 || N % GROUP != 0 || K % GROUP != 0 || ldw < K || ldq < K)
        return FP8FG_EINVAL;
    if (N == 0 || K == 0)
        return FP8FG_OK;
    if (!w || !q || !scales)
        return FP8FG_EINVAL;
    if (!aligned16(w) || !aligned16(q) || ldw % 8 != 0 || ldq % 16 != 0 ||
        (reinterpret_cast<uintptr_t>(scales) & 3u) != 0)
        return FP8FG_EALIGN;
    if (!device_supported())
        return FP8FG_EUNSUPPORTED;
    const int64_t gx = K / GROUP, gy = N / GROUP;
    if (gx > 0x7FFFFFFF || gy > 65535)
        return FP8FG_EINVAL;
    quant_blocks_kernel<P2, false><<<dim3((unsigned)gx, (unsigned)gy), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t *>(w), N, K, ldw, q, ldq, scales, nullptr, 0, nullptr);
    return launch_status();
}

template <bool P2>
int quant_128x128_dual(const void *w, int64_t N, int64_t K, int64_t ldw, uint8_t *q, int64_t ldq, float *scales,
                       uint8_t *qT, int64_t ldqT, float *scalesT, void *stream)
{
    if (N < 0 || K < 0 || N % GROUP != 0 || K % GROUP != 0 || ldw < K || ldq < K || ldqT < N)
        return FP8FG_EINVAL;
    if (N == 0 || K == 0)
        return FP8FG_OK;
    if (!w || !q || !scales || !qT || !scalesT)
        return FP8FG_EINVAL;
    if (!aligned16(w) || !aligned16(q) || !aligned16(qT) || ldw % 8 != 0 || ldq % 16 != 0 || ldqT % 16 != 0 ||
        (reinterpret_cast<uintptr_t>(scales) & 3u) != 0 || (reinterpret_cast<uintptr_t>(scalesT) & 3u) != 0)
        return FP8FG_EALIGN;
    if (!device_supported())
        return FP8FG_EUNSUPPORTED;
    const int64_t gx = K / GROUP, gy = N / GROUP;
    if (gx > 0x7FFFFFFF || gy > 65535)
        return FP8FG_EINVAL;
    quant_blocks_kernel<P2, true><<<dim3((unsigned)gx, (unsigned)gy), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t *>(w), N, K, ldw, q, ldq, scales, qT, ldqT, scalesT);
    return launch_status();
}

}  // namespace
}  // namespace fp8fg

using namespace fp8fg;

extern "C" int fp8_quant_1x128(const void *x, int64_t rows, int64_t cols, int64_t ldx, uint8_t *q, int64_t ldq,
                               float *scales, int64_t ld_s, int transpose, void *stream)
{
    return quant_1x128<false>(x, rows, cols, ldx, q, ldq, scales, ld_s, transpose, stream);
}

extern "C" int fp8_quant_1x128_gather(const void *x, int64_t n_src, int64_t cols, int64_t ldx,
                                      const int32_t *row_index, int64_t rows, uint8_t *q, int64_t ldq, float *scales,
                                      int64_t ld_s, void *stream)
{
    return quant_1x128_gather<false>(x, n_src, cols, ldx, row_index, rows, q, ldq, scales, ld_s, stream);
}

extern "C" int fp8_quant_1x128_scatter(const void *x, int64_t n_src, int64_t cols, int64_t ldx,
                                       const int32_t *dest_index, int k, int64_t n_out, uint8_t *q, int64_t ldq,
                                       float *scales, int64_t ld_s, void *stream)
{
    return quant_1x128_scatter<false>(x, n_src, cols, ldx, dest_index, k, n_out, q, ldq, scales, ld_s, stream);
}

extern "C" int fp8_quant_1x128_scatter_pow2(const void *x, int64_t n_src, int64_t cols, int64_t ldx,
                                            const int32_t *dest_index, int k, int64_t n_out, uint8_t *q,
                                            int64_t ldq, float *scales, int64_t ld_s, void *stream)
{
    return quant_1x128_scatter<true>(x, n_src, cols, ldx, dest_index, k, n_out, q, ldq, scales, ld_s, stream);
}

extern "C" int fp8_quant_1x128_dual(const void *x, int64_t rows, int64_t cols, int64_t ldx, uint8_t *q,
                                    int64_t ldq, float *scales, int64_t ld_s, uint8_t *qT, int64_t ldqT,
                                    float *scalesT, int64_t ld_sT, void *stream)
{
    return quant_1x128_dual<false>(x, rows, cols, ldx, q, ldq, scales, ld_s, qT, ldqT, scalesT, ld_sT, stream);
}

extern "C" int fp8_quant_128x128(const void *w, int64_t N, int64_t K, int64_t ldw, uint8_t *q, int64_t ldq,
                                 float *scales, void *stream)
{
    return quant_128x128<false>(w, N, K, ldw, q, ldq, scales, stream);
}

extern "C" int fp8_quant_1x128_pow2(const void *x, int64_t rows, int64_t cols, int64_t ldx, uint8_t *q, int64_t ldq,
                                    float *scales, int64_t ld_s, int transpose, void *stream)
{
    return quant_1x128<true>(x, rows, cols, ldx, q, ldq, scales, ld_s, transpose, stream);
}

extern "C" int fp8_quant_1x128_gather_pow2(const void *x, int64_t n_src, int64_t cols, int64_t ldx,
                                           const int32_t *row_index, int64_t rows, uint8_t *q, int64_t ldq,
                                           float *scales, int64_t ld_s, void *stream)
{
    return quant_1x128_gather<true>(x, n_src, cols, ldx, row_index, rows, q, ldq, scales, ld_s, stream);
}

extern "C" int fp8_quant_1x128_dual_pow2(const void *x, int64_t rows, int64_t cols, int64_t ldx, uint8_t *q,
                                         int64_t ldq, float *scales, int64_t ld_s, uint8_t *qT, int64_t ldqT,
                                         float *scalesT, int64_t ld_sT, void *stream)
{
    return quant_1x128_dual<true>(x, rows, cols, ldx, q, ldq, scales, ld_s, qT, ldqT, scalesT, ld_sT, stream);
}

extern "C" int fp8_quant_128x128_pow2(const void *w, int64_t N, int64_t K, int64_t ldw, uint8_t *q, int64_t ldq,
                                      float *scales, void *stream)
{
    return quant_128x128<true>(w, N, K, ldw, q, ldq, scales, stream);
}

extern "C" int fp8_quant_128x128_dual(const void *w, int64_t N, int64_t K, int64_t ldw, uint8_t *q, int64_t ldq,
                                      float *scales, uint8_t *qT, int64_t ldqT, float *scalesT, void *stream)
{
    return quant_128x128_dual<false>(w, N, K, ldw, q, ldq, scales, qT, ldqT, scalesT, stream);
}

extern "C" int fp8_quant_128x128_dual_pow2(const void *w, int64_t N, int64_t K, int64_t ldw, uint8_t *q,
                                           int64_t ldq, float *scales, uint8_t *qT, int64_t ldqT, float *scalesT,
                                           void *stream)
{
    return quant_128x128_dual<true>(w, N, K, ldw, q, ldq, scales, qT, ldqT, scalesT, stream);
}
