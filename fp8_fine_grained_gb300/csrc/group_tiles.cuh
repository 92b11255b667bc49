// Tile space of a grouped (MoE expert) GEMM: the experts' row ranges from
// expert_offsets, each cut into BM-row tiles times the N tiles, laid out
// expert after expert with the m-tiles fastest inside an expert (CTAs
// running together then share the expert's weight tiles in L2). Shared by
// the grouped GEMM kernels.
#pragma once

#include <stdint.h>

#include "fp8fg.h"

namespace fp8fg {

struct GroupTile {
    int64_t m0;       // first output row of the tile
    int64_t row_end;  // one past the expert's last row
    int64_t n0;       // first output column
    int expert;
};

// Which experts a prefix counts: those with more than `small` rows
// (small = 0: every non-empty expert), or the non-empty ones with at most
// `small` rows.
enum GroupSet { ROWS_ABOVE = 0, ROWS_UP_TO = 1 };

// Block-wide exclusive prefix over experts of (m-tiles x n-tiles) into
// prefix[0..E] (prefix[E] = total tiles), counting only the experts of
// `which`; malformed offsets are reported as FP8FG_EDEVICE and clamped. All
// NT threads of the block call it; warp_sums is NT/32 ints of shared
// scratch (the kernels lend a region that is idle during their prologue, so
// they declare no static shared memory that would push their aligned
// dynamic region).
template <int NT>
__device__ void build_group_prefix(const int32_t *offsets, int E, int64_t n_rows, int64_t n_tiles_n, int bm,
                                   int *status, int32_t *prefix, int32_t *warp_sums, int64_t small = 0,
                                   GroupSet which = ROWS_ABOVE)
{
    const int per = (E + NT - 1) / NT;
    const int e0 = threadIdx.x * per;
    int32_t local[16];  // per <= 4096 / NT + 1
    int32_t sum = 0;
    for (int i = 0; i < per && i < 16; ++i) {
        const int e = e0 + i;
        int32_t v = 0;
        if (e < E) {
            int64_t r0 = offsets[e], r1 = offsets[e + 1];
            if (r0 < 0 || r1 < r0 || r1 > n_rows)
                atomicCAS(status, 0, FP8FG_EDEVICE);
            r0 = r0 < 0 ? 0 : (r0 > n_rows ? n_rows : r0);
            r1 = r1 > n_rows ? n_rows : r1;
            const int64_t m = r1 > r0 ? r1 - r0 : 0;
            if (which == ROWS_ABOVE ? m > small : m <= small)
                v = (int32_t)(((m + bm - 1) / bm) * n_tiles_n);
        }
        local[i] = v;
        sum += v;
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t x = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o)
            x += y;
    }
    if (lane == 31)
        warp_sums[warp] = x;
    __syncthreads();
    int32_t base = 0;
    for (int w = 0; w < warp; ++w)
        base += warp_sums[w];
    int32_t run = base + x - sum;  // exclusive prefix of this thread
    for (int i = 0; i < per && i < 16; ++i) {
        const int e = e0 + i;
        if (e < E)
            prefix[e] = run;
        run += local[i];
    }
    if (threadIdx.x == NT - 1)
        prefix[E] = run;  // the last thread's run ends at the total
    __syncthreads();
}

// Tile t of the grouped tile space (0 <= t < prefix[E]).
__device__ __forceinline__ GroupTile decode_group_tile(int64_t t, const int32_t *prefix, const int32_t *offsets,
                                                       int E, int64_t n_rows, int bm, int bn)
{
    int lo = 0, hi = E;  // last e with prefix[e] <= t
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid] <= t)
            lo = mid;
        else
            hi = mid;
    }
    const int e = lo;
    const int64_t local = t - prefix[e];
    int64_t r0 = offsets[e], r1 = offsets[e + 1];
    r0 = r0 < 0 ? 0 : (r0 > n_rows ? n_rows : r0);
    r1 = r1 > n_rows ? n_rows : r1;
    const int64_t mt = (r1 - r0 + bm - 1) / bm;
    GroupTile g;
    g.expert = e;
    g.m0 = r0 + (local % mt) * bm;
    g.row_end = r1;
    g.n0 = (local / mt) * bn;
    return g;
}

}  // namespace fp8fg
