// Block-scaled FP8 GEMM with promotion every 128 of the contraction
// dimension, on sm_103a tensor cores (tcgen05), for the forward, data-
// gradient and weight-gradient products and for MoE experts over a row
// index.
//
// Method (innerforce.co.kr, increased-precision accumulation paragraph;
// yunhecapital.com 2.2.3; tonho.wtf DeepSeek-V3 entry, "como funciona"):
// the tensor cores form the FP8 x FP8 product of one 128-wide contraction
// block; that partial sum is then moved off the tensor cores, multiplied by
// the block's two dequantisation scales and added to an FP32 accumulator.
//
// GB300 design (one CTA per SM, persistent over 128x256 output tiles):
//   warp 0      TMA producer: A tile 128x128 B and B tile 256x128 B per
//               contraction block into a 4-stage shared-memory ring
//               (128-byte swizzle), signalled on mbarriers. The block's
//               dequantisation scales travel in the same stage: the tile's
//               128 row scales (and, for the weight gradient, its 256 column
//               scales) by TMA, the two 128x128 weight-block scales by 4-byte
//               cp.async from the producer, so the promotion warps read them
//               from shared memory instead of waiting on L2 once per block.
//   warps 1..3  MMA issuers: warp 1 allocates all 512 tensor-memory
//               columns; per contraction block one of them (in turn) issues
//               4 x tcgen05.mma (M128 N256 K32, E4M3 -> FP32) into one of two
//               256-column TMEM partial buffers and commits to the buffer's
//               "full" barrier (the promotion warps free the stage once they
//               have seen that commit). Three issuers spread the issue cost
//               over three SMSPs. MoE rows gathered through a row index:
//               warp 1 issues every block and warps 2..3 gather the tile's
//               token rows and their scales into the stage with cp.async.
//   warps 4..11 promotion/epilogue: each thread owns one output row and 128
//               columns; per block it reads its scales from the stage, loads
//               the partial from TMEM (tcgen05.ld 32x32b, 16 columns per
//               load), releases the buffer once all 128 columns are in
//               registers, and does acc = fma(P, sA*sB, acc) in FP32
//               registers (paired FP32 FMAs), half before the release and
//               half after it, so the MMA of block kb+2 overlaps the end of
//               the promotion of block kb. After the last block it rounds
//               its rows and stores them through a shared-memory staging
//               block, 8 rows x 64 bytes per store.
// Every wait is bounded (global timer); a wait that runs out records
// FP8FG_ETIMEOUT in the device status word and all roles leave their loops,
// drain their own in-flight copies and MMAs, and release tensor memory.
#include <cuda_bf16.h>

#include "group_rule.cuh"
#include "group_tiles.cuh"
#include "host_common.h"
#include "ptx.cuh"
#include "tensor_map.h"

namespace fp8fg {
namespace {

constexpr int BM = 128;        // output rows per tile (TMEM lanes)
constexpr int BN = 256;        // output columns per tile
constexpr int BK = 128;        // contraction block = promotion interval = scale group
constexpr int STAGES = 4;
constexpr int EPI_WARPS = 8;
constexpr int EPI_WARP0 = 4;                  // promotion warps are warpgroups 1 and 2
constexpr int NUM_THREADS = (EPI_WARP0 + EPI_WARPS) * 32;
constexpr int CHUNK = 16;                     // TMEM columns per tcgen05.ld in the promotion loop
// Register split (setmaxnreg): warpgroup 0 (TMA, MMA and the gather or
// idle warps) gives registers to the two promotion warpgroups, which hold
// 128 FP32 sums per thread plus four 16-column partial chunks. The launch
// holds NUM_THREADS x (compiled register count) registers; the split must
// fit in it, which the host checks before every launch. (A 40/232 split for
// the contiguous MoE mode measured 0.5 % slower than this one.)
template <int MODE> struct Regs {
    static constexpr int LOW = 56;
    static constexpr int EPI = 224;
    static constexpr int LAUNCH_MIN = (4 * 32 * LOW + EPI_WARPS * 32 * EPI + NUM_THREADS - 1) / NUM_THREADS;
};
constexpr uint32_t A_STAGE_BYTES = BM * BK;   // 16 KB
constexpr uint32_t B_STAGE_BYTES = BN * BK;   // 32 KB
constexpr uint32_t TMEM_COLS = 512;           // two 256-column partial buffers
constexpr int MAX_EXPERTS = 4096;
constexpr int MMA_K = 32;                     // K per tcgen05.mma for 8-bit operands
constexpr int GATHER_WARPS = 2;               // grouped mode: warps 2..3 gather A rows
// Epilogue staging: a promotion warp passes its 32 rows through a 2 KB
// shared-memory block, 64 bytes of each row at a time, so that its global
// stores cover 8 rows x 64 contiguous bytes each instead of 32 rows x 16.
constexpr uint32_t STAGE_C_BYTES = 32 * 64;

// GROUPED: MoE experts, A rows gathered through a row index by warps 2..3.
// GROUPED_C: MoE experts, A rows already in expert order (TMA tiles). Two
// instantiations, so that neither carries the other's registers.
enum Mode { FPROP = 0, DGRAD = 1, WGRAD = 2, GROUPED = 3, GROUPED_C = 4 };
// Output element: FP32, bf16 (RNE), or E4M3 with 1x128 scales along N (the
// bf16 value of each element quantised by the group rule, i.e. what
// fp8_quant_1x128 of the bf16 output would write).
enum Out { OUT_F32 = 0, OUT_BF16 = 1, OUT_E4M3 = 2 };
constexpr bool is_grouped(int mode) { return mode == GROUPED || mode == GROUPED_C; }

struct Params {
    int64_t M, N, K;
    const uint8_t *A;  // grouped mode: token rows gathered by cp.async
    const float *sA;
    int64_t ld_sA;
    const float *sB;
    int64_t ld_sB;
    void *C;
    int64_t ldc;
    int64_t num_m_tiles, num_n_tiles;
    // tile order of the dense modes: bands of `band` m-tiles (m fastest)
    // or, with n_major, bands of `band` n-tiles (n fastest)
    int64_t band;
    int n_major;
    int *status;
    uint64_t wait_limit_ns;
    int skip_first_load;
    // grouped mode
    const int32_t *row_index;
    const int32_t *expert_offsets;
    int n_experts;
    int64_t n_rows;
    int64_t n_tokens;
    // E4M3 output: scales [N/128][ld_sC]
    float *sC;
    int64_t ld_sC;
    // experts with rows in expert order: experts with at most skinny_rows
    // rows take skinny tiles (0: none), and the SM time of a skinny tile
    // relative to a full one, in percent, divides the CTAs between the two
    int skinny_rows;
    int skinny_cost_pct;
};

// Scale slot of one pipeline stage: the A row scales of the block (a box of
// 132 FP32 from the 4-aligned row at or below the tile's first row, so that
// the TMA start coordinate is 16-byte aligned; the tile's rows begin at
// offset m0 % 4), then the B scales: the two 128x128 weight-block scales of
// the tile's column halves, or (weight gradient) the tile's 256 column scales.
// Gathered MoE rows receive their row scales by cp.async instead (128 FP32,
// one per tile row).
constexpr uint32_t SA_BOX = 132;
template <int MODE> struct ScaleSlot {
    static constexpr uint32_t a_bytes = MODE == GROUPED ? 4 * BM : 4 * SA_BOX;
    static constexpr uint32_t b_off = MODE == WGRAD ? 640 : a_bytes;              // TMA destination: 128-byte aligned
    static constexpr uint32_t b_bytes = MODE == WGRAD ? 4 * BN : 16;
    static constexpr uint32_t bytes = MODE == GROUPED ? b_off + b_bytes : (b_off + b_bytes + 127) / 128 * 128;
};

// Shared memory, from a 1024-byte aligned base (the 128-byte swizzle atoms of
// the operand stages need it): B stages, A stages, barriers, the promotion
// warps' epilogue staging blocks, the stages' scale slots and, for MoE
// experts, the tile's token rows and the experts' tile prefix.
template <int MODE> struct SmemLayout {
    // B stages first: every operand read stays well inside the allocation
    static constexpr uint32_t b_off = 0;
    static constexpr uint32_t a_off = b_off + STAGES * B_STAGE_BYTES;
    static constexpr uint32_t bar_off = a_off + STAGES * A_STAGE_BYTES;
    static constexpr uint32_t full_off = bar_off;
    static constexpr uint32_t empty_off = full_off + 8 * STAGES;
    static constexpr uint32_t tfull_off = empty_off + 8 * STAGES;
    static constexpr uint32_t tempty_off = tfull_off + 8 * 2;          // one per stage (block g: g % STAGES)
    static constexpr uint32_t tmem_ptr_off = tempty_off + 8 * STAGES;
    static constexpr uint32_t abort_off = tmem_ptr_off + 4;
    static constexpr uint32_t sched_off = (abort_off + 4 + 7) & ~7u;   // the CTA's tile schedule
    static constexpr uint32_t misc_end = sched_off + 16;
    // per promotion warp: epilogue staging block
    static constexpr uint32_t stage_c_off = (misc_end + 15) & ~15u;
    static constexpr uint32_t stage_c_end = stage_c_off + EPI_WARPS * STAGE_C_BYTES;
    static constexpr uint32_t scale_off = (stage_c_end + 127) & ~127u;
    static constexpr uint32_t scale_end = scale_off + STAGES * ScaleSlot<MODE>::bytes;
    static constexpr uint32_t tok_off = scale_end;                              // GROUPED: the tile's token rows
    static constexpr uint32_t tok_end = tok_off + (MODE == GROUPED ? 4 * BM : 0);
    static constexpr uint32_t prefix_off = tok_end;                             // grouped: tile prefix
    static constexpr uint32_t prefix_end = prefix_off + (is_grouped(MODE) ? 4 * (MAX_EXPERTS + 1) : 0);
    static constexpr uint32_t total = prefix_end;
};
static_assert(SmemLayout<FPROP>::total <= 232448, "shared memory budget");
static_assert(SmemLayout<WGRAD>::total <= 232448, "shared memory budget");
static_assert(SmemLayout<GROUPED>::total <= 232448, "shared memory budget");
static_assert(SmemLayout<GROUPED_C>::total <= 232448, "shared memory budget");

// Arrivals that complete a stage's "full" barrier: the producer's
// arrive.expect_tx; the completion of its 4-byte weight-scale copies
// (fprop, dgrad, experts with rows in expert order; the weight gradient's
// scales all come by TMA); or, for MoE rows gathered through a row index,
// the two gather warps (whose copies include the weight-block scales).
// Threads issuing MMAs: warps 1..3 take the blocks in turn, except for MoE
// rows gathered through a row index, where warps 2 and 3 gather A rows.
template <int MODE> constexpr int MMA_ISSUERS() { return MODE == GROUPED ? 1 : 3; }

template <int MODE> constexpr uint32_t full_arrivals()
{
    return MODE == GROUPED ? 1 + GATHER_WARPS : (MODE == WGRAD ? 1 : 2);
}

// A CTA's tiles: t = first, first + stride, ... below count. The roles read
// it from shared memory at each tile, so that no register holds it through
// the contraction loop.
struct Sched {
    int64_t count;
    int first, stride;
};

struct Tile {
    int64_t m0;       // first A row (dense) / first output row (grouped)
    int64_t row_end;  // one past the last valid output row of the tile's group
    int64_t n0;       // first output column
    int expert;
};

// Weight-block scale of column half h of tile tl for contraction block kb:
// sB is [N/128][ld_sB] (fprop), [K/128][ld_sB] (dgrad) or
// [E][N/128][K/128] (experts).
template <int MODE>
__device__ __forceinline__ const float *weight_scale(const Params &p, const Tile &tl, int kb, int h)
{
    const int64_t nb = tl.n0 / 128 + h;
    if constexpr (MODE == FPROP)
        return p.sB + nb * p.ld_sB + kb;
    else if constexpr (MODE == DGRAD)
        return p.sB + (int64_t)kb * p.ld_sB + nb;
    else
        return p.sB + ((int64_t)tl.expert * (p.N / 128) + nb) * (p.K / 128) + kb;
}

template <int MODE>
__device__ __forceinline__ Tile decode_tile(int64_t t, const Params &p, const int32_t *prefix)
{
    Tile tl;
    if constexpr (is_grouped(MODE)) {
        const GroupTile g = decode_group_tile(t, prefix, p.expert_offsets, p.n_experts, p.n_rows, BM, BN);
        tl.expert = g.expert;
        tl.m0 = g.m0;
        tl.row_end = g.row_end;
        tl.n0 = g.n0;
    } else {
        // Bands of p.band tiles along one dimension, that dimension fastest:
        // the band's panel of that operand stays in L2 while the other
        // operand streams past once per band (the host picks the side and
        // the band from the operand sizes).
        const int64_t nb = p.n_major ? p.num_n_tiles : p.num_m_tiles;   // tiles along the banded side
        const int64_t no = p.n_major ? p.num_m_tiles : p.num_n_tiles;   // tiles along the other side
        const int64_t per_band = p.band * no;
        const int64_t band = t / per_band, r = t % per_band;
        const int64_t first = band * p.band;
        const int64_t g = (nb - first) < p.band ? (nb - first) : p.band;
        const int64_t fast = first + r % g, slow = r / g;
        tl.m0 = (p.n_major ? slow : fast) * BM;
        tl.n0 = (p.n_major ? fast : slow) * BN;
        tl.row_end = p.M;
        tl.expert = 0;
    }
    return tl;
}

// ---------------------------------------------------------------- skinny ----
// Experts with at most SK_TOK rows (rows in expert order). A full tile of
// such an expert is 128 token rows of which at most 32 are real. A skinny
// tile turns the product around: the weight gives the MMA's 128-row side
// and the tokens its N = 32 side, so one tile is 256 weight rows (two MMAs
// of M = 128) x 32 tokens, and one pipeline stage carries 32 KB of weights
// and 4 KB of token codes; five stages fit where the full tiles have four.
// Both kinds of tile of a small expert stream its weights from DRAM once,
// and one CTA's stream runs at about 65 GB/s (measured on the MoE layer:
// about 29 us per skinny tile of 1.8 MB, 31 us per full tile of the same
// weights); prefetching the boxes into L2 ahead of the ring made both
// slower. The skinny CTAs run beside the full-tile CTAs, which are bound by
// their promotion chain instead.
//
// The sums are the same: for output (token t, column n), per contraction
// block kb the tensor cores give P = sum_k W[n,k] X[t,k] and the promotion
// adds P * (sX[t,kb] * sW[n/128,kb]) into an FP32 sum, with the scale
// product formed first, as in the full tiles. Roles: warp 0 loads (weights
// through the B map, tokens through a 32-row map, token scales through the
// row-scale map, the weight-block scales by cp.async), warp 1 issues, warps
// 4..11 promote (warp w: TMEM lane quarter w % 4 = 32 weight rows of MMA
// half (w - 4) / 4, one weight row and the 32 token columns per thread) and
// store Y[t, n] directly: a warp's 32 consecutive columns of one token row
// per store.
constexpr int SK_TOK = 32;                          // token columns of a skinny tile
constexpr uint32_t SK_X_BYTES = SK_TOK * BK;        // 4 KB of token codes per stage

// CTAs given to the skinny tiles: the grid's share of the estimated SM time
// (skinny tiles x cost_pct / 100 against full tiles x 1), at least one CTA
// when there are skinny tiles and one left for the full tiles when there
// are full tiles; never more CTAs than skinny tiles. Every CTA computes the
// same value from the same offsets.
__device__ __forceinline__ int skinny_cta_count(int64_t full_tiles, int64_t skinny_tiles, int grid, int cost_pct)
{
    if (skinny_tiles == 0)
        return 0;
    int64_t s;
    if (full_tiles == 0) {
        s = grid;
    } else {
        const int64_t ws = skinny_tiles * cost_pct, wf = full_tiles * 100;
        s = ((int64_t)grid * ws + (ws + wf) / 2) / (ws + wf);
        s = s < 1 ? 1 : (s > grid - 1 ? grid - 1 : s);
    }
    return (int)(s < skinny_tiles ? s : skinny_tiles);
}

// Shared memory of a skinny CTA, in the full tiles' allocation: five
// stages of 32 KB of weights (the four B stages and the first half of the A
// stages) and 4 KB of token codes (after those, in the A stages), and its
// barriers and scale slots in the region of the full tiles' epilogue
// staging blocks, which a skinny CTA does not use. Four TMEM partial
// buffers of 64 columns (two MMA halves of 32); a buffer's "read" barrier is
// its block's stage's, which needs no more buffers than stages (see the
// full tiles' "partial read" barriers).
struct SkLayout {
    using L = SmemLayout<GROUPED_C>;
    static constexpr int STAGES_ = 5;
    static constexpr int BUFS = 4;
    static constexpr uint32_t full_off = L::stage_c_off;
    static constexpr uint32_t empty_off = full_off + 8 * STAGES_;
    static constexpr uint32_t tfull_off = empty_off + 8 * STAGES_;
    static constexpr uint32_t tempty_off = tfull_off + 8 * BUFS;
    static constexpr uint32_t scale_off = (tempty_off + 8 * STAGES_ + 127) & ~127u;
    static constexpr uint32_t scale_end = scale_off + STAGES_ * ScaleSlot<GROUPED_C>::bytes;
    static constexpr uint32_t x_off = L::a_off + B_STAGE_BYTES;
    __device__ static constexpr uint32_t w(int s) { return s < STAGES ? L::b_off + s * B_STAGE_BYTES : L::a_off; }
    __device__ static constexpr uint32_t x(int s) { return x_off + s * SK_X_BYTES; }
};
static_assert(SkLayout::STAGES_ == STAGES + 1, "one weight stage in the A stages");
static_assert(SkLayout::scale_end <= SmemLayout<GROUPED_C>::stage_c_end, "skinny barriers and scale slots");
static_assert(SkLayout::x_off + SkLayout::STAGES_ * SK_X_BYTES <= SmemLayout<GROUPED_C>::a_off + STAGES * A_STAGE_BYTES,
              "skinny token stages");
static_assert(SkLayout::BUFS <= SkLayout::STAGES_ && SkLayout::BUFS * 2 * SK_TOK <= (int)TMEM_COLS, "skinny buffers");

__device__ __forceinline__ void skinny_init_barriers(uint32_t sbase)
{
    for (int s = 0; s < SkLayout::STAGES_; ++s) {
        mbar_init(sbase + SkLayout::full_off + 8 * s, full_arrivals<GROUPED_C>());
        mbar_init(sbase + SkLayout::empty_off + 8 * s, EPI_WARPS);
        mbar_init(sbase + SkLayout::tempty_off + 8 * s, EPI_WARPS);
    }
    for (int b = 0; b < SkLayout::BUFS; ++b)
        mbar_init(sbase + SkLayout::tfull_off + 8 * b, 1);
    fence_mbar_init();
}

template <int OUT>
__device__ __forceinline__ void skinny_roles(const CUtensorMap *tmX, const CUtensorMap *tmW, const CUtensorMap *tmSA,
                                             const Params &p, uint8_t *smem, const int32_t *prefix,
                                             volatile const Sched *sched, uint32_t tmem_base, const WaitCtl &wc,
                                             int warp, int lane)
{
    using SK = SkLayout;
    using SS = ScaleSlot<GROUPED_C>;
    constexpr int NS = SK::STAGES_, NB = SK::BUFS;
    const uint32_t sbase = smem_u32(smem);
    const uint32_t full_bar = sbase + SK::full_off;
    const uint32_t empty_bar = sbase + SK::empty_off;
    const uint32_t tfull_bar = sbase + SK::tfull_off;
    const uint32_t tempty_bar = sbase + SK::tempty_off;
    const uint32_t scale_base = sbase + SK::scale_off;
    const int num_kb = (int)(p.K / BK);

    if (warp == 0) {
        // ------------------------------------------------------ producer ----
        uint32_t stage = 0, phase = 0;
        uint32_t filled_mask = 0, fill_parity = 0;
        bool ok = true;
        for (int64_t t = sched->first; t < sched->count && ok; t += sched->stride) {
            const Tile tl = decode_tile<GROUPED_C>(t, p, prefix);
            for (int kb = 0; kb < num_kb; ++kb) {
                bool got = true;
                if (lane == 0)
                    got = mbar_wait(empty_bar + 8 * stage, phase ^ 1, wc, FP8FG_ETIMEOUT);
                got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
                if (!got) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    const uint32_t fb = full_bar + 8 * stage;
                    const uint32_t sc_dst = scale_base + stage * SS::bytes;
                    mbar_arrive_expect_tx(fb, B_STAGE_BYTES + SK_X_BYTES + 4 * SA_BOX);
                    filled_mask |= 1u << stage;
                    fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
                    tma_load_2d(sc_dst, tmSA, (int32_t)(tl.m0 & ~int64_t(3)), kb, fb);
                    cp_async4(sc_dst + SS::b_off, weight_scale<GROUPED_C>(p, tl, kb, 0));
                    if (tl.n0 + 128 < p.N)
                        cp_async4(sc_dst + SS::b_off + 4, weight_scale<GROUPED_C>(p, tl, kb, 1));
                    cp_async_mbar_arrive_noinc(fb);
                    tma_load_2d(sbase + SK::x(stage), tmX, kb * BK, (int32_t)tl.m0, fb);
                    tma_load_2d(sbase + SK::w(stage), tmW, kb * BK, (int32_t)(tl.expert * p.N + tl.n0), fb);
                }
                __syncwarp();
                if (++stage == NS) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        if (!ok && lane == 0) {
            for (int s = 0; s < NS; ++s) {
                if (!(filled_mask & (1u << s)))
                    continue;
                const uint32_t bar = full_bar + 8 * s, par = (fill_parity >> s) & 1u;
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(bar, par) && global_timer_ns() - t0 < wc.limit_ns) {
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA ----
        constexpr uint32_t IDESC = idesc_e4m3_f32(BM, SK_TOK, false);
        int committed = 0;
        uint32_t last_buf = 0, last_par = 0;
        bool ok = true;
        int64_t g = 0;
        uint32_t stage = 0, phase = 0, buf = 0, tphase = 0;
        for (int64_t t = sched->first; t < sched->count && ok; t += sched->stride) {
            for (int kb = 0; kb < num_kb; ++kb, ++g) {
                // buffer `buf` is free once block g - NB has been read out
                if (g >= NB) {
                    const int64_t h = g - NB;
                    const bool got = mbar_wait(tempty_bar + 8 * (uint32_t)(h % NS), (uint32_t)((h / NS) & 1), wc,
                                               FP8FG_ETIMEOUT);
                    if (!__all_sync(0xffffffffu, got)) {
                        ok = false;
                        break;
                    }
                }
                tc_fence_after();
                const bool got = mbar_wait(full_bar + 8 * stage, phase, wc, FP8FG_ETIMEOUT);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t w_addr = sbase + SK::w(stage);
                const uint32_t x_addr = sbase + SK::x(stage);
                if (elect_one_sync()) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
#pragma unroll
                        for (int k = 0; k < BK / MMA_K; ++k) {
                            // both operands K-major with 128-byte rows; the
                            // weight half h is 128 rows = 16 KB further on
                            const uint64_t adesc = smem_desc_sw128(w_addr + h * (BM * BK) + k * MMA_K, 0, 1024);
                            const uint64_t bdesc = smem_desc_sw128(x_addr + k * MMA_K, 0, 1024);
                            mma_f8f6f4(tmem_base + buf * (2 * SK_TOK) + h * SK_TOK, adesc, bdesc, IDESC,
                                       k > 0 ? 1u : 0u);
                        }
                    }
                    mma_commit(tfull_bar + 8 * buf);
                }
                __syncwarp();
                committed = 1;
                last_buf = buf;
                last_par = tphase;
                if (++stage == NS) {
                    stage = 0;
                    phase ^= 1;
                }
                if (++buf == NB) {
                    buf = 0;
                    tphase ^= 1;
                }
            }
        }
        if (!ok && committed && lane == 0) {
            const uint32_t bar = tfull_bar + 8 * last_buf;
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(bar, last_par) && global_timer_ns() - t0 < wc.limit_ns) {
            }
        }
        __syncwarp();
    } else if (warp >= EPI_WARP0) {
        // ------------------------------------------------- promotion ----
        const int quarter = warp & 3;
        const int half = (warp - EPI_WARP0) >> 2;
        uint32_t buf = 0, tphase = 0, stage = 0, phase = 0;
        bool ok = true;
        for (int64_t t = sched->first; t < sched->count && ok; t += sched->stride) {
            const Tile tl = decode_tile<GROUPED_C>(t, p, prefix);
            const int64_t n = tl.n0 + half * 128 + quarter * 32 + lane;  // this thread's weight row = output column
            const bool half_ok = tl.n0 + half * 128 < p.N;
            const int64_t left = tl.row_end - tl.m0;
            const int nrows = left < SK_TOK ? (int)left : SK_TOK;
            const uint32_t x0 = 4 * (uint32_t)(tl.m0 & 3);               // first token scale in the slot
            float2 acc[SK_TOK / 2];
#pragma unroll
            for (int j = 0; j < SK_TOK / 2; ++j)
                acc[j] = make_float2(0.0f, 0.0f);
            for (int kb = 0; kb < num_kb; ++kb) {
                bool got = mbar_wait(full_bar + 8 * stage, phase, wc, FP8FG_ETIMEOUT);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                const uint8_t *slot = smem + SK::scale_off + stage * SS::bytes;
                const float sw = reinterpret_cast<const float *>(slot + SS::b_off)[half];
                const float *sx = reinterpret_cast<const float *>(slot + x0);
                float2 sc[SK_TOK / 2];
#pragma unroll
                for (int j = 0; j < SK_TOK / 2; ++j)
                    sc[j] = make_float2(__fmul_rn(sx[2 * j], sw), __fmul_rn(sx[2 * j + 1], sw));
                got = mbar_wait(tfull_bar + 8 * buf, tphase, wc, FP8FG_ETIMEOUT);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                // the block's MMAs are complete and its scales read
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(empty_bar + 8 * stage);
                tc_fence_after();
                uint32_t r[SK_TOK];
                tmem_ld_chunk(tmem_base + ((uint32_t)(quarter * 32) << 16) + buf * (2 * SK_TOK) + half * SK_TOK, r);
                tmem_wait_ld_chunk(r);
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(tempty_bar + 8 * stage);
#pragma unroll
                for (int j = 0; j < SK_TOK / 2; ++j)
                    acc[j] = __ffma2_rn(make_float2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1])), sc[j],
                                        acc[j]);
                if (++buf == NB) {
                    buf = 0;
                    tphase ^= 1;
                }
                if (++stage == NS) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (!ok || !half_ok)
                continue;
#pragma unroll
            for (int j = 0; j < SK_TOK; ++j) {
                if (j < nrows) {
                    const float v = (j & 1) ? acc[j >> 1].y : acc[j >> 1].x;
                    const int64_t at = (tl.m0 + j) * p.ldc + n;
                    if constexpr (OUT == OUT_BF16)
                        static_cast<__nv_bfloat16 *>(p.C)[at] = __float2bfloat16_rn(v);
                    else
                        static_cast<float *>(p.C)[at] = v;
                }
            }
        }
    }
}

template <int MODE, int OUT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB, const Params p)
{
    using L = SmemLayout<MODE>;
    using SS = ScaleSlot<MODE>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw;
    // the layout assumes the 1024-byte alignment requested above; refuse to
    // run (before any barrier or tensor memory is set up) if it is missing
    if (smem_u32(smem) & 1023u) {
        if (threadIdx.x == 0)
            atomicCAS(p.status, 0, FP8FG_EUNSUPPORTED);
        return;
    }
    const uint32_t sbase = smem_u32(smem);
    const uint32_t full_bar = sbase + L::full_off;
    const uint32_t empty_bar = sbase + L::empty_off;
    const uint32_t tfull_bar = sbase + L::tfull_off;
    const uint32_t tempty_bar = sbase + L::tempty_off;
    volatile uint32_t *tmem_ptr = reinterpret_cast<volatile uint32_t *>(smem + L::tmem_ptr_off);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::abort_off);
    int32_t *prefix = reinterpret_cast<int32_t *>(smem + L::prefix_off);
    const uint32_t scale_base = sbase + L::scale_off;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const WaitCtl wc{abort_flag, p.status, p.wait_limit_ns};
    // GROUPED: A rows gathered through row_index by warps 2..3; GROUPED_C:
    // A rows already in expert order, loaded by TMA like the dense modes
    constexpr bool gathered = MODE == GROUPED;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar + 8 * s, full_arrivals<MODE>());
            // freed by the promotion warps: each arrives once it has read
            // the stage's scales and seen the block's MMAs complete (which
            // covers the tensor cores' reads of the stage), so the MMA
            // issuer needs no commit of its own for the stage
            mbar_init(empty_bar + 8 * s, EPI_WARPS);
        }
        for (int b = 0; b < 2; ++b)
            mbar_init(tfull_bar + 8 * b, 1);
        // "partial read" barriers, one per stage rather than per TMEM buffer:
        // an issuer may be a few blocks ahead of the others, and with one
        // barrier per buffer it could test a phase two behind the one it
        // needs, which a parity wait cannot tell apart
        for (int s = 0; s < STAGES; ++s)
            mbar_init(tempty_bar + 8 * s, EPI_WARPS);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        if constexpr (!gathered)
            tma_prefetch_desc(&tmSA);
        if constexpr (MODE == WGRAD || MODE == GROUPED_C)
            tma_prefetch_desc(&tmSB);
    }
    if (warp == 1) {
        tmem_alloc(sbase + L::tmem_ptr_off, TMEM_COLS);
        tmem_relinquish();
    }
    // Everything above touches only this CTA's shared and tensor memory;
    // inputs written by the previous kernel in the stream (for example the
    // quantiser, which lets this grid launch under its last wave) are read
    // only after this wait.
    griddep_wait();
    // This CTA's tiles: t = cta, cta + ncta, ... below num_tiles. With
    // skinny tiles the first `s` CTAs take the skinny experts and the rest
    // the others (every CTA derives the same split from the offsets).
    int64_t num_tiles = p.num_m_tiles * p.num_n_tiles;
    int cta = (int)blockIdx.x, ncta = (int)gridDim.x;
    bool skinny = false;
    if constexpr (is_grouped(MODE)) {
        int32_t *scan = reinterpret_cast<int32_t *>(smem + L::stage_c_off);
        if (MODE == GROUPED_C && p.skinny_rows > 0) {
            build_group_prefix<NUM_THREADS>(p.expert_offsets, p.n_experts, p.n_rows, p.num_n_tiles, BM, p.status,
                                            prefix, scan, p.skinny_rows, ROWS_UP_TO);
            const int64_t skinny_tiles = prefix[p.n_experts];
            build_group_prefix<NUM_THREADS>(p.expert_offsets, p.n_experts, p.n_rows, p.num_n_tiles, BM, p.status,
                                            prefix, scan, p.skinny_rows, ROWS_ABOVE);
            const int64_t full_tiles = prefix[p.n_experts];
            const int s = skinny_cta_count(full_tiles, skinny_tiles, (int)gridDim.x, p.skinny_cost_pct);
            if ((int)blockIdx.x < s) {
                skinny = true;
                ncta = s;
                num_tiles = skinny_tiles;
                build_group_prefix<NUM_THREADS>(p.expert_offsets, p.n_experts, p.n_rows, p.num_n_tiles, BM,
                                                p.status, prefix, scan, p.skinny_rows, ROWS_UP_TO);
                // (after the last pass has read its scratch, which these
                // barriers overwrite)
                if (threadIdx.x == 0)
                    skinny_init_barriers(sbase);
            } else {
                cta = (int)blockIdx.x - s;
                ncta = (int)gridDim.x - s;
                num_tiles = full_tiles;
            }
        } else {
            build_group_prefix<NUM_THREADS>(p.expert_offsets, p.n_experts, p.n_rows, p.num_n_tiles, BM, p.status,
                                            prefix, scan);
            num_tiles = prefix[p.n_experts];
        }
    }
    volatile Sched *sched = reinterpret_cast<volatile Sched *>(smem + L::sched_off);
    if (threadIdx.x == 0) {
        sched->count = num_tiles;
        sched->first = cta;
        sched->stride = ncta;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_ptr;
    const int num_kb = (int)(p.K / BK);

    if (MODE == GROUPED_C && skinny) {
        if constexpr (MODE == GROUPED_C)
            skinny_roles<OUT>(&tmSB, &tmB, &tmSA, p, smem, prefix, sched, tmem_base, wc, warp, lane);
    } else if (warp == 0) {
        // ------------------------------------------------------ producer ----
        setmaxnreg_dec<Regs<MODE>::LOW>();
        uint32_t stage = 0, phase = 0;
        uint32_t filled_mask = 0, fill_parity = 0;  // per stage: a fill was issued, and its parity
        bool skip = p.skip_first_load && blockIdx.x == 0;
        bool ok = true;
        for (int64_t t = sched->first; t < sched->count && ok; t += sched->stride) {
            const Tile tl = decode_tile<MODE>(t, p, prefix);
            for (int kb = 0; kb < num_kb; ++kb) {
                bool got = true;
                if (lane == 0)
                    got = mbar_wait(empty_bar + 8 * stage, phase ^ 1, wc, FP8FG_ETIMEOUT);
                got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
                if (!got) {
                    ok = false;
                    break;
                }
                const uint32_t fb = full_bar + 8 * stage;
                const uint32_t a_dst = sbase + L::a_off + stage * A_STAGE_BYTES;
                const uint32_t b_dst = sbase + L::b_off + stage * B_STAGE_BYTES;
                const uint32_t sc_dst = scale_base + stage * SS::bytes;
                if (skip) {
                    skip = false;  // withhold this load: consumers must time out
                } else {
                    // gathered rows (and their scales) arrive through the
                    // gather warps, not TMA
                    uint32_t bytes = (gathered ? 0 : A_STAGE_BYTES + 4 * SA_BOX) + B_STAGE_BYTES;
                    if constexpr (MODE == WGRAD)
                        bytes += 4 * BN;
                    bool second_half = true;
                    if constexpr (MODE == DGRAD) {
                        second_half = tl.n0 + 128 < p.N;
                        if (!second_half)
                            bytes -= B_STAGE_BYTES / 2;
                    }
                    if (lane == 0) {
                        mbar_arrive_expect_tx(fb, bytes);
                        filled_mask |= 1u << stage;
                        fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
                        if constexpr (!gathered)
                            // the block's row scales: 132 from the 4-aligned row
                            tma_load_2d(sc_dst, &tmSA, (int32_t)(tl.m0 & ~int64_t(3)), kb, fb);
                        if constexpr (MODE == WGRAD) {
                            tma_load_2d(sc_dst + SS::b_off, &tmSB, (int32_t)tl.n0, kb, fb);
                        } else if constexpr (!gathered) {
                            // the weight-block scales of the tile's two column
                            // halves (4-byte copies: one FP32 per block and half)
                            cp_async4(sc_dst + SS::b_off, weight_scale<MODE>(p, tl, kb, 0));
                            if (tl.n0 + 128 < p.N)
                                cp_async4(sc_dst + SS::b_off + 4, weight_scale<MODE>(p, tl, kb, 1));
                            cp_async_mbar_arrive_noinc(fb);
                        }
                    }
                    __syncwarp();
                    if constexpr (is_grouped(MODE)) {
                        if (lane == 0) {
                            if (!gathered)
                                tma_load_2d(a_dst, &tmA, kb * BK, (int32_t)tl.m0, fb);
                            tma_load_2d(b_dst, &tmB, kb * BK, (int32_t)(tl.expert * p.N + tl.n0), fb);
                        }
                    } else if (lane == 0) {
                        tma_load_2d(a_dst, &tmA, kb * BK, (int32_t)tl.m0, fb);
                        if constexpr (MODE == DGRAD) {
                            // B is the weight [K][N] read N-contiguous: two
                            // 128(K) x 128(N) boxes, one per 128-column half.
                            tma_load_2d(b_dst, &tmB, (int32_t)tl.n0, kb * BK, fb);
                            if (second_half)
                                tma_load_2d(b_dst + B_STAGE_BYTES / 2, &tmB, (int32_t)tl.n0 + 128, kb * BK, fb);
                        } else {
                            tma_load_2d(b_dst, &tmB, kb * BK, (int32_t)tl.n0, fb);
                        }
                    }
                }
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
        // the weight-scale copies of the last stages land before the CTA exits
        asm volatile("cp.async.wait_all;" ::: "memory");
        if (!ok && lane == 0) {
            // drain: every issued fill must land before the CTA exits
            WaitCtl drain{abort_flag, p.status, p.wait_limit_ns};
            for (int s = 0; s < STAGES; ++s) {
                if (!(filled_mask & (1u << s)))
                    continue;
                const uint32_t bar = full_bar + 8 * s, par = (fill_parity >> s) & 1u;
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(bar, par) && global_timer_ns() - t0 < drain.limit_ns) {
                }
            }
        }
    } else if (warp >= 1 && warp <= MMA_ISSUERS<MODE>()) {
        // ---------------------------------------------------------- MMA ----
        // Issuing a block's four MMAs and its commit keeps the issuing
        // warp's SMSP busy for about 400 cycles, time the promotion warps on
        // that SMSP (bound to its TMEM lane quarter) lose. The blocks are
        // dealt round-robin to three issuers on three SMSPs (warps 1, 2, 3):
        // MMAs of different blocks are independent (each block starts with
        // accumulate off), and each issuer's commits track its own MMAs.
        setmaxnreg_dec<Regs<MODE>::LOW>();
        // The whole warp runs the loop and waits (so that the descriptors
        // are warp-uniform values); one elected lane issues the MMAs and
        // the commit.
        {
            constexpr uint32_t IDESC = idesc_e4m3_f32(BM, BN, MODE == DGRAD);
            constexpr int NI = MMA_ISSUERS<MODE>();
            const int issuer = warp - 1;
            int committed = 0;
            uint32_t last_buf = 0, last_par = 0;
            bool ok = true;
            int64_t g = 0;  // the CTA's block counter (tile-major)
            for (int64_t t = sched->first; t < sched->count && ok; t += sched->stride) {
                for (int kb = 0; kb < num_kb; ++kb, ++g) {
                    if ((int)(g % NI) != issuer)
                        continue;
                    const uint32_t stage = (uint32_t)(g % STAGES), phase = (uint32_t)((g / STAGES) & 1);
                    const uint32_t buf = (uint32_t)(g & 1), tphase = (uint32_t)((g >> 1) & 1);
                    // the buffer is free once block g-2's partial has been
                    // read out (its barrier: stage (g-2) % STAGES, that
                    // block's phase); the first two blocks find it free
                    if (g >= 2) {
                        const int64_t h = g - 2;
                        const bool got = mbar_wait(tempty_bar + 8 * (uint32_t)(h % STAGES),
                                                   (uint32_t)((h / STAGES) & 1), wc, FP8FG_ETIMEOUT);
                        if (!__all_sync(0xffffffffu, got)) {
                            ok = false;
                            break;
                        }
                    }
                    tc_fence_after();
                    const bool got = mbar_wait(full_bar + 8 * stage, phase, wc, FP8FG_ETIMEOUT);
                    if (!__all_sync(0xffffffffu, got)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = sbase + L::a_off + stage * A_STAGE_BYTES;
                    const uint32_t b_addr = sbase + L::b_off + stage * B_STAGE_BYTES;
                    const uint32_t d = tmem_base + buf * BN;
                    if (elect_one_sync()) {
#pragma unroll
                        for (int k = 0; k < BK / MMA_K; ++k) {
                            // K-major, 128-byte rows: step K by 32 bytes inside the swizzle atom
                            const uint64_t adesc = smem_desc_sw128(a_addr + k * MMA_K, 0, 1024);
                            uint64_t bdesc;
                            if constexpr (MODE == DGRAD)
                                // N-major: 32 K-rows = 4 groups of 8 rows (1024 B each);
                                // the two 128-column halves are 16 KB apart.
                                bdesc = smem_desc_sw128(b_addr + k * MMA_K * 128, B_STAGE_BYTES / 2, 1024);
                            else
                                bdesc = smem_desc_sw128(b_addr + k * MMA_K, 0, 1024);
                            mma_f8f6f4(d, adesc, bdesc, IDESC, k > 0 ? 1u : 0u);
                        }
                        mma_commit(tfull_bar + 8 * buf);
                    }
                    __syncwarp();
                    committed = 1;
                    last_buf = buf;
                    last_par = tphase;
                }
            }
            if (!ok && committed && lane == 0) {
                // drain: the last commit covers every MMA this warp issued before it
                const uint32_t bar = tfull_bar + 8 * last_buf;
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(bar, last_par) && global_timer_ns() - t0 < p.wait_limit_ns) {
                }
            }
        }
        __syncwarp();
    } else if (warp >= EPI_WARP0) {
        // ------------------------------------------ promotion / epilogue ----
        setmaxnreg_inc<Regs<MODE>::EPI>();
        const int ew = warp - EPI_WARP0;
        const int quarter = warp & 3;        // TMEM lanes 32*quarter .. +31
        const int half = ew >> 2;            // output columns half*128 .. +127 of the tile
        const int row_in_tile = quarter * 32 + lane;
        // weight gradient: the block's 128 column scales of this warp's half,
        // in the first 512 bytes of its epilogue staging block (idle until
        // the tile's last block has been folded)
        float *wscale = reinterpret_cast<float *>(smem + L::stage_c_off + ew * STAGE_C_BYTES);
        uint32_t buf = 0, tphase = 0;        // TMEM partial buffer
        uint32_t stage = 0, phase = 0;       // pipeline stage holding the block's scales
        bool ok = true;
        for (int64_t t = sched->first; t < sched->count && ok; t += sched->stride) {
            const Tile tl = decode_tile<MODE>(t, p, prefix);
            const int64_t row = tl.m0 + row_in_tile;  // A row (dense) / output row (grouped)
            const bool row_ok = row < tl.row_end;
            const int64_t col0 = tl.n0 + half * 128;
            const bool cols_ok = col0 < p.N;
            // this thread's row scale inside a stage's slot (TMA boxes start
            // at the 4-aligned row at or below the tile's first row)
            const uint32_t sa_off = 4 * (uint32_t)((gathered ? 0 : (tl.m0 & 3)) + row_in_tile);

            // running FP32 sums of this thread's row, 128 columns as 64 pairs
            float2 acc[64];
#pragma unroll
            for (int j = 0; j < 64; ++j)
                acc[j] = make_float2(0.0f, 0.0f);

            for (int kb = 0; kb < num_kb; ++kb) {
                // the stage's scales landed before its MMA was issued, so
                // this wait only orders the reads after the copies
                const uint8_t *slot = smem + L::scale_off + stage * SS::bytes;
                bool got = mbar_wait(full_bar + 8 * stage, phase, wc, FP8FG_ETIMEOUT);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                float sa = *reinterpret_cast<const float *>(slot + sa_off);
                if (gathered && !row_ok)
                    sa = 0.0f;  // gathered slots of rows past the expert's end are not written
                // B scales: the weight-block scale of this half, or (weight
                // gradient) the half's 128 column scales, copied to the
                // warp's own shared block for the fold
                const float *bslot = reinterpret_cast<const float *>(slot + SS::b_off);
                const float sb = MODE == WGRAD ? 0.0f : bslot[half];
                if constexpr (MODE == WGRAD)
                    reinterpret_cast<float4 *>(wscale)[lane] = reinterpret_cast<const float4 *>(bslot + half * 128)[lane];
                got = mbar_wait(tfull_bar + 8 * buf, tphase, wc, FP8FG_ETIMEOUT);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                // the block's MMAs are complete and its scales read (the
                // weight gradient's column scales copied): the stage may be
                // refilled
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(empty_bar + 8 * stage);
                tc_fence_after();
                const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + buf * BN + half * 128;
                const float sab = sa * sb;
                const float2 s2 = make_float2(sab, sab);
                const float2 sa2 = make_float2(sa, sa);
                // fold one 16-column chunk c (held in r) into the sums
                auto fold = [&](int c, const uint32_t(&r)[CHUNK]) {
#pragma unroll
                    for (int j = 0; j < CHUNK / 2; ++j) {
                        const float2 pv = make_float2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
                        const int a = c * (CHUNK / 2) + j;
                        if constexpr (MODE == WGRAD) {
                            const float2 sc = reinterpret_cast<const float2 *>(wscale)[a];
                            acc[a] = __ffma2_rn(pv, __fmul2_rn(sa2, sc), acc[a]);
                        } else {
                            acc[a] = __ffma2_rn(pv, s2, acc[a]);
                        }
                    }
                };
                // The partial buffer is released as soon as all of its
                // columns sit in registers: chunks 0..3 are loaded, then
                // each is folded in while the load of chunk 4..7 takes its
                // registers; once those four loads land the buffer goes back
                // to the MMA and chunks 4..7 are folded after the release,
                // off the MMA's critical path.
                constexpr int HELD = 4;  // chunks in registers at a time
                static_assert(HELD * 2 * CHUNK == 128, "two rounds of HELD chunks cover the half");
                uint32_t r[HELD][CHUNK];
#pragma unroll
                for (int c = 0; c < HELD; ++c)
                    tmem_ld_chunk(taddr + c * CHUNK, r[c]);
#pragma unroll
                for (int c = 0; c < HELD; ++c)
                    tmem_wait_ld_chunk(r[c]);  // one wait; each call ties its registers to it
#pragma unroll
                for (int c = 0; c < HELD; ++c) {
                    fold(c, r[c]);
                    tmem_ld_chunk(taddr + (HELD + c) * CHUNK, r[c]);
                }
#pragma unroll
                for (int c = 0; c < HELD; ++c)
                    tmem_wait_ld_chunk(r[c]);
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(tempty_bar + 8 * stage);
#pragma unroll
                for (int c = 0; c < HELD; ++c)
                    fold(HELD + c, r[c]);
                if constexpr (MODE == WGRAD)
                    __syncwarp();  // the column scales are read before the next block overwrites them
                if (++buf == 2) {
                    buf = 0;
                    tphase ^= 1;
                }
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (!ok)
                break;
            if (!cols_ok)
                continue;
            // Round and store the warp's 32 rows x 128 columns, 64 bytes of
            // each row per pass: each lane writes its row's piece into the
            // staging block (16-byte piece c of row r at c ^ ((r / 2) % 4),
            // conflict-free), then the warp reads it back 8 rows x 64 bytes
            // per instruction and stores those runs. Rows past the tile's
            // group (the next expert, or past M) are skipped.
            float qinv = 1.0f;
            if constexpr (OUT == OUT_E4M3) {
                // round to bf16 in place (the values a bf16 store keeps), then
                // the group rule over this thread's 128 columns: one 1x128
                // group of its row
                float amax = 0.0f;
#pragma unroll
                for (int a = 0; a < 64; ++a) {
                    acc[a] = __bfloat1622float2(__float22bfloat162_rn(acc[a]));
                    amax = fmaxf(amax, fmaxf(fabsf(acc[a].x), fabsf(acc[a].y)));
                }
                const ScalePair sp = group_scale(amax);
                qinv = sp.inv;
                if (row_ok)
                    p.sC[(col0 / 128) * p.ld_sC + row] = sp.s;
            }
            {
                constexpr int CW = OUT == OUT_BF16 ? 32 : (OUT == OUT_F32 ? 16 : 64);  // columns per 64-byte piece
                constexpr int ESZ = OUT == OUT_BF16 ? 2 : (OUT == OUT_F32 ? 4 : 1);
                uint8_t *const stg = smem + L::stage_c_off + ew * STAGE_C_BYTES;
                // write side: this lane's row, pieces swizzled by (lane / 2) % 4
                uint8_t *const w_row = stg + lane * 64;
                const int w_sw = (lane >> 1) & 3;
                // read side: row 8i + lane / 4, piece lane % 4 (the swizzle
                // term of those rows does not depend on i)
                const int cc = lane & 3;
                const uint8_t *const r_ptr = stg + (lane >> 2) * 64 + ((cc ^ ((lane >> 3) & 3)) << 4);
                const int rrow0 = row - lane + (lane >> 2);  // output row read back at i = 0
                uint8_t *const out0 =
                    static_cast<uint8_t *>(p.C) + ((int64_t)rrow0 * p.ldc + col0) * ESZ + cc * 16;
                const int64_t row8 = 8 * p.ldc * ESZ;        // bytes between the rows of i and i + 1
#pragma unroll
                for (int q = 0; q < 128 / CW; ++q) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint4 o;
                        if constexpr (OUT == OUT_E4M3) {
                            const int a = q * 32 + c * 8;
                            uint32_t w[4];
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                w[k] = cvt_e4m3x2(__fmul_rn(acc[a + 2 * k].x, qinv), __fmul_rn(acc[a + 2 * k].y, qinv)) |
                                       (cvt_e4m3x2(__fmul_rn(acc[a + 2 * k + 1].x, qinv),
                                                   __fmul_rn(acc[a + 2 * k + 1].y, qinv))
                                        << 16);
                            o = make_uint4(w[0], w[1], w[2], w[3]);
                        } else if constexpr (OUT == OUT_BF16) {
                            const int a = q * 16 + c * 4;
                            __nv_bfloat162 h0 = __float22bfloat162_rn(acc[a + 0]);
                            __nv_bfloat162 h1 = __float22bfloat162_rn(acc[a + 1]);
                            __nv_bfloat162 h2 = __float22bfloat162_rn(acc[a + 2]);
                            __nv_bfloat162 h3 = __float22bfloat162_rn(acc[a + 3]);
                            o.x = *reinterpret_cast<uint32_t *>(&h0);
                            o.y = *reinterpret_cast<uint32_t *>(&h1);
                            o.z = *reinterpret_cast<uint32_t *>(&h2);
                            o.w = *reinterpret_cast<uint32_t *>(&h3);
                        } else {
                            const int a = q * 8 + c * 2;
                            o = make_uint4(__float_as_uint(acc[a].x), __float_as_uint(acc[a].y),
                                           __float_as_uint(acc[a + 1].x), __float_as_uint(acc[a + 1].y));
                        }
                        *reinterpret_cast<uint4 *>(w_row + ((c ^ w_sw) << 4)) = o;
                    }
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint4 v = *reinterpret_cast<const uint4 *>(r_ptr + i * 512);
                        if (rrow0 + 8 * i < tl.row_end)
                            *reinterpret_cast<uint4 *>(out0 + i * row8 + q * 64) = v;
                    }
                    __syncwarp();
                }
            }
        }
    } else if (gathered) {
        // ------------------------------------------------ row gather (A) ----
        // Warps 2..3 copy the tile's token rows, 128 bytes per row and
        // contraction block, with 16-byte cp.async into the 128-byte
        // swizzled layout TMA would produce (chunk c of row r at c ^ (r % 8)).
        // Warp w owns tile rows 64(w-2) .. +63; one instruction copies 4 whole
        // rows (8 lanes per row), so each request is a full 128-byte line.
        // The tile's token indices sit in shared memory; rows past the
        // expert's end are not copied (their outputs are never stored, and an
        // MMA row depends on its own A row only). Up to three blocks stay in
        // flight; when a block's copies have landed the warp fences them for
        // the tensor cores' async proxy and arrives on the stage's "full"
        // barrier.
        setmaxnreg_dec<Regs<MODE>::LOW>();
        const int wrow = (warp - 2) * 64;          // first tile row of this warp
        const int chunk = lane & 7;                // 16-byte chunk of the row
        int32_t *tok = reinterpret_cast<int32_t *>(smem + L::tok_off);
        uint32_t stage = 0, phase = 0;
        int64_t issued = 0, arrived = 0;          // blocks issued / blocks signalled
        uint32_t arrive_stage = 0;
        bool ok = true;
        auto signal_oldest = [&]() {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(full_bar + 8 * arrive_stage);
            arrive_stage = arrive_stage + 1 == STAGES ? 0 : arrive_stage + 1;
            ++arrived;
        };
        for (int64_t t = sched->first; t < sched->count && ok; t += sched->stride) {
            const Tile tl = decode_tile<MODE>(t, p, prefix);
            const int64_t left = tl.row_end - tl.m0;
            const int nvalid = left < BM ? (int)left : BM;  // valid rows of the tile
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int rr = wrow + 32 * j + lane;
                if (rr < nvalid) {
                    int32_t v = p.row_index[tl.m0 + rr];
                    if (v < 0 || v >= p.n_tokens) {
                        atomicCAS(p.status, 0, FP8FG_EDEVICE);
                        v = 0;
                    }
                    tok[rr] = v;
                }
            }
            __syncwarp();
            for (int kb = 0; kb < num_kb; ++kb) {
                bool got = true;
                if (lane == 0)
                    got = mbar_wait(empty_bar + 8 * stage, phase ^ 1, wc, FP8FG_ETIMEOUT);
                got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
                if (!got) {
                    ok = false;
                    break;
                }
                const uint32_t a_dst = sbase + L::a_off + stage * A_STAGE_BYTES;
                const uint8_t *a_src = p.A + (int64_t)kb * BK + chunk * 16;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int rr = wrow + 4 * i + (lane >> 3);
                    if (rr < nvalid)
                        cp_async16(a_dst + rr * 128 + ((chunk ^ (rr & 7)) << 4), a_src + (int64_t)tok[rr] * p.K);
                }
                // the rows' scales of this block, into the stage's scale slot,
                // and (warp 2) the tile's two weight-block scales
                const uint32_t sa_dst = scale_base + stage * SS::bytes;
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int rr = wrow + 32 * j + lane;
                    if (rr < nvalid)
                        cp_async4(sa_dst + 4 * rr, p.sA + (int64_t)kb * p.ld_sA + tok[rr]);
                }
                if (warp == 2 && lane < 2 && tl.n0 + 128 * lane < p.N)
                    cp_async4(sa_dst + SS::b_off + 4 * lane, weight_scale<MODE>(p, tl, kb, lane));
                cp_async_commit();
                ++issued;
                cp_async_wait<2>();  // all but the two newest blocks have landed
                while (arrived < issued - 2)
                    signal_oldest();
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            __syncwarp();  // every lane has read this tile's token rows
        }
        cp_async_wait<0>();
        while (arrived < issued)
            signal_oldest();
    } else {
        // completes warpgroup 0 (warps 2..3 when warp 1 issues every block);
        // no role here
        setmaxnreg_dec<Regs<MODE>::LOW>();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ------------------------------------------------------------ host side ----

// Tensor maps of one launch: operands A and B, and the scale rows read by
// TMA (A's row scales; the weight gradient's column scales).
struct Maps {
    CUtensorMap a, b, sa, sb;
};

template <int MODE, int OUT>
int launch(const Maps &m, const Params &p, int grid, cudaStream_t s)
{
    auto k = gemm_kernel<MODE, OUT>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SmemLayout<MODE>::total) !=
        cudaSuccess) {
        cudaGetLastError();
        return FP8FG_ECUDA;
    }
    // The setmaxnreg split must fit in the registers the launch holds, or
    // the promotion warps' increase would never be granted.
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, k) != cudaSuccess) {
        cudaGetLastError();
        return FP8FG_ECUDA;
    }
    if (fa.numRegs < Regs<MODE>::LAUNCH_MIN)
        return FP8FG_EUNSUPPORTED;
    // programmatic stream serialization: the grid may launch while the
    // previous kernel's last CTAs run; the kernel waits (griddep_wait)
    // before it reads anything that kernel wrote
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = SmemLayout<MODE>::total;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, k, m.a, m.b, m.sa, m.sb, p) != cudaSuccess) {
        cudaGetLastError();
        return FP8FG_ECUDA;
    }
    return launch_status();
}

template <int MODE>
int launch_out(int out, const Maps &m, const Params &p, int grid, cudaStream_t s)
{
    return out == FP8FG_OUT_BF16 ? launch<MODE, OUT_BF16>(m, p, grid, s) : launch<MODE, OUT_F32>(m, p, grid, s);
}

// Tile order of a dense GEMM: bands of m-tiles, m fastest inside a band;
// the band's A panel is shared by the waves of the band and each B panel is
// read once per band. Bands of 32 m-tiles (the 152 CTAs that run at once
// cover 32 m-tiles x 4.75 n-tiles) halve the B re-reads of 16: the trio's
// fprop reads 331 MB of DRAM instead of 590, the weight gradient 708
// instead of 749. The data gradient (contraction 18432: A panels of 2.4
// MB, B panels of 4.7 MB) keeps bands of 16: with 32 its band's A panel no
// longer survives in L2 across the band's waves (1272 MB read against
// 1077), and n-major bands of 4, 7 or 14 n-tiles read 1103-1420 MB.
// (Keeping a whole operand resident in L2 measured 2x the DRAM reads: the
// output stream evicts it.)
void choose_raster(Params &p, int mode)
{
    p.n_major = 0;
    p.band = mode == DGRAD ? 16 : 32;
}

bool fill_runtime(Params &p)
{
    p.status = status_word_ptr();
    p.wait_limit_ns = wait_limit_ns();
    p.skip_first_load = take_skip_first_load() ? 1 : 0;
    return p.status != nullptr;
}

}  // namespace
}  // namespace fp8fg

using namespace fp8fg;

namespace fp8fg {
namespace {

// shared by the two GEMM entry points; out is an Out kind (sC and ld_sC are
// read for OUT_E4M3 only)
int gemm_entry(int mode, const uint8_t *A, const float *sA, int64_t lda, int64_t ld_sA, const uint8_t *B,
               const float *sB, int64_t ldb, int64_t ld_sB, int64_t M, int64_t N, int64_t K, void *C, int out,
               int64_t ldc, float *sC, int64_t ld_sC, void *stream)
{
    if (mode < FPROP || mode > WGRAD)
        return FP8FG_EINVAL;
    if (M < 0 || N < 0 || K < BK || N % 128 != 0 || K % BK != 0)
        return FP8FG_EINVAL;
    if (M >= (1ll << 31) || N >= (1ll << 31) || K >= (1ll << 31))
        return FP8FG_EINVAL;
    const int64_t esz = out == OUT_BF16 ? 2 : (out == OUT_F32 ? 4 : 1);
    if (lda < K || ldc < N || ld_sA < M)
        return FP8FG_EINVAL;
    if (out == OUT_E4M3 && ld_sC < M)
        return FP8FG_EINVAL;
    if (mode == DGRAD ? (ldb < N || ld_sB < N / 128) : (ldb < K))
        return FP8FG_EINVAL;
    if (mode == FPROP && ld_sB < K / 128)
        return FP8FG_EINVAL;
    if (mode == WGRAD && ld_sB < N)
        return FP8FG_EINVAL;
    if (M == 0 || N == 0)
        return FP8FG_OK;
    if (!A || !sA || !B || !sB || !C || (out == OUT_E4M3 && !sC))
        return FP8FG_EINVAL;
    if (!aligned16(A) || !aligned16(B) || !aligned16(C) || !aligned16(sA) || !aligned16(sB) || lda % 16 != 0 ||
        ldb % 16 != 0 || (ldc * esz) % 16 != 0 || ld_sA % 4 != 0 || (mode == WGRAD && ld_sB % 4 != 0))
        return FP8FG_EALIGN;
    if (out == OUT_E4M3 && (!aligned16(sC) || ld_sC % 4 != 0))
        return FP8FG_EALIGN;
    if (!device_supported())
        return FP8FG_EUNSUPPORTED;

    Params p{};
    p.M = M;
    p.N = N;
    p.K = K;
    p.sA = sA;
    p.ld_sA = ld_sA;
    p.sB = sB;
    p.ld_sB = ld_sB;
    p.C = C;
    p.ldc = ldc;
    p.sC = sC;
    p.ld_sC = ld_sC;
    p.num_m_tiles = (M + BM - 1) / BM;
    p.num_n_tiles = (N + BN - 1) / BN;
    choose_raster(p, mode);
    if (!fill_runtime(p))
        return FP8FG_ECUDA;

    Maps m;
    if (!make_map(&m.a, A, (uint64_t)K, (uint64_t)M, (uint64_t)lda, BK, BM))
        return FP8FG_ECUDA;
    bool okb;
    if (mode == DGRAD)  // weight [K][N], N contiguous: boxes of 128 N x 128 K
        okb = make_map(&m.b, B, (uint64_t)N, (uint64_t)K, (uint64_t)ldb, 128, BK);
    else
        okb = make_map(&m.b, B, (uint64_t)K, (uint64_t)N, (uint64_t)ldb, BK, BN);
    if (!okb)
        return FP8FG_ECUDA;
    // row scales [K/128][ld_sA]: one box of SA_BOX per block; the weight
    // gradient's column scales [K/128][ld_sB]: one box of BN per block
    if (!make_map_f32_row(&m.sa, sA, (uint64_t)M, (uint64_t)(K / BK), (uint64_t)ld_sA, SA_BOX))
        return FP8FG_ECUDA;
    if (mode == WGRAD) {
        if (!make_map_f32_row(&m.sb, sB, (uint64_t)N, (uint64_t)(K / BK), (uint64_t)ld_sB, BN))
            return FP8FG_ECUDA;
    } else {
        m.sb = m.sa;  // unused
    }

    const int64_t tiles = p.num_m_tiles * p.num_n_tiles;
    const int sms = sm_count();
    const int grid = (int)(tiles < sms ? tiles : sms);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (out == OUT_E4M3)
        return mode == FPROP ? launch<FPROP, OUT_E4M3>(m, p, grid, s) : launch<DGRAD, OUT_E4M3>(m, p, grid, s);
    switch (mode) {
    case FPROP: return launch_out<FPROP>(out, m, p, grid, s);
    case DGRAD: return launch_out<DGRAD>(out, m, p, grid, s);
    default: return launch_out<WGRAD>(out, m, p, grid, s);
    }
}

}  // namespace
}  // namespace fp8fg

extern "C" int fp8_gemm_blockscaled(int mode, const uint8_t *A, const float *sA, int64_t lda, int64_t ld_sA,
                                    const uint8_t *B, const float *sB, int64_t ldb, int64_t ld_sB, int64_t M,
                                    int64_t N, int64_t K, void *C, int out, int64_t ldc, void *stream)
{
    if (out != FP8FG_OUT_F32 && out != FP8FG_OUT_BF16)
        return FP8FG_EINVAL;
    return gemm_entry(mode, A, sA, lda, ld_sA, B, sB, ldb, ld_sB, M, N, K, C, out == FP8FG_OUT_BF16 ? OUT_BF16 : OUT_F32,
                      ldc, nullptr, 0, stream);
}

extern "C" int fp8_gemm_blockscaled_e4m3(int mode, const uint8_t *A, const float *sA, int64_t lda, int64_t ld_sA,
                                         const uint8_t *B, const float *sB, int64_t ldb, int64_t ld_sB, int64_t M,
                                         int64_t N, int64_t K, uint8_t *Cq, int64_t ldc, float *sC, int64_t ld_sC,
                                         void *stream)
{
    if (mode != FPROP && mode != DGRAD)  // the weight gradient stays FP32
        return FP8FG_EINVAL;
    return gemm_entry(mode, A, sA, lda, ld_sA, B, sB, ldb, ld_sB, M, N, K, Cq, OUT_E4M3, ldc, sC, ld_sC, stream);
}

extern "C" int fp8_grouped_gemm(const uint8_t *Xq, const float *sX, int64_t ld_sX, int64_t n_tokens,
                                const int32_t *row_index, const int32_t *expert_offsets, int32_t n_experts,
                                int64_t n_rows, const uint8_t *Wq, const float *sW, int64_t N, int64_t K, void *Y,
                                int out, int64_t ldy, void *stream)
{
    if (out != FP8FG_OUT_F32 && out != FP8FG_OUT_BF16)
        return FP8FG_EINVAL;
    if (n_tokens < 0 || n_rows < 0 || N < 0 || K < BK || N % 128 != 0 || K % BK != 0)
        return FP8FG_EINVAL;
    if (n_experts < 1 || n_experts > MAX_EXPERTS)
        return FP8FG_EINVAL;
    if (n_tokens >= (1ll << 31) || n_rows >= (1ll << 31) || K >= (1ll << 31) ||
        (int64_t)n_experts * N >= (1ll << 31))
        return FP8FG_EINVAL;
    // the kernels keep the experts' tile prefix in int32: reject any call
    // whose largest possible tile count (every expert ending in a partial
    // row tile) would not fit
    if (((n_rows + (int64_t)n_experts * (BM - 1)) / BM) * ((N + BN - 1) / BN) >= (1ll << 31))
        return FP8FG_EINVAL;
    const int64_t esz = out == FP8FG_OUT_BF16 ? 2 : 4;
    if (ld_sX < n_tokens || ldy < N)
        return FP8FG_EINVAL;
    if (!expert_offsets)
        return FP8FG_EINVAL;
    if (n_rows == 0 || N == 0 || n_tokens == 0) {
        // nothing can be written; offsets are not inspected
        return FP8FG_OK;
    }
    if (!Xq || !sX || !Wq || !sW || !Y)
        return FP8FG_EINVAL;
    if (!row_index && n_tokens < n_rows)  // rows already in expert order: row r is Xq row r
        return FP8FG_EINVAL;
    if (!aligned16(Xq) || !aligned16(Wq) || !aligned16(sX) || !aligned16(Y) || K % 16 != 0 || ld_sX % 4 != 0 ||
        (ldy * esz) % 16 != 0)
        return FP8FG_EALIGN;
    if (!device_supported())
        return FP8FG_EUNSUPPORTED;

    Params p{};
    p.M = n_rows;
    p.N = N;
    p.K = K;
    p.sA = sX;
    p.ld_sA = ld_sX;
    p.sB = sW;
    p.ld_sB = K / 128;
    p.C = Y;
    p.ldc = ldy;
    p.num_m_tiles = 0;
    p.num_n_tiles = (N + BN - 1) / BN;
    p.row_index = row_index;
    p.expert_offsets = expert_offsets;
    p.n_experts = n_experts;
    p.n_rows = n_rows;
    p.n_tokens = n_tokens;
    if (!fill_runtime(p))
        return FP8FG_ECUDA;
    p.skip_first_load = 0;

    Maps m;
    p.A = Xq;
    // with a row index the A rows and their scales are gathered with
    // cp.async (the A and row-scale maps are then unused but kept valid);
    // without one, TMA loads 128-row A tiles and their row scales
    if (!make_map(&m.a, Xq, (uint64_t)K, (uint64_t)n_tokens, (uint64_t)K, BK, row_index ? 1 : BM))
        return FP8FG_ECUDA;
    if (!make_map(&m.b, Wq, (uint64_t)K, (uint64_t)n_experts * (uint64_t)N, (uint64_t)K, BK, BN))
        return FP8FG_ECUDA;
    if (!make_map_f32_row(&m.sa, sX, (uint64_t)n_tokens, (uint64_t)(K / BK), (uint64_t)ld_sX, SA_BOX))
        return FP8FG_ECUDA;
    const int grid = sm_count();
    if (row_index) {
        m.sb = m.sa;  // unused
    } else {
        // the skinny tiles' token rows: 32-row boxes (the fourth map, which
        // carries column scales only for the weight gradient)
        if (!make_map(&m.sb, Xq, (uint64_t)K, (uint64_t)n_tokens, (uint64_t)K, BK, SK_TOK))
            return FP8FG_ECUDA;
        p.skinny_rows = grid >= 2 ? grouped_skinny_rows() : 0;
        p.skinny_cost_pct = grouped_skinny_cost_pct();
    }
    if (row_index)
        return launch_out<GROUPED>(out, m, p, grid > 0 ? grid : 1, static_cast<cudaStream_t>(stream));
    return launch_out<GROUPED_C>(out, m, p, grid > 0 ? grid : 1, static_cast<cudaStream_t>(stream));
}
