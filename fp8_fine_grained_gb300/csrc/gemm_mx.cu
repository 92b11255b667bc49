// Block-scaled FP8 GEMM on the tensor cores' own group scaling, for
// power-of-two group scales (the microscaling variant).
//
// Method: the same operands and group shapes as the promoted GEMM (1x128
// activation tiles, 128x128 weight blocks, groups of 128 tokens for the
// weight gradient), with every group scale a power of two. innerforce.co.kr
// (the paragraph relating the fine-grained groups to microscaling formats)
// notes that Blackwell tensor cores support microscaling; tonho.wtf
// ("o que isso custou") lists MMA with group scaling among the hardware
// requests. tcgen05.mma kind::mxf8f6f4 takes one UE8M0 scale per row of A
// and per column of B for each 32-wide contraction step and applies them
// inside the MMA, so the whole contraction accumulates in tensor memory and
// no partial sum leaves the tensor cores until the epilogue. A 128-wide
// group's scale is one byte in TMEM that all four of its K steps read.
// Modes: fprop, dgrad, wgrad, and MoE experts over rows already in expert
// order (the tiles of group_tiles.cuh).
//
// GB300 design (one CTA per SM, persistent over 128x256 output tiles, 16
// warps):
//   warp 0       TMA producer: A tile 128x128 B and B tile 256x128 B per
//                contraction block into a 4-stage shared-memory ring.
//   warp 1       MMA issuer: 4 x tcgen05.mma (M128 N256 K32) per block into
//                one 256-column FP32 accumulator; commits each block to its
//                stage's "empty" barrier and each tile to "accumulator full".
//   warps 2..3   no role.
//   warps 4..11  epilogue: 32 rows x 128 columns per warp from TMEM
//                (tcgen05.ld, 32 columns at a time), rounded and stored
//                through a shared-memory staging block; the accumulator is
//                released as soon as the last columns are loaded.
//   warps 12..15 scale writers, one per TMEM lane quarter: per group of
//                four blocks, the tiles' 128 A-row and 256 B-column scales
//                as UE8M0 bytes (the FP32 exponent field of a power of two),
//                block j in byte j % 4, into a scale slot in TMEM
//                (tcgen05.st), then "scales full"; the MMA selects the byte.
// TMEM: columns 0..255 accumulator; scale slot s at 256 + 64 s: A scales in
// columns +0..+3, B scales in +32..+39 (the layout mma_mxf8f6f4 reads).
// Every wait is bounded; a wait that runs out records FP8FG_ETIMEOUT and all
// roles leave their loops, drain their in-flight work and free TMEM.
#include <cuda_bf16.h>

#include "group_tiles.cuh"
#include "host_common.h"
#include "ptx.cuh"
#include "tensor_map.h"

namespace fp8fg {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 128;
constexpr int STAGES = 4;
constexpr int MMA_K = 32;
constexpr int EPI_WARP0 = 4;
constexpr int EPI_WARPS = 8;
constexpr int SF_WARP0 = 12;
constexpr int SF_WARPS = 4;
constexpr int NUM_THREADS = 16 * 32;
constexpr uint32_t A_STAGE_BYTES = BM * BK;
constexpr uint32_t B_STAGE_BYTES = BN * BK;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COL = 0;
constexpr uint32_t SF_COL0 = 256;
constexpr uint32_t SF_SLOT_COLS = 64;
constexpr uint32_t SFA_OFF = 0;
constexpr uint32_t SFB_OFF = 32;
// A scale slot serves SF_GROUP consecutive blocks of the CTA: block j's
// scales are byte j % 4 of every cell, selected by the MMA's scale-byte
// fields. SF_SLOTS slots let the writers run up to 12 blocks ahead.
constexpr int SF_GROUP = 4;
constexpr int SF_SLOTS = 4;
constexpr uint32_t STAGE_C_BYTES = 32 * 64;
static_assert(SF_COL0 + SF_SLOTS * SF_SLOT_COLS <= TMEM_COLS, "scale slots inside the allocation");

// GROUPED_C: MoE experts over rows already in expert order (as the gather
// quantiser writes them); B is the experts' weights [E][N][K].
enum Mode { FPROP = 0, DGRAD = 1, WGRAD = 2, GROUPED_C = 3 };
constexpr int MAX_EXPERTS = 4096;
enum Out { OUT_F32 = 0, OUT_BF16 = 1 };

struct Params {
    int64_t M, N, K;
    const float *sA;
    int64_t ld_sA;
    const float *sB;
    int64_t ld_sB;
    void *C;
    int64_t ldc;
    int64_t num_m_tiles, num_n_tiles;
    int *status;
    uint64_t wait_limit_ns;
    int skip_first_load;
    // grouped mode
    const int32_t *expert_offsets;
    int n_experts;
    int64_t n_rows;
};

struct SmemLayout {
    static constexpr uint32_t b_off = 0;
    static constexpr uint32_t a_off = b_off + STAGES * B_STAGE_BYTES;
    static constexpr uint32_t full_off = a_off + STAGES * A_STAGE_BYTES;
    static constexpr uint32_t empty_off = full_off + 8 * STAGES;
    static constexpr uint32_t sfull_off = empty_off + 8 * STAGES;
    static constexpr uint32_t sempty_off = sfull_off + 8 * SF_SLOTS;
    static constexpr uint32_t tfull_off = sempty_off + 8 * SF_SLOTS;
    static constexpr uint32_t tempty_off = tfull_off + 8;
    static constexpr uint32_t tmem_ptr_off = tempty_off + 8;
    static constexpr uint32_t abort_off = tmem_ptr_off + 4;
    static constexpr uint32_t stage_c_off = (abort_off + 4 + 15) & ~15u;
    static constexpr uint32_t prefix_off = stage_c_off + EPI_WARPS * STAGE_C_BYTES;  // grouped: tile prefix
    static constexpr uint32_t total = prefix_off + 4 * (MAX_EXPERTS + 1) + 1024;     // + alignment slack
};
static_assert(SmemLayout::total <= 232448, "shared memory budget");

// Dense modes: bands of m-tiles, m fastest inside a band (A and B tiles of
// CTAs that run together stay in L2): 32 m-tiles per band, 16 for the data
// gradient, whose long contraction makes its panels too large for a band of
// 32 to stay in L2 (as in the promoted kernel). Grouped: the experts' tiles.
template <int MODE>
__device__ __forceinline__ GroupTile decode_tile(int64_t t, const Params &p, const int32_t *prefix)
{
    if constexpr (MODE == GROUPED_C) {
        return decode_group_tile(t, prefix, p.expert_offsets, p.n_experts, p.n_rows, BM, BN);
    } else {
        constexpr int64_t BAND = MODE == DGRAD ? 16 : 32;
        const int64_t per_band = BAND * p.num_n_tiles;
        const int64_t band = t / per_band, r = t % per_band;
        const int64_t mfirst = band * BAND;
        const int64_t gm = (p.num_m_tiles - mfirst) < BAND ? (p.num_m_tiles - mfirst) : BAND;
        GroupTile g;
        g.m0 = (mfirst + r % gm) * BM;
        g.n0 = (r / gm) * BN;
        g.row_end = p.M;
        g.expert = 0;
        return g;
    }
}

// UE8M0 byte of a power-of-two scale: its biased FP32 exponent (2^-127, an
// FP32 subnormal, gives 0 = 2^-127).
__device__ __forceinline__ uint32_t ue8m0(float s)
{
    return (__float_as_uint(s) >> 23) & 0xFFu;
}

template <int MODE, int OUT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_mx_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const Params p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t full_bar = sbase + SmemLayout::full_off;
    const uint32_t empty_bar = sbase + SmemLayout::empty_off;
    const uint32_t sfull_bar = sbase + SmemLayout::sfull_off;
    const uint32_t sempty_bar = sbase + SmemLayout::sempty_off;
    const uint32_t tfull_bar = sbase + SmemLayout::tfull_off;
    const uint32_t tempty_bar = sbase + SmemLayout::tempty_off;
    volatile uint32_t *tmem_ptr = reinterpret_cast<volatile uint32_t *>(smem + SmemLayout::tmem_ptr_off);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + SmemLayout::abort_off);
    int32_t *prefix = reinterpret_cast<int32_t *>(smem + SmemLayout::prefix_off);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const WaitCtl wc{abort_flag, p.status, p.wait_limit_ns};

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar + 8 * s, 1);
            mbar_init(empty_bar + 8 * s, 1);
        }
        for (int s = 0; s < SF_SLOTS; ++s) {
            mbar_init(sfull_bar + 8 * s, SF_WARPS);
            mbar_init(sempty_bar + 8 * s, 1);
        }
        mbar_init(tfull_bar, 1);
        mbar_init(tempty_bar, EPI_WARPS);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(sbase + SmemLayout::tmem_ptr_off, TMEM_COLS);
        tmem_relinquish();
    }
    // Everything above touches only this CTA's shared and tensor memory;
    // inputs written by the previous kernel in the stream (for example the
    // quantiser, which lets this grid launch under its last wave) are read
    // only after this wait.
    griddep_wait();
    if constexpr (MODE == GROUPED_C)
        build_group_prefix<NUM_THREADS>(p.expert_offsets, p.n_experts, p.n_rows, p.num_n_tiles, BM, p.status, prefix,
                                        reinterpret_cast<int32_t *>(smem + SmemLayout::stage_c_off));
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_ptr;

    const int64_t num_tiles = MODE == GROUPED_C ? (int64_t)prefix[p.n_experts] : p.num_m_tiles * p.num_n_tiles;
    const int num_kb = (int)(p.K / BK);
    // this CTA's blocks, counted over its tiles in order
    const int64_t my_tiles = num_tiles > blockIdx.x ? (num_tiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    const int64_t total = my_tiles * num_kb;

    if (warp == 0) {
        // ------------------------------------------------------ producer ----
        uint32_t stage = 0, phase = 0;
        uint32_t filled_mask = 0, fill_parity = 0;
        bool skip = p.skip_first_load && blockIdx.x == 0;
        bool ok = true;
        for (int64_t t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
            const GroupTile tl = decode_tile<MODE>(t, p, prefix);
            const int64_t m0 = tl.m0, n0 = tl.n0;
            const int64_t brow0 = MODE == GROUPED_C ? (int64_t)tl.expert * p.N + n0 : n0;  // first B row
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
                const uint32_t a_dst = sbase + SmemLayout::a_off + stage * A_STAGE_BYTES;
                const uint32_t b_dst = sbase + SmemLayout::b_off + stage * B_STAGE_BYTES;
                if (skip) {
                    skip = false;  // withhold this load: consumers must time out
                } else if (lane == 0) {
                    bool second_half = true;
                    uint32_t bytes = A_STAGE_BYTES + B_STAGE_BYTES;
                    if constexpr (MODE == DGRAD) {
                        second_half = n0 + 128 < p.N;
                        if (!second_half)
                            bytes = A_STAGE_BYTES + B_STAGE_BYTES / 2;
                    }
                    mbar_arrive_expect_tx(fb, bytes);
                    filled_mask |= 1u << stage;
                    fill_parity = (fill_parity & ~(1u << stage)) | (phase << stage);
                    tma_load_2d(a_dst, &tmA, kb * BK, (int32_t)m0, fb);
                    if constexpr (MODE == DGRAD) {
                        // B is the weight [K][N] read N-contiguous: one 128 x 128
                        // box per 128-column half of the tile
                        tma_load_2d(b_dst, &tmB, (int32_t)n0, kb * BK, fb);
                        if (second_half)
                            tma_load_2d(b_dst + B_STAGE_BYTES / 2, &tmB, (int32_t)n0 + 128, kb * BK, fb);
                    } else {
                        tma_load_2d(b_dst, &tmB, kb * BK, (int32_t)brow0, fb);
                    }
                }
                __syncwarp();
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
        if (!ok && lane == 0) {
            // every issued fill must land before the CTA exits
            for (int s = 0; s < STAGES; ++s) {
                if (!(filled_mask & (1u << s)))
                    continue;
                const uint32_t bar = full_bar + 8 * s, par = (fill_parity >> s) & 1u;
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(bar, par) && global_timer_ns() - t0 < p.wait_limit_ns) {
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA ----
        if (lane == 0) {
            constexpr uint32_t IDESC = idesc_mx_e4m3(BM, BN, MODE == DGRAD);
            uint32_t stage = 0, phase = 0, tphase = 0, sslot = 0, sphase = 0;
            uint32_t last_bar = 0, last_par = 0;
            int64_t g = 0;  // block of the CTA
            bool issued = false, ok = true;
            for (int64_t t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                // the epilogue has read the previous tile's accumulator
                if (!mbar_wait(tempty_bar, tphase ^ 1, wc, FP8FG_ETIMEOUT)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int kb = 0; kb < num_kb; ++kb) {
                    const uint32_t byte = (uint32_t)(g % SF_GROUP);
                    if (!mbar_wait(full_bar + 8 * stage, phase, wc, FP8FG_ETIMEOUT) ||
                        (byte == 0 && !mbar_wait(sfull_bar + 8 * sslot, sphase, wc, FP8FG_ETIMEOUT))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = sbase + SmemLayout::a_off + stage * A_STAGE_BYTES;
                    const uint32_t b_addr = sbase + SmemLayout::b_off + stage * B_STAGE_BYTES;
                    const uint32_t sf = tmem_base + SF_COL0 + sslot * SF_SLOT_COLS;
                    const uint32_t idesc = IDESC | (byte << 29) | (byte << 4);  // scale bytes of this block
#pragma unroll
                    for (int k = 0; k < BK / MMA_K; ++k) {
                        const uint64_t adesc = smem_desc_sw128(a_addr + k * MMA_K, 0, 1024);
                        uint64_t bdesc;
                        if constexpr (MODE == DGRAD)
                            // N-major: 32 K-rows = 4 groups of 8 rows (1024 B
                            // each); the two 128-column halves are 16 KB apart
                            bdesc = smem_desc_sw128(b_addr + k * MMA_K * 128, B_STAGE_BYTES / 2, 1024);
                        else
                            bdesc = smem_desc_sw128(b_addr + k * MMA_K, 0, 1024);
                        mma_mxf8f6f4(tmem_base + ACC_COL, adesc, bdesc, idesc, sf + SFA_OFF, sf + SFB_OFF,
                                     (kb > 0 || k > 0) ? 1u : 0u);
                    }
                    mma_commit(empty_bar + 8 * stage);
                    issued = true;
                    last_bar = empty_bar + 8 * stage;
                    last_par = phase;
                    if (byte == SF_GROUP - 1 || g == total - 1) {
                        // the slot's blocks are done with its scales
                        mma_commit(sempty_bar + 8 * sslot);
                        last_bar = sempty_bar + 8 * sslot;
                        last_par = sphase;
                        if (++sslot == SF_SLOTS) {
                            sslot = 0;
                            sphase ^= 1;
                        }
                    }
                    ++g;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok)
                    break;
                mma_commit(tfull_bar);
                last_bar = tfull_bar;
                last_par = tphase;
                tphase ^= 1;
            }
            if (!ok && issued) {
                // the last commit covers every MMA issued before it
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(last_bar, last_par) && global_timer_ns() - t0 < p.wait_limit_ns) {
                }
            }
        }
        __syncwarp();
    } else if (warp >= SF_WARP0) {
        // ------------------------------------------------ scale writers ----
        // The CTA's blocks in order (its tiles, then kb), four to a scale
        // slot. A cursor that decodes each tile once loads a group's raw
        // scales one group ahead (the load latency, about 1000 cycles from
        // L2, stays off the path); they are converted only when written.
        const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
        // raw scale values of one block: the A row's and, for the weight
        // gradient, 8 column scales (else the tile's two weight-block scales)
        constexpr int NB = MODE == WGRAD ? 8 : 2;
        struct Sf {
            float a, b[NB];
        };
        int64_t ct = blockIdx.x, cm0 = 0, cn0 = 0, crow_end = 0;  // cursor: tile, its origin, block
        int cexp = 0, ckb = 0;
        auto seek = [&]() {
            if (ct < num_tiles) {
                const GroupTile tl = decode_tile<MODE>(ct, p, prefix);
                cm0 = tl.m0;
                cn0 = tl.n0;
                crow_end = tl.row_end;
                cexp = tl.expert;
            }
        };
        seek();
        auto load_sf = [&]() -> Sf {
            Sf v;
            v.a = 1.0f;
#pragma unroll
            for (int c = 0; c < NB; ++c)
                v.b[c] = 1.0f;
            if (ct >= num_tiles)
                return v;
            const int kb = ckb;
            const int64_t row = cm0 + quarter * 32 + lane;
            if (row < crow_end)
                v.a = __ldg(p.sA + (int64_t)kb * p.ld_sA + row);
            if constexpr (MODE == WGRAD) {
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const int64_t n = cn0 + 32 * c + lane;
                    if (n < p.N)
                        v.b[c] = __ldg(p.sB + (int64_t)kb * p.ld_sB + n);
                }
            } else {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int64_t nb = cn0 / 128 + h;
                    if (nb * 128 < p.N) {
                        if constexpr (MODE == GROUPED_C)  // expert block scales [E][N/128][K/128]
                            v.b[h] = __ldg(p.sB + ((int64_t)cexp * (p.N / 128) + nb) * p.ld_sB + kb);
                        else
                            v.b[h] = MODE == FPROP ? __ldg(p.sB + nb * p.ld_sB + kb)
                                                   : __ldg(p.sB + (int64_t)kb * p.ld_sB + nb);
                    }
                }
            }
            if (++ckb == num_kb) {
                ckb = 0;
                ct += gridDim.x;
                seek();
            }
            return v;
        };
        struct Grp {
            Sf blk[SF_GROUP];
        };
        auto load_grp = [&]() -> Grp {
            Grp r;
#pragma unroll
            for (int b = 0; b < SF_GROUP; ++b)
                r.blk[b] = load_sf();
            return r;
        };
        const int64_t groups = (total + SF_GROUP - 1) / SF_GROUP;
        Grp cur = load_grp();
        uint32_t sslot = 0, sphase = 0;
        for (int64_t G = 0; G < groups; ++G) {
            const Grp nxt = load_grp();
            bool got = true;
            if (lane == 0)
                got = mbar_wait(sempty_bar + 8 * sslot, sphase ^ 1, wc, FP8FG_ETIMEOUT);
            got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
            if (!got)
                break;
            tc_fence_after();
            uint32_t wa = 0, wb[8];
#pragma unroll
            for (int c = 0; c < 8; ++c)
                wb[c] = 0;
#pragma unroll
            for (int b = 0; b < SF_GROUP; ++b) {
                wa |= ue8m0(cur.blk[b].a) << (8 * b);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    wb[c] |= ue8m0(cur.blk[b].b[MODE == WGRAD ? c : c >> 2]) << (8 * b);
            }
            const uint32_t slot = tmem_base + ((uint32_t)(quarter * 32) << 16) + SF_COL0 + sslot * SF_SLOT_COLS;
            tmem_st_x1(slot + SFA_OFF + quarter, wa);
            tmem_st_x8(slot + SFB_OFF, wb);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(sfull_bar + 8 * sslot);
            if (++sslot == SF_SLOTS) {
                sslot = 0;
                sphase ^= 1;
            }
            cur = nxt;
        }
    } else if (warp >= EPI_WARP0) {
        // ------------------------------------------------------ epilogue ----
        const int ew = warp - EPI_WARP0;
        const int quarter = warp & 3;
        const int half = ew >> 2;
        constexpr int ESZ = OUT == OUT_BF16 ? 2 : 4;
        uint8_t *const stg = smem + SmemLayout::stage_c_off + ew * STAGE_C_BYTES;
        // staging: lane writes its row's 64-byte piece (16-byte chunk c at
        // c ^ ((row / 2) % 4)); the warp reads back 8 rows x 64 bytes per
        // instruction (row 8i + lane / 4, chunk lane % 4)
        uint8_t *const w_row = stg + lane * 64;
        const int w_sw = (lane >> 1) & 3;
        const int cc = lane & 3;
        const uint8_t *const r_ptr = stg + (lane >> 2) * 64 + ((cc ^ ((lane >> 3) & 3)) << 4);
        uint32_t tphase = 0;
        bool ok = true;
        for (int64_t t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
            const GroupTile tl = decode_tile<MODE>(t, p, prefix);
            const int64_t m0 = tl.m0, n0 = tl.n0, row_end = tl.row_end;
            const int64_t col0 = n0 + half * 128;
            const bool cols_ok = col0 < p.N;
            const int64_t rrow0 = m0 + quarter * 32 + (lane >> 2);  // row read back at i = 0
            uint8_t *const out0 = static_cast<uint8_t *>(p.C) + (rrow0 * p.ldc + col0) * ESZ + cc * 16;
            const int64_t row8 = 8 * p.ldc * ESZ;
            const bool got = mbar_wait(tfull_bar, tphase, wc, FP8FG_ETIMEOUT);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + ACC_COL + half * 128;
            auto store_piece = [&](const uint4 (&o)[4], int64_t colb) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    *reinterpret_cast<uint4 *>(w_row + ((c ^ w_sw) << 4)) = o[c];
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(r_ptr + i * 512);
                    if (rrow0 + 8 * i < row_end)
                        *reinterpret_cast<uint4 *>(out0 + i * row8 + colb) = v;
                }
                __syncwarp();
            };
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                uint32_t r[32];
                if (cols_ok) {
                    tmem_ld_chunk(taddr + 32 * c, r);
                    tmem_wait_ld_chunk(r);
                }
                if (c == 3) {
                    // the accumulator has been read: the next tile may start
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(tempty_bar);
                }
                if (!cols_ok)
                    continue;
                if constexpr (OUT == OUT_BF16) {
                    uint4 o[4];
                    uint32_t *ow = reinterpret_cast<uint32_t *>(o);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        __nv_bfloat162 h =
                            __float22bfloat162_rn(make_float2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1])));
                        ow[j] = *reinterpret_cast<uint32_t *>(&h);
                    }
                    store_piece(o, (int64_t)c * 32 * ESZ);
                } else {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint4 o[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            o[j] = make_uint4(r[16 * h + 4 * j], r[16 * h + 4 * j + 1], r[16 * h + 4 * j + 2],
                                              r[16 * h + 4 * j + 3]);
                        store_piece(o, (int64_t)c * 32 * ESZ + h * 64);
                    }
                }
            }
            tphase ^= 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

template <int MODE, int OUT>
int launch(const CUtensorMap &ta, const CUtensorMap &tb, const Params &p, int grid, cudaStream_t s)
{
    auto k = gemm_mx_kernel<MODE, OUT>;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SmemLayout::total) !=
        cudaSuccess) {
        cudaGetLastError();
        return FP8FG_ECUDA;
    }
    // programmatic stream serialization: the grid may launch while the
    // previous kernel's last CTAs run; the kernel waits (griddep_wait)
    // before it reads anything that kernel wrote
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = SmemLayout::total;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, k, ta, tb, p) != cudaSuccess) {
        cudaGetLastError();
        return FP8FG_ECUDA;
    }
    return launch_status();
}

template <int MODE>
int launch_out(int out, const CUtensorMap &ta, const CUtensorMap &tb, const Params &p, int grid, cudaStream_t s)
{
    return out == FP8FG_OUT_BF16 ? launch<MODE, OUT_BF16>(ta, tb, p, grid, s) : launch<MODE, OUT_F32>(ta, tb, p, grid, s);
}

}  // namespace
}  // namespace fp8fg

using namespace fp8fg;

extern "C" int fp8_gemm_mx(int mode, const uint8_t *A, const float *sA, int64_t lda, int64_t ld_sA, const uint8_t *B,
                           const float *sB, int64_t ldb, int64_t ld_sB, int64_t M, int64_t N, int64_t K, void *C,
                           int out, int64_t ldc, void *stream)
{
    if (mode < FPROP || mode > WGRAD || (out != FP8FG_OUT_F32 && out != FP8FG_OUT_BF16))
        return FP8FG_EINVAL;
    if (M < 0 || N < 0 || K < BK || N % 128 != 0 || K % BK != 0)
        return FP8FG_EINVAL;
    if (M >= (1ll << 31) || N >= (1ll << 31) || K >= (1ll << 31))
        return FP8FG_EINVAL;
    const int64_t esz = out == FP8FG_OUT_BF16 ? 2 : 4;
    if (lda < K || ldc < N || ld_sA < M)
        return FP8FG_EINVAL;
    if (mode == DGRAD ? (ldb < N || ld_sB < N / 128) : (ldb < K))
        return FP8FG_EINVAL;
    if (mode == FPROP && ld_sB < K / 128)
        return FP8FG_EINVAL;
    if (mode == WGRAD && ld_sB < N)
        return FP8FG_EINVAL;
    if (M == 0 || N == 0)
        return FP8FG_OK;
    if (!A || !sA || !B || !sB || !C)
        return FP8FG_EINVAL;
    if (!aligned16(A) || !aligned16(B) || !aligned16(C) || !aligned16(sA) || !aligned16(sB) || lda % 16 != 0 ||
        ldb % 16 != 0 || (ldc * esz) % 16 != 0 || ld_sA % 4 != 0 || (mode == WGRAD && ld_sB % 4 != 0))
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
    p.num_m_tiles = (M + BM - 1) / BM;
    p.num_n_tiles = (N + BN - 1) / BN;
    p.status = status_word_ptr();
    p.wait_limit_ns = wait_limit_ns();
    p.skip_first_load = take_skip_first_load() ? 1 : 0;
    if (!p.status)
        return FP8FG_ECUDA;

    CUtensorMap ta, tb;
    if (!make_map(&ta, A, (uint64_t)K, (uint64_t)M, (uint64_t)lda, BK, BM))
        return FP8FG_ECUDA;
    bool okb;
    if (mode == DGRAD)  // weight [K][N], N contiguous: boxes of 128 N x 128 K
        okb = make_map(&tb, B, (uint64_t)N, (uint64_t)K, (uint64_t)ldb, 128, BK);
    else
        okb = make_map(&tb, B, (uint64_t)K, (uint64_t)N, (uint64_t)ldb, BK, BN);
    if (!okb)
        return FP8FG_ECUDA;

    const int64_t tiles = p.num_m_tiles * p.num_n_tiles;
    const int sms = sm_count();
    const int grid = (int)(tiles < sms ? tiles : sms);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (mode) {
    case FPROP: return launch_out<FPROP>(out, ta, tb, p, grid, s);
    case DGRAD: return launch_out<DGRAD>(out, ta, tb, p, grid, s);
    default: return launch_out<WGRAD>(out, ta, tb, p, grid, s);
    }
}

extern "C" int fp8_grouped_gemm_mx(const uint8_t *Xq, const float *sX, int64_t ld_sX,
                                   const int32_t *expert_offsets, int32_t n_experts, int64_t n_rows,
                                   const uint8_t *Wq, const float *sW, int64_t N, int64_t K, void *Y, int out,
                                   int64_t ldy, void *stream)
{
    if (out != FP8FG_OUT_F32 && out != FP8FG_OUT_BF16)
        return FP8FG_EINVAL;
    if (n_rows < 0 || N < 0 || K < BK || N % 128 != 0 || K % BK != 0)
        return FP8FG_EINVAL;
    if (n_experts < 1 || n_experts > MAX_EXPERTS)
        return FP8FG_EINVAL;
    if (n_rows >= (1ll << 31) || K >= (1ll << 31) || (int64_t)n_experts * N >= (1ll << 31))
        return FP8FG_EINVAL;
    // the kernels keep the experts' tile prefix in int32: reject any call
    // whose largest possible tile count (every expert ending in a partial
    // row tile) would not fit
    if (((n_rows + (int64_t)n_experts * (BM - 1)) / BM) * ((N + BN - 1) / BN) >= (1ll << 31))
        return FP8FG_EINVAL;
    const int64_t esz = out == FP8FG_OUT_BF16 ? 2 : 4;
    if (ld_sX < n_rows || ldy < N || !expert_offsets)
        return FP8FG_EINVAL;
    if (n_rows == 0 || N == 0)
        return FP8FG_OK;
    if (!Xq || !sX || !Wq || !sW || !Y)
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
    p.expert_offsets = expert_offsets;
    p.n_experts = n_experts;
    p.n_rows = n_rows;
    p.status = status_word_ptr();
    p.wait_limit_ns = wait_limit_ns();
    p.skip_first_load = take_skip_first_load() ? 1 : 0;
    if (!p.status)
        return FP8FG_ECUDA;

    CUtensorMap ta, tb;
    if (!make_map(&ta, Xq, (uint64_t)K, (uint64_t)n_rows, (uint64_t)K, BK, BM))
        return FP8FG_ECUDA;
    if (!make_map(&tb, Wq, (uint64_t)K, (uint64_t)n_experts * (uint64_t)N, (uint64_t)K, BK, BN))
        return FP8FG_ECUDA;
    const int grid = sm_count();
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return out == FP8FG_OUT_BF16 ? launch<GROUPED_C, OUT_BF16>(ta, tb, p, grid > 0 ? grid : 1, s)
                                 : launch<GROUPED_C, OUT_F32>(ta, tb, p, grid > 0 ? grid : 1, s);
}
