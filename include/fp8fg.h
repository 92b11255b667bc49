/*
 * fp8fg.h - fine-grained FP8 quantisation and block-scaled FP8 GEMM on
 * GB300 (sm_103a). C ABI of libfp8fg.so.
 *
 * What the operations compute comes from web pages describing DeepSeek-V3's
 * FP8 mixed-precision training framework:
 *   - innerforce.co.kr, paragraph on fine-grained quantization (Figure
 *     7(a)): activations are scaled per 1x128 tile (one token, 128
 *     channels), weights per 128x128 block; each group's largest magnitude
 *     is mapped onto FP8's largest representable value. The following
 *     paragraph: FP8 GEMM partial sums are promoted and accumulated in FP32,
 *     and dequantisation rides on that promotion.
 *   - yunhecapital.com, section 2.2.3 (FP8 mixed-precision framework):
 *     the same 1x128 / 128x128 grouping; at each accumulation interval the
 *     tensor-core partials move to FP32 registers on CUDA cores.
 *   - tonho.wtf DeepSeek-V3 entry, section "como funciona": scale factors
 *     are computed online, tensors are always E4M3, partials are promoted
 *     every 128 elements. Section "o que isso custou": activation gradients
 *     diverge under 128x128 blocks (so they use 1x128 tiles), and a fused
 *     cast and a transposed read are on the hardware wish list.
 *
 * Numerics shared by every entry point:
 *   E4M3      OCP FP8 E4M3 ("fn"): bias 7, no infinities, max finite +-448.
 *   scale     per group: amax = max |x| over the group's bf16 values;
 *             s = amax / 448 and inv = 448 / amax, both IEEE FP32 divisions
 *             rounded to nearest. If amax == 0, or 448/amax overflows FP32,
 *             s = inv = 1.
 *   code      q = E4M3(x * inv): one FP32 product, then round to nearest
 *             even into E4M3, saturating at +-448; the sign of zero is kept.
 *   GEMM      C[i,j] = sum over 128-wide contraction blocks kb of
 *             sA(i,kb) * sB(j,kb) * P(i,j,kb), P the block's FP8 x FP8 dot
 *             product from the tensor cores (FP32 in tensor memory), the sum
 *             over kb kept in FP32 registers.
 *   inputs    bf16 inputs must be finite. A NaN or an infinity in a group is
 *             outside the contract: the call still returns, no kernel hangs
 *             or touches memory outside its arguments, but that group's
 *             codes and scale (and every GEMM output that reads them) are
 *             unspecified. The pages give no rule for non-finite values.
 *
 * Conventions for every call:
 *   - All pointers are DEVICE pointers owned by the caller. The library
 *     allocates no device memory and keeps no state beyond per-device
 *     kernel attributes and a device status word.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Work is enqueued asynchronously; no call synchronises.
 *   - Leading dimensions are in ELEMENTS. Matrices are row-major.
 *   - Synchronous validation returns FP8FG_EINVAL (null pointer, negative or
 *     unsupported size, leading dimension too small), FP8FG_EALIGN (a pointer
 *     not 16-byte aligned or a row pitch not a multiple of 16 bytes) before
 *     anything is launched; FP8FG_ECUDA if a launch fails. A zero-sized
 *     problem returns FP8FG_OK and launches nothing.
 *   - Errors found on the device (a bounded wait that ran out, an expert row
 *     index out of range) are recorded in a per-device status word and
 *     reported by fp8fg_device_status(). Kernels never trap.
 *   - No C++ exception crosses this interface.
 */
#ifndef FP8FG_H
#define FP8FG_H

#include <stdint.h>

#if defined(__GNUC__)
#define FP8FG_API __attribute__((visibility("default")))
#else
#define FP8FG_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP8FG_OK = 0,
    FP8FG_EINVAL = 1,       /* invalid argument */
    FP8FG_EALIGN = 2,       /* pointer or pitch not 16-byte aligned */
    FP8FG_EUNSUPPORTED = 3, /* device is not sm_103 / feature unavailable */
    FP8FG_ECUDA = 4,        /* CUDA runtime or driver error */
    FP8FG_ETIMEOUT = 5,     /* a device-side bounded wait ran out */
    FP8FG_EDEVICE = 6       /* invalid data found on the device */
} fp8fg_status;

typedef enum { FP8FG_OUT_F32 = 0, FP8FG_OUT_BF16 = 1 } fp8fg_out;

typedef enum { FP8FG_FPROP = 0, FP8FG_DGRAD = 1, FP8FG_WGRAD = 2 } fp8fg_mode;

/* ---------------------------------------------------------------------
 * fp8_quant_1x128: activation quantisation in 1x128 tiles.
 * Source: innerforce.co.kr, fine-grained quantization paragraph (Figure
 * 7(a)), "per token per 128 channels"; tonho.wtf "como funciona" (online
 * scale, E4M3); for transpose = 1, tonho.wtf "o que isso custou"
 * (transposed read for the weight-gradient operands, which are grouped
 * along tokens).
 *
 *   x       bf16 [rows][ldx], row-major, ldx >= cols.
 *   transpose = 0: groups are 128 consecutive COLUMNS of one row.
 *           cols % 128 == 0, rows >= 0 arbitrary.
 *           q      E4M3 bytes [rows][ldq], ldq >= cols.
 *           scales FP32 [cols/128][ld_s], ld_s >= rows: scale of row r,
 *                  group g at scales[g*ld_s + r] (groups outer, rows
 *                  contiguous: the layout the GEMM reads).
 *   transpose = 1: groups are 128 consecutive ROWS of one column and the
 *           output is transposed. rows % 128 == 0, cols >= 0 arbitrary;
 *           rows are read in 16-byte pieces, so with cols % 8 != 0 each
 *           row of x must be readable up to cols rounded up to a multiple
 *           of 8 (within ldx; the extra columns do not affect the output).
 *           q      E4M3 bytes [cols][ldq], ldq >= rows: q[c*ldq + r].
 *           scales FP32 [rows/128][ld_s], ld_s >= cols: scale of column c,
 *                  group g at scales[g*ld_s + c].
 *           (This is exactly the transpose=0 output for the matrix x^T.)
 *   Alignment: x, q, scales 16-byte aligned; ldx % 8 == 0, ldq % 16 == 0,
 *   ld_s % 4 == 0.
 * ------------------------------------------------------------------- */
FP8FG_API int fp8_quant_1x128(const void *x, int64_t rows, int64_t cols, int64_t ldx,
                    uint8_t *q, int64_t ldq, float *scales, int64_t ld_s,
                    int transpose, void *stream);

/* ---------------------------------------------------------------------
 * fp8_quant_1x128_dual: both activation layouts from one read of x.
 * Source: the 1x128 rule of fp8_quant_1x128 (innerforce.co.kr, fine-grained
 * quantization paragraph); tonho.wtf "o que isso custou" (the transposed read
 * for the weight-gradient operands, and the wish to fuse the cast with the
 * memory transfer).
 *
 * Writes exactly what fp8_quant_1x128(x, transpose = 0) and
 * fp8_quant_1x128(x, transpose = 1) write, bit for bit, reading x once.
 *   x       bf16 [rows][ldx], rows % 128 == 0, cols % 128 == 0, ldx >= cols.
 *   q       E4M3 [rows][ldq] (ldq >= cols); scales FP32 [cols/128][ld_s],
 *           ld_s >= rows: row r, group g at scales[g*ld_s + r].
 *   qT      E4M3 [cols][ldqT] (ldqT >= rows): qT[c*ldqT + r]; scalesT FP32
 *           [rows/128][ld_sT], ld_sT >= cols: column c, group g at
 *           scalesT[g*ld_sT + c].
 *   Alignment: x, q, scales, qT, scalesT 16-byte aligned; ldx % 8 == 0,
 *   ldq % 16 == 0, ldqT % 16 == 0, ld_s % 4 == 0, ld_sT % 4 == 0.
 *   All buffers belong to the caller; nothing is allocated. rows == 0 or
 *   cols == 0 is a no-op.
 * ------------------------------------------------------------------- */
FP8FG_API int fp8_quant_1x128_dual(const void *x, int64_t rows, int64_t cols, int64_t ldx,
                         uint8_t *q, int64_t ldq, float *scales, int64_t ld_s,
                         uint8_t *qT, int64_t ldqT, float *scalesT, int64_t ld_sT,
                         void *stream);

/* ---------------------------------------------------------------------
 * fp8_quant_1x128_gather: 1x128 activation quantisation of selected rows,
 * written in the order of a row index (MoE rows grouped by expert).
 * Source: the 1x128 rule of fp8_quant_1x128 (innerforce.co.kr, fine-grained
 * quantization paragraph); yunhecapital.com 2.2.2 (each token is routed to
 * 8 of 256 experts). The tiles are per row, so the result is exactly the
 * rows row_index[0..rows) of fp8_quant_1x128(x): the quantised tokens
 * dispatched to their experts in one pass.
 *
 *   x         bf16 [n_src][ldx], ldx >= cols, cols % 128 == 0.
 *   row_index int32 [rows], device: source row of output row r. Entries
 *             outside [0, n_src) are reported as FP8FG_EDEVICE through
 *             fp8fg_device_status and read source row 0.
 *   q         E4M3 bytes [rows][ldq], ldq >= cols.
 *   scales    FP32 [cols/128][ld_s], ld_s >= rows (the GEMM's layout).
 *   Alignment: x, q, scales 16-byte aligned; ldx % 8 == 0, ldq % 16 == 0,
 *   ld_s % 4 == 0. All buffers are owned by the caller; nothing is
 *   allocated. rows == 0 or cols == 0 is a no-op; n_src == 0 with rows > 0
 *   is FP8FG_EINVAL.
 * ------------------------------------------------------------------- */
FP8FG_API int fp8_quant_1x128_gather(const void *x, int64_t n_src, int64_t cols, int64_t ldx,
                           const int32_t *row_index, int64_t rows,
                           uint8_t *q, int64_t ldq, float *scales, int64_t ld_s,
                           void *stream);

/* ---------------------------------------------------------------------
 * fp8_quant_1x128_scatter: the same dispatch in token order.
 * Source: as fp8_quant_1x128_gather (yunhecapital.com 2.2.3: FP8 for the
 * dispatch; 2.2.2 and tonho.wtf "como funciona": 8 of 256 routed experts
 * per token).
 *
 * Every source row r of x is read and quantised once (1x128 rule) and
 * written to its k destination rows d = dest_index[r*k + j], j < k:
 * q[d][:] and scales[g*ld_s + d]. The result equals
 * fp8_quant_1x128_gather with the inverse index, while each token is read
 * once instead of once per copy.
 *   x           bf16 [n_src][ldx]; cols % 128 == 0.
 *   dest_index  int32 [n_src][k], device; 1 <= k <= 16. A negative entry
 *               is not written; an entry >= n_out is reported as
 *               FP8FG_EDEVICE through fp8fg_device_status and not written.
 *   q           E4M3 [n_out][ldq]; scales FP32 [cols/128][ld_s],
 *               ld_s >= n_out. Rows no entry points to are left untouched.
 *   Alignment as fp8_quant_1x128. fp8_quant_1x128_scatter_pow2 is the
 *   power-of-two variant (see below).
 * ------------------------------------------------------------------- */
FP8FG_API int fp8_quant_1x128_scatter(const void *x, int64_t n_src, int64_t cols, int64_t ldx,
                           const int32_t *dest_index, int k, int64_t n_out,
                           uint8_t *q, int64_t ldq, float *scales, int64_t ld_s,
                           void *stream);

/* ---------------------------------------------------------------------
 * fp8_quant_128x128: weight quantisation in 128x128 blocks.
 * Source: innerforce.co.kr, fine-grained quantization paragraph ("per 128
 * input channels per 128 output channels"); yunhecapital.com 2.2.3;
 * tonho.wtf "como funciona".
 *
 *   w       bf16 [N][ldw], ldw >= K; N % 128 == 0, K % 128 == 0.
 *   q       E4M3 bytes [N][ldq], ldq >= K.
 *   scales  FP32 [N/128][K/128], dense: scale of block (i, j) at
 *           scales[i*(K/128) + j].
 *   Alignment: w, q 16-byte aligned; ldw % 8 == 0, ldq % 16 == 0.
 * ------------------------------------------------------------------- */
FP8FG_API int fp8_quant_128x128(const void *w, int64_t N, int64_t K, int64_t ldw,
                      uint8_t *q, int64_t ldq, float *scales, void *stream);

/* ---------------------------------------------------------------------
 * fp8_quant_128x128_dual: the weight's 128x128 blocks and those of its
 * transpose from one read of w.
 * Source: innerforce.co.kr, fine-grained quantization paragraph (128x128
 * weight blocks); tonho.wtf "o que isso custou" (a fused cast and a
 * transposed read on the wish list). The block (j, i) of W^T is the
 * transpose of block (i, j) of W with the same scale, so qT and scalesT
 * equal fp8_quant_128x128 of the materialised transpose, byte for byte.
 *
 *   w, q, scales  as fp8_quant_128x128 (W [N][K]).
 *   qT       E4M3 bytes [K][ldqT], ldqT >= N: qT[k][n] = q[n][k].
 *   scalesT  FP32 [K/128][N/128], dense: scalesT[j*(N/128) + i] =
 *            scales[i*(K/128) + j].
 *   Alignment: w, q, qT 16-byte aligned; ldw % 8 == 0, ldq % 16 == 0,
 *   ldqT % 16 == 0; scales and scalesT 4-byte aligned.
 *   Errors: FP8FG_EINVAL for N or K not a multiple of 128 or a leading
 *   dimension below its minimum; FP8FG_EALIGN as above. All buffers are
 *   owned by the caller. fp8_quant_128x128_dual_pow2 is the power-of-two
 *   variant (see below).
 * ------------------------------------------------------------------- */
FP8FG_API int fp8_quant_128x128_dual(const void *w, int64_t N, int64_t K, int64_t ldw,
                      uint8_t *q, int64_t ldq, float *scales,
                      uint8_t *qT, int64_t ldqT, float *scalesT, void *stream);

/* ---------------------------------------------------------------------
 * fp8_gemm_blockscaled: block-scaled FP8 GEMM, promotion every 128 of the
 * contraction dimension K.
 * Source: innerforce.co.kr, increased-precision accumulation paragraph
 * (FP32 accumulation, dequantisation folded into the promotion);
 * yunhecapital.com 2.2.3; tonho.wtf "como funciona" (every 128 elements);
 * tonho.wtf "o que isso custou" (activation gradients in 1x128 tiles).
 *
 * All modes compute C[M][N] (ldc >= N) with K % 128 == 0, N % 128 == 0,
 * M >= 0 arbitrary; out = FP8FG_OUT_F32 (C is float) or FP8FG_OUT_BF16 (C
 * is bf16, rounded to nearest even from the FP32 sum).
 *
 *   FP8FG_FPROP  C = A . B^T. A: activations quantised 1x128,
 *                E4M3 [M][lda], scales sA [K/128][ld_sA] (ld_sA >= M).
 *                B: weight quantised 128x128, E4M3 [N][ldb], scales
 *                sB [N/128][ld_sB] (ld_sB >= K/128).
 *   FP8FG_DGRAD  C = A . B. A: gradient dY quantised 1x128 along K (the
 *                layer's output channels), [M][lda], sA [K/128][ld_sA].
 *                B: the forward weight exactly as fp8_quant_128x128 stored
 *                it, E4M3 [K][ldb] (ldb >= N), scales sB [K/128][ld_sB]
 *                (ld_sB >= N/128). B is read N-contiguous; no transposed
 *                copy is needed.
 *   FP8FG_WGRAD  C = A . B^T with both operands quantised in groups of
 *                128 along K (tokens), i.e. fp8_quant_1x128 outputs with
 *                transpose = 1: A E4M3 [M][lda], sA [K/128][ld_sA]
 *                (ld_sA >= M); B E4M3 [N][ldb], sB [K/128][ld_sB]
 *                (ld_sB >= N). Each output element uses its row's and its
 *                column's scale.
 *   Alignment: A, B, C, sA, sB 16-byte aligned; lda, ldb % 16 == 0;
 *   ldc*sizeof(out) % 16 == 0; ld_sA % 4 == 0 (and ld_sB % 4 == 0 for
 *   WGRAD).
 * ------------------------------------------------------------------- */
FP8FG_API int fp8_gemm_blockscaled(int mode,
                         const uint8_t *A, const float *sA, int64_t lda, int64_t ld_sA,
                         const uint8_t *B, const float *sB, int64_t ldb, int64_t ld_sB,
                         int64_t M, int64_t N, int64_t K,
                         void *C, int out, int64_t ldc, void *stream);

/* ---------------------------------------------------------------------
 * fp8_gemm_blockscaled_e4m3: the forward or data-gradient GEMM of
 * fp8_gemm_blockscaled with its output quantised in the epilogue.
 * Source: the GEMM above; tonho.wtf "o que isso custou" (the wish to fuse
 * the FP8 cast with the producer of the activation, so that activations are
 * stored in FP8 and scaled online); the 1x128 group rule of
 * fp8_quant_1x128 (innerforce.co.kr, fine-grained quantization paragraph).
 *
 * Every element is first rounded to bf16 (RNE), then each row's groups of
 * 128 consecutive columns are quantised by the 1x128 rule: the outputs are
 * bit-identical to fp8_quant_1x128 applied to the bf16 result of
 * fp8_gemm_blockscaled with out = FP8FG_OUT_BF16, without that bf16 matrix
 * ever being written.
 *   mode    FP8FG_FPROP or FP8FG_DGRAD (operands as in fp8_gemm_blockscaled;
 *           FP8FG_WGRAD is EINVAL: the weight gradient stays FP32).
 *   Cq      E4M3 [M][ldc], ldc >= N, ldc % 16 == 0.
 *   sC      FP32 [N/128][ld_sC], ld_sC >= M, ld_sC % 4 == 0: scale of row
 *           r, group g at sC[g*ld_sC + r].
 *   Other arguments, alignment and errors as fp8_gemm_blockscaled; Cq and sC
 *   16-byte aligned. Buffers belong to the caller; nothing is allocated.
 * ------------------------------------------------------------------- */
FP8FG_API int fp8_gemm_blockscaled_e4m3(int mode,
                         const uint8_t *A, const float *sA, int64_t lda, int64_t ld_sA,
                         const uint8_t *B, const float *sB, int64_t ldb, int64_t ld_sB,
                         int64_t M, int64_t N, int64_t K,
                         uint8_t *Cq, int64_t ldc, float *sC, int64_t ld_sC, void *stream);

/* ---------------------------------------------------------------------
 * fp8_grouped_gemm: MoE expert GEMM over a per-expert row index.
 * Source: yunhecapital.com 2.2.2 and tonho.wtf "como funciona" (one shared
 * and 256 routed experts, 8 active per token) with the FP8 GEMM above
 * (expert GEMMs are FP8 GEMMs).
 *
 *   For each expert e and each row r in [off[e], off[e+1]):
 *       Y[r][:] = fprop(Xq[row_index[r]], Wq[e])
 *   Xq        E4M3 [n_tokens][K] (lda = K), quantised once per token 1x128.
 *   sX        FP32 [K/128][ld_sX], ld_sX >= n_tokens (fp8_quant_1x128 layout).
 *   row_index int32 [n_rows], device: token of each row, rows grouped by
 *             expert. Entries outside [0, n_tokens) are reported as
 *             FP8FG_EDEVICE through fp8fg_device_status and read token 0.
 *             NULL: Xq and sX already hold the rows in expert order (as
 *             fp8_quant_1x128_gather writes them); output row r reads Xq
 *             row r, and n_tokens >= n_rows is required (else EINVAL).
 *             A tile's rows are then loaded by TMA instead of gathered.
 *   expert_offsets int32 [n_experts+1], device, non-decreasing, off[0] = 0,
 *             off[n_experts] <= n_rows. Rows at or beyond off[n_experts] are
 *             not written.
 *   Wq        E4M3 [n_experts][N][K]; sW FP32 [n_experts][N/128][K/128].
 *   Y         [n_rows][ldy], FP32 or bf16 per `out`.
 *   K % 128 == 0, N % 128 == 0, 1 <= n_experts <= 4096, and the largest
 *   possible tile count ((n_rows + 127 n_experts) / 128) x ceil(N / 256)
 *   below 2^31 (else EINVAL).
 *   Alignment: Xq, Wq, sX, Y 16-byte aligned; K % 16 == 0; ld_sX % 4 == 0;
 *   ldy*sizeof(out) % 16 == 0.
 *   Tiles: 128 rows of an expert x 256 columns. With row_index == NULL,
 *   experts with at most 32 rows (fp8fg_set_grouped_schedule) are computed
 *   instead as 256 weight rows x their (up to) 32 token rows per tile, with
 *   the weight as the tensor cores' 128-row operand; the sum and its
 *   promotion per 128-wide contraction block are the same. Part of the SMs
 *   takes those tiles while the others take the rest.
 * ------------------------------------------------------------------- */
FP8FG_API int fp8_grouped_gemm(const uint8_t *Xq, const float *sX, int64_t ld_sX, int64_t n_tokens,
                     const int32_t *row_index, const int32_t *expert_offsets,
                     int32_t n_experts, int64_t n_rows,
                     const uint8_t *Wq, const float *sW, int64_t N, int64_t K,
                     void *Y, int out, int64_t ldy, void *stream);

/* ---------------------------------------------------------------------
 * Microscaling variant: power-of-two group scales and the tensor cores'
 * own block scaling.
 * Source: innerforce.co.kr, the paragraph relating the fine-grained groups
 * to microscaling formats, which Blackwell tensor cores support; tonho.wtf
 * "o que isso custou" (MMA with group scaling on the hardware wish list) and
 * "onde isso aparece hoje" (microscaling announced for Blackwell).
 * Microscaling shares a power-of-two scale per group; the pages give no
 * rounding for it. Reading used here: the groups stay the pages' (1x128,
 * 128x1, 128x128) and
 *   scale   s = 2^e, the smallest power of two with amax <= 448 * 2^e,
 *           e >= -127 (the UE8M0 range); amax == 0 gives s = 1. inv = 2^-e.
 *   code    q = E4M3(x * inv), one rounding (x * inv is exact), never
 *           saturating since |x * inv| <= 448.
 * Scales are stored as FP32 values (exact powers of two) in the same layouts
 * as the entry points above, so either GEMM accepts them.
 *
 * fp8_quant_1x128_pow2, fp8_quant_1x128_dual_pow2,
 * fp8_quant_1x128_gather_pow2, fp8_quant_1x128_scatter_pow2,
 * fp8_quant_128x128_pow2, fp8_quant_128x128_dual_pow2: arguments,
 * layouts, alignment and errors exactly as fp8_quant_1x128,
 * fp8_quant_1x128_dual, fp8_quant_1x128_gather, fp8_quant_1x128_scatter,
 * fp8_quant_128x128 and fp8_quant_128x128_dual; only the scale rule
 * differs.
 * ------------------------------------------------------------------- */
FP8FG_API int fp8_quant_1x128_pow2(const void *x, int64_t rows, int64_t cols, int64_t ldx,
                         uint8_t *q, int64_t ldq, float *scales, int64_t ld_s,
                         int transpose, void *stream);
FP8FG_API int fp8_quant_1x128_dual_pow2(const void *x, int64_t rows, int64_t cols, int64_t ldx,
                         uint8_t *q, int64_t ldq, float *scales, int64_t ld_s,
                         uint8_t *qT, int64_t ldqT, float *scalesT, int64_t ld_sT,
                         void *stream);
FP8FG_API int fp8_quant_1x128_gather_pow2(const void *x, int64_t n_src, int64_t cols, int64_t ldx,
                         const int32_t *row_index, int64_t rows,
                         uint8_t *q, int64_t ldq, float *scales, int64_t ld_s, void *stream);
FP8FG_API int fp8_quant_1x128_scatter_pow2(const void *x, int64_t n_src, int64_t cols, int64_t ldx,
                         const int32_t *dest_index, int k, int64_t n_out,
                         uint8_t *q, int64_t ldq, float *scales, int64_t ld_s, void *stream);
FP8FG_API int fp8_quant_128x128_pow2(const void *w, int64_t N, int64_t K, int64_t ldw,
                         uint8_t *q, int64_t ldq, float *scales, void *stream);
FP8FG_API int fp8_quant_128x128_dual_pow2(const void *w, int64_t N, int64_t K, int64_t ldw,
                      uint8_t *q, int64_t ldq, float *scales,
                      uint8_t *qT, int64_t ldqT, float *scalesT, void *stream);

/* ---------------------------------------------------------------------
 * fp8_gemm_mx: the GEMM of fp8_gemm_blockscaled (same modes, operands,
 * layouts, alignment and errors) for power-of-two scales, with the scales
 * applied inside the tensor cores' block-scaled MMA (one UE8M0 scale per
 * A row and per B column for every 32-wide contraction step; a 128-wide
 * group repeats its scale over its four steps). The whole contraction
 * accumulates in FP32 in tensor memory; there is no per-block promotion.
 * Mathematically C is the same sum as fp8_gemm_blockscaled computes:
 *     C[i,j] = sum_kb sA(i,kb) sB(j,kb) P(i,j,kb),
 * rounded differently (the tolerance is the same).
 *   Every scale must be a power of two in [2^-127, 2^127] (the *_pow2
 *   quantisers write only such values); a scale's FP32 exponent field is
 *   what the tensor cores receive, so other values are taken as the power
 *   of two at or below them.
 * ------------------------------------------------------------------- */
FP8FG_API int fp8_gemm_mx(int mode,
                         const uint8_t *A, const float *sA, int64_t lda, int64_t ld_sA,
                         const uint8_t *B, const float *sB, int64_t ldb, int64_t ld_sB,
                         int64_t M, int64_t N, int64_t K,
                         void *C, int out, int64_t ldc, void *stream);

/* ---------------------------------------------------------------------
 * fp8_moe_combine: the MoE layer's output from its experts' rows.
 * Source: yunhecapital.com 2.2.2 and tonho.wtf "como funciona" (8 of 256
 * routed experts per token: a token's output is the gate-weighted sum of
 * its routed experts' outputs); innerforce.co.kr, the mixed-precision
 * framework paragraph (activations are dispatched to the experts in FP8;
 * the expert outputs come back in bf16). The pages fix no precision for
 * the combine; the reading taken: FP32 products and sums in slot order.
 *
 *   out[t][n] = sum_{j < k} w[t][j] * y[dest[t][j]][n]
 *   y       bf16 [y_rows][ldy] (for example fp8_grouped_gemm's output).
 *   dest    int32 [T][k], device: row of y for token t's slot j; a negative
 *           entry skips the slot (a token routed to fewer experts); an entry
 *           >= y_rows is reported as FP8FG_EDEVICE through
 *           fp8fg_device_status and skipped.
 *   w       FP32 [T][k], device: gate weights.
 *   out     [T][ldo], FP32 or bf16 per out_kind (FP8FG_OUT_F32 or
 *           FP8FG_OUT_BF16; bf16: the FP32 sum
 *           rounded to nearest even).
 *   Each product w*y and each partial sum is an IEEE FP32 operation, in
 *   slot order j = 0..k-1, with no fused multiply-add, so the result does
 *   not depend on the launch.
 *   1 <= k <= 16, N % 8 == 0, ldy >= N, ldo >= N.
 *   Alignment: y and out 16-byte aligned, ldy % 8 == 0,
 *   ldo*sizeof(out) % 16 == 0. T == 0 or N == 0 is a no-op.
 * ------------------------------------------------------------------- */
FP8FG_API int fp8_moe_combine(const void *y, int64_t ldy, int64_t y_rows, const int32_t *dest, const float *w,
                    int64_t T, int k, int64_t N, void *out, int out_kind, int64_t ldo, void *stream);

/* ---------------------------------------------------------------------
 * fp8_grouped_gemm_mx: the MoE expert GEMM of fp8_grouped_gemm (rows
 * already in expert order, i.e. row_index = NULL) for power-of-two scales,
 * on the tensor cores' block-scaled MMA as fp8_gemm_mx.
 *   For each expert e and each row r in [off[e], off[e+1]):
 *       Y[r][:] = fprop(Xq[r], Wq[e])
 *   Xq        E4M3 [n_rows][K] (lda = K), e.g. fp8_quant_1x128_gather_pow2.
 *   sX        FP32 [K/128][ld_sX], ld_sX >= n_rows, powers of two.
 *   expert_offsets, n_experts, Wq, sW (powers of two), N, K, Y, out, ldy:
 *             as fp8_grouped_gemm.
 *   Errors and alignment as fp8_grouped_gemm (malformed offsets are
 *   reported as FP8FG_EDEVICE through fp8fg_device_status).
 * ------------------------------------------------------------------- */
FP8FG_API int fp8_grouped_gemm_mx(const uint8_t *Xq, const float *sX, int64_t ld_sX,
                         const int32_t *expert_offsets, int32_t n_experts, int64_t n_rows,
                         const uint8_t *Wq, const float *sW, int64_t N, int64_t K,
                         void *Y, int out, int64_t ldy, void *stream);

/* ---------------------------------------------------------------------
 * Status and diagnostics (no counterpart on the pages).
 * ------------------------------------------------------------------- */

/* Human-readable name of a status code; never NULL. */
FP8FG_API const char *fp8fg_status_str(int status);

/* Synchronises `stream`, then returns and clears the current device's
 * status word: FP8FG_OK, FP8FG_ETIMEOUT or FP8FG_EDEVICE (or FP8FG_ECUDA if
 * the synchronisation itself failed). */
FP8FG_API int fp8fg_device_status(void *stream);

/* Library version (major*10000 + minor*100 + patch). */
FP8FG_API int fp8fg_version(void);

/* Test hook: when `skip` != 0, the next fp8_gemm_blockscaled, fp8_gemm_mx,
 * fp8_grouped_gemm_mx or fp8_quant_1x128_dual(_pow2) launch on the current
 * device withholds its first operand load (a fp8_grouped_gemm launch
 * clears the request without using it), so the consumers' bounded waits
 * run out and the launch reports FP8FG_ETIMEOUT. One-shot; returns
 * FP8FG_OK. For exercising failure detection without a GPU fault. */
FP8FG_API int fp8fg_test_skip_first_load(int skip);

/* Wait limit of the device-side bounded waits, in nanoseconds (default two
 * seconds). Values below 1e6 are raised to 1e6. Returns FP8FG_OK. */
FP8FG_API int fp8fg_set_wait_limit_ns(int64_t ns);

/* Schedule of fp8_grouped_gemm with rows in expert order (row_index ==
 * NULL); results do not depend on it. Experts with at most `skinny_rows`
 * rows take skinny tiles (0 turns them off; default 32, at most 32), and
 * `skinny_cost_pct` is the SM time of one skinny tile relative to a full
 * tile, in percent (default 100), which sets the share of the SMs the
 * skinny tiles get. Process-wide; read at each launch. Returns FP8FG_OK,
 * or FP8FG_EINVAL (nothing changed) unless 0 <= skinny_rows <= 32 and
 * 1 <= skinny_cost_pct <= 1000. */
FP8FG_API int fp8fg_set_grouped_schedule(int skinny_rows, int skinny_cost_pct);

#ifdef __cplusplus
}
#endif

#endif /* FP8FG_H */
