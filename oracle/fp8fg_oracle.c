/*
 * Plain CPU oracle for fine-grained FP8 quantisation and the block-scaled
 * FP8 GEMM.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path links, loads or calls
 * this file; only the tests, the package's smoke check and the bench's CPU
 * baseline leg do. It shares no code, header, table or constant generator
 * with the CUDA kernels.
 *
 * Sources followed (web pages on DeepSeek-V3's FP8 training framework):
 *   [innerforce]  innerforce.co.kr, the paragraph on fine-grained quantization
 *                 (Figure 7(a)): activations are grouped per token per 128
 *                 channels (1x128), weights per 128x128 block; each group's
 *                 maximum absolute value is scaled to FP8's maximum
 *                 representable value. The following paragraph: partial
 *                 sums are promoted and accumulated in FP32.
 *   [yunhecapital 2.2.3]  yunhecapital.com, section 2.2.3 (mixed-precision
 *                 framework for FP8 training): 1x128 group-wise activations,
 *                 128x128 block-wise weights; at each accumulation interval
 *                 the partial results move to FP32 registers on CUDA cores.
 *   [tonho]       tonho.wtf DeepSeek-V3 entry, section "como funciona":
 *                 scale factor computed online, always E4M3, partials
 *                 promoted every 128 elements and summed in FP32; section
 *                 "o que isso custou": activation gradients must not use
 *                 128x128 blocks.
 * E4M3 itself is taken from the OCP 8-bit floating point specification
 * (E4M3 "fn": bias 7, no infinities, NaN = S.1111.111, max finite 448).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - stored scale s = amax/448, quantise multiplies by inv = 448/amax,
 *     both IEEE FP32 divisions rounded to nearest;
 *   - a group whose amax is 0, or whose 448/amax overflows FP32, uses
 *     s = inv = 1;
 *   - rounding into E4M3 is round-to-nearest-even from FP32 in one step,
 *     saturating at +-448; the sign of zero is kept;
 *   - the promotion interval is 128, equal to the scale group width;
 *   - the cross-block FP32 sum runs over blocks in ascending order with a
 *     separate multiply and add (no fused multiply-add).
 *
 * Microscaling variant ([innerforce], the paragraph that relates the
 * fine-grained groups to microscaling formats and to the Blackwell tensor
 * cores that support them; [tonho] "o que isso custou": tensor-core MMA with
 * group scaling is on the wish list, "onde isso aparece hoje": microscaling
 * announced for Blackwell). Microscaling shares one power-of-two scale per
 * group. Reading: the same 1x128 / 128x128 groups, each scale the smallest
 * power of two 2^e (e >= -127) with amax <= 448 * 2^e; amax = 0 gives s = 1.
 * x * 2^-e is exact, so a code is one rounding of x/s into E4M3.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fopenmp -shared -fPIC.
 * -ffp-contract=off matters: the FP32 accumulation below is specified as a
 * rounded product followed by a rounded sum.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <omp.h>

#define ORC_GROUP 128

/* ---------------------------------------------------------------------- */
/* E4M3 codec (OCP FP8 E4M3fn, the format [tonho] names).                  */
/* ---------------------------------------------------------------------- */

/* Value of an E4M3 code, from the bit fields: sign S, exponent E (bias 7),
 * mantissa M. E = 0 is subnormal: 2^-6 * M/8. S.1111.111 is NaN. */
static double e4m3_value(unsigned code)
{
    unsigned s = (code >> 7) & 1u, e = (code >> 3) & 0xFu, m = code & 7u;
    double v;
    if (e == 15u && m == 7u)
        return NAN;
    if (e == 0u)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return s ? -v : v;
}

void orc_e4m3_decode_table(float out[256])
{
    for (unsigned c = 0; c < 256u; ++c)
        out[c] = (float)e4m3_value(c);
}

/* Nearest E4M3 code to a finite FP32 value: round to nearest, ties to the
 * code whose last mantissa bit is 0, magnitudes of 448 and above saturate to
 * 448 (code 0x7E). Implemented as a linear walk over the 127 non-negative
 * finite codes, comparing against the midpoint of each adjacent pair; every
 * midpoint is exact in double. NaN input is outside the contract; it maps to
 * the NaN code so that callers can see it. */
uint8_t orc_e4m3_encode(float v)
{
    uint8_t sign = signbit(v) ? 0x80u : 0x00u;
    double a = fabs((double)v);
    if (isnan(v))
        return (uint8_t)(sign | 0x7Fu);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7Eu);
    for (unsigned c = 0; c < 126u; ++c) {
        double lo = e4m3_value(c), hi = e4m3_value(c + 1u);
        double mid = 0.5 * (lo + hi);
        if (a < mid)
            return (uint8_t)(sign | c);
        if (a == mid)
            return (uint8_t)(sign | ((c & 1u) ? c + 1u : c));
    }
    return (uint8_t)(sign | 0x7Eu);
}

void orc_e4m3_encode_array(const float *v, int64_t n, uint8_t *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_e4m3_encode(v[i]);
}

/* ---------------------------------------------------------------------- */
/* Group scale and quantisation ([innerforce] fine-grained quantization,   */
/* [tonho] "como funciona": online amax scale, E4M3).                      */
/* ---------------------------------------------------------------------- */

static float bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Scale of one group from its amax: the amax is mapped onto 448.
 * s is the dequantisation multiplier stored beside the codes, inv the
 * quantisation multiplier. */
void orc_group_scale(float amax, float *s, float *inv)
{
    float i;
    if (amax == 0.0f) {
        *s = 1.0f;
        *inv = 1.0f;
        return;
    }
    i = 448.0f / amax;
    if (isinf(i)) {
        *s = 1.0f;
        *inv = 1.0f;
        return;
    }
    *s = amax / 448.0f;
    *inv = i;
}

/* Power-of-two scale of one group (the microscaling variant): the smallest
 * s = 2^e, e >= -127, with amax <= 448 * s; inv = 1/s. Both are exact.
 * frexpf gives amax = f * 2^x with f in [0.5, 1), so amax * 2^-(x-9) lies in
 * [256, 512): e is x-9, or x-8 when that product exceeds 448. */
void orc_group_scale_pow2(float amax, float *s, float *inv)
{
    int x, e;
    if (amax == 0.0f) {
        *s = 1.0f;
        *inv = 1.0f;
        return;
    }
    (void)frexpf(amax, &x);
    e = x - 9;
    if (ldexpf(amax, -e) > 448.0f)
        e += 1;
    if (e < -127)
        e = -127;
    *s = ldexpf(1.0f, e);
    *inv = ldexpf(1.0f, -e);
}

typedef void (*scale_rule_fn)(float, float *, float *);

/* rule 0: s = amax/448 (the pages' method); rule 1: power of two */
static scale_rule_fn scale_rule(int rule)
{
    return rule ? orc_group_scale_pow2 : orc_group_scale;
}

/* One element: a single FP32 product by inv, then one rounding into E4M3. */
static uint8_t quantise_one(float x, float inv)
{
    float y = x * inv;
    return orc_e4m3_encode(y);
}

/* 1x128 tiles: per row, per group of 128 consecutive columns.
 * x: bf16 bits [rows][cols]; q: codes [rows][cols]; s: scales [rows][cols/128].
 * cols must be a multiple of 128. */
void orc_quant_1x128_rule(const uint16_t *x, int64_t rows, int64_t cols,
                          uint8_t *q, float *s, int rule)
{
    int64_t groups = cols / ORC_GROUP;
    scale_rule_fn group_scale = scale_rule(rule);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t g = 0; g < groups; ++g) {
            const uint16_t *xg = x + r * cols + g * ORC_GROUP;
            float amax = 0.0f, sc, inv;
            for (int k = 0; k < ORC_GROUP; ++k) {
                float a = fabsf(bf16_to_f32(xg[k]));
                if (a > amax)
                    amax = a;
            }
            group_scale(amax, &sc, &inv);
            s[r * groups + g] = sc;
            for (int k = 0; k < ORC_GROUP; ++k)
                q[r * cols + g * ORC_GROUP + k] = quantise_one(bf16_to_f32(xg[k]), inv);
        }
    }
}

/* 128x1 tiles along the row (token) dimension, output transposed: the
 * operands of the weight-gradient GEMM, which contracts over tokens.
 * x: bf16 bits [rows][cols]; qT: codes [cols][rows]; s: scales
 * [rows/128][cols]. rows must be a multiple of 128. */
void orc_quant_128x1_t_rule(const uint16_t *x, int64_t rows, int64_t cols,
                            uint8_t *qT, float *s, int rule)
{
    int64_t groups = rows / ORC_GROUP;
    scale_rule_fn group_scale = scale_rule(rule);
#pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < cols; ++c) {
        for (int64_t g = 0; g < groups; ++g) {
            float amax = 0.0f, sc, inv;
            for (int k = 0; k < ORC_GROUP; ++k) {
                float a = fabsf(bf16_to_f32(x[(g * ORC_GROUP + k) * cols + c]));
                if (a > amax)
                    amax = a;
            }
            group_scale(amax, &sc, &inv);
            s[g * cols + c] = sc;
            for (int k = 0; k < ORC_GROUP; ++k) {
                int64_t r = g * ORC_GROUP + k;
                qT[c * rows + r] = quantise_one(bf16_to_f32(x[r * cols + c]), inv);
            }
        }
    }
}

/* 128x128 blocks ([innerforce]: per 128 input channels per 128 output
 * channels). w: bf16 bits [N][K]; q: codes [N][K]; s: scales [N/128][K/128].
 * N and K must be multiples of 128. */
void orc_quant_128x128_rule(const uint16_t *w, int64_t N, int64_t K,
                            uint8_t *q, float *s, int rule)
{
    int64_t nb = N / ORC_GROUP, kb = K / ORC_GROUP;
    scale_rule_fn group_scale = scale_rule(rule);
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t bi = 0; bi < nb; ++bi) {
        for (int64_t bj = 0; bj < kb; ++bj) {
            float amax = 0.0f, sc, inv;
            for (int i = 0; i < ORC_GROUP; ++i)
                for (int j = 0; j < ORC_GROUP; ++j) {
                    float a = fabsf(bf16_to_f32(w[(bi * ORC_GROUP + i) * K + bj * ORC_GROUP + j]));
                    if (a > amax)
                        amax = a;
                }
            group_scale(amax, &sc, &inv);
            s[bi * kb + bj] = sc;
            for (int i = 0; i < ORC_GROUP; ++i)
                for (int j = 0; j < ORC_GROUP; ++j) {
                    int64_t o = (bi * ORC_GROUP + i) * K + bj * ORC_GROUP + j;
                    q[o] = quantise_one(bf16_to_f32(w[o]), inv);
                }
        }
    }
}

/* The pages' scale rule (rule 0) under the original names. */
void orc_quant_1x128(const uint16_t *x, int64_t rows, int64_t cols, uint8_t *q, float *s)
{
    orc_quant_1x128_rule(x, rows, cols, q, s, 0);
}

void orc_quant_128x1_t(const uint16_t *x, int64_t rows, int64_t cols, uint8_t *qT, float *s)
{
    orc_quant_128x1_t_rule(x, rows, cols, qT, s, 0);
}

void orc_quant_128x128(const uint16_t *w, int64_t N, int64_t K, uint8_t *q, float *s)
{
    orc_quant_128x128_rule(w, N, K, q, s, 0);
}

/* ---------------------------------------------------------------------- */
/* Block-scaled GEMM with promotion every 128 K ([innerforce] increased-   */
/* precision accumulation; [yunhecapital 2.2.3]; [tonho] "como funciona"). */
/* ---------------------------------------------------------------------- */

/* C[i][j] = sum over k-blocks kb of (sa[i][kb] * sb[j][kb]) * P[i][j][kb],
 * P[i][j][kb] = sum over k in block kb of dec(qa[i][k]) * dec(qb[j][k]).
 *
 * Both operands are K-contiguous with one scale per (row, k-block); a
 * 128x128-block operand passes its block scale repeated for each of its
 * rows. The block sum P is formed in double, where it is exact in any order:
 * every E4M3 value is an integer multiple of 2^-9 of magnitude at most 448,
 * so a product is an integer multiple of 2^-18 below 2^18 and a sum of 128
 * of them needs fewer than 53 bits. Promotion then rounds P to FP32 and
 * accumulates in FP32, blocks ascending:
 *     acc = acc + fl32( fl32(P) * fl32(sa * sb) ).
 *
 * Outputs, for the selected rows (rows == NULL selects all M):
 *   c       FP32 result as above                      [nsel][N]
 *   c_exact sum of P * (sa * sb) in double             [nsel][N] (may be NULL)
 *   tol     sum of |sa*sb| * sum |dec(qa) dec(qb)|     [nsel][N] (may be NULL)
 * qa: [M][K]; sa: [M][K/128]; qb: [N][K]; sb: [N][K/128]; K % 128 == 0. */
void orc_gemm_blockscaled(const uint8_t *qa, const float *sa,
                          const uint8_t *qb, const float *sb,
                          int64_t M, int64_t N, int64_t K,
                          const int64_t *rows, int64_t nsel,
                          float *c, double *c_exact, double *tol)
{
    double dec[256];
    int64_t nkb = K / ORC_GROUP;
    if (rows == NULL)
        nsel = M;
    for (unsigned v = 0; v < 256u; ++v)
        dec[v] = e4m3_value(v);

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t t = 0; t < nsel; ++t) {
        int64_t i = rows ? rows[t] : t;
        const uint8_t *a = qa + i * K;
        for (int64_t j = 0; j < N; ++j) {
            const uint8_t *b = qb + j * K;
            float acc = 0.0f;
            double ex = 0.0, tl = 0.0;
            for (int64_t kb = 0; kb < nkb; ++kb) {
                double p = 0.0, pabs = 0.0;
                float sab, pf, term;
                for (int64_t k = kb * ORC_GROUP; k < (kb + 1) * ORC_GROUP; ++k) {
                    double prod = dec[a[k]] * dec[b[k]];
                    p += prod;
                    pabs += fabs(prod);
                }
                sab = sa[i * nkb + kb] * sb[j * nkb + kb];
                pf = (float)p;
                term = pf * sab;
                acc = acc + term;
                ex += p * ((double)sa[i * nkb + kb] * (double)sb[j * nkb + kb]);
                tl += pabs * fabs((double)sa[i * nkb + kb] * (double)sb[j * nkb + kb]);
            }
            c[t * N + j] = acc;
            if (c_exact)
                c_exact[t * N + j] = ex;
            if (tol)
                tol[t * N + j] = tl;
        }
    }
}

/* FP32 -> bf16 bits, round to nearest even (finite inputs). */
void orc_f32_to_bf16(const float *v, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) {
        uint32_t u;
        memcpy(&u, &v[i], sizeof u);
        if ((u & 0x7F800000u) == 0x7F800000u) { /* inf / NaN: truncate */
            out[i] = (uint16_t)(u >> 16);
            continue;
        }
        out[i] = (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
    }
}

/*
 * MoE combine: the output of token t is the gate-weighted sum of the rows
 * its k routed experts produced for it,
 *     out[t][n] = sum_{j < k} w[t][j] * y[dest[t][j]][n],
 * the MoE layer's definition, with the expert rows dispatched in FP8 and
 * returned in bf16 ([innerforce], the mixed-precision framework paragraph:
 * activations are cached and dispatched in FP8; [yunhecapital 2.2.2] and
 * [tonho] "como funciona": 8 of 256 routed experts per token). The pages fix
 * no precision for the combine. Reading: y is bf16 (the experts' output
 * format), each product w*y and each partial sum an IEEE FP32 operation in
 * slot order j = 0, 1, ..., k-1 (no fused multiply-add), slots with
 * dest < 0 skipped, then the FP32 sum rounded to bf16 (nearest even) or
 * kept in FP32 when out_f32 is set.
 *   y    bf16 bits [rows][ldy]; dest int32 [T][k]; w FP32 [T][k]
 *   out  bf16 bits [T][N] (out_f32 = 0) or FP32 [T][N] (out_f32 = 1)
 */
void orc_moe_combine(const uint16_t *y, int64_t ldy, const int32_t *dest, const float *w, int64_t T, int k,
                     int64_t N, void *out, int out_f32)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t n = 0; n < N; ++n) {
            float acc = 0.0f;
            for (int j = 0; j < k; ++j) {
                const int32_t d = dest[t * k + j];
                if (d < 0)
                    continue;
                uint32_t u = (uint32_t)y[(int64_t)d * ldy + n] << 16;
                float v;
                memcpy(&v, &u, sizeof v);
                const float prod = w[t * k + j] * v;
                acc = acc + prod;
            }
            if (out_f32)
                ((float *)out)[t * N + n] = acc;
            else
                orc_f32_to_bf16(&acc, 1, (uint16_t *)out + t * N + n);
        }
    }
}

int orc_version(void) { return 1; }

/* Threads the following OpenMP regions of this library use (n >= 1); for
 * timing the oracle on one core against all of them. */
void orc_set_num_threads(int n)
{
    if (n >= 1)
        omp_set_num_threads(n);
}

/* Threads an OpenMP parallel region of this library uses. */
int orc_num_threads(void)
{
    int n = 1;
#pragma omp parallel
    {
#pragma omp single
        n = omp_get_num_threads();
    }
    return n;
}
