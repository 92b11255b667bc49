"""Pins for the CPU oracle: checks against what the pages and the mathematics
fix, never against the oracle's own formulas retyped.

- the E4M3 code points of the OCP format the pages name (golden fixture);
- the codec against two library routines (torch float8_e4m3fn, ml_dtypes);
- the scale rule's closed forms and the exactness on FP8-representable input;
- the tile shapes (1x128, 128x1 transposed, 128x128) through invariants that a
  wrong group membership breaks;
- the GEMM against exact-rational brute force and closed forms (constant
  operands, a permutation weight that exposes a transposed operand, a single
  non-zero block that isolates one promotion interval).
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from tests import _brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_bits_of(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bits_to_f32(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def torch_e4m3(v):
    """Library rounding to E4M3 (RNE). torch does not saturate, so clamp first."""
    t = torch.from_numpy(np.asarray(v, np.float32)).clamp(-448.0, 448.0)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def finite_codes():
    return np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)


# ------------------------------------------------------------------ codec ----

def test_decode_golden_ocp_values():
    dec = oracle.e4m3_decode_table()
    n = 0
    with open(os.path.join(GOLDEN, "e4m3_ocp.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            code, val = line.split()
            code = int(code, 16)
            if val == "nan":
                assert np.isnan(dec[code])
            else:
                assert dec[code] == np.float32(float(val)), (hex(code), dec[code], val)
                if val.startswith("-"):
                    assert np.signbit(dec[code])
            n += 1
    assert n >= 15
    # NaN only at S.1111.111; largest finite 448
    assert np.isnan(dec).sum() == 2
    assert np.nanmax(dec) == 448.0 and np.nanmin(dec) == -448.0


def test_decode_matches_torch_exhaustive():
    dec = oracle.e4m3_decode_table()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    assert np.array_equal(np.isnan(dec), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(dec[ok].view(np.uint32), ref[ok].view(np.uint32))


def test_decode_matches_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    dec = oracle.e4m3_decode_table()
    ref = np.arange(256, dtype=np.uint8).view(ml.float8_e4m3fn).astype(np.float32)
    ok = ~np.isnan(ref)
    assert np.array_equal(np.isnan(dec), np.isnan(ref))
    assert np.array_equal(dec[ok].view(np.uint32), ref[ok].view(np.uint32))


def test_decode_against_bitfield_brute_force():
    dec = oracle.e4m3_decode_table()
    for c in range(256):
        v = _brute.e4m3_exact(c)
        if v is None:
            assert np.isnan(dec[c])
        else:
            assert Fraction(float(dec[c])) == v


def test_encode_roundtrip_every_finite_code():
    dec = oracle.e4m3_decode_table()
    codes = finite_codes()
    assert np.array_equal(oracle.e4m3_encode(dec[codes]), codes)


def test_encode_all_bf16_values_times_scales_vs_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = bits_to_f32(bits)
    x = x[np.isfinite(x)]
    rng = np.random.default_rng(0)
    factors = [1.0, 448.0, 1.0 / 448.0, 3.5, 2.0 ** -20, 2.0 ** 20, 448.0 / 3.0]
    factors += list(rng.uniform(1e-3, 1e3, 4))
    for f in factors:
        with np.errstate(over="ignore"):
            y = (x * np.float32(f)).astype(np.float32)
        y = y[np.isfinite(y)]
        got = oracle.e4m3_encode(y)
        assert np.array_equal(got, torch_e4m3(y)), f


def test_encode_midpoints_and_neighbours_vs_torch():
    dec = oracle.e4m3_decode_table().astype(np.float64)
    pos = np.array([dec[c] for c in range(0x7F)])
    mids = (pos[:-1] + pos[1:]) / 2
    vals = []
    for m in mids:
        m32 = np.float32(m)
        assert float(m32) == m  # every midpoint is exact in FP32
        vals += [np.nextafter(m32, np.float32(-1)), m32, np.nextafter(m32, np.float32(1e9))]
    vals = np.array(vals, np.float32)
    vals = np.concatenate([vals, -vals, np.array([448, 449, 463.99, 464, 464.01, 480, 1e30, 3e38], np.float32)])
    assert np.array_equal(oracle.e4m3_encode(vals), torch_e4m3(vals))
    # ties go to the even code: 464 (between 448 and the absent 480) -> 448,
    # 2^-10 (between 0 and 2^-9) -> 0, 17/16*2^-6... checked by torch above
    assert oracle.e4m3_encode(np.array([464.0, 2.0 ** -10, -2.0 ** -10], np.float32)).tolist() == [0x7E, 0x00, 0x80]


def test_encode_saturates_and_keeps_sign_of_zero():
    v = np.array([448.0, 1e6, -1e6, 0.0, -0.0, 1e-30, -1e-30], np.float32)
    assert oracle.e4m3_encode(v).tolist() == [0x7E, 0x7E, 0xFE, 0x00, 0x80, 0x00, 0x80]


# ------------------------------------------------------------- scale rule ----

def test_scale_of_power_of_two_multiples_of_448_is_exact():
    for e in range(-40, 40):
        amax = np.float32(448.0 * 2.0 ** e)
        s, inv = oracle.group_scale(amax)
        assert s == np.float32(2.0 ** e) and inv == np.float32(2.0 ** -e)


def test_scale_degenerate_groups():
    assert oracle.group_scale(0.0) == (1.0, 1.0)
    # 448/amax overflows FP32 for the smallest bf16 subnormals: treated like zero
    tiny = bits_to_f32(np.array([1], np.uint16))[0]
    with np.errstate(over="ignore"):
        assert not np.isfinite(np.float32(448.0) / tiny)
    assert oracle.group_scale(tiny) == (1.0, 1.0)
    x = np.zeros((1, 128), np.float32)
    x[0, 5] = -tiny
    q, s = oracle.quant_1x128(bf16_bits_of(x))
    assert s[0, 0] == 1.0 and q[0, 5] == 0x80 and q[0, 0] == 0x00


def test_amax_element_maps_to_448():
    rng = np.random.default_rng(1)
    for _ in range(20):
        x = rng.standard_normal((4, 256)).astype(np.float32) * np.float32(rng.uniform(1e-6, 1e6))
        b = bf16_bits_of(x)
        q, s = oracle.quant_1x128(b)
        xf = bits_to_f32(b)
        for r in range(4):
            for g in range(2):
                seg = xf[r, g * 128:(g + 1) * 128]
                k = int(np.argmax(np.abs(seg)))
                assert q[r, g * 128 + k] & 0x7F == 0x7E
                assert s[r, g] == np.float32(np.float32(np.abs(seg).max()) / np.float32(448.0))


def test_fp8_representable_groups_quantise_to_their_own_codes():
    """A group of E4M3 values scaled by 2^e whose amax is 448*2^e is
    reproduced exactly: codes equal the source codes and s = 2^e."""
    dec = oracle.e4m3_decode_table()
    rng = np.random.default_rng(2)
    codes = finite_codes()
    for e in (-8, 0, 3):
        src = rng.choice(codes, size=(3, 256))
        src[:, 0] = 0x7E
        src[:, 128] = 0xFE
        x = dec[src] * np.float32(2.0 ** e)
        q, s = oracle.quant_1x128(bf16_bits_of(x))
        # -0 and +0 both decode to zero; compare values, and codes off zero
        assert np.array_equal(dec[q], dec[src])
        nz = dec[src] != 0
        assert np.array_equal(q[nz], src[nz])
        assert np.all(s == np.float32(2.0 ** e))


def test_quantisation_error_bound():
    """|x - s*dec(q)| <= s * (half an E4M3 ulp of x*inv) + rounding of the scale."""
    dec = oracle.e4m3_decode_table().astype(np.float64)
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((64, 512)) * np.exp(rng.standard_normal(512))).astype(np.float32)
    b = bf16_bits_of(x)
    q, s = oracle.quant_1x128(b)
    xf = bits_to_f32(b).astype(np.float64)
    sr = np.repeat(s, 128, axis=1).astype(np.float64)
    y = np.abs(xf) / sr                       # x * inv up to FP32 rounding
    e = np.floor(np.log2(np.maximum(y, 2.0 ** -6)))
    half_ulp = 0.5 * 2.0 ** (e - 3)           # 3 mantissa bits; subnormal quantum 2^-9
    err = np.abs(xf - sr * dec[q])
    assert np.all(err <= sr * half_ulp * (1 + 1e-6) + np.abs(xf) * 2.0 ** -22)


# ------------------------------------------------------------- tile shapes ----

def test_1x128_groups_are_per_row_and_per_128_columns():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((8, 512)).astype(np.float32)
    b = bf16_bits_of(x)
    q0, s0 = oracle.quant_1x128(b)
    # a new maximum in (row 3, group 2) changes only that group
    b2 = b.copy()
    b2[3, 2 * 128 + 7] = bf16_bits_of(np.array([1000.0], np.float32))[0]
    q1, s1 = oracle.quant_1x128(b2)
    diff_s = np.argwhere(s0 != s1)
    assert diff_s.tolist() == [[3, 2]]
    dq = np.argwhere(q0 != q1)
    assert set(map(tuple, dq[:, :1].tolist())) == {(3,)}
    assert dq[:, 1].min() >= 256 and dq[:, 1].max() < 384
    # row permutation commutes with quantisation (a token's tiles are its own)
    perm = rng.permutation(8)
    qp, sp = oracle.quant_1x128(b[perm])
    assert np.array_equal(qp, q0[perm]) and np.array_equal(sp, s0[perm])


def test_transposed_quant_equals_rowwise_of_transpose():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((384, 200)) * np.exp(rng.standard_normal(200))).astype(np.float32)
    b = bf16_bits_of(x)
    qT, sT = oracle.quant_128x1_t(b)
    # materialise the transpose (200 rows of 384 tokens) and quantise per row
    bt = np.ascontiguousarray(b.T)
    q_ref, s_ref = oracle.quant_1x128(bt)
    assert np.array_equal(qT, q_ref)
    assert np.array_equal(sT, s_ref.T)


def test_128x128_block_membership_and_transpose():
    rng = np.random.default_rng(6)
    w = (rng.standard_normal((256, 384)) * 0.02).astype(np.float32)
    b = bf16_bits_of(w)
    q, s = oracle.quant_128x128(b)
    # transpose of the weight: blocks are square, so codes transpose and
    # the block-scale grid transposes
    qt, st = oracle.quant_128x128(np.ascontiguousarray(b.T))
    assert np.array_equal(qt, q.T) and np.array_equal(st, s.T)
    # when every row of a block holds the block's maximum, the 128x128 block
    # quantises exactly like 1x128 tiles of its rows
    w2 = w.copy()
    for bi in range(2):
        for bj in range(3):
            w2[bi * 128:(bi + 1) * 128, bj * 128] = 0.5 + 0.25 * bi + 0.125 * bj
    b2 = bf16_bits_of(w2)
    q2, s2 = oracle.quant_128x128(b2)
    q1, s1 = oracle.quant_1x128(b2)
    assert np.array_equal(q2, q1)
    assert np.array_equal(np.repeat(s2, 128, axis=0), s1)
    # a single large element raises exactly one block's scale
    b3 = b.copy()
    b3[200, 300] = bf16_bits_of(np.array([64.0], np.float32))[0]
    _, s3 = oracle.quant_128x128(b3)
    assert np.argwhere(s3 != s).tolist() == [[1, 2]]
    assert s3[1, 2] == np.float32(64.0 / 448.0)


# ------------------------------------------- power-of-two scale variant ----
# The microscaling variant keeps the pages' groups but shares one power-of-two
# scale per group: s = 2^e, the smallest with amax <= 448 * 2^e (e >= -127).

def test_pow2_scale_hand_derived_values():
    # (amax, e) worked out by hand from "smallest e with amax <= 448 * 2^e"
    cases = [
        (448.0, 0),                      # exactly 448 * 2^0
        (450.0, 1),                      # next bf16 above 448
        (224.0, -1),                     # 448 * 2^-1 = 224 covers it, 112 does not
        (1.0, -8),                       # 448/256 = 1.75 >= 1 > 448/512
        (1.75, -8),                      # 448 * 2^-8 = 1.75 exactly
        (1.7578125, -7),                 # the bf16 just above 1.75
        (0.01, -15),                     # 448 * 2^-16 = 0.00684 < 0.01 <= 0.01367
        (3.3895313892515355e38, 120),    # largest finite bf16, 1.9921875 * 2^127
        (1.75 * 2.0 ** -119, -127),      # 448 * 2^-127 exactly
        (2.0 ** -120, -127),             # below 448 * 2^-128: clamped to -127
        (2.0 ** -133, -127),             # smallest bf16 subnormal
    ]
    for amax, e in cases:
        s, inv = oracle.group_scale(np.float32(amax), pow2=True)
        assert Fraction(float(s)) == Fraction(2) ** e, (amax, e, s)
        assert Fraction(float(inv)) == Fraction(2) ** -e, (amax, e, inv)
    assert oracle.group_scale(0.0, pow2=True) == (1.0, 1.0)


def test_pow2_scale_is_the_smallest_power_covering_amax():
    rng = np.random.default_rng(11)
    bits = rng.integers(1, 0x7F80, size=4000, dtype=np.int64).astype(np.uint16)  # finite positive bf16
    for a in bits_to_f32(bits):
        s, inv = oracle.group_scale(a, pow2=True)
        fa, fs = Fraction(float(a)), Fraction(float(s))
        m, x = np.frexp(float(s))
        assert m == 0.5 and Fraction(float(inv)) * fs == 1
        assert fa <= 448 * fs
        e = x - 1
        assert e == -127 or fa > 448 * fs / 2


def test_pow2_codes_are_one_rounding_of_x_over_s():
    """code = RNE(x / s) with s = 2^e; x/s <= 448 so nothing saturates."""
    rng = np.random.default_rng(12)
    x = (rng.standard_normal((6, 512)) * np.exp(3 * rng.standard_normal(512))).astype(np.float32)
    x[0, :128] = 0.0
    x[1, 128:256] *= np.float32(1e-30)
    b = bf16_bits_of(x)
    q, s = oracle.quant_1x128(b, pow2=True)
    xf = bits_to_f32(b).astype(np.float64)
    sr = np.repeat(s, 128, axis=1).astype(np.float64)
    y = xf / sr                                   # exact: division by a power of two
    assert np.all(np.abs(y) <= 448.0)
    assert np.array_equal(q, torch_e4m3(y.astype(np.float32)))
    assert s[0, 0] == 1.0 and np.all(q[0, :128] == 0)


def test_pow2_fp8_representable_groups_roundtrip():
    dec = oracle.e4m3_decode_table()
    rng = np.random.default_rng(13)
    codes = finite_codes()
    for e in (-20, -8, 0, 5):
        src = rng.choice(codes, size=(3, 256))
        src[:, 3] = 0x7E
        src[:, 200] = 0xFE
        x = dec[src] * np.float32(2.0 ** e)
        q, s = oracle.quant_1x128(bf16_bits_of(x), pow2=True)
        assert np.array_equal(dec[q], dec[src])
        assert np.all(s == np.float32(2.0 ** e))
    # an amax one bf16 step above 448 * 2^e moves the scale to 2^(e+1)
    x = dec[rng.choice(codes, size=(1, 128))].astype(np.float32)
    x[0, 7] = 450.0
    _, s = oracle.quant_1x128(bf16_bits_of(x), pow2=True)
    assert s[0, 0] == 2.0


def test_pow2_layouts_agree_with_rowwise():
    rng = np.random.default_rng(14)
    x = (rng.standard_normal((256, 384)) * np.exp(rng.standard_normal(384))).astype(np.float32)
    b = bf16_bits_of(x)
    qT, sT = oracle.quant_128x1_t(b, pow2=True)
    q_ref, s_ref = oracle.quant_1x128(np.ascontiguousarray(b.T), pow2=True)
    assert np.array_equal(qT, q_ref) and np.array_equal(sT, s_ref.T)
    qb, sb = oracle.quant_128x128(b, pow2=True)
    xf = bits_to_f32(b)
    for bi in range(2):
        for bj in range(3):
            blk = xf[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128]
            s, inv = oracle.group_scale(np.abs(blk).max(), pow2=True)
            assert sb[bi, bj] == s
            assert np.array_equal(qb[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128],
                                  torch_e4m3(blk.astype(np.float64) / float(s)))


# ------------------------------------------------------------------- GEMM ----

def _rand_codes(rng, shape):
    return rng.choice(finite_codes(), size=shape).astype(np.uint8)


def test_gemm_matches_exact_rational_brute_force():
    rng = np.random.default_rng(7)
    M, N, K = 3, 4, 256
    qa = _rand_codes(rng, (M, K))
    qb = _rand_codes(rng, (N, K))
    sa = rng.uniform(1e-3, 10, (M, K // 128)).astype(np.float32)
    sb = rng.uniform(1e-3, 10, (N, K // 128)).astype(np.float32)
    c, ce, t = oracle.gemm_rowscaled(qa, sa, qb, sb)
    P, ex, T, c32 = _brute.gemm_exact(qa, sa, qb, sb)
    for i in range(M):
        for j in range(N):
            assert Fraction(float(t[i, j])) == pytest.approx(T[i][j], rel=1e-15)
            assert abs(Fraction(float(ce[i, j])) - ex[i][j]) <= T[i][j] * Fraction(1, 2 ** 50)
            # FP32 promotion sequence, every rounding exact
            assert c[i, j].view(np.uint32) == c32[i, j].view(np.uint32)
            # and the result is within the oracle's stated bound of the exact value
            assert abs(Fraction(float(c[i, j])) - ex[i][j]) <= (K // 128) * Fraction(1, 2 ** 23) * T[i][j]


def test_gemm_block_sum_exact_at_extremes():
    """Extreme codes: the double block sum must still be exact (43-bit sums)."""
    M, N, K = 2, 2, 128
    qa = np.full((M, K), 0x7E, np.uint8)
    qb = np.full((N, K), 0x7E, np.uint8)
    qa[0, ::2] = 0x01     # 2^-9 alternating with 448
    qb[1, 1::2] = 0x81    # -2^-9
    ones = np.ones((M, 1), np.float32)
    c, ce, t = oracle.gemm_rowscaled(qa, ones, qb, ones[:N])
    P, ex, T, c32 = _brute.gemm_exact(qa, ones, qb, ones[:N])
    for i in range(M):
        for j in range(N):
            assert Fraction(float(ce[i, j])) == ex[i][j]
            assert c[i, j] == c32[i, j]


def test_gemm_constant_operands_closed_form():
    """X = a everywhere, W = w everywhere: every code is 0x7E, s = a/448 and
    w/448, so C = K * 448^2 * (a/448)*(w/448) = K*a*w up to scale rounding."""
    M, N, K = 5, 256, 384
    a, wv = 1.75, -0.0234375
    xq, sx = oracle.quant_1x128(bf16_bits_of(np.full((M, K), a, np.float32)))
    wq, sw = oracle.quant_128x128(bf16_bits_of(np.full((N, K), wv, np.float32)))
    assert np.all(xq == 0x7E) and np.all(wq == 0xFE)
    c, ce, t = oracle.fprop(xq, sx, wq, sw)
    assert np.allclose(c, K * a * wv, rtol=4e-7, atol=0)


def test_gemm_permutation_weight_exposes_transposition():
    """W[n, k] = 1 iff k = pi(n): fprop gives Y[m, n] = dequant(X)[m, pi(n)];
    dgrad (dX = dY W) gives dX[m, k] = dequant(dY)[m, pi^-1(k)]."""
    rng = np.random.default_rng(8)
    M, N = 7, 256
    pi = rng.permutation(N)
    assert np.any(pi[pi] != np.arange(N))  # not an involution
    w = np.zeros((N, N), np.float32)
    w[np.arange(N), pi] = 1.0
    wq, sw = oracle.quant_128x128(bf16_bits_of(w))
    x = (rng.standard_normal((M, N)) * 3).astype(np.float32)
    xq, sx = oracle.quant_1x128(bf16_bits_of(x))
    dec = oracle.e4m3_decode_table()
    xdq = dec[xq].astype(np.float64) * np.repeat(sx, 128, axis=1)
    y, _, _ = oracle.fprop(xq, sx, wq, sw)
    assert np.allclose(y, xdq[:, pi], rtol=1e-6, atol=0)
    dx, _, _ = oracle.dgrad(xq, sx, wq, sw)
    inv = np.argsort(pi)
    assert np.allclose(dx, xdq[:, inv], rtol=1e-6, atol=0)


def test_wgrad_token_permutation_closed_form():
    """X[m, k] = 1 iff m = sigma(k): dW = dY^T X gives dW[n, k] = dequant(dY)[sigma(k), n]
    with dY quantised in groups of 128 tokens."""
    rng = np.random.default_rng(9)
    M, K, N = 256, 256, 3 * 128
    sigma = rng.permutation(M)
    x = np.zeros((M, K), np.float32)
    x[sigma, np.arange(K)] = 1.0
    dy = (rng.standard_normal((M, N)) * 1e-3).astype(np.float32)
    xqT, sxT = oracle.quant_128x1_t(bf16_bits_of(x))
    dyqT, sdyT = oracle.quant_128x1_t(bf16_bits_of(dy))
    dec = oracle.e4m3_decode_table()
    dy_dq = (dec[dyqT].astype(np.float64) * np.repeat(sdyT.T, 128, axis=1)).T  # [M, N]
    dw, _, _ = oracle.wgrad(dyqT, sdyT, xqT, sxT)
    assert dw.shape == (N, K)
    assert np.allclose(dw, dy_dq[sigma, :].T, rtol=1e-6, atol=0)


def test_single_nonzero_block_isolates_one_promotion_interval():
    """Only k-block 2 of 4 is non-zero: C equals that block's scaled sum, and
    changing another block's scale changes nothing."""
    rng = np.random.default_rng(10)
    M, N, K = 4, 3, 512
    qa = np.zeros((M, K), np.uint8)
    qb = _rand_codes(rng, (N, K))
    qa[:, 256:384] = _rand_codes(rng, (M, 128))
    sa = rng.uniform(0.1, 2, (M, 4)).astype(np.float32)
    sb = rng.uniform(0.1, 2, (N, 4)).astype(np.float32)
    c, _, _ = oracle.gemm_rowscaled(qa, sa, qb, sb)
    c1, _, _ = oracle.gemm_rowscaled(qa[:, 256:384], sa[:, 2:3], qb[:, 256:384], sb[:, 2:3])
    assert np.array_equal(c, c1)
    sa2 = sa.copy()
    sa2[:, [0, 1, 3]] *= 7
    c2, _, _ = oracle.gemm_rowscaled(qa, sa2, qb, sb)
    assert np.array_equal(c, c2)


def test_gemm_row_selection_matches_full():
    rng = np.random.default_rng(11)
    qa = _rand_codes(rng, (20, 256))
    qb = _rand_codes(rng, (9, 256))
    sa = rng.uniform(0.1, 2, (20, 2)).astype(np.float32)
    sb = rng.uniform(0.1, 2, (9, 2)).astype(np.float32)
    c, ce, t = oracle.gemm_rowscaled(qa, sa, qb, sb)
    rows = np.array([19, 0, 7, 7])
    cs, ces, ts = oracle.gemm_rowscaled(qa, sa, qb, sb, rows=rows)
    assert np.array_equal(cs, c[rows]) and np.array_equal(ts, t[rows])


# ---------------------------------------------------------------- grouped ----

def test_grouped_reduces_to_dense_per_expert_and_handles_empty_experts():
    rng = np.random.default_rng(12)
    T, K, N, E = 50, 256, 256, 5
    x = rng.standard_normal((T, K)).astype(np.float32)
    xq, sx = oracle.quant_1x128(bf16_bits_of(x))
    w = (rng.standard_normal((E, N, K)) * 0.02).astype(np.float32)
    wq = np.empty((E, N, K), np.uint8)
    sw = np.empty((E, N // 128, K // 128), np.float32)
    for e in range(E):
        wq[e], sw[e] = oracle.quant_128x128(bf16_bits_of(w[e]))
    counts = [0, 17, 0, 40, 3]        # experts 0 and 2 empty
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    row_index = np.concatenate([np.sort(rng.choice(T, c, replace=False)) for c in counts]).astype(np.int32)
    y, _, _ = oracle.grouped(xq, sx, row_index, off, wq, sw)
    assert y.shape == (60, N)
    for e in range(E):
        r0, r1 = off[e], off[e + 1]
        if r0 == r1:
            continue
        ye, _, _ = oracle.fprop(xq[row_index[r0:r1]], sx[row_index[r0:r1]], wq[e], sw[e])
        assert np.array_equal(y[r0:r1], ye)
    # permuting rows inside an expert permutes the outputs
    perm = np.arange(60)
    perm[17:57] = 17 + rng.permutation(40)
    y2, _, _ = oracle.grouped(xq, sx, row_index[perm], off, wq, sw)
    assert np.array_equal(y2, y[perm])
    # sampled rows equal the full result
    rows = np.array([59, 0, 20, 18])
    ys, _, _ = oracle.grouped(xq, sx, row_index, off, wq, sw, rows=rows)
    assert np.array_equal(ys, y[rows])


def test_bf16_output_rounding_matches_torch():
    rng = np.random.default_rng(13)
    v = (rng.standard_normal(100000) * np.exp(rng.standard_normal(100000) * 5)).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.to_bf16_bits(v), ref)


def test_page_constants_fixture():
    consts = {}
    with open(os.path.join(GOLDEN, "page_constants.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                k, v = line.split()
                consts[k] = int(v)
    assert consts["activation_group_rows"] == 1 and consts["activation_group_cols"] == oracle.GROUP
    assert consts["weight_block_rows"] == consts["weight_block_cols"] == oracle.GROUP
    assert consts["promotion_interval"] == oracle.GROUP
    assert consts["e4m3_max"] == oracle.E4M3_MAX == float(np.nanmax(oracle.e4m3_decode_table()))


def test_results_do_not_depend_on_the_thread_count():
    # the oracle's OpenMP loops split rows and output elements only, so one
    # thread and all threads must give the same bytes, scales and sums
    rng = np.random.default_rng(21)
    x = (rng.standard_normal((256, 512)) * np.exp(rng.standard_normal(512))).astype(np.float32)
    w = (rng.standard_normal((384, 512)) * 0.02).astype(np.float32)
    xb, wb = bf16_bits_of(x), bf16_bits_of(w)
    n = oracle.num_threads()

    def run():
        xq, sx = oracle.quant_1x128(xb)
        xt, st = oracle.quant_128x1_t(xb)
        wq, sw = oracle.quant_128x128(wb)
        c, ce, t = oracle.fprop(xq, sx, wq, sw)
        return [xq, sx, xt, st, wq, sw, c, ce, t]

    many = run()
    oracle.set_num_threads(1)
    try:
        one = run()
    finally:
        oracle.set_num_threads(n)
    for a, b in zip(many, one):
        assert a.dtype == b.dtype and np.array_equal(a.view(np.uint8), b.view(np.uint8))
