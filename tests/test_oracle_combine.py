"""Pins of the oracle's MoE combine (CPU): out[t] = sum_j w[t, j] *
y[dest[t, j]], FP32 products and sums in slot order, slots with dest < 0
skipped, bf16 (nearest even) or FP32 output.

The combine follows the MoE layer's definition (each token's output is the
gate-weighted sum of its routed experts' outputs; yunhecapital.com 2.2.2,
tonho.wtf "como funciona": 8 of 256 routed experts per token), with the
expert rows dispatched in FP8 and returned in bf16 (innerforce.co.kr, the
mixed-precision framework paragraph: activations cached and dispatched in
FP8). The pins below do not restate the formula: they check cases whose
result is fixed independently (a copy, skipped slots, exact integer sums in
any slot order, an FP32 error bound against exact rational arithmetic, and
the bf16 rounding against torch's conversion)."""
from fractions import Fraction

import numpy as np
import torch

import oracle


def bf16_bits(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(
        np.uint16)


def bits_to_f32(b):
    return (np.asarray(b, np.uint32) << 16).view(np.float32)


def test_single_slot_weight_one_is_a_copy():
    rng = np.random.default_rng(0)
    y = bf16_bits(rng.standard_normal((50, 96)).astype(np.float32) * 10)
    dest = rng.permutation(50)[:40].astype(np.int32).reshape(40, 1)
    out = oracle.moe_combine(y, dest, np.ones((40, 1), np.float32))
    assert np.array_equal(out, y[dest[:, 0]])


def test_skipped_slots_contribute_nothing():
    rng = np.random.default_rng(1)
    y = bf16_bits(rng.standard_normal((30, 64)).astype(np.float32))
    dest = rng.integers(0, 30, (20, 4)).astype(np.int32)
    w = rng.standard_normal((20, 4)).astype(np.float32)
    full = oracle.moe_combine(y, dest, w, out_f32=True)
    d2 = dest.copy()
    d2[:, 3] = -1                    # drop the last slot: equals a 3-slot combine
    assert np.array_equal(oracle.moe_combine(y, d2, w, out_f32=True),
                          oracle.moe_combine(y, dest[:, :3], w[:, :3], out_f32=True))
    d3 = np.full_like(dest, -1)      # no slot at all: zero
    assert np.all(oracle.moe_combine(y, d3, w, out_f32=True) == 0.0)
    assert not np.array_equal(full, oracle.moe_combine(y, d2, w, out_f32=True))


def test_exact_integer_sums_in_any_slot_order():
    """Integer rows (|y| <= 64, exact in bf16) and power-of-two weights: every
    product and partial sum is exact in FP32, so the result is the exact sum,
    whatever the slot order."""
    rng = np.random.default_rng(2)
    y = bf16_bits(rng.integers(-64, 65, (40, 48)).astype(np.float32))
    T, k = 25, 8
    dest = rng.integers(0, 40, (T, k)).astype(np.int32)
    w = np.ldexp(1.0, rng.integers(-3, 4, (T, k))).astype(np.float32) * rng.choice([-1, 1], (T, k))
    out = oracle.moe_combine(y, dest, w, out_f32=True)
    yf = bits_to_f32(y).astype(np.int64)
    for t in range(T):
        for n in range(48):
            exact = sum(Fraction(float(w[t, j])) * int(yf[dest[t, j], n]) for j in range(k))
            assert Fraction(float(out[t, n])) == exact
    perm = rng.permutation(k)
    assert np.array_equal(out, oracle.moe_combine(y, dest[:, perm], w[:, perm], out_f32=True))


def test_fp32_result_within_the_recursive_summation_bound():
    """General inputs: |out - exact| <= k * 2^-24 * sum_j |w_j y_j| (k rounded
    products and sums, each with relative error at most 2^-24, to first
    order), the exact value computed with rationals."""
    rng = np.random.default_rng(3)
    y = bf16_bits(rng.standard_normal((60, 32)).astype(np.float32) * np.exp(rng.standard_normal((60, 1))))
    T, k = 30, 8
    dest = rng.integers(0, 60, (T, k)).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    out = oracle.moe_combine(y, dest, w, out_f32=True)
    yf = bits_to_f32(y)
    for t in range(T):
        for n in range(32):
            terms = [Fraction(float(w[t, j])) * Fraction(float(yf[dest[t, j], n])) for j in range(k)]
            exact = sum(terms)
            bound = k * Fraction(1, 2 ** 24) * sum(abs(v) for v in terms) * Fraction(101, 100)
            assert abs(Fraction(float(out[t, n])) - exact) <= bound


def test_bf16_output_is_the_rounded_fp32_result():
    rng = np.random.default_rng(4)
    y = bf16_bits(rng.standard_normal((50, 80)).astype(np.float32))
    dest = rng.integers(-1, 50, (33, 8)).astype(np.int32)
    w = rng.random((33, 8)).astype(np.float32)
    f32 = oracle.moe_combine(y, dest, w, out_f32=True)
    b16 = oracle.moe_combine(y, dest, w)
    assert np.array_equal(b16, bf16_bits(f32))
