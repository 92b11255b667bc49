"""Exact-rational brute force for tiny cases (pins the oracle from outside).

Written independently of the oracle: E4M3 values come from the bit fields as
Python Fractions, block sums and scale products are exact rationals, and the
one FP32 rounding helper below rounds an exact rational to the nearest FP32
value (ties to even) without going through double.
"""
from fractions import Fraction

import numpy as np


def e4m3_exact(code):
    s = -1 if code & 0x80 else 1
    e = (code >> 3) & 0xF
    m = code & 7
    if e == 15 and m == 7:
        return None  # NaN
    if e == 0:
        return s * Fraction(m, 8) * Fraction(1, 2 ** 6)
    v = (1 + Fraction(m, 8))
    return s * (v * 2 ** (e - 7) if e >= 7 else v / 2 ** (7 - e))


def f32_exact(x):
    """Exact rational value of a float32."""
    return Fraction(float(np.float32(x)))


def round_f32(fr):
    """Nearest float32 to the rational ``fr``, ties to even (no overflow handling)."""
    if fr == 0:
        return np.float32(0.0)
    sign = -1 if fr < 0 else 1
    a = abs(fr)
    # exponent e with 2^e <= a < 2^(e+1)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    elif Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)            # subnormal range has the fixed quantum 2^-149
    quantum = Fraction(2) ** (e - 23)
    n = a / quantum
    lo = n.numerator // n.denominator
    rem = n - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    return np.float32(sign * float(lo * quantum))


def gemm_exact(qa, sa, qb, sb):
    """Exact block sums for per-(row, k-block) scaled operands.

    Returns (P, exact_C, T, fp32_C):
      P[i][j][kb]   exact block sums (Fractions)
      exact_C[i][j] sum_kb P * sa * sb (exact)
      T[i][j]       sum_kb |sa*sb| * sum_k |a*b| (exact)
      fp32_C[i][j]  promotion sequence acc = rn(acc + rn(rn(P) * rn(sa*sb))),
                    kb ascending, each rounding done exactly.
    """
    M, K = qa.shape
    N = qb.shape[0]
    nkb = K // 128
    P = [[[None] * nkb for _ in range(N)] for _ in range(M)]
    ex = [[Fraction(0)] * N for _ in range(M)]
    T = [[Fraction(0)] * N for _ in range(M)]
    c32 = np.zeros((M, N), np.float32)
    for i in range(M):
        for j in range(N):
            acc = np.float32(0.0)
            for kb in range(nkb):
                p = Fraction(0)
                pa = Fraction(0)
                for k in range(kb * 128, kb * 128 + 128):
                    prod = e4m3_exact(int(qa[i, k])) * e4m3_exact(int(qb[j, k]))
                    p += prod
                    pa += abs(prod)
                P[i][j][kb] = p
                sab_exact = f32_exact(sa[i, kb]) * f32_exact(sb[j, kb])
                ex[i][j] += p * sab_exact
                T[i][j] += pa * abs(sab_exact)
                sab32 = round_f32(sab_exact)
                p32 = round_f32(p)
                term = round_f32(Fraction(float(p32)) * Fraction(float(sab32)))
                acc = round_f32(Fraction(float(acc)) + Fraction(float(term)))
            c32[i, j] = acc
    return P, ex, T, c32
