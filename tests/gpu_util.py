"""Helpers for the GPU parity tests: layout conversion between the library's
scale arrays and the oracle's, and the GEMM tolerance.

GEMM tolerance (per output element), from the arithmetic:
    |C_gpu - C_ref| <= 1e-5 * T  (+ half a bf16 ulp of the larger magnitude
                                   when the output is rounded to bf16)
with T = sum_kb |sA*sB| * sum_k |dec(qa)*dec(qb)| from the oracle. The 1e-5
factor is the bound the benchmark states for the FP32-promoted result; the
bf16 term is the output rounding, which the FP32 bound does not cover (two
FP32 values inside the band can round to neighbouring bf16 values).
"""
import numpy as np

import oracle
from fp8_fine_grained_gb300 import synth

REL_TOL = 1e-5


def bf16_ulp(v):
    """Spacing of bf16 values at |v| (8 significant bits)."""
    v = np.abs(np.asarray(v, np.float64))
    _, e = np.frexp(np.where(v > 0, v, 2.0 ** -126))
    return np.ldexp(1.0, e - 8)


def check_gemm(c_gpu, c_ref, t, bf16_out, what=""):
    g = np.asarray(c_gpu, np.float64)
    r = np.asarray(c_ref, np.float64)
    tol = REL_TOL * np.asarray(t, np.float64)
    if bf16_out:
        tol = tol + 0.5 * bf16_ulp(np.maximum(np.abs(g), np.abs(r)))
    err = np.abs(g - r)
    bad = ~(err <= tol)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError("%s: %d/%d elements outside tolerance; first at %s: gpu=%r ref=%r T=%r" % (
            what, int(bad.sum()), bad.size, tuple(i), g[tuple(i)], r[tuple(i)], float(np.asarray(t)[tuple(i)])))
    return float(np.max(err / np.maximum(np.asarray(t, np.float64), 1e-300))) if err.size else 0.0


def to_np(t):
    import torch
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy()
    return t.cpu().numpy()


def rows_scales(s_gpu, rows):
    """Library scale layout [groups, ld_s] -> oracle layout [rows, groups]."""
    return np.ascontiguousarray(to_np(s_gpu)[:, :rows].T)


def bits(t):
    return synth.bf16_bits(t)


def assert_quant_1x128(x, q, s):
    qo, so = oracle.quant_1x128(bits(x))
    qg = to_np(q)
    sg = rows_scales(s, x.shape[0])
    if not np.array_equal(qg, qo):
        bad = np.argwhere(qg != qo)
        raise AssertionError("1x128 codes differ at %d positions, first %s: gpu %d oracle %d" % (
            len(bad), tuple(bad[0]), qg[tuple(bad[0])], qo[tuple(bad[0])]))
    assert np.array_equal(sg.view(np.uint32), so.view(np.uint32)), "1x128 scales differ"
    return qo, so
