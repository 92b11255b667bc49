"""CPU oracle for fine-grained FP8 quantisation and the block-scaled FP8 GEMM.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the package smoke check
and by the bench's CPU-baseline leg, never by the product path. It shares no
code with the CUDA library and does not import it.

The arithmetic lives in ``fp8fg_oracle.c`` (plain C, IEEE, no FMA
contraction); this module marshals numpy arrays and holds the layout-only
wrappers that express dgrad, wgrad and the grouped (MoE) GEMM in terms of the
one block-scaled GEMM definition:

    C[i, j] = sum_kb  (sa[i, kb] * sb[j, kb]) * sum_{k in kb} dec(qa[i, k]) * dec(qb[j, k])

with both operands K-contiguous and one scale per (row, 128-wide k-block).

Sources: innerforce.co.kr, paragraph on fine-grained quantization (Figure
7(a)) and the following one on increased-precision accumulation;
yunhecapital.com section 2.2.3; tonho.wtf DeepSeek-V3 entry, sections "como
funciona" (1x128 / 128x128, online scale, E4M3, promotion every 128
elements) and "o que isso custou" (activation gradients are not quantised in
128x128 blocks).
"""
import ctypes
import os

import numpy as np

from . import build as _build

GROUP = 128
E4M3_MAX = 448.0

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        L.orc_e4m3_decode_table.argtypes = [P]
        L.orc_e4m3_encode.argtypes = [ctypes.c_float]
        L.orc_e4m3_encode.restype = ctypes.c_uint8
        L.orc_e4m3_encode_array.argtypes = [P, I64, P]
        L.orc_group_scale.argtypes = [ctypes.c_float, P, P]
        L.orc_group_scale_pow2.argtypes = [ctypes.c_float, P, P]
        L.orc_quant_1x128_rule.argtypes = [P, I64, I64, P, P, ctypes.c_int]
        L.orc_quant_128x1_t_rule.argtypes = [P, I64, I64, P, P, ctypes.c_int]
        L.orc_quant_128x128_rule.argtypes = [P, I64, I64, P, P, ctypes.c_int]
        L.orc_gemm_blockscaled.argtypes = [P, P, P, P, I64, I64, I64, P, I64, P, P, P]
        L.orc_f32_to_bf16.argtypes = [P, I64, P]
        L.orc_moe_combine.argtypes = [P, I64, P, P, I64, ctypes.c_int, I64, P, ctypes.c_int]
        L.orc_num_threads.restype = ctypes.c_int
        L.orc_set_num_threads.argtypes = [ctypes.c_int]
        _lib = L
    return _lib


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- codec ----

def e4m3_decode_table():
    """float32[256]: value of every E4M3 code (OCP E4M3fn; NaN at 0x7F/0xFF)."""
    out = np.empty(256, np.float32)
    lib().orc_e4m3_decode_table(_ptr(out))
    return out


def e4m3_encode(v):
    """Round float32 values to E4M3 codes: nearest, ties to even, saturating."""
    v = _c(v, np.float32)
    out = np.empty(v.shape, np.uint8)
    lib().orc_e4m3_encode_array(_ptr(v), v.size, _ptr(out))
    return out


def group_scale(amax, pow2=False):
    """(s, inv) for one group with the given amax (float32 scalars).

    pow2=False: the pages' rule, s = amax/448. pow2=True: the microscaling
    variant, s = the smallest power of two 2^e (e >= -127) with
    amax <= 448 * s."""
    s = np.zeros(1, np.float32)
    inv = np.zeros(1, np.float32)
    fn = lib().orc_group_scale_pow2 if pow2 else lib().orc_group_scale
    fn(ctypes.c_float(float(np.float32(amax))), _ptr(s), _ptr(inv))
    return s[0], inv[0]


# ------------------------------------------------------------ quantise ----

def quant_1x128(x_bits, pow2=False):
    """Per-row 1x128 quantisation.

    x_bits: uint16 bf16 bit patterns [rows, cols], cols % 128 == 0.
    pow2 selects the power-of-two scale rule (see group_scale).
    Returns (q uint8 [rows, cols], s float32 [rows, cols/128]).
    """
    x = _c(x_bits, np.uint16)
    rows, cols = x.shape
    assert cols % GROUP == 0
    q = np.empty((rows, cols), np.uint8)
    s = np.empty((rows, cols // GROUP), np.float32)
    lib().orc_quant_1x128_rule(_ptr(x), rows, cols, _ptr(q), _ptr(s), 1 if pow2 else 0)
    return q, s


def quant_128x1_t(x_bits, pow2=False):
    """Groups of 128 rows per column, output transposed (pow2: see group_scale).

    x_bits: uint16 [rows, cols], rows % 128 == 0.
    Returns (qT uint8 [cols, rows], s float32 [rows/128, cols]).
    """
    x = _c(x_bits, np.uint16)
    rows, cols = x.shape
    assert rows % GROUP == 0
    qT = np.empty((cols, rows), np.uint8)
    s = np.empty((rows // GROUP, cols), np.float32)
    lib().orc_quant_128x1_t_rule(_ptr(x), rows, cols, _ptr(qT), _ptr(s), 1 if pow2 else 0)
    return qT, s


def quant_128x128(w_bits, pow2=False):
    """128x128 block quantisation (pow2: see group_scale).

    w_bits: uint16 [N, K], both multiples of 128.
    Returns (q uint8 [N, K], s float32 [N/128, K/128]).
    """
    w = _c(w_bits, np.uint16)
    N, K = w.shape
    assert N % GROUP == 0 and K % GROUP == 0
    q = np.empty((N, K), np.uint8)
    s = np.empty((N // GROUP, K // GROUP), np.float32)
    lib().orc_quant_128x128_rule(_ptr(w), N, K, _ptr(q), _ptr(s), 1 if pow2 else 0)
    return q, s


# ---------------------------------------------------------------- GEMM ----

def gemm_rowscaled(qa, sa, qb, sb, rows=None, want_exact=True):
    """The block-scaled GEMM definition with per-(row, k-block) scales.

    qa uint8 [M, K], sa float32 [M, K/128], qb uint8 [N, K], sb float32
    [N, K/128]. ``rows`` selects rows of A (default: all).
    Returns (C float32, C_exact float64 or None, T float64 or None), each
    [len(rows), N]; T is the per-element tolerance base
    sum_kb |sa*sb| * sum_k |dec(qa)*dec(qb)|.
    """
    qa = _c(qa, np.uint8)
    qb = _c(qb, np.uint8)
    sa = _c(sa, np.float32)
    sb = _c(sb, np.float32)
    M, K = qa.shape
    N, K2 = qb.shape
    assert K == K2 and K % GROUP == 0
    assert sa.shape == (M, K // GROUP) and sb.shape == (N, K // GROUP)
    if rows is None:
        sel = None
        nsel = M
    else:
        sel = _c(rows, np.int64)
        assert sel.ndim == 1 and (sel.size == 0 or (sel.min() >= 0 and sel.max() < M))
        nsel = sel.size
    c = np.empty((nsel, N), np.float32)
    ce = np.empty((nsel, N), np.float64) if want_exact else None
    tl = np.empty((nsel, N), np.float64) if want_exact else None
    if nsel and N:
        lib().orc_gemm_blockscaled(_ptr(qa), _ptr(sa), _ptr(qb), _ptr(sb), M, N, K,
                                   _ptr(sel), nsel, _ptr(c), _ptr(ce), _ptr(tl))
    return c, ce, tl


def expand_block_scales(s_blocks, n_rows):
    """Per-row scales of a 128x128-block operand: row j uses block row j//128.

    s_blocks float32 [ceil(n_rows/128), K/128] -> float32 [n_rows, K/128].
    """
    s_blocks = np.asarray(s_blocks, np.float32)
    return np.repeat(s_blocks, GROUP, axis=0)[:n_rows]


def fprop(xq, sx, wq, sw, rows=None, want_exact=True):
    """Y = X W^T. X 1x128-scaled: xq [M, K], sx [M, K/128].
    W 128x128-scaled: wq [N, K], sw [N/128, K/128]."""
    return gemm_rowscaled(xq, sx, wq, expand_block_scales(sw, wq.shape[0]), rows, want_exact)


def dgrad(dyq, sdy, wq, sw, rows=None, want_exact=True):
    """dX = dY W, contraction over the layer's output channels N.

    dY is 1x128-scaled along N: dyq [M, N], sdy [M, N/128].
    W is the forward weight [N, K] with its 128x128 scales sw [N/128, K/128];
    its transpose W^T [K, N] carries the transposed block scales."""
    wqT = np.ascontiguousarray(np.asarray(wq, np.uint8).T)
    swT = np.ascontiguousarray(np.asarray(sw, np.float32).T)
    return gemm_rowscaled(dyq, sdy, wqT, expand_block_scales(swT, wqT.shape[0]), rows, want_exact)


def wgrad(dyqT, sdyT, xqT, sxT, rows=None, want_exact=True):
    """dW = dY^T X, contraction over tokens M.

    Both operands are quantised in groups of 128 tokens and stored
    transposed: dyqT [N, M] with scales sdyT [M/128, N]; xqT [K, M] with
    scales sxT [M/128, K] (the layout of quant_128x1_t)."""
    return gemm_rowscaled(dyqT, np.ascontiguousarray(np.asarray(sdyT).T), xqT,
                          np.ascontiguousarray(np.asarray(sxT).T), rows, want_exact)


def grouped(xq, sx, row_index, expert_offsets, wq, sw, rows=None, want_exact=True):
    """MoE expert GEMM: for expert e and every row r in
    [expert_offsets[e], expert_offsets[e+1]), Y[r] = fprop(X[row_index[r]], W_e).

    xq [T, K], sx [T, K/128] (1x128, one quantisation per token);
    row_index int [R]; expert_offsets int [E+1]; wq [E, N, K]; sw [E, N/128, K/128].
    ``rows`` selects output rows r (default: all R). Returns arrays [len(rows), N].
    """
    row_index = np.asarray(row_index, np.int64)
    off = np.asarray(expert_offsets, np.int64)
    E = off.size - 1
    R = int(off[-1])
    N = wq.shape[1]
    sel = np.arange(R, dtype=np.int64) if rows is None else np.asarray(rows, np.int64)
    c = np.zeros((sel.size, N), np.float32)
    ce = np.zeros((sel.size, N), np.float64)
    tl = np.zeros((sel.size, N), np.float64)
    expert_of = np.searchsorted(off, sel, side="right") - 1
    for e in range(E):
        pick = np.nonzero(expert_of == e)[0]
        if pick.size == 0:
            continue
        toks = row_index[sel[pick]]
        ci, cei, tli = fprop(xq[toks], sx[toks], wq[e], sw[e], None, want_exact)
        c[pick] = ci
        if want_exact:
            ce[pick] = cei
            tl[pick] = tli
    return (c, ce, tl) if want_exact else (c, None, None)


def num_threads():
    """Threads the oracle's OpenMP regions run on."""
    return int(lib().orc_num_threads())


def set_num_threads(n):
    """Run the oracle's OpenMP regions on n threads from now on."""
    lib().orc_set_num_threads(int(n))


def to_bf16_bits(c):
    """float32 -> bf16 bit patterns (round to nearest even)."""
    c = _c(c, np.float32)
    out = np.empty(c.shape, np.uint16)
    lib().orc_f32_to_bf16(_ptr(c), c.size, _ptr(out))
    return out


def moe_combine(y_bits, dest, w, out_f32=False):
    """MoE combine: out[t] = sum_{j<k} w[t, j] * y[dest[t, j]] (FP32 products
    and sums in slot order, no FMA; slots with dest < 0 skipped), rounded to
    bf16 bits (or FP32 with out_f32). y_bits uint16 bf16 bit patterns
    [rows, N]; dest int32 [T, k]; w float32 [T, k]."""
    y = _c(y_bits, np.uint16)
    d = _c(dest, np.int32)
    ww = _c(w, np.float32)
    T, k = d.shape
    assert ww.shape == (T, k)
    N = y.shape[1]
    assert d.size == 0 or d.max() < y.shape[0]
    out = np.empty((T, N), np.float32 if out_f32 else np.uint16)
    if T and N:
        lib().orc_moe_combine(_ptr(y), N, _ptr(d), _ptr(ww), T, k, N, _ptr(out), 1 if out_f32 else 0)
    return out
