"""Fine-grained FP8 quantisation and block-scaled FP8 GEMM for GB300 (sm_103a).

Thin ctypes binding over ``libfp8fg.so`` (C ABI declared in
``include/fp8fg.h``). This module only marshals arguments: it takes torch
tensors that live on the GPU, allocates outputs with torch, and passes raw
device pointers, sizes and the current CUDA stream to the library. Every step
of the computation runs in the library's CUDA kernels; there is no fallback.
If the library is missing or fails to load, every call raises.

Entry points (same names as the C ABI):
    fp8_quant_1x128(x, transpose=False)     -> (q, scales)
    fp8_quant_128x128(w)                    -> (q, scales)
    fp8_quant_128x128_dual(w)               -> (q, scales, qT, scalesT)
    fp8_gemm_blockscaled(mode, a, sa, b, sb, out_dtype) -> C
    fp8_grouped_gemm(xq, sx, row_index, expert_offsets, wq, sw, n_rows, out_dtype) -> Y
plus the convenience wrappers fprop / dgrad / wgrad and device_status().
"""
import ctypes
import os

FPROP, DGRAD, WGRAD = 0, 1, 2
OUT_F32, OUT_BF16 = 0, 1

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfp8fg.so")
_lib = None


class Fp8fgError(RuntimeError):
    def __init__(self, code, what):
        self.code = code
        super().__init__("%s: %s (status %d)" % (what, status_str(code) if _lib else "?", code))


def lib():
    """Load libfp8fg.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                "libfp8fg.so is not built; run `python fp8_fine_grained_gb300/build.py` "
                "(or __graft_entry__.build()) first")
        L = ctypes.CDLL(LIB_PATH)
        P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.fp8_quant_1x128.argtypes = [P, I64, I64, I64, P, I64, P, I64, I32, P]
        L.fp8_quant_1x128_gather.argtypes = [P, I64, I64, I64, P, I64, P, I64, P, I64, P]
        L.fp8_quant_1x128_dual.argtypes = [P, I64, I64, I64, P, I64, P, I64, P, I64, P, I64, P]
        L.fp8_quant_128x128.argtypes = [P, I64, I64, I64, P, I64, P, P]
        L.fp8_quant_128x128_dual.argtypes = [P, I64, I64, I64, P, I64, P, P, I64, P, P]
        L.fp8_quant_128x128_dual_pow2.argtypes = [P, I64, I64, I64, P, I64, P, P, I64, P, P]
        L.fp8_quant_1x128_pow2.argtypes = L.fp8_quant_1x128.argtypes
        L.fp8_quant_1x128_gather_pow2.argtypes = L.fp8_quant_1x128_gather.argtypes
        L.fp8_quant_1x128_dual_pow2.argtypes = L.fp8_quant_1x128_dual.argtypes
        L.fp8_quant_128x128_pow2.argtypes = L.fp8_quant_128x128.argtypes
        L.fp8_quant_1x128_scatter.argtypes = [P, I64, I64, I64, P, I32, I64, P, I64, P, I64, P]
        L.fp8_quant_1x128_scatter_pow2.argtypes = L.fp8_quant_1x128_scatter.argtypes
        L.fp8_gemm_mx.argtypes = [I32, P, P, I64, I64, P, P, I64, I64, I64, I64, I64, P, I32, I64, P]
        L.fp8_grouped_gemm_mx.argtypes = [P, P, I64, P, ctypes.c_int32, I64, P, P, I64, I64, P, I32, I64, P]
        L.fp8_gemm_blockscaled.argtypes = [I32, P, P, I64, I64, P, P, I64, I64, I64, I64, I64, P, I32, I64, P]
        L.fp8_gemm_blockscaled_e4m3.argtypes = [I32, P, P, I64, I64, P, P, I64, I64, I64, I64, I64, P, I64, P, I64, P]
        L.fp8_grouped_gemm.argtypes = [P, P, I64, I64, P, P, ctypes.c_int32, I64, P, P, I64, I64, P, I32, I64, P]
        L.fp8_moe_combine.argtypes = [P, I64, I64, P, P, I64, I32, I64, P, I32, I64, P]
        L.fp8fg_status_str.argtypes = [I32]
        L.fp8fg_status_str.restype = ctypes.c_char_p
        L.fp8fg_device_status.argtypes = [P]
        L.fp8fg_version.argtypes = []
        L.fp8fg_test_skip_first_load.argtypes = [I32]
        L.fp8fg_set_wait_limit_ns.argtypes = [I64]
        L.fp8fg_set_grouped_schedule.argtypes = [I32, I32]
        for f in ("fp8_quant_1x128", "fp8_quant_128x128", "fp8_gemm_blockscaled", "fp8_grouped_gemm",
                  "fp8fg_device_status", "fp8fg_version", "fp8fg_test_skip_first_load",
                  "fp8fg_set_wait_limit_ns", "fp8fg_set_grouped_schedule"):
            getattr(L, f).restype = I32
        _lib = L
    return _lib


def status_str(code):
    return lib().fp8fg_status_str(int(code)).decode()


def _check(rc, what):
    if rc != 0:
        raise Fp8fgError(rc, what)


def _torch():
    import torch
    return torch


def _stream(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _layout(t, name):
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("%s must be a 2-D row-major tensor (unit inner stride)" % name)


def _on_gpu(*named):
    for t, name in named:
        if t is not None and not t.is_cuda:
            raise ValueError("%s must be a CUDA tensor" % name)


def _rowmajor(t, name):
    _layout(t, name)
    _on_gpu((t, name))


def _pad(n, m):
    return (n + m - 1) // m * m


def _dtype(t, dtype, name):
    if t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))


def _at_least(t, rows, cols, name):
    """A 2-D tensor must cover [rows, cols] (the kernels read or write that
    extent through raw pointers, so a smaller tensor would be overrun)."""
    if t.dim() != 2 or t.shape[0] < rows or t.shape[1] < cols:
        raise ValueError("%s must cover [%d, %d], got %s" % (name, rows, cols, tuple(t.shape)))


def _quant_out(q, scales, q_shape, s_rows, s_cols, qn="q", sn="scales"):
    """Caller-supplied outputs of a quantiser: E4M3 bytes of q_shape and
    FP32 scales covering [s_rows, s_cols]."""
    torch = _torch()
    _dtype(q, torch.uint8, qn)
    _dtype(scales, torch.float32, sn)
    _layout(q, qn)
    _layout(scales, sn)
    _at_least(q, q_shape[0], q_shape[1], qn)
    _at_least(scales, s_rows, s_cols, sn)


def _gemm_operands(mode, a, sa, b, sb):
    """Dtypes and extents of a block-scaled GEMM's operands; returns (M, N, K).

    FPROP: a [M,K], sa [K/128, >=M], b [N,K], sb [N/128, K/128]
    DGRAD: a [M,K], sa [K/128, >=M], b [K,N], sb [K/128, N/128]
    WGRAD: a [M,K], sa [K/128, >=M], b [N,K], sb [K/128, >=N]
    """
    torch = _torch()
    if mode not in (FPROP, DGRAD, WGRAD):
        raise ValueError("mode must be FPROP, DGRAD or WGRAD")
    for t, n in ((a, "a"), (b, "b"), (sa, "sa"), (sb, "sb")):
        _layout(t, n)
    _dtype(a, torch.uint8, "a")
    _dtype(b, torch.uint8, "b")
    _dtype(sa, torch.float32, "sa")
    _dtype(sb, torch.float32, "sb")
    M, K = a.shape
    if mode == DGRAD:
        if b.shape[0] != K:
            raise ValueError("dgrad: b must be [K, N] with K = a.shape[1] = %d, got %s" % (K, tuple(b.shape)))
        N = b.shape[1]
    else:
        if b.shape[1] != K:
            raise ValueError("b must be [N, K] with K = a.shape[1] = %d, got %s" % (K, tuple(b.shape)))
        N = b.shape[0]
    kb = K // 128
    _at_least(sa, kb, M, "sa")
    if mode == FPROP:
        _at_least(sb, N // 128, kb, "sb")
    elif mode == DGRAD:
        _at_least(sb, kb, N // 128, "sb")
    else:
        _at_least(sb, kb, N, "sb")
    return M, N, K


def _gemm_out(c, M, N):
    _layout(c, "c")
    if tuple(c.shape) != (M, N):
        raise ValueError("c must be [%d, %d], got %s" % (M, N, tuple(c.shape)))


def _grouped_operands(xq, sx, expert_offsets, wq, sw, n_rows, row_index):
    """Dtypes and extents of a grouped GEMM's operands; returns (T, E, N, K)."""
    torch = _torch()
    _layout(xq, "xq")
    _layout(sx, "sx")
    _dtype(xq, torch.uint8, "xq")
    _dtype(sx, torch.float32, "sx")
    _dtype(wq, torch.uint8, "wq")
    _dtype(sw, torch.float32, "sw")
    if expert_offsets.dtype != torch.int32 or (row_index is not None and row_index.dtype != torch.int32):
        raise ValueError("row_index and expert_offsets must be int32")
    if not ((row_index is None or row_index.is_contiguous()) and expert_offsets.is_contiguous()
            and wq.is_contiguous() and sw.is_contiguous()):
        raise ValueError("row_index, expert_offsets, wq, sw must be contiguous")
    if wq.dim() != 3:
        raise ValueError("wq must be [E, N, K]")
    T, K = xq.shape
    E, N, K2 = wq.shape
    if K2 != K or xq.stride(0) != K:
        raise ValueError("xq must be [T, K] contiguous with the experts' K")
    if n_rows < 0:
        raise ValueError("n_rows must be >= 0")
    if expert_offsets.dim() != 1 or expert_offsets.numel() != E + 1:
        raise ValueError("expert_offsets must hold E + 1 = %d entries" % (E + 1))
    if tuple(sw.shape) != (E, N // 128, K // 128):
        raise ValueError("sw must be [%d, %d, %d], got %s" % (E, N // 128, K // 128, tuple(sw.shape)))
    _at_least(sx, K // 128, T, "sx")
    if row_index is None:
        if T < n_rows:
            raise ValueError("without a row index xq and sx must hold n_rows = %d rows" % n_rows)
    elif row_index.dim() != 1 or row_index.numel() < n_rows:
        raise ValueError("row_index must hold n_rows = %d entries" % n_rows)
    return T, E, N, K


# ------------------------------------------------------------- quantise ----

def fp8_quant_1x128(x, transpose=False, q=None, scales=None, stream=None, pow2=False):
    """E4M3 codes and FP32 scales of a bf16 matrix in 1x128 tiles.

    pow2=True selects the power-of-two scale rule (fp8_quant_1x128_pow2).

    transpose=False: x [rows, cols] grouped per row along cols (cols % 128 == 0);
        returns q uint8 [rows, cols], scales float32 [cols/128, ld_s>=rows].
    transpose=True: groups of 128 rows per column, output transposed
        (rows % 128 == 0); returns q uint8 [cols, rows], scales [rows/128, ld_s>=cols].
    """
    torch = _torch()
    _layout(x, "x")
    if x.dtype != torch.bfloat16:
        raise ValueError("x must be bfloat16")
    rows, cols = x.shape
    if not transpose:
        if q is None:
            q = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
        if scales is None:
            scales = torch.empty((cols // 128, _pad(max(rows, 1), 4)), dtype=torch.float32, device=x.device)
        _quant_out(q, scales, (rows, cols), cols // 128, rows)
    else:
        if q is None:
            q = torch.empty((cols, rows), dtype=torch.uint8, device=x.device)
        if scales is None:
            scales = torch.empty((rows // 128, _pad(max(cols, 1), 4)), dtype=torch.float32, device=x.device)
        _quant_out(q, scales, (cols, rows), rows // 128, cols)
    _on_gpu((x, "x"), (q, "q"), (scales, "scales"))
    fn = lib().fp8_quant_1x128_pow2 if pow2 else lib().fp8_quant_1x128
    rc = fn(_ptr(x), rows, cols, x.stride(0), _ptr(q), q.stride(0), _ptr(scales),
            scales.stride(0), 1 if transpose else 0, _stream(stream))
    _check(rc, "fp8_quant_1x128_pow2" if pow2 else "fp8_quant_1x128")
    return q, scales


def fp8_quant_1x128_dual(x, q=None, scales=None, qT=None, scalesT=None, stream=None, pow2=False):
    """Both layouts of fp8_quant_1x128 from one read of x (rows and cols
    multiples of 128): returns (q, scales, qT, scalesT), equal to
    fp8_quant_1x128(x) and fp8_quant_1x128(x, transpose=True) (with the
    same pow2 choice)."""
    torch = _torch()
    _layout(x, "x")
    if x.dtype != torch.bfloat16:
        raise ValueError("x must be bfloat16")
    rows, cols = x.shape
    dev = x.device
    if q is None:
        q = torch.empty((rows, cols), dtype=torch.uint8, device=dev)
    if scales is None:
        scales = torch.empty((cols // 128, _pad(max(rows, 1), 4)), dtype=torch.float32, device=dev)
    if qT is None:
        qT = torch.empty((cols, rows), dtype=torch.uint8, device=dev)
    if scalesT is None:
        scalesT = torch.empty((rows // 128, _pad(max(cols, 1), 4)), dtype=torch.float32, device=dev)
    _quant_out(q, scales, (rows, cols), cols // 128, rows)
    _quant_out(qT, scalesT, (cols, rows), rows // 128, cols, "qT", "scalesT")
    _on_gpu((x, "x"), (q, "q"), (scales, "scales"), (qT, "qT"), (scalesT, "scalesT"))
    fn = lib().fp8_quant_1x128_dual_pow2 if pow2 else lib().fp8_quant_1x128_dual
    rc = fn(_ptr(x), rows, cols, x.stride(0), _ptr(q), q.stride(0), _ptr(scales),
            scales.stride(0), _ptr(qT), qT.stride(0), _ptr(scalesT), scalesT.stride(0),
            _stream(stream))
    _check(rc, "fp8_quant_1x128_dual_pow2" if pow2 else "fp8_quant_1x128_dual")
    return q, scales, qT, scalesT


def fp8_quant_1x128_gather(x, row_index, q=None, scales=None, stream=None, pow2=False):
    """1x128 quantisation of the rows x[row_index[r]], written in row_index
    order (MoE rows grouped by expert): q uint8 [n_rows, cols], scales
    float32 [cols/128, ld_s>=n_rows]. Equal to gathering the rows of
    fp8_quant_1x128(x); feeds fp8_grouped_gemm with row_index=None."""
    torch = _torch()
    _layout(x, "x")
    if x.dtype != torch.bfloat16:
        raise ValueError("x must be bfloat16")
    if row_index.dtype != torch.int32 or not row_index.is_contiguous():
        raise ValueError("row_index must be contiguous int32")
    n_src, cols = x.shape
    rows = row_index.numel()
    if q is None:
        q = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty((cols // 128, _pad(max(rows, 1), 4)), dtype=torch.float32, device=x.device)
    _quant_out(q, scales, (rows, cols), cols // 128, rows)
    _on_gpu((x, "x"), (row_index, "row_index"), (q, "q"), (scales, "scales"))
    fn = lib().fp8_quant_1x128_gather_pow2 if pow2 else lib().fp8_quant_1x128_gather
    rc = fn(_ptr(x), n_src, cols, x.stride(0), _ptr(row_index), rows, _ptr(q),
            q.stride(0), _ptr(scales), scales.stride(0), _stream(stream))
    _check(rc, "fp8_quant_1x128_gather_pow2" if pow2 else "fp8_quant_1x128_gather")
    return q, scales


def fp8_quant_1x128_scatter(x, dest_index, n_out, q=None, scales=None, stream=None, pow2=False):
    """1x128 quantisation of every row of x, written to its k destination
    rows dest_index[r, :] (int32 [n_src, k]; negative = not written):
    q uint8 [n_out, cols], scales float32 [cols/128, ld_s>=n_out]. Equal to
    fp8_quant_1x128_gather with the inverse index; each row is read once."""
    torch = _torch()
    _layout(x, "x")
    if x.dtype != torch.bfloat16:
        raise ValueError("x must be bfloat16")
    if dest_index.dtype != torch.int32 or not dest_index.is_contiguous() or dest_index.dim() != 2:
        raise ValueError("dest_index must be contiguous int32 [n_src, k]")
    n_src, cols = x.shape
    if dest_index.shape[0] != n_src:
        raise ValueError("dest_index needs one row per source row")
    k = dest_index.shape[1]
    if q is None:
        q = torch.empty((n_out, cols), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty((cols // 128, _pad(max(n_out, 1), 4)), dtype=torch.float32, device=x.device)
    _quant_out(q, scales, (n_out, cols), cols // 128, n_out)
    _on_gpu((x, "x"), (dest_index, "dest_index"), (q, "q"), (scales, "scales"))
    fn = lib().fp8_quant_1x128_scatter_pow2 if pow2 else lib().fp8_quant_1x128_scatter
    rc = fn(_ptr(x), n_src, cols, x.stride(0), _ptr(dest_index), k, n_out, _ptr(q), q.stride(0), _ptr(scales),
            scales.stride(0), _stream(stream))
    _check(rc, "fp8_quant_1x128_scatter_pow2" if pow2 else "fp8_quant_1x128_scatter")
    return q, scales


def fp8_quant_128x128(w, q=None, scales=None, stream=None, pow2=False):
    """E4M3 codes and FP32 scales of a bf16 weight [N, K] in 128x128 blocks.
    A 3-D weight [E, N, K] (MoE experts) is quantised as [E*N, K]."""
    torch = _torch()
    shape = w.shape
    w2 = w.reshape(-1, shape[-1]) if w.dim() == 3 else w
    _layout(w2, "w")
    if w.dtype != torch.bfloat16:
        raise ValueError("w must be bfloat16")
    N, K = w2.shape
    if q is None:
        q = torch.empty(shape, dtype=torch.uint8, device=w.device)
    if scales is None:
        scales = torch.empty(tuple(shape[:-2]) + (shape[-2] // 128, K // 128), dtype=torch.float32,
                             device=w.device)
    q2 = q.reshape(-1, K)
    _dtype(q, torch.uint8, "q")
    _dtype(scales, torch.float32, "scales")
    if tuple(q2.shape) != (N, K) or not q2.is_contiguous() or not scales.is_contiguous() \
            or scales.numel() < (N // 128) * (K // 128):
        raise ValueError("q must be %s uint8 and scales hold [N/128, K/128] float32" % (tuple(shape),))
    _on_gpu((w2, "w"), (q, "q"), (scales, "scales"))
    fn = lib().fp8_quant_128x128_pow2 if pow2 else lib().fp8_quant_128x128
    rc = fn(_ptr(w2), N, K, w2.stride(0), _ptr(q2), q2.stride(0), _ptr(scales), _stream(stream))
    _check(rc, "fp8_quant_128x128_pow2" if pow2 else "fp8_quant_128x128")
    return q, scales


def fp8_quant_128x128_dual(w, q=None, scales=None, qT=None, scalesT=None, stream=None, pow2=False):
    """128x128 blocks of a bf16 weight [N, K] and of its transpose from one
    read: returns (q [N, K], scales [N/128, K/128], qT [K, N], scalesT
    [K/128, N/128]), equal to fp8_quant_128x128(w) and
    fp8_quant_128x128(w.t()) (with the same pow2 choice)."""
    torch = _torch()
    _layout(w, "w")
    if w.dim() != 2 or w.dtype != torch.bfloat16:
        raise ValueError("w must be a 2-D bfloat16 tensor")
    N, K = w.shape
    dev = w.device
    q = torch.empty((N, K), dtype=torch.uint8, device=dev) if q is None else q
    scales = torch.empty((N // 128, K // 128), dtype=torch.float32, device=dev) if scales is None else scales
    qT = torch.empty((K, N), dtype=torch.uint8, device=dev) if qT is None else qT
    scalesT = torch.empty((K // 128, N // 128), dtype=torch.float32, device=dev) if scalesT is None else scalesT
    for t, name, dt in ((q, "q", torch.uint8), (qT, "qT", torch.uint8), (scales, "scales", torch.float32),
                        (scalesT, "scalesT", torch.float32)):
        _dtype(t, dt, name)
    _layout(q, "q")
    _layout(qT, "qT")
    _at_least(q, N, K, "q")
    _at_least(qT, K, N, "qT")
    if not scales.is_contiguous() or not scalesT.is_contiguous() or scales.numel() < (N // 128) * (K // 128) \
            or scalesT.numel() < (N // 128) * (K // 128):
        raise ValueError("scales and scalesT must be contiguous and hold [N/128, K/128] float32")
    _on_gpu((w, "w"), (q, "q"), (scales, "scales"), (qT, "qT"), (scalesT, "scalesT"))
    fn = lib().fp8_quant_128x128_dual_pow2 if pow2 else lib().fp8_quant_128x128_dual
    rc = fn(_ptr(w), N, K, w.stride(0), _ptr(q), q.stride(0), _ptr(scales), _ptr(qT), qT.stride(0), _ptr(scalesT),
            _stream(stream))
    _check(rc, "fp8_quant_128x128_dual_pow2" if pow2 else "fp8_quant_128x128_dual")
    return q, scales, qT, scalesT


# ----------------------------------------------------------------- GEMM ----

def _out_code(dtype):
    torch = _torch()
    if dtype == torch.bfloat16:
        return OUT_BF16
    if dtype == torch.float32:
        return OUT_F32
    raise ValueError("output dtype must be bfloat16 or float32")


def fp8_gemm_blockscaled(mode, a, sa, b, sb, out_dtype=None, c=None, stream=None):
    """Block-scaled FP8 GEMM (see include/fp8fg.h for the three modes).

    FPROP: a [M,K] 1x128 + sa [K/128, >=M]; b [N,K] 128x128 + sb [N/128, K/128] -> C [M,N]
    DGRAD: a [M,K] 1x128 + sa [K/128, >=M]; b [K,N] 128x128 + sb [K/128, N/128] -> C [M,N]
    WGRAD: a [M,K] + sa [K/128, >=M]; b [N,K] + sb [K/128, >=N] (both grouped along K) -> C [M,N]
    """
    torch = _torch()
    M, N, K = _gemm_operands(mode, a, sa, b, sb)
    if out_dtype is None:
        out_dtype = torch.float32 if mode == WGRAD else torch.bfloat16
    if c is None:
        c = torch.empty((M, N), dtype=out_dtype, device=a.device)
    _gemm_out(c, M, N)
    _on_gpu((a, "a"), (b, "b"), (sa, "sa"), (sb, "sb"), (c, "c"))
    rc = lib().fp8_gemm_blockscaled(mode, _ptr(a), _ptr(sa), a.stride(0), sa.stride(0), _ptr(b), _ptr(sb),
                                    b.stride(0), sb.stride(0), M, N, K, _ptr(c), _out_code(c.dtype),
                                    c.stride(0), _stream(stream))
    _check(rc, "fp8_gemm_blockscaled")
    return c


def fp8_gemm_mx(mode, a, sa, b, sb, out_dtype=None, c=None, stream=None):
    """fp8_gemm_blockscaled's GEMM for power-of-two scales (the *_pow2
    quantisers' output), with the scales applied by the tensor cores'
    block-scaled MMA; same modes, shapes and layouts."""
    torch = _torch()
    M, N, K = _gemm_operands(mode, a, sa, b, sb)
    if out_dtype is None:
        out_dtype = torch.float32 if mode == WGRAD else torch.bfloat16
    if c is None:
        c = torch.empty((M, N), dtype=out_dtype, device=a.device)
    _gemm_out(c, M, N)
    _on_gpu((a, "a"), (b, "b"), (sa, "sa"), (sb, "sb"), (c, "c"))
    rc = lib().fp8_gemm_mx(mode, _ptr(a), _ptr(sa), a.stride(0), sa.stride(0), _ptr(b), _ptr(sb),
                           b.stride(0), sb.stride(0), M, N, K, _ptr(c), _out_code(c.dtype),
                           c.stride(0), _stream(stream))
    _check(rc, "fp8_gemm_mx")
    return c


def fp8_gemm_blockscaled_e4m3(mode, a, sa, b, sb, c=None, scales=None, stream=None):
    """FPROP or DGRAD with the output quantised in the epilogue: returns
    (C E4M3 [M,N], scales [N/128, ld_s>=M]), equal to fp8_quant_1x128 of
    the bf16 output of fp8_gemm_blockscaled."""
    torch = _torch()
    if mode not in (FPROP, DGRAD):
        raise ValueError("the E4M3 output exists for FPROP and DGRAD only")
    M, N, K = _gemm_operands(mode, a, sa, b, sb)
    if c is None:
        c = torch.empty((M, N), dtype=torch.uint8, device=a.device)
    if scales is None:
        scales = torch.empty((N // 128, _pad(max(M, 1), 4)), dtype=torch.float32, device=a.device)
    _dtype(c, torch.uint8, "c")
    _gemm_out(c, M, N)
    _dtype(scales, torch.float32, "scales")
    _layout(scales, "scales")
    _at_least(scales, N // 128, M, "scales")
    _on_gpu((a, "a"), (b, "b"), (sa, "sa"), (sb, "sb"), (c, "c"), (scales, "scales"))
    rc = lib().fp8_gemm_blockscaled_e4m3(mode, _ptr(a), _ptr(sa), a.stride(0), sa.stride(0), _ptr(b), _ptr(sb),
                                         b.stride(0), sb.stride(0), M, N, K, _ptr(c), c.stride(0), _ptr(scales),
                                         scales.stride(0), _stream(stream))
    _check(rc, "fp8_gemm_blockscaled_e4m3")
    return c, scales


def fprop(xq, sx, wq, sw, out_dtype=None, c=None, stream=None):
    """Y = X W^T from fp8_quant_1x128(X) and fp8_quant_128x128(W)."""
    return fp8_gemm_blockscaled(FPROP, xq, sx, wq, sw, out_dtype, c, stream)


def dgrad(dyq, sdy, wq, sw, out_dtype=None, c=None, stream=None):
    """dX = dY W from fp8_quant_1x128(dY) and the forward weight's fp8_quant_128x128."""
    return fp8_gemm_blockscaled(DGRAD, dyq, sdy, wq, sw, out_dtype, c, stream)


def wgrad(dyqT, sdyT, xqT, sxT, out_dtype=None, c=None, stream=None):
    """dW = dY^T X from fp8_quant_1x128(dY, transpose=True) and fp8_quant_1x128(X, transpose=True)."""
    return fp8_gemm_blockscaled(WGRAD, dyqT, sdyT, xqT, sxT, out_dtype, c, stream)


def fp8_grouped_gemm(xq, sx, row_index, expert_offsets, wq, sw, n_rows, out_dtype=None, y=None, stream=None):
    """MoE expert GEMM: Y[r] = fprop(Xq[row_index[r]], Wq[e]) for r in expert e's range.

    xq [T, K] uint8, sx [K/128, >=T]; row_index int32 [n_rows]; expert_offsets
    int32 [E+1]; wq uint8 [E, N, K]; sw float32 [E, N/128, K/128].
    row_index=None: xq/sx already hold the rows in expert order (for example
    from fp8_quant_1x128_gather), row r of xq feeds output row r (T >= n_rows).
    """
    torch = _torch()
    T, E, N, K = _grouped_operands(xq, sx, expert_offsets, wq, sw, n_rows, row_index)
    if out_dtype is None:
        out_dtype = torch.bfloat16
    if y is None:
        y = torch.empty((n_rows, N), dtype=out_dtype, device=xq.device)
    _layout(y, "y")
    _at_least(y, n_rows, N, "y")
    _on_gpu((xq, "xq"), (sx, "sx"), (wq, "wq"), (sw, "sw"), (expert_offsets, "expert_offsets"),
            (row_index, "row_index"), (y, "y"))
    ri = None if row_index is None else _ptr(row_index)
    rc = lib().fp8_grouped_gemm(_ptr(xq), _ptr(sx), sx.stride(0), T, ri, _ptr(expert_offsets), E,
                                n_rows, _ptr(wq), _ptr(sw), N, K, _ptr(y), _out_code(y.dtype), y.stride(0),
                                _stream(stream))
    _check(rc, "fp8_grouped_gemm")
    return y


def fp8_grouped_gemm_mx(xq, sx, expert_offsets, wq, sw, n_rows, out_dtype=None, y=None, stream=None):
    """fp8_grouped_gemm with rows already in expert order (row_index=None)
    for power-of-two scales, on the tensor cores' block-scaled MMA."""
    torch = _torch()
    T, E, N, K = _grouped_operands(xq, sx, expert_offsets, wq, sw, n_rows, None)
    if out_dtype is None:
        out_dtype = torch.bfloat16
    if y is None:
        y = torch.empty((n_rows, N), dtype=out_dtype, device=xq.device)
    _layout(y, "y")
    _at_least(y, n_rows, N, "y")
    _on_gpu((xq, "xq"), (sx, "sx"), (wq, "wq"), (sw, "sw"), (expert_offsets, "expert_offsets"), (y, "y"))
    rc = lib().fp8_grouped_gemm_mx(_ptr(xq), _ptr(sx), sx.stride(0), _ptr(expert_offsets), E, n_rows, _ptr(wq),
                                   _ptr(sw), N, K, _ptr(y), _out_code(y.dtype), y.stride(0), _stream(stream))
    _check(rc, "fp8_grouped_gemm_mx")
    return y


def fp8_moe_combine(y, dest, w, out_dtype=None, out=None, stream=None):
    """MoE combine: out[t] = sum_{j<k} w[t, j] * y[dest[t, j]] with FP32
    products and sums in slot order (no FMA); a negative dest skips the
    slot. y bf16 [rows, N]; dest int32 [T, k]; w float32 [T, k]; returns
    out [T, N] (bf16 by default, or float32)."""
    torch = _torch()
    _layout(y, "y")
    _dtype(y, torch.bfloat16, "y")
    _dtype(dest, torch.int32, "dest")
    _dtype(w, torch.float32, "w")
    if dest.dim() != 2 or not dest.is_contiguous() or not w.is_contiguous() or tuple(w.shape) != tuple(dest.shape):
        raise ValueError("dest and w must be contiguous [T, k] tensors of the same shape")
    T, k = dest.shape
    N = y.shape[1]
    if out_dtype is None:
        out_dtype = torch.bfloat16 if out is None else out.dtype
    if out is None:
        out = torch.empty((T, N), dtype=out_dtype, device=y.device)
    _layout(out, "out")
    _at_least(out, T, N, "out")
    _on_gpu((y, "y"), (dest, "dest"), (w, "w"), (out, "out"))
    rc = lib().fp8_moe_combine(_ptr(y), y.stride(0), y.shape[0], _ptr(dest), _ptr(w), T, k, N, _ptr(out),
                               _out_code(out.dtype), out.stride(0), _stream(stream))
    _check(rc, "fp8_moe_combine")
    return out


def device_status(stream=None):
    """Synchronise the stream and return (and clear) the device status word."""
    return lib().fp8fg_device_status(_stream(stream))


def set_wait_limit_ns(ns):
    _check(lib().fp8fg_set_wait_limit_ns(int(ns)), "fp8fg_set_wait_limit_ns")


def set_grouped_schedule(skinny_rows=32, skinny_cost_pct=100):
    """Schedule of fp8_grouped_gemm with rows in expert order (results do
    not depend on it): experts with at most `skinny_rows` rows (0: none, at
    most 32) are computed as 256 weight rows x 32 token rows per tile;
    `skinny_cost_pct` is such a tile's SM time relative to a full tile, in
    percent, which sets their share of the SMs. Process-wide."""
    _check(lib().fp8fg_set_grouped_schedule(int(skinny_rows), int(skinny_cost_pct)), "fp8fg_set_grouped_schedule")


def inject_skip_first_load(skip=True):
    _check(lib().fp8fg_test_skip_first_load(1 if skip else 0), "fp8fg_test_skip_first_load")


def version():
    return lib().fp8fg_version()
