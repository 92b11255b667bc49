"""Host-side checks of the Python binding's argument validation (no GPU).

The C ABI receives bare pointers and cannot see how large the tensors
behind them are, so the binding compares dtypes and extents before it calls
into the library: an undersized operand, scale array or output must raise
ValueError instead of letting a kernel read or write past its allocation.
These tests use CPU tensors; every check on extents and dtypes runs before
the check that the tensors live on the GPU, so each case raises the error
that names the faulty argument."""
import ctypes

import pytest
import torch

import fp8_fine_grained_gb300 as fg
from fp8_fine_grained_gb300 import build as libbuild

U8, F32, BF16, I32 = torch.uint8, torch.float32, torch.bfloat16, torch.int32


def z(shape, dtype):
    return torch.zeros(shape, dtype=dtype)


def gemm_args(mode, M=256, N=512, K=384):
    """Well-formed operands of one mode (CPU tensors)."""
    a = z((M, K), U8)
    sa = z((K // 128, M), F32)
    if mode == fg.FPROP:
        b, sb = z((N, K), U8), z((N // 128, K // 128), F32)
    elif mode == fg.DGRAD:
        b, sb = z((K, N), U8), z((K // 128, N // 128), F32)
    else:
        b, sb = z((N, K), U8), z((K // 128, N), F32)
    return a, sa, b, sb


def expect(msg, fn, *a, **kw):
    with pytest.raises(ValueError, match=msg):
        fn(*a, **kw)


@pytest.mark.parametrize("mode", [fg.FPROP, fg.DGRAD, fg.WGRAD])
@pytest.mark.parametrize("entry", ["fp8_gemm_blockscaled", "fp8_gemm_mx"])
def test_gemm_operand_extents(mode, entry):
    f = getattr(fg, entry)
    a, sa, b, sb = gemm_args(mode)
    # well-formed CPU operands reach only the device check
    expect("CUDA tensor", f, mode, a, sa, b, sb)
    # B with the wrong contraction extent
    bad_b = z((b.shape[0] - 128, b.shape[1]), U8) if mode == fg.DGRAD else z((b.shape[0], b.shape[1] - 128), U8)
    expect("K = a.shape", f, mode, a, sa, bad_b, sb)
    # too few row scales, too few contraction blocks of row scales
    expect("sa must cover", f, mode, a, sa[:, :-1], b, sb)
    expect("sa must cover", f, mode, a, sa[:-1], b, sb)
    # too few B scales
    expect("sb must cover", f, mode, a, sa, b, sb[:-1])
    expect("sb must cover", f, mode, a, sa, b, sb[:, :-1])
    # dtypes
    expect("a must be", f, mode, a.to(F32), sa, b, sb)
    expect("b must be", f, mode, a, sa, b.to(I32), sb)
    expect("sa must be", f, mode, a, sa.to(BF16), b, sb)
    expect("sb must be", f, mode, a, sa, b, sb.to(torch.float64))
    # an output of the wrong shape
    M, N = a.shape[0], (b.shape[1] if mode == fg.DGRAD else b.shape[0])
    expect("c must be", f, mode, a, sa, b, sb, c=z((M, N - 128), F32))


def test_gemm_rejects_unknown_mode():
    a, sa, b, sb = gemm_args(fg.FPROP)
    expect("mode", fg.fp8_gemm_blockscaled, 7, a, sa, b, sb)


def test_gemm_e4m3_output_checks():
    a, sa, b, sb = gemm_args(fg.FPROP)
    expect("FPROP and DGRAD", fg.fp8_gemm_blockscaled_e4m3, fg.WGRAD, a, sa, b, sb)
    expect("sa must cover", fg.fp8_gemm_blockscaled_e4m3, fg.FPROP, a, sa[:, :10], b, sb)
    expect("scales must cover", fg.fp8_gemm_blockscaled_e4m3, fg.FPROP, a, sa, b, sb,
           c=z((256, 512), U8), scales=z((4, 255), F32))


def grouped_args(E=4, N=256, K=384, T=300, R=200):
    xq = z((T, K), U8)
    sx = z((K // 128, T), F32)
    wq = z((E, N, K), U8)
    sw = z((E, N // 128, K // 128), F32)
    off = torch.tensor([0, 50, 50, 120, R], dtype=I32)
    ri = z((R,), I32)
    return xq, sx, ri, off, wq, sw, R


def test_grouped_operand_extents():
    xq, sx, ri, off, wq, sw, R = grouped_args()
    f = fg.fp8_grouped_gemm
    expect("CUDA tensor", f, xq, sx, ri, off, wq, sw, R)
    expect("row_index must hold", f, xq, sx, ri[:-1], off, wq, sw, R)
    expect("expert_offsets must hold", f, xq, sx, ri, off[:-1], wq, sw, R)
    expect("sw must be", f, xq, sx, ri, off, wq, sw[:, :, :-1].contiguous(), R)
    expect("sw must be", f, xq, sx, ri, off, wq, sw[:-1].contiguous(), R)
    expect("sx must cover", f, xq, sx[:-1], ri, off, wq, sw, R)
    expect("sx must cover", f, xq, sx[:, :-1], ri, off, wq, sw, R)
    expect("xq must be", f, xq.to(F32), sx, ri, off, wq, sw, R)
    expect("wq must be", f, xq, sx, ri, off, wq.to(I32), sw, R)
    expect("int32", f, xq, sx, ri.to(torch.int64), off, wq, sw, R)
    expect("n_rows", f, xq, sx, ri, off, wq, sw, -1)
    # rows already in expert order: xq and sx must hold every output row
    expect("n_rows", f, xq[:150], sx[:, :150], None, off, wq, sw, R)
    # output too small
    expect("y must cover", f, xq, sx, ri, off, wq, sw, R, y=z((R - 1, 256), BF16))


def test_grouped_mx_operand_extents():
    xq, sx, _, off, wq, sw, R = grouped_args()
    f = fg.fp8_grouped_gemm_mx
    expect("CUDA tensor", f, xq, sx, off, wq, sw, R)
    expect("expert_offsets must hold", f, xq, sx, off[:-1], wq, sw, R)
    expect("sw must be", f, xq, sx, off, wq, sw[:-1].contiguous(), R)
    expect("n_rows", f, xq[:100], sx[:, :100], off, wq, sw, R)
    expect("sx must cover", f, xq, sx[:-1], off, wq, sw, R)


def test_quantiser_outputs_checked():
    x = z((256, 384), BF16)
    expect("CUDA tensor", fg.fp8_quant_1x128, x)
    expect("q must cover", fg.fp8_quant_1x128, x, q=z((255, 384), U8), scales=z((3, 256), F32))
    expect("scales must cover", fg.fp8_quant_1x128, x, q=z((256, 384), U8), scales=z((3, 252), F32))
    expect("q must be", fg.fp8_quant_1x128, x, q=z((256, 384), I32), scales=z((3, 256), F32))
    expect("scales must cover", fg.fp8_quant_1x128, x, transpose=True, q=z((384, 256), U8),
           scales=z((1, 380), F32))
    expect("qT must cover", fg.fp8_quant_1x128_dual, x, qT=z((383, 256), U8))
    expect("scalesT must cover", fg.fp8_quant_1x128_dual, x, scalesT=z((2, 380), F32))
    w = z((256, 384), BF16)
    expect("q must be", fg.fp8_quant_128x128, w, q=z((128, 384), U8))
    expect("qT must cover", fg.fp8_quant_128x128_dual, w, qT=z((384, 128), U8))
    expect("q must cover", fg.fp8_quant_128x128_dual, w, q=z((256, 256), U8))
    expect("scales and scalesT", fg.fp8_quant_128x128_dual, w, scalesT=z((3, 1), F32))
    expect("qT must be", fg.fp8_quant_128x128_dual, w, qT=z((384, 256), I32))
    expect("w must be a 2-D", fg.fp8_quant_128x128_dual, z((2, 256, 384), BF16))


def test_grouped_tile_count_limit_in_the_abi():
    """The experts' tile prefix is int32 in the kernels: a call whose largest
    possible tile count reaches 2^31 is rejected before anything runs."""
    libbuild.build()
    L = fg.lib()
    A16 = ctypes.c_void_p(0x10000)
    # one expert of 2^30 - 128 columns and 2^30 rows: every other limit
    # holds (E*N, n_rows < 2^31), but 2^23 m-tiles x 2^22 n-tiles do not fit
    n_rows, E, N, K = (1 << 30), 1, (1 << 30) - 128, 128
    rc = L.fp8_grouped_gemm(A16, A16, n_rows, n_rows, None, A16, E, n_rows, A16, A16, N, K, A16, 1, N, None)
    assert rc == 1  # FP8FG_EINVAL
    rc = L.fp8_grouped_gemm_mx(A16, A16, n_rows, A16, E, n_rows, A16, A16, N, K, A16, 1, N, None)
    assert rc == 1


def test_combine_argument_checks():
    y = z((100, 256), BF16)
    dest = z((64, 8), I32)
    w = z((64, 8), F32)
    expect("CUDA tensor", fg.fp8_moe_combine, y, dest, w)
    expect("y must be", fg.fp8_moe_combine, y.to(F32), dest, w)
    expect("dest must be", fg.fp8_moe_combine, y, dest.to(torch.int64), w)
    expect("w must be", fg.fp8_moe_combine, y, dest, w.to(BF16))
    expect("same shape", fg.fp8_moe_combine, y, dest, w[:, :4].contiguous())
    expect("out must cover", fg.fp8_moe_combine, y, dest, w, out=z((63, 256), BF16))
