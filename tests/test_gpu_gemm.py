"""GPU parity of the block-scaled GEMM (fprop, dgrad, wgrad) and the grouped
MoE GEMM against the CPU oracle, on the same seeded inputs.

Small shapes span several 128x256 output tiles and ragged row tails and are
checked element by element; the full-size workloads are checked on sampled
output rows that the oracle computes one by one. Quantised operands are
first checked bit-exact, so the GEMM comparison starts from identical codes.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_fine_grained_gb300 import synth
from tests.gpu_util import assert_quant_1x128, bits, check_gemm, rows_scales, to_np

pytestmark = pytest.mark.gpu

fg = pytest.importorskip("fp8_fine_grained_gb300")
DEV = "cuda"


def _gen(seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    return g


def _act(M, K, seed):
    g = _gen(seed)
    c = torch.exp(torch.randn(K, generator=g, device=DEV))
    return (torch.randn(M, K, generator=g, device=DEV) * c).to(torch.bfloat16)


def _wt(N, K, seed, std=0.02):
    return (torch.randn(N, K, generator=_gen(seed), device=DEV) * std).to(torch.bfloat16)


def _quant_w(w):
    wq, sw = fg.fp8_quant_128x128(w)
    torch.cuda.synchronize()
    wo, swo = oracle.quant_128x128(bits(w))
    assert np.array_equal(to_np(wq), wo) and np.array_equal(to_np(sw), swo)
    return wq, sw, wo, swo


FPROP_SHAPES = [(1, 128, 128), (127, 256, 256), (129, 384, 512), (300, 512, 1024), (256, 1024, 384)]


@pytest.mark.parametrize("M,N,K", FPROP_SHAPES)
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_fprop(M, N, K, out):
    x = _act(M, K, seed=M + N + K)
    w = _wt(N, K, seed=M * N + K)
    xq, sx = fg.fp8_quant_1x128(x)
    torch.cuda.synchronize()
    xo, sxo = assert_quant_1x128(x, xq, sx)
    wq, sw, wo, swo = _quant_w(w)
    dt = torch.float32 if out == "f32" else torch.bfloat16
    y = fg.fprop(xq, sx, wq, sw, out_dtype=dt)
    assert fg.device_status() == 0
    c, _, t = oracle.fprop(xo, sxo, wo, swo)
    check_gemm(to_np(y), c, t, out == "bf16", "fprop %dx%dx%d" % (M, N, K))


def test_fprop_tiny_config():
    """The tiny fprop workload (X 128x256 with 1% x100 outliers, W 128x256), FP32 out."""
    x, w = synth.tiny(seed=0, device=DEV)
    xq, sx = fg.fp8_quant_1x128(x)
    torch.cuda.synchronize()
    xo, sxo = assert_quant_1x128(x, xq, sx)
    wq, sw, wo, swo = _quant_w(w)
    y = fg.fprop(xq, sx, wq, sw, out_dtype=torch.float32)
    c, ce, t = oracle.fprop(xo, sxo, wo, swo)
    check_gemm(to_np(y), c, t, False, "tiny")
    # the exact value is inside the same band
    check_gemm(to_np(y), ce, t, False, "tiny vs exact")


def test_fprop_output_pitch_and_sampled_rows_of_large_m():
    M, N, K = 2000, 768, 640
    x = _act(M, K, seed=11)
    w = _wt(N, K, seed=12)
    xq, sx = fg.fp8_quant_1x128(x)
    wq, sw, wo, swo = _quant_w(w)
    c_full = torch.full((M, N + 64), 7.0, dtype=torch.bfloat16, device=DEV)
    fg.fprop(xq, sx, wq, sw, c=c_full[:, :N])
    torch.cuda.synchronize()
    assert torch.all(c_full[:, N:] == 7.0)
    xo, sxo = assert_quant_1x128(x, xq, sx)
    rows = np.array([0, 1, 127, 128, 1000, 1919, 1920, 1999])
    c, _, t = oracle.fprop(xo, sxo, wo, swo, rows=rows)
    check_gemm(to_np(c_full[:, :N])[rows], c, t, True, "pitched")


@pytest.mark.parametrize("M,Kout,Ncontract", [(1, 128, 128), (130, 256, 384), (257, 384, 256), (64, 640, 1024)])
def test_dgrad(M, Kout, Ncontract):
    """dX[M, Kout] = dY[M, Ncontract] . W[Ncontract, Kout], W read as stored."""
    g = _gen(M + Kout)
    dy = (torch.randn(M, Ncontract, generator=g, device=DEV) * 1e-3).to(torch.bfloat16)
    w = _wt(Ncontract, Kout, seed=Kout * 3 + Ncontract)
    dyq, sdy = fg.fp8_quant_1x128(dy)
    torch.cuda.synchronize()
    dyo, sdyo = assert_quant_1x128(dy, dyq, sdy)
    wq, sw, wo, swo = _quant_w(w)
    dx = fg.dgrad(dyq, sdy, wq, sw, out_dtype=torch.float32)
    assert fg.device_status() == 0
    c, _, t = oracle.dgrad(dyo, sdyo, wo, swo)
    check_gemm(to_np(dx), c, t, False, "dgrad")


@pytest.mark.parametrize("tokens,N,K", [(128, 128, 128), (256, 384, 256), (384, 256, 640)])
def test_wgrad(tokens, N, K):
    """dW[N, K] = dY^T X over tokens, both quantised in groups of 128 tokens."""
    x = _act(tokens, K, seed=tokens + K)
    dy = (torch.randn(tokens, N, generator=_gen(N), device=DEV) * 1e-3).to(torch.bfloat16)
    xqT, sxT = fg.fp8_quant_1x128(x, transpose=True)
    dyqT, sdyT = fg.fp8_quant_1x128(dy, transpose=True)
    torch.cuda.synchronize()
    xo, sxo = oracle.quant_128x1_t(bits(x))
    dyo, sdyo = oracle.quant_128x1_t(bits(dy))
    assert np.array_equal(to_np(xqT), xo) and np.array_equal(to_np(dyqT), dyo)
    dw = fg.wgrad(dyqT, sdyT, xqT, sxT)
    assert fg.device_status() == 0
    c, _, t = oracle.wgrad(dyo, sdyo, xo, sxo)
    check_gemm(to_np(dw), c, t, False, "wgrad")


@pytest.mark.parametrize("mode,M,N,K", [(0, 300, 512, 1024), (0, 129, 384, 512), (1, 200, 384, 640)])
def test_gemm_e4m3_output(mode, M, N, K):
    """The GEMM with its output quantised in the epilogue writes exactly
    what the oracle's 1x128 quantiser makes of the bf16 output of the same
    GEMM (which itself is checked against the oracle GEMM elsewhere)."""
    x = _act(M, K, seed=40 + mode)
    if mode == 0:
        w = _wt(N, K, seed=41)
    else:
        w = _wt(K, N, seed=42)          # dgrad: B is the weight [K_contract][N]
    xq, sx = fg.fp8_quant_1x128(x)
    wq, sw = fg.fp8_quant_128x128(w)
    y = fg.fp8_gemm_blockscaled(mode, xq, sx, wq, sw, out_dtype=torch.bfloat16)
    yq, sy = fg.fp8_gemm_blockscaled_e4m3(mode, xq, sx, wq, sw)
    assert fg.device_status() == 0
    qo, so = oracle.quant_1x128(bits(y))
    assert np.array_equal(to_np(yq), qo)
    assert np.array_equal(rows_scales(sy, M).view(np.uint32), so.view(np.uint32))


def _moe_small(seed, T=300, K=384, N=256, E=9, counts=None):
    g = _gen(seed)
    x = torch.randn(T, K, generator=g, device=DEV).to(torch.bfloat16)
    w = (torch.randn(E, N, K, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    if counts is None:
        counts = [0, 1, 129, 0, 300, 5, 128, 0, 257]
    rng = np.random.default_rng(seed)
    row_index = np.concatenate([np.sort(rng.choice(T, c, replace=False)) if c else np.zeros(0, np.int64)
                                for c in counts]).astype(np.int32)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return x, w, row_index, off


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_grouped_small(out):
    x, w, row_index, off = _moe_small(seed=21)
    xq, sx = fg.fp8_quant_1x128(x)
    wq, sw = fg.fp8_quant_128x128(w)
    ri = torch.from_numpy(row_index).to(DEV)
    of = torch.from_numpy(off).to(DEV)
    dt = torch.float32 if out == "f32" else torch.bfloat16
    y = fg.fp8_grouped_gemm(xq, sx, ri, of, wq, sw, n_rows=int(off[-1]), out_dtype=dt)
    assert fg.device_status() == 0
    xo, sxo = assert_quant_1x128(x, xq, sx)
    wo = to_np(wq)
    swo = to_np(sw)
    for e in range(w.shape[0]):
        qe, se = oracle.quant_128x128(bits(w[e]))
        assert np.array_equal(wo[e], qe) and np.array_equal(swo[e], se)
    c, _, t = oracle.grouped(xo, sxo, row_index, off, wo, swo)
    check_gemm(to_np(y), c, t, out == "bf16", "grouped")


@pytest.mark.parametrize("out,counts", [("f32", None), ("bf16", None),
                                        ("bf16", [40, 64, 2, 65, 17, 33, 32, 0, 1]),
                                        ("f32", [64, 63, 31, 129, 1])])
def test_grouped_rows_in_expert_order(out, counts):
    """Without a row index: the rows are quantised straight into expert
    order (fp8_quant_1x128_gather) and the GEMM loads 128-row A tiles with
    TMA, across expert sizes of 0..300 rows (tiles that straddle the next
    expert's rows included). Rows past the last offset stay untouched."""
    x, w, row_index, off = _moe_small(seed=24, counts=counts, E=9 if counts is None else len(counts))
    R = int(off[-1])
    ri = torch.from_numpy(row_index).to(DEV)
    xg, sxg = fg.fp8_quant_1x128_gather(x, ri)
    wq, sw = fg.fp8_quant_128x128(w)
    dt = torch.float32 if out == "f32" else torch.bfloat16
    y = torch.full((R + 40, w.shape[1]), 5.0, dtype=dt, device=DEV)
    xg_pad = torch.zeros((R + 40, x.shape[1]), dtype=torch.uint8, device=DEV)
    xg_pad[:R] = xg
    sxg_pad = torch.zeros((sxg.shape[0], (R + 40 + 3) // 4 * 4), dtype=torch.float32, device=DEV)
    sxg_pad[:, :R] = sxg[:, :R]
    fg.fp8_grouped_gemm(xg_pad, sxg_pad, None, torch.from_numpy(off).to(DEV), wq, sw, n_rows=R + 40, y=y)
    assert fg.device_status() == 0
    assert torch.all(y[R:] == 5.0)
    xo, sxo = oracle.quant_1x128(bits(x))
    assert np.array_equal(to_np(xg), xo[row_index])
    wo, swo = to_np(wq), to_np(sw)
    c, _, t = oracle.grouped(xo, sxo, row_index, off, wo, swo)
    check_gemm(to_np(y[:R]), c, t, out == "bf16", "grouped, rows in expert order")


def test_grouped_rows_beyond_last_offset_untouched():
    x, w, row_index, off = _moe_small(seed=22, counts=[3, 0, 130])
    xq, sx = fg.fp8_quant_1x128(x)
    wq, sw = fg.fp8_quant_128x128(w[:3])
    n_rows = int(off[-1]) + 40
    y = torch.full((n_rows, w.shape[1]), 5.0, dtype=torch.float32, device=DEV)
    ri = torch.from_numpy(np.concatenate([row_index, np.zeros(40, np.int32)])).to(DEV)
    fg.fp8_grouped_gemm(xq, sx, ri, torch.from_numpy(off).to(DEV), wq, sw, n_rows=n_rows, y=y)
    assert fg.device_status() == 0
    assert torch.all(y[int(off[-1]):] == 5.0)


def test_grouped_bad_row_index_reported():
    x, w, row_index, off = _moe_small(seed=23, counts=[4, 4])
    xq, sx = fg.fp8_quant_1x128(x)
    wq, sw = fg.fp8_quant_128x128(w[:2])
    bad = row_index.copy()
    bad[2] = 10 ** 6
    fg.fp8_grouped_gemm(xq, sx, torch.from_numpy(bad).to(DEV), torch.from_numpy(off).to(DEV), wq, sw,
                        n_rows=8)
    assert fg.device_status() == 6  # FP8FG_EDEVICE
    assert fg.device_status() == 0  # cleared


def test_dense_config_sampled():
    """Dense projection workload at full size (4096 x 7168 x 7168, bf16 out):
    quantisation bit-exact, GEMM on sampled rows."""
    x, w = synth.dense(seed=0, device=DEV)
    xq, sx = fg.fp8_quant_1x128(x)
    wq, sw = fg.fp8_quant_128x128(w)
    y = fg.fprop(xq, sx, wq, sw)
    assert fg.device_status() == 0
    xo, sxo = assert_quant_1x128(x, xq, sx)
    wo, swo = oracle.quant_128x128(bits(w))
    assert np.array_equal(to_np(wq), wo)
    rows = np.random.default_rng(0).choice(4096, 6, replace=False)
    rows = np.concatenate([rows, [0, 4095]])
    c, _, t = oracle.fprop(xo, sxo, wo, swo, rows=rows)
    check_gemm(to_np(y[torch.from_numpy(rows).to(DEV)]), c, t, True, "dense config")


def test_timeout_is_reported_not_hung():
    """A withheld operand load makes the consumers' bounded waits run out:
    the launch reports FP8FG_ETIMEOUT and the next launch is clean."""
    x = _act(256, 256, seed=1)
    w = _wt(256, 256, seed=2)
    xq, sx = fg.fp8_quant_1x128(x)
    wq, sw = fg.fp8_quant_128x128(w)
    fg.set_wait_limit_ns(50_000_000)
    try:
        fg.inject_skip_first_load(True)
        fg.fprop(xq, sx, wq, sw)
        assert fg.device_status() == 5  # FP8FG_ETIMEOUT
        y = fg.fprop(xq, sx, wq, sw, out_dtype=torch.float32)
        assert fg.device_status() == 0
    finally:
        fg.set_wait_limit_ns(2_000_000_000)
    xo, sxo = assert_quant_1x128(x, xq, sx)
    wo, swo = oracle.quant_128x128(bits(w))
    c, _, t = oracle.fprop(xo, sxo, wo, swo)
    check_gemm(to_np(y), c, t, False, "after timeout")
