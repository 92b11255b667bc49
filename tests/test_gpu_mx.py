"""GPU parity of the microscaling variant: the power-of-two quantisers
(bit-exact against the oracle's power-of-two rule) and the GEMM on the
tensor cores' block-scaled MMA (within the GEMM tolerance of the oracle's
block-scaled GEMM on the same codes and scales).

Shapes span several 128x256 output tiles, ragged row tails and an N that
ends half-way through a tile; the full-size dense workload is checked on
sampled rows.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_fine_grained_gb300 import synth
from tests.gpu_util import bits, check_gemm, rows_scales, to_np

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


def _same(a, b, what):
    a, b = np.asarray(a), np.asarray(b)
    if a.dtype == np.float32:
        a, b = a.view(np.uint32), b.view(np.uint32)
    if not np.array_equal(a, b):
        bad = np.argwhere(a != b)
        raise AssertionError("%s: %d differences, first at %s: gpu %r oracle %r" % (
            what, len(bad), tuple(bad[0]), a[tuple(bad[0])], b[tuple(bad[0])]))


def _quant_rows(x):
    q, s = fg.fp8_quant_1x128(x, pow2=True)
    torch.cuda.synchronize()
    qo, so = oracle.quant_1x128(bits(x), pow2=True)
    _same(to_np(q), qo, "1x128 pow2 codes")
    _same(rows_scales(s, x.shape[0]), so, "1x128 pow2 scales")
    return q, s, qo, so


def _quant_w(w):
    wq, sw = fg.fp8_quant_128x128(w, pow2=True)
    torch.cuda.synchronize()
    wo, swo = oracle.quant_128x128(bits(w), pow2=True)
    _same(to_np(wq), wo, "128x128 pow2 codes")
    _same(to_np(sw), swo, "128x128 pow2 scales")
    return wq, sw, wo, swo


def _hard_rows(M, K, seed):
    """Activations with an all-zero group, bf16 subnormals, values near the
    top of the bf16 range and a group whose amax sits at 448 * 2^e exactly."""
    x = _act(M, K, seed).float()
    x[0, :128] = 0.0
    x[1, 128:256] *= 1e-38
    x[2, :128] = 1e36 * torch.sign(x[2, :128])
    x[3, :128] = 0.5
    x[3, 5] = 448.0 * 2.0 ** -3
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("M,K", [(1, 128), (5, 384), (257, 640), (300, 7168)])
def test_quant_1x128_pow2(M, K):
    x = _hard_rows(max(M, 4), K, seed=M + K)[:M].contiguous()
    _quant_rows(x)


@pytest.mark.parametrize("rows,cols", [(128, 64), (256, 200), (384, 1000)])
def test_quant_128x1_pow2(rows, cols):
    x = _act(rows, cols, seed=rows * cols).float()
    x[:128, 0] = 0.0
    x[:, 1] *= 1e-38
    x = x.to(torch.bfloat16)
    qT, sT = fg.fp8_quant_1x128(x, transpose=True, pow2=True)
    torch.cuda.synchronize()
    qo, so = oracle.quant_128x1_t(bits(x), pow2=True)
    _same(to_np(qT), qo, "128x1 pow2 codes")
    _same(to_np(sT)[:, :cols], so, "128x1 pow2 scales")


@pytest.mark.parametrize("rows,cols", [(128, 128), (256, 384), (640, 512)])
def test_quant_dual_pow2(rows, cols):
    x = _hard_rows(rows, cols, seed=rows + 7 * cols)
    q, s, qT, sT = fg.fp8_quant_1x128_dual(x, pow2=True)
    torch.cuda.synchronize()
    qo, so = oracle.quant_1x128(bits(x), pow2=True)
    qTo, sTo = oracle.quant_128x1_t(bits(x), pow2=True)
    _same(to_np(q), qo, "dual rows codes")
    _same(rows_scales(s, rows), so, "dual rows scales")
    _same(to_np(qT), qTo, "dual cols codes")
    _same(to_np(sT)[:, :cols], sTo, "dual cols scales")


def test_quant_gather_pow2():
    x = _hard_rows(50, 384, seed=3)
    idx = torch.tensor([7, 0, 3, 3, 49, 1, 2, 20], dtype=torch.int32, device=DEV)
    q, s = fg.fp8_quant_1x128_gather(x, idx, pow2=True)
    torch.cuda.synchronize()
    qo, so = oracle.quant_1x128(bits(x), pow2=True)
    sel = idx.cpu().numpy()
    _same(to_np(q), qo[sel], "gather pow2 codes")
    _same(rows_scales(s, len(sel)), so[sel], "gather pow2 scales")


@pytest.mark.parametrize("N,K", [(128, 128), (384, 640), (256, 7168)])
def test_quant_128x128_pow2(N, K):
    w = _wt(N, K, seed=N + K).float()
    w[:128, :128] = 0.0
    if N > 128 and K > 128:
        w[128:256, 128:256] *= 1e-37
    _quant_w(w.to(torch.bfloat16))


FPROP_SHAPES = [(1, 128, 128), (127, 256, 256), (129, 384, 512), (300, 512, 1024), (256, 1024, 384)]


@pytest.mark.parametrize("M,N,K", FPROP_SHAPES)
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_gemm_mx_fprop(M, N, K, out):
    x = _act(M, K, seed=M + N + K)
    w = _wt(N, K, seed=M * N + K)
    xq, sx, xo, sxo = _quant_rows(x)
    wq, sw, wo, swo = _quant_w(w)
    dt = torch.float32 if out == "f32" else torch.bfloat16
    y = fg.fp8_gemm_mx(fg.FPROP, xq, sx, wq, sw, out_dtype=dt)
    assert fg.device_status() == 0
    c, ce, t = oracle.fprop(xo, sxo, wo, swo)
    check_gemm(to_np(y), c, t, out == "bf16", "mx fprop %dx%dx%d" % (M, N, K))
    if out == "f32":
        check_gemm(to_np(y), ce, t, False, "mx fprop vs exact")


def test_gemm_mx_hard_scales():
    """Zero groups, subnormal-scaled groups and large groups in one GEMM:
    every scale exponent from 2^-127 up to the top of the range."""
    M, N, K = 200, 256, 512
    x = _hard_rows(M, K, seed=5)
    w = _wt(N, K, seed=6).float()
    w[:128, 256:384] *= 1e-30
    w[128:, 128:256] *= 1e20
    xq, sx, xo, sxo = _quant_rows(x)
    wq, sw, wo, swo = _quant_w(w.to(torch.bfloat16))
    y = fg.fp8_gemm_mx(fg.FPROP, xq, sx, wq, sw, out_dtype=torch.float32)
    assert fg.device_status() == 0
    c, _, t = oracle.fprop(xo, sxo, wo, swo)
    g = to_np(y)
    assert np.all(np.isfinite(c)) and np.all(np.isfinite(g))
    check_gemm(g, c, t, False, "mx hard scales")


@pytest.mark.parametrize("M,Kout,Ncontract", [(1, 128, 128), (130, 256, 384), (257, 384, 256), (64, 640, 1024)])
def test_gemm_mx_dgrad(M, Kout, Ncontract):
    g = _gen(M + Kout)
    dy = (torch.randn(M, Ncontract, generator=g, device=DEV) * 1e-3).to(torch.bfloat16)
    w = _wt(Ncontract, Kout, seed=Kout * 3 + Ncontract)
    dyq, sdy, dyo, sdyo = _quant_rows(dy)
    wq, sw, wo, swo = _quant_w(w)
    dx = fg.fp8_gemm_mx(fg.DGRAD, dyq, sdy, wq, sw, out_dtype=torch.float32)
    assert fg.device_status() == 0
    c, _, t = oracle.dgrad(dyo, sdyo, wo, swo)
    check_gemm(to_np(dx), c, t, False, "mx dgrad")


@pytest.mark.parametrize("tokens,N,K", [(128, 128, 128), (256, 384, 256), (384, 256, 640)])
def test_gemm_mx_wgrad(tokens, N, K):
    x = _act(tokens, K, seed=tokens + K)
    dy = (torch.randn(tokens, N, generator=_gen(N), device=DEV) * 1e-3).to(torch.bfloat16)
    xqT, sxT = fg.fp8_quant_1x128(x, transpose=True, pow2=True)
    dyqT, sdyT = fg.fp8_quant_1x128(dy, transpose=True, pow2=True)
    torch.cuda.synchronize()
    xo, sxo = oracle.quant_128x1_t(bits(x), pow2=True)
    dyo, sdyo = oracle.quant_128x1_t(bits(dy), pow2=True)
    _same(to_np(xqT), xo, "wgrad X^T codes")
    _same(to_np(dyqT), dyo, "wgrad dY^T codes")
    dw = fg.fp8_gemm_mx(fg.WGRAD, dyqT, sdyT, xqT, sxT)
    assert fg.device_status() == 0
    c, _, t = oracle.wgrad(dyo, sdyo, xo, sxo)
    check_gemm(to_np(dw), c, t, False, "mx wgrad")


def test_gemm_mx_dense_config_sampled():
    """Dense projection workload at full size (4096 x 7168 x 7168, bf16 out)
    with power-of-two scales: quantisation bit-exact, GEMM on sampled rows."""
    x, w = synth.dense(seed=0, device=DEV)
    xq, sx, xo, sxo = _quant_rows(x)
    wq, sw, wo, swo = _quant_w(w)
    y = fg.fp8_gemm_mx(fg.FPROP, xq, sx, wq, sw)
    assert fg.device_status() == 0
    rows = np.concatenate([np.random.default_rng(1).choice(4096, 6, replace=False), [0, 4095]])
    c, _, t = oracle.fprop(xo, sxo, wo, swo, rows=rows)
    check_gemm(to_np(y[torch.from_numpy(rows).to(DEV)]), c, t, True, "mx dense config")


def test_gemm_mx_timeout_is_reported_not_hung():
    x = _act(256, 256, seed=1)
    w = _wt(256, 256, seed=2)
    xq, sx = fg.fp8_quant_1x128(x, pow2=True)
    wq, sw = fg.fp8_quant_128x128(w, pow2=True)
    fg.set_wait_limit_ns(50_000_000)
    try:
        fg.inject_skip_first_load(True)
        fg.fp8_gemm_mx(fg.FPROP, xq, sx, wq, sw)
        assert fg.device_status() == 5  # FP8FG_ETIMEOUT
        y = fg.fp8_gemm_mx(fg.FPROP, xq, sx, wq, sw, out_dtype=torch.float32)
        assert fg.device_status() == 0
    finally:
        fg.set_wait_limit_ns(2_000_000_000)
    xo, sxo = oracle.quant_1x128(bits(x), pow2=True)
    wo, swo = oracle.quant_128x128(bits(w), pow2=True)
    c, _, t = oracle.fprop(xo, sxo, wo, swo)
    check_gemm(to_np(y), c, t, False, "mx after timeout")


def _moe_small(seed, T=300, K=384, N=256, counts=(0, 1, 129, 0, 300, 5, 128, 0, 257)):
    g = _gen(seed)
    x = torch.randn(T, K, generator=g, device=DEV).to(torch.bfloat16)
    w = (torch.randn(len(counts), N, K, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    rng = np.random.default_rng(seed)
    row_index = np.concatenate([np.sort(rng.choice(T, c, replace=False)) if c else np.zeros(0, np.int64)
                                for c in counts]).astype(np.int32)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return x, w, row_index, off


@pytest.mark.parametrize("out,counts", [("f32", (0, 1, 129, 0, 300, 5, 128, 0, 257)),
                                        ("bf16", (40, 64, 2, 65, 17, 33, 32, 0, 1)),
                                        ("f32", (64, 63, 31, 129, 1))])
def test_grouped_gemm_mx(out, counts):
    """MoE experts in the microscaling variant: rows quantised into expert
    order with power-of-two scales, the grouped GEMM on the block-scaled
    MMA; expert sizes 0..300 (tiles straddling the next expert's rows);
    rows past the last offset untouched."""
    x, w, row_index, off = _moe_small(seed=31, counts=counts)
    R = int(off[-1])
    ri = torch.from_numpy(row_index).to(DEV)
    xg, sxg = fg.fp8_quant_1x128_gather(x, ri, pow2=True)
    wq, sw = fg.fp8_quant_128x128(w, pow2=True)
    dt = torch.float32 if out == "f32" else torch.bfloat16
    y = torch.full((R + 40, w.shape[1]), 5.0, dtype=dt, device=DEV)
    xg_pad = torch.zeros((R + 40, x.shape[1]), dtype=torch.uint8, device=DEV)
    xg_pad[:R] = xg
    sxg_pad = torch.zeros((sxg.shape[0], (R + 40 + 3) // 4 * 4), dtype=torch.float32, device=DEV)
    sxg_pad[:, :R] = sxg[:, :R]
    fg.fp8_grouped_gemm_mx(xg_pad, sxg_pad, torch.from_numpy(off).to(DEV), wq, sw, n_rows=R + 40, y=y)
    assert fg.device_status() == 0
    assert torch.all(y[R:] == 5.0)
    xo, sxo = oracle.quant_1x128(bits(x), pow2=True)
    _same(to_np(xg), xo[row_index], "gathered pow2 codes")
    wo, swo = to_np(wq), to_np(sw)
    for e in range(w.shape[0]):
        qe, se = oracle.quant_128x128(bits(w[e]), pow2=True)
        _same(wo[e], qe, "expert codes")
        _same(swo[e], se, "expert scales")
    c, _, t = oracle.grouped(xo, sxo, row_index, off, wo, swo)
    check_gemm(to_np(y[:R]), c, t, out == "bf16", "mx grouped")


def test_grouped_gemm_mx_bad_offsets_reported():
    x, w, row_index, off = _moe_small(seed=32, counts=(10, 20))
    xq, sx = fg.fp8_quant_1x128(x, pow2=True)
    wq, sw = fg.fp8_quant_128x128(w, pow2=True)
    bad = torch.tensor([0, 40, 30], dtype=torch.int32, device=DEV)  # decreasing
    fg.fp8_grouped_gemm_mx(xq, sx, bad, wq, sw, n_rows=300)
    assert fg.device_status() == 6  # FP8FG_EDEVICE
    fg.fp8_grouped_gemm_mx(xq, sx, torch.from_numpy(off).to(DEV), wq, sw, n_rows=300)
    assert fg.device_status() == 0
