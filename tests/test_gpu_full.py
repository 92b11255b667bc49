"""Parity at the benchmark's full sizes, in the launch configuration bench.py
times: every quantised tensor bit-exact against the oracle, GEMM outputs on
sampled rows that the oracle computes one by one.

Workloads: the linear-layer training trio (7168 -> 18432 at 8192 tokens:
fprop, dgrad, wgrad), the MoE expert GEMM (4096 tokens, 256 experts of
2048 x 7168, top-8 with a Zipf(1.1) bias; with a row index, and in the
dispatch form bench.py times) and the outlier-heavy fprop (16384 x 7168 x
7168); the trio and the MoE step also in the microscaling variant."""
import numpy as np
import pytest
import torch

import oracle
from fp8_fine_grained_gb300 import synth
from tests.gpu_util import assert_quant_1x128, bits, check_gemm, to_np

pytestmark = pytest.mark.gpu

fg = pytest.importorskip("fp8_fine_grained_gb300")
DEV = "cuda"


def _sample(n, k, seed):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([rng.choice(n, k, replace=False), [0, n - 1]]))


def test_trio_weight_dual_full_size():
    """The trio's weight (18432 x 7168) and its transpose from one read,
    both bit-exact: the transposed blocks against the oracle's quantisation
    of the materialised W^T."""
    _, w, _ = synth.trio(seed=0, device=DEV)
    q, s, qT, sT = fg.fp8_quant_128x128_dual(w)
    torch.cuda.synchronize()
    qo, so = oracle.quant_128x128(bits(w))
    assert np.array_equal(to_np(q), qo) and np.array_equal(to_np(s).view(np.uint32), so.view(np.uint32))
    qTo, sTo = oracle.quant_128x128(bits(w.t().contiguous()))
    assert np.array_equal(to_np(qT), qTo) and np.array_equal(to_np(sT).view(np.uint32), sTo.view(np.uint32))


def test_trio_full_size():
    x, w, dy = synth.trio(seed=0, device=DEV)
    M, K = x.shape
    N = w.shape[0]
    wq, sw = fg.fp8_quant_128x128(w)
    xq, sx = fg.fp8_quant_1x128(x)
    xqT, sxT = fg.fp8_quant_1x128(x, transpose=True)
    dyq, sdy = fg.fp8_quant_1x128(dy)
    dyqT, sdyT = fg.fp8_quant_1x128(dy, transpose=True)
    y = fg.fprop(xq, sx, wq, sw)
    dx = fg.dgrad(dyq, sdy, wq, sw)
    dw = fg.wgrad(dyqT, sdyT, xqT, sxT)
    assert fg.device_status() == 0
    torch.cuda.synchronize()

    wo, swo = oracle.quant_128x128(bits(w))
    assert np.array_equal(to_np(wq), wo) and np.array_equal(to_np(sw), swo)
    xo, sxo = assert_quant_1x128(x, xq, sx)
    dyo, sdyo = assert_quant_1x128(dy, dyq, sdy)
    xoT, sxoT = oracle.quant_128x1_t(bits(x))
    assert np.array_equal(to_np(xqT), xoT) and np.array_equal(to_np(sxT)[:, :K], sxoT)
    dyoT, sdyoT = oracle.quant_128x1_t(bits(dy))
    assert np.array_equal(to_np(dyqT), dyoT) and np.array_equal(to_np(sdyT)[:, :N], sdyoT)

    rows = _sample(M, 4, 1)
    idx = torch.from_numpy(rows).to(DEV)
    c, _, t = oracle.fprop(xo, sxo, wo, swo, rows=rows)
    check_gemm(to_np(y[idx]), c, t, True, "trio fprop")
    c, _, t = oracle.dgrad(dyo, sdyo, wo, swo, rows=rows)
    check_gemm(to_np(dx[idx]), c, t, True, "trio dgrad")
    wrows = _sample(N, 4, 2)
    c, _, t = oracle.wgrad(dyoT, sdyoT, xoT, sxoT, rows=wrows)
    check_gemm(to_np(dw[torch.from_numpy(wrows).to(DEV)]), c, t, False, "trio wgrad")


def test_moe_full_size():
    mo = synth.moe(seed=0, device=DEV)
    E, N, K = mo.w.shape
    R = int(mo.expert_offsets[-1].item())
    assert R == 4096 * 8
    xq, sx = fg.fp8_quant_1x128(mo.x)
    wq, sw = fg.fp8_quant_128x128(mo.w)
    y = fg.fp8_grouped_gemm(xq, sx, mo.row_index, mo.expert_offsets, wq, sw, R)
    assert fg.device_status() == 0
    torch.cuda.synchronize()

    xo, sxo = assert_quant_1x128(mo.x, xq, sx)
    off = mo.expert_offsets.cpu().numpy().astype(np.int64)
    ri = mo.row_index.cpu().numpy().astype(np.int64)
    counts = np.diff(off)
    # rows from the largest expert, a mid-sized one and single-row experts
    order = np.argsort(-counts, kind="stable")
    picks = [order[0], order[len(order) // 8], order[np.nonzero(counts[order] == 1)[0][0]]]
    rows = []
    for e in picks:
        rows += [off[e], off[e + 1] - 1]
    rows = np.unique(np.array(rows, np.int64))
    experts = np.searchsorted(off, rows, side="right") - 1
    wq_h, sw_h = {}, {}
    for e in np.unique(experts):
        e = int(e)
        wq_h[e], sw_h[e] = to_np(wq[e]), to_np(sw[e])
        we, swe = oracle.quant_128x128(bits(mo.w[e]))
        assert np.array_equal(wq_h[e], we) and np.array_equal(sw_h[e], swe)
    yh = to_np(y[torch.from_numpy(rows).to(DEV)])
    for r, e, yr in zip(rows, experts, yh):
        tok = ri[r:r + 1]
        c, _, t = oracle.fprop(xo[tok], sxo[tok], wq_h[int(e)], sw_h[int(e)])
        check_gemm(yr[None], c, t, True, "moe row %d expert %d" % (r, e))


def test_outliers_full_size():
    x, w, ch, bl = synth.outliers(seed=0, device=DEV)
    xq, sx = fg.fp8_quant_1x128(x)
    wq, sw = fg.fp8_quant_128x128(w)
    y = fg.fprop(xq, sx, wq, sw)
    assert fg.device_status() == 0
    torch.cuda.synchronize()
    xo, sxo = assert_quant_1x128(x, xq, sx)
    wo, swo = oracle.quant_128x128(bits(w))
    assert np.array_equal(to_np(wq), wo) and np.array_equal(to_np(sw), swo)
    # the scaled-up weight blocks carry 50x larger scales
    assert np.median(swo.reshape(-1)[bl.cpu().numpy()]) > 20 * np.median(swo)
    rows = _sample(x.shape[0], 5, 3)
    c, _, t = oracle.fprop(xo, sxo, wo, swo, rows=rows)
    check_gemm(to_np(y[torch.from_numpy(rows).to(DEV)]), c, t, True, "outliers")


def _moe_dest(mo):
    """The routing's token -> row index: the 8 rows of every token."""
    T = mo.x.shape[0]
    R = mo.row_index.numel()
    return torch.argsort(mo.row_index.long(), stable=True).to(torch.int32).reshape(T, R // T).contiguous()


def _moe_check_rows(mo, xo, sxo, wq, sw, y, pow2, what):
    """Sampled output rows (largest, a mid-sized and a single-row expert)
    against the oracle, token by token."""
    off = mo.expert_offsets.cpu().numpy().astype(np.int64)
    ri = mo.row_index.cpu().numpy().astype(np.int64)
    counts = np.diff(off)
    order = np.argsort(-counts, kind="stable")
    picks = [order[0], order[len(order) // 8], order[np.nonzero(counts[order] == 1)[0][0]]]
    rows = np.unique(np.array([r for e in picks for r in (off[e], off[e + 1] - 1)], np.int64))
    experts = np.searchsorted(off, rows, side="right") - 1
    yh = to_np(y[torch.from_numpy(rows).to(DEV)])
    for r, e, yr in zip(rows, experts, yh):
        e = int(e)
        we, swe = oracle.quant_128x128(bits(mo.w[e]), pow2=pow2)
        assert np.array_equal(to_np(wq[e]), we) and np.array_equal(to_np(sw[e]), swe)
        tok = ri[r:r + 1]
        c, _, t = oracle.fprop(xo[tok], sxo[tok], we, swe)
        check_gemm(yr[None], c, t, True, "%s row %d expert %d" % (what, r, e))


@pytest.mark.parametrize("pow2", [False, True])
def test_moe_full_size_dispatch_path(pow2):
    """The MoE step as bench.py times it: every token quantised once and
    scattered into expert order, then the grouped GEMM on contiguous rows
    (the promoted kernel, or the block-scaled one for power-of-two scales)."""
    mo = synth.moe(seed=0, device=DEV)
    R = mo.row_index.numel()
    xg, sxg = fg.fp8_quant_1x128_scatter(mo.x, _moe_dest(mo), R, pow2=pow2)
    wq, sw = fg.fp8_quant_128x128(mo.w, pow2=pow2)
    if pow2:
        y = fg.fp8_grouped_gemm_mx(xg, sxg, mo.expert_offsets, wq, sw, R)
    else:
        y = fg.fp8_grouped_gemm(xg, sxg, None, mo.expert_offsets, wq, sw, R)
    assert fg.device_status() == 0
    torch.cuda.synchronize()
    xo, sxo = oracle.quant_1x128(bits(mo.x), pow2=pow2)
    ri = mo.row_index.cpu().numpy().astype(np.int64)
    assert np.array_equal(to_np(xg), xo[ri])
    assert np.array_equal(to_np(sxg)[:, :R].T, sxo[ri])
    _moe_check_rows(mo, xo, sxo, wq, sw, y, pow2, "moe dispatch")


def test_trio_mx_full_size():
    """The training trio in the microscaling variant at full size."""
    x, w, dy = synth.trio(seed=0, device=DEV)
    M, K = x.shape
    N = w.shape[0]
    wq, sw = fg.fp8_quant_128x128(w, pow2=True)
    xq, sx, xqT, sxT = fg.fp8_quant_1x128_dual(x, pow2=True)
    dyq, sdy, dyqT, sdyT = fg.fp8_quant_1x128_dual(dy, pow2=True)
    y = fg.fp8_gemm_mx(fg.FPROP, xq, sx, wq, sw)
    dx = fg.fp8_gemm_mx(fg.DGRAD, dyq, sdy, wq, sw)
    dw = fg.fp8_gemm_mx(fg.WGRAD, dyqT, sdyT, xqT, sxT)
    assert fg.device_status() == 0
    torch.cuda.synchronize()

    wo, swo = oracle.quant_128x128(bits(w), pow2=True)
    assert np.array_equal(to_np(wq), wo) and np.array_equal(to_np(sw), swo)
    xo, sxo = oracle.quant_1x128(bits(x), pow2=True)
    assert np.array_equal(to_np(xq), xo) and np.array_equal(to_np(sx)[:, :M].T, sxo)
    dyo, sdyo = oracle.quant_1x128(bits(dy), pow2=True)
    assert np.array_equal(to_np(dyq), dyo) and np.array_equal(to_np(sdy)[:, :M].T, sdyo)
    xoT, sxoT = oracle.quant_128x1_t(bits(x), pow2=True)
    assert np.array_equal(to_np(xqT), xoT) and np.array_equal(to_np(sxT)[:, :K], sxoT)
    dyoT, sdyoT = oracle.quant_128x1_t(bits(dy), pow2=True)
    assert np.array_equal(to_np(dyqT), dyoT) and np.array_equal(to_np(sdyT)[:, :N], sdyoT)

    rows = _sample(M, 4, 4)
    idx = torch.from_numpy(rows).to(DEV)
    c, _, t = oracle.fprop(xo, sxo, wo, swo, rows=rows)
    check_gemm(to_np(y[idx]), c, t, True, "trio_mx fprop")
    c, _, t = oracle.dgrad(dyo, sdyo, wo, swo, rows=rows)
    check_gemm(to_np(dx[idx]), c, t, True, "trio_mx dgrad")
    wrows = _sample(N, 4, 5)
    c, _, t = oracle.wgrad(dyoT, sdyoT, xoT, sxoT, rows=wrows)
    check_gemm(to_np(dw[torch.from_numpy(wrows).to(DEV)]), c, t, False, "trio_mx wgrad")
