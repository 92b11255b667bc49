"""Element-by-element parity of the persistent GEMMs when every CTA runs
several output tiles.

The GEMM kernels keep one CTA per SM and walk the tile space with a stride
of the grid size, carrying the tensor-memory buffer index and its barrier
phases from one tile to the next. These cases give every CTA two to four
tiles, an odd number of 128-wide contraction blocks (so a CTA's second tile
starts on the other accumulator buffer), a ragged last row tile, and they
compare every output element with the oracle:

- fprop, dgrad and wgrad at about 3x the SM count in 128x256 tiles with
  three contraction blocks;
- the grouped MoE GEMM (row-index and expert-order forms) with more than
  400 tiles over experts of 0..400 rows; with 100 experts all inside one
  128-row tile (500 tiles); and with 2100 and 4096 experts, 40 of them
  routed (some past expert 2047);
- the whole dense projection workload (4096 x 7168 x 7168, bf16 out), all
  rows;
- the full-size training trio quantised by the dual-output quantiser, as
  the benchmark times it (both layouts bit-exact at full size).
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

# 4000 rows = 31 full 128-row tiles + a 32-row tail; 3840 columns = 15 tiles
# of 256; 32 x 15 = 480 tiles, more than three per SM on a 152-SM part
MW_M, MW_N, MW_K = 4000, 3840, 384


def _gen(seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    return g


def _act(M, K, seed):
    g = _gen(seed)
    c = torch.exp(torch.randn(K, generator=g, device=DEV))
    return (torch.randn(M, K, generator=g, device=DEV) * c).to(torch.bfloat16)


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def test_shapes_give_several_tiles_per_sm():
    tiles = -(-MW_M // 128) * (MW_N // 256)
    assert tiles >= 3 * _sms()
    assert (MW_K // 128) % 2 == 1


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_fprop_multiwave(out):
    x = _act(MW_M, MW_K, seed=101)
    w = (torch.randn(MW_N, MW_K, generator=_gen(102), device=DEV) * 0.02).to(torch.bfloat16)
    xq, sx = fg.fp8_quant_1x128(x)
    wq, sw = fg.fp8_quant_128x128(w)
    dt = torch.float32 if out == "f32" else torch.bfloat16
    y = fg.fprop(xq, sx, wq, sw, out_dtype=dt)
    assert fg.device_status() == 0
    xo, sxo = assert_quant_1x128(x, xq, sx)
    wo, swo = oracle.quant_128x128(bits(w))
    assert np.array_equal(to_np(wq), wo) and np.array_equal(to_np(sw), swo)
    c, _, t = oracle.fprop(xo, sxo, wo, swo)
    check_gemm(to_np(y), c, t, out == "bf16", "fprop multiwave")


def test_dgrad_multiwave():
    """dX[4000, 3840] = dY[4000, 384] . W[384, 3840], W read as stored."""
    dy = (torch.randn(MW_M, MW_K, generator=_gen(103), device=DEV) * 1e-3).to(torch.bfloat16)
    w = (torch.randn(MW_K, MW_N, generator=_gen(104), device=DEV) * 0.02).to(torch.bfloat16)
    dyq, sdy = fg.fp8_quant_1x128(dy)
    wq, sw = fg.fp8_quant_128x128(w)
    dx = fg.dgrad(dyq, sdy, wq, sw, out_dtype=torch.float32)
    assert fg.device_status() == 0
    dyo, sdyo = assert_quant_1x128(dy, dyq, sdy)
    wo, swo = oracle.quant_128x128(bits(w))
    assert np.array_equal(to_np(wq), wo) and np.array_equal(to_np(sw), swo)
    c, _, t = oracle.dgrad(dyo, sdyo, wo, swo)
    check_gemm(to_np(dx), c, t, False, "dgrad multiwave")


def test_wgrad_multiwave():
    """dW[4000, 3840] = dY^T X over 384 tokens (three token groups)."""
    x = _act(MW_K, MW_N, seed=105)
    dy = (torch.randn(MW_K, MW_M, generator=_gen(106), device=DEV) * 1e-3).to(torch.bfloat16)
    xqT, sxT = fg.fp8_quant_1x128(x, transpose=True)
    dyqT, sdyT = fg.fp8_quant_1x128(dy, transpose=True)
    dw = fg.wgrad(dyqT, sdyT, xqT, sxT)
    assert fg.device_status() == 0
    xo, sxo = oracle.quant_128x1_t(bits(x))
    dyo, sdyo = oracle.quant_128x1_t(bits(dy))
    assert np.array_equal(to_np(xqT), xo) and np.array_equal(to_np(dyqT), dyo)
    assert np.array_equal(to_np(sxT)[:, :MW_N], sxo) and np.array_equal(to_np(sdyT)[:, :MW_M], sdyo)
    c, _, t = oracle.wgrad(dyo, sdyo, xo, sxo)
    check_gemm(to_np(dw), c, t, False, "wgrad multiwave")


def _moe_many(seed, T=1000, K=384, N=1280, E=48):
    g = _gen(seed)
    x = torch.randn(T, K, generator=g, device=DEV).to(torch.bfloat16)
    w = (torch.randn(E, N, K, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    rng = np.random.default_rng(seed)
    counts = rng.integers(0, 401, E)
    counts[[3, 17, 30]] = 0                      # empty experts
    counts[[5, 6]] = [1, 128]                    # a single row, an exact tile
    row_index = np.concatenate([np.sort(rng.choice(T, c, replace=False)) if c else np.zeros(0, np.int64)
                                for c in counts]).astype(np.int32)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return x, w, row_index, off


def test_grouped_multiwave_shape():
    _, _, _, off = _moe_many(seed=31)
    tiles = int(sum(-(-int(c) // 128) for c in np.diff(off))) * (1280 // 256)
    assert tiles >= 400


@pytest.mark.parametrize("form", ["row_index", "expert_order"])
def test_grouped_multiwave(form):
    x, w, row_index, off = _moe_many(seed=31)
    R = int(off[-1])
    wq, sw = fg.fp8_quant_128x128(w)
    of = torch.from_numpy(off).to(DEV)
    ri = torch.from_numpy(row_index).to(DEV)
    if form == "row_index":
        xq, sx = fg.fp8_quant_1x128(x)
        y = fg.fp8_grouped_gemm(xq, sx, ri, of, wq, sw, n_rows=R, out_dtype=torch.float32)
    else:
        xg, sxg = fg.fp8_quant_1x128_gather(x, ri)
        y = fg.fp8_grouped_gemm(xg, sxg, None, of, wq, sw, n_rows=R, out_dtype=torch.float32)
    assert fg.device_status() == 0
    xo, sxo = oracle.quant_1x128(bits(x))
    if form == "row_index":
        assert np.array_equal(to_np(xq), xo)
    else:
        assert np.array_equal(to_np(xg), xo[row_index])
    wo, swo = to_np(wq), to_np(sw)
    for e in (0, 5, 6, w.shape[0] - 1):
        qe, se = oracle.quant_128x128(bits(w[e]))
        assert np.array_equal(wo[e], qe) and np.array_equal(swo[e], se)
    c, _, t = oracle.grouped(xo, sxo, row_index, off, wo, swo)
    check_gemm(to_np(y), c, t, False, "grouped multiwave (%s)" % form)


def _grouped_against_oracle(x, w, row_index, off, form, what):
    R = int(off[-1])
    wq, sw = fg.fp8_quant_128x128(w)
    of = torch.from_numpy(off).to(DEV)
    ri = torch.from_numpy(row_index).to(DEV)
    if form == "row_index":
        xq, sx = fg.fp8_quant_1x128(x)
        y = fg.fp8_grouped_gemm(xq, sx, ri, of, wq, sw, n_rows=R, out_dtype=torch.float32)
    else:
        xq, sx = fg.fp8_quant_1x128_gather(x, ri)
        y = fg.fp8_grouped_gemm(xq, sx, None, of, wq, sw, n_rows=R, out_dtype=torch.float32)
    assert fg.device_status() == 0
    xo, sxo = oracle.quant_1x128(bits(x))
    wo, swo = to_np(wq), to_np(sw)
    for e in np.flatnonzero(np.diff(off))[:3]:
        qe, se = oracle.quant_128x128(bits(w[int(e)]))
        assert np.array_equal(wo[e], qe) and np.array_equal(swo[e], se)
    c, _, t = oracle.grouped(xo, sxo, row_index, off, wo, swo)
    check_gemm(to_np(y), c, t, False, what)


def _routing(rng, T, counts):
    row_index = np.concatenate([np.sort(rng.choice(T, c, replace=False)) if c else np.zeros(0, np.int64)
                                for c in counts]).astype(np.int32)
    return row_index, np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)


@pytest.mark.parametrize("form", ["row_index", "expert_order"])
def test_grouped_multiwave_single_class(form):
    """100 experts of 1..128 rows: every expert is one m-tile."""
    E, T, K, N = 100, 1000, 384, 1280
    g = _gen(41)
    x = torch.randn(T, K, generator=g, device=DEV).to(torch.bfloat16)
    w = (torch.randn(E, N, K, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    rng = np.random.default_rng(41)
    counts = rng.integers(1, 129, E)
    counts[[0, 1]] = [1, 128]
    row_index, off = _routing(rng, T, counts)
    assert E * (N // 256) >= 400
    _grouped_against_oracle(x, w, row_index, off, form, "grouped, one-m-tile experts (%s)" % form)


@pytest.mark.parametrize("form", ["row_index", "expert_order"])
@pytest.mark.parametrize("E", [2100, 4096])
def test_grouped_many_experts_plain_order(form, E):
    """2100 or 4096 experts (the most the ABI takes), 40 of them routed,
    some past expert 2047."""
    T, K, N = 1000, 384, 256
    g = _gen(42)
    x = torch.randn(T, K, generator=g, device=DEV).to(torch.bfloat16)
    w = (torch.randn(E, N, K, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    rng = np.random.default_rng(42)
    counts = np.zeros(E, np.int64)
    used = np.concatenate([rng.choice(2048, 30, replace=False), 2048 + rng.choice(E - 2048, 10, replace=False)])
    counts[used] = rng.integers(1, 400, used.size)
    counts[E - 1] = 129
    row_index, off = _routing(rng, T, counts)
    _grouped_against_oracle(x, w, row_index, off, form, "grouped, %d experts (%s)" % (E, form))


def test_dense_config_every_element():
    """The dense projection workload at full size, every output element."""
    x, w = synth.dense(seed=0, device=DEV)
    xq, sx = fg.fp8_quant_1x128(x)
    wq, sw = fg.fp8_quant_128x128(w)
    y = fg.fprop(xq, sx, wq, sw)
    assert fg.device_status() == 0
    xo, sxo = assert_quant_1x128(x, xq, sx)
    wo, swo = oracle.quant_128x128(bits(w))
    assert np.array_equal(to_np(wq), wo) and np.array_equal(to_np(sw), swo)
    c, _, t = oracle.fprop(xo, sxo, wo, swo)
    check_gemm(to_np(y), c, t, True, "dense config, all rows")


def test_trio_full_size_dual_quantiser():
    """The training trio as the benchmark times it: X and dY quantised by
    the dual-output quantiser (both layouts from one read, bit-exact at full
    size), W in 128x128 blocks; GEMMs on sampled rows."""
    x, w, dy = synth.trio(seed=0, device=DEV)
    M, K = x.shape
    N = w.shape[0]
    wq, sw = fg.fp8_quant_128x128(w)
    xq, sx, xqT, sxT = fg.fp8_quant_1x128_dual(x)
    dyq, sdy, dyqT, sdyT = fg.fp8_quant_1x128_dual(dy)
    y = fg.fprop(xq, sx, wq, sw)
    dx = fg.dgrad(dyq, sdy, wq, sw)
    dw = fg.wgrad(dyqT, sdyT, xqT, sxT)
    assert fg.device_status() == 0

    wo, swo = oracle.quant_128x128(bits(w))
    assert np.array_equal(to_np(wq), wo) and np.array_equal(to_np(sw), swo)
    xo, sxo = assert_quant_1x128(x, xq, sx)
    dyo, sdyo = assert_quant_1x128(dy, dyq, sdy)
    xoT, sxoT = oracle.quant_128x1_t(bits(x))
    assert np.array_equal(to_np(xqT), xoT)
    assert np.array_equal(to_np(sxT)[:, :K].view(np.uint32), sxoT.view(np.uint32))
    dyoT, sdyoT = oracle.quant_128x1_t(bits(dy))
    assert np.array_equal(to_np(dyqT), dyoT)
    assert np.array_equal(to_np(sdyT)[:, :N].view(np.uint32), sdyoT.view(np.uint32))

    rng = np.random.default_rng(7)
    rows = np.unique(np.concatenate([rng.choice(M, 6, replace=False), [0, 127, 128, M - 1]]))
    idx = torch.from_numpy(rows).to(DEV)
    c, _, t = oracle.fprop(xo, sxo, wo, swo, rows=rows)
    check_gemm(to_np(y[idx]), c, t, True, "trio fprop (dual-quantised X)")
    c, _, t = oracle.dgrad(dyo, sdyo, wo, swo, rows=rows)
    check_gemm(to_np(dx[idx]), c, t, True, "trio dgrad (dual-quantised dY)")
    wrows = np.unique(np.concatenate([rng.choice(N, 6, replace=False), [0, 255, 256, N - 1]]))
    c, _, t = oracle.wgrad(dyoT, sdyoT, xoT, sxoT, rows=wrows)
    check_gemm(to_np(dw[torch.from_numpy(wrows).to(DEV)]), c, t, False, "trio wgrad (dual-quantised)")


@pytest.mark.parametrize("form", ["row_index", "expert_order"])
def test_grouped_half_width_last_tile(form):
    """N = 384: every expert's last n-tile holds 128 columns of 256."""
    E, T, K, N = 6, 700, 256, 384
    g = _gen(43)
    x = torch.randn(T, K, generator=g, device=DEV).to(torch.bfloat16)
    w = (torch.randn(E, N, K, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    rng = np.random.default_rng(43)
    counts = np.array([0, 1, 127, 128, 129, 300])
    row_index, off = _routing(rng, T, counts)
    _grouped_against_oracle(x, w, row_index, off, form, "grouped, N = 384 (%s)" % form)
