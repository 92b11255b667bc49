"""Element-by-element parity of the grouped GEMM's skinny tiles.

With rows in expert order, experts with at most 32 rows are computed as
256 weight rows x 32 token rows per tile (the weight as the tensor cores'
128-row operand), by part of the grid, while the other CTAs run the
128-row x 256-column tiles of the other experts. The cases:

- a routing with every row count at the boundaries (1, 2, 31, 32, 33, 64,
  127, 128, 129 and empty experts), skinny tiles on and off, FP32 and bf16
  output, an odd number of contraction blocks;
- only skinny experts (no full tiles: the whole grid takes skinny tiles),
  more skinny tiles than CTAs;
- N = 384 (the last skinny tile's second 128-row half lies past N) with
  an output pitch wider than N whose padding must stay untouched;
- the last expert's rows ending at the last token row (the 32-row token
  box runs past the buffer and is zero-filled);
- first rows of experts at every offset modulo 4 (the token-scale box
  starts at the 4-aligned row below);
- the MoE workload at full size, rows of skinny experts sampled against the
  oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_fine_grained_gb300 import synth
from tests.gpu_util import bits, check_gemm, to_np

pytestmark = pytest.mark.gpu

fg = pytest.importorskip("fp8_fine_grained_gb300")
DEV = "cuda"


@pytest.fixture
def schedule():
    """Restores the default schedule after the test."""
    yield fg.set_grouped_schedule
    fg.set_grouped_schedule()


def _gen(seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    return g


def _problem(seed, counts, K, N, T=None):
    """Token rows already in expert order: row r of Xq is output row r."""
    counts = np.asarray(counts, np.int64)
    R = int(counts.sum())
    T = R if T is None else T
    E = counts.size
    g = _gen(seed)
    x = torch.randn(T, K, generator=g, device=DEV) * torch.exp(torch.randn(T, 1, generator=g, device=DEV))
    x = x.to(torch.bfloat16)
    w = (torch.randn(E, N, K, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return x, w, off


def _run(x, w, off, out_dtype=torch.float32, y=None):
    R = int(off[-1])
    xq, sx = fg.fp8_quant_1x128(x)
    wq, sw = fg.fp8_quant_128x128(w)
    of = torch.from_numpy(off).to(DEV)
    y = fg.fp8_grouped_gemm(xq, sx, None, of, wq, sw, R, out_dtype=out_dtype, y=y)
    assert fg.device_status() == 0
    return xq, sx, wq, sw, y


def _check(x, w, xq, sx, wq, sw, off, y, bf16, what):
    """The oracle quantises X and every expert's weight itself (the
    kernels' codes and scales must equal its own) and forms every output
    row from its own operands."""
    R = int(off[-1])
    xo, sxo = oracle.quant_1x128(bits(x))
    assert np.array_equal(to_np(xq), xo)
    assert np.array_equal(to_np(sx)[:, :x.shape[0]].T.view(np.uint32), sxo.view(np.uint32))
    E = w.shape[0]
    wo = np.empty(tuple(w.shape), np.uint8)
    swo = np.empty(tuple(sw.shape), np.float32)
    for e in range(E):
        wo[e], swo[e] = oracle.quant_128x128(bits(w[e]))
    assert np.array_equal(to_np(wq), wo) and np.array_equal(to_np(sw), swo)
    c, _, t = oracle.grouped(xo, sxo, np.arange(R), off, wo, swo)
    check_gemm(to_np(y), c, t, bf16, what)


BOUNDARY = [1, 2, 31, 32, 33, 0, 64, 127, 128, 129, 0, 17, 5, 300, 32, 3]


@pytest.mark.parametrize("rows", [32, 0])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_boundary_row_counts(schedule, rows, out):
    schedule(rows, 100)
    x, w, off = _problem(61, BOUNDARY, K=384, N=768)
    dt = torch.float32 if out == "f32" else torch.bfloat16
    xq, sx, wq, sw, y = _run(x, w, off, dt)
    _check(x, w, xq, sx, wq, sw, off, y, out == "bf16", "boundary counts, skinny rows %d, %s" % (rows, out))


@pytest.mark.parametrize("cost", [1, 100, 1000])
def test_split_of_the_grid_does_not_change_results(schedule, cost):
    """The CTA split follows cost_pct (from one skinny CTA to all but one
    for the full tiles); every split gives the oracle's sums."""
    schedule(32, cost)
    rng = np.random.default_rng(62)
    counts = np.concatenate([rng.integers(1, 33, 150), rng.integers(100, 400, 6)])
    rng.shuffle(counts)
    x, w, off = _problem(62, counts, K=256, N=512)
    xq, sx, wq, sw, y = _run(x, w, off)
    _check(x, w, xq, sx, wq, sw, off, y, False, "split with cost %d%%" % cost)


@pytest.mark.parametrize("K", [256, 384])
def test_only_skinny_experts(K):
    """No full tiles: every CTA takes skinny tiles; 400 experts of 1..32
    rows x 2 tiles each, more than two per SM."""
    rng = np.random.default_rng(63)
    counts = rng.integers(1, 33, 400)
    counts[[0, 1, 2]] = [1, 32, 31]
    x, w, off = _problem(63 + K, counts, K=K, N=512)
    xq, sx, wq, sw, y = _run(x, w, off)
    _check(x, w, xq, sx, wq, sw, off, y, False, "only skinny experts, K %d" % K)


def test_half_width_n_and_output_pitch():
    """N = 384: the last skinny tile covers weight rows 256..511, of which
    the second 128-row half is past N; Y has a pitch of 400 columns whose
    last 16 must stay untouched."""
    counts = [5, 40, 32, 1, 0, 19]
    x, w, off = _problem(64, counts, K=256, N=384)
    R = int(off[-1])
    ybuf = torch.full((R, 400), 7.0, dtype=torch.float32, device=DEV)
    xq, sx, wq, sw, y = _run(x, w, off, y=ybuf[:, :384])
    assert torch.all(ybuf[:, 384:] == 7.0)
    _check(x, w, xq, sx, wq, sw, off, ybuf[:, :384], False, "N = 384, pitched output")


def test_last_rows_end_at_the_buffer_end():
    """The last expert's 3 rows are the last rows of Xq (T = R): its 32-row
    token box reads 29 rows past the end (zero-filled)."""
    counts = [200, 7, 3]
    x, w, off = _problem(65, counts, K=384, N=256)
    assert x.shape[0] == int(off[-1])
    xq, sx, wq, sw, y = _run(x, w, off)
    _check(x, w, xq, sx, wq, sw, off, y, False, "rows ending at the buffer end")


def test_expert_starts_at_every_offset_mod_4():
    counts = [1, 1, 1, 30, 2, 3, 29, 33, 4, 0, 6, 31]
    x, w, off = _problem(66, counts, K=256, N=256)
    assert set(int(v) % 4 for v in off[:-1]) == {0, 1, 2, 3}
    xq, sx, wq, sw, y = _run(x, w, off)
    _check(x, w, xq, sx, wq, sw, off, y, False, "expert starts modulo 4")


def test_moe_workload_skinny_experts_full_size():
    """The MoE workload (4096 tokens, 256 experts of 2048 x 7168, top-8)
    with rows in expert order: every row of the four smallest non-empty
    experts and first/last rows of others up to 32 rows, all 2048 columns,
    against the oracle."""
    mo = synth.moe(seed=0, device=DEV)
    R = mo.row_index.numel()
    xg, sxg = fg.fp8_quant_1x128_gather(mo.x, mo.row_index)
    wq, sw = fg.fp8_quant_128x128(mo.w)
    y = fg.fp8_grouped_gemm(xg, sxg, None, mo.expert_offsets, wq, sw, R)
    assert fg.device_status() == 0
    torch.cuda.synchronize()
    off = mo.expert_offsets.cpu().numpy().astype(np.int64)
    counts = np.diff(off)
    skinny = np.nonzero((counts > 0) & (counts <= 32))[0]
    assert skinny.size > 50
    order = skinny[np.argsort(counts[skinny], kind="stable")]
    rows = [r for e in order[:4] for r in range(off[e], off[e + 1])]
    for e in order[4::12]:
        rows += [off[e], off[e + 1] - 1]
    rows = np.unique(np.array(rows, np.int64))
    xo, sxo = oracle.quant_1x128(bits(mo.x))
    ri = mo.row_index.cpu().numpy().astype(np.int64)
    experts = np.searchsorted(off, rows, side="right") - 1
    yh = to_np(y[torch.from_numpy(rows).to(DEV)])
    for e in np.unique(experts):
        e = int(e)
        we, swe = oracle.quant_128x128(bits(mo.w[e]))
        assert np.array_equal(to_np(wq[e]), we) and np.array_equal(to_np(sw[e]), swe)
        pick = np.nonzero(experts == e)[0]
        toks = ri[rows[pick]]
        c, _, t = oracle.fprop(xo[toks], sxo[toks], we, swe)
        check_gemm(yh[pick], c, t, True, "moe skinny expert %d (%d rows)" % (e, counts[e]))
