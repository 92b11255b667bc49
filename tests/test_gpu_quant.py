"""GPU parity of the quantisation kernels against the CPU oracle: codes and
scales must match bit for bit (every case on the same seeded bf16 input)."""
import numpy as np
import pytest
import torch

import oracle
from fp8_fine_grained_gb300 import synth
from tests.gpu_util import assert_quant_1x128, bits, rows_scales, to_np

pytestmark = pytest.mark.gpu

fg = pytest.importorskip("fp8_fine_grained_gb300")
DEV = "cuda"


def _x(rows, cols, seed, std=1.0):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    c = torch.exp(torch.randn(cols, generator=g, device=DEV))
    return (torch.randn(rows, cols, generator=g, device=DEV) * c * std).to(torch.bfloat16)


@pytest.mark.parametrize("rows,cols", [(1, 128), (31, 256), (32, 512), (33, 640), (127, 128), (129, 1024),
                                       (300, 896), (1000, 7168)])
def test_quant_1x128_rows(rows, cols):
    x = _x(rows, cols, seed=rows * 7 + cols)
    q, s = fg.fp8_quant_1x128(x)
    torch.cuda.synchronize()
    assert_quant_1x128(x, q, s)


def test_quant_1x128_strided_input_and_padded_outputs():
    base = _x(70, 384 + 64, seed=3)
    x = base[:, :384]                     # ldx = 448
    q = torch.full((70, 512), 0xAA, dtype=torch.uint8, device=DEV)   # ldq = 512
    s = torch.full((3, 76), -1.0, dtype=torch.float32, device=DEV)     # ld_s = 76
    fg.fp8_quant_1x128(x, q=q[:, :384], scales=s)
    torch.cuda.synchronize()
    assert_quant_1x128(x.contiguous(), q[:, :384], s)
    assert torch.all(q[:, 384:] == 0xAA) and torch.all(s[:, 70:] == -1.0)   # padding untouched


def test_quant_1x128_special_values():
    rows, cols = 8, 512
    x = torch.zeros(rows, cols, dtype=torch.float32)
    x[1, :128] = -0.0                               # all-zero group with negative zeros
    x[2, 5] = 2.0 ** -133                           # smallest bf16 subnormal: 448/amax overflows
    x[3, :] = 448.0 * 2.0 ** -3                     # amax = 448 * 2^e
    x[4, 128:256] = torch.linspace(-1.0, 1.0, 128) * 3e38  # near the bf16 maximum (finite)
    x[5, :] = torch.arange(cols) * 1e-30            # tiny normals
    x[6, 256:] = 1e-39                              # fp32 subnormal inputs
    x[7, :] = torch.tensor([(-1.0) ** i * (i % 17) for i in range(cols)])
    xb = x.to(torch.bfloat16).to(DEV)
    q, s = fg.fp8_quant_1x128(xb)
    torch.cuda.synchronize()
    assert_quant_1x128(xb, q, s)


@pytest.mark.parametrize("rows,cols", [(128, 1), (128, 64), (128, 100), (256, 200), (384, 640), (1024, 7168)])
def test_quant_transposed(rows, cols):
    # the row pitch must be a multiple of 8 elements: ragged widths are views
    # into a wider buffer
    pitch = (cols + 7) // 8 * 8
    x = _x(rows, pitch, seed=rows + cols)[:, :cols]
    q, s = fg.fp8_quant_1x128(x, transpose=True)
    torch.cuda.synchronize()
    qo, so = oracle.quant_128x1_t(bits(x))
    assert np.array_equal(to_np(q), qo)
    assert np.array_equal(to_np(s)[:, :cols].view(np.uint32), so.view(np.uint32))


@pytest.mark.parametrize("N,K", [(128, 128), (384, 640), (1024, 7168)])
def test_quant_128x128(N, K):
    g = torch.Generator(device=DEV)
    g.manual_seed(N + K)
    w = (torch.randn(N, K, generator=g, device=DEV) * 0.02)
    w[:128, :128] *= 50
    w[128:, :128] = 0.0 if N > 128 else w[128:, :128]
    w = w.to(torch.bfloat16)
    q, s = fg.fp8_quant_128x128(w)
    torch.cuda.synchronize()
    qo, so = oracle.quant_128x128(bits(w))
    assert np.array_equal(to_np(q), qo)
    assert np.array_equal(to_np(s).view(np.uint32), so.view(np.uint32))


@pytest.mark.parametrize("N,K", [(128, 128), (256, 384), (384, 256), (1024, 2048)])
@pytest.mark.parametrize("pow2", [False, True])
def test_quant_128x128_dual(N, K, pow2):
    """Both the weight's blocks and those of its transpose from one read:
    q and scales equal the oracle's quantisation of W, qT and scalesT the
    oracle's quantisation of the materialised W^T (computed independently,
    not by transposing q)."""
    g = torch.Generator(device=DEV)
    g.manual_seed(N * 3 + K + pow2)
    w = (torch.randn(N, K, generator=g, device=DEV) * 0.02)
    w[:128, -128:] *= 40
    w = w.to(torch.bfloat16)
    q, s, qT, sT = fg.fp8_quant_128x128_dual(w, pow2=pow2)
    torch.cuda.synchronize()
    qo, so = oracle.quant_128x128(bits(w), pow2=pow2)
    qTo, sTo = oracle.quant_128x128(bits(w.t().contiguous()), pow2=pow2)
    assert np.array_equal(to_np(q), qo)
    assert np.array_equal(to_np(s).view(np.uint32), so.view(np.uint32))
    assert np.array_equal(to_np(qT), qTo)
    assert np.array_equal(to_np(sT).view(np.uint32), sTo.view(np.uint32))


def test_quant_128x128_dual_pitched_outputs():
    """Output pitches larger than the matrix: the padding stays untouched."""
    g = torch.Generator(device=DEV)
    g.manual_seed(9)
    w = (torch.randn(256, 384, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    qbuf = torch.full((256, 400), 7, dtype=torch.uint8, device=DEV)
    qTbuf = torch.full((384, 272), 7, dtype=torch.uint8, device=DEV)
    q, s, qT, sT = fg.fp8_quant_128x128_dual(w, q=qbuf[:, :384], qT=qTbuf[:, :256])
    torch.cuda.synchronize()
    assert torch.all(qbuf[:, 384:] == 7) and torch.all(qTbuf[:, 256:] == 7)
    qo, _ = oracle.quant_128x128(bits(w))
    assert np.array_equal(to_np(qbuf[:, :384]), qo) and np.array_equal(to_np(qTbuf[:, :256]), qo.T)


def test_quant_128x128_experts_3d():
    g = torch.Generator(device=DEV)
    g.manual_seed(5)
    w = (torch.randn(3, 256, 384, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    q, s = fg.fp8_quant_128x128(w)
    torch.cuda.synchronize()
    for e in range(3):
        qo, so = oracle.quant_128x128(bits(w[e]))
        assert np.array_equal(to_np(q[e]), qo)
        assert np.array_equal(to_np(s[e]), so)


def test_quant_dense_full_size():
    """Full-size activation of the dense projection workload (4096 x 7168,
    log-normal channel magnitudes), bit-exact against the oracle."""
    x, w = synth.dense(seed=0, device=DEV)
    q, s = fg.fp8_quant_1x128(x)
    torch.cuda.synchronize()
    assert_quant_1x128(x, q, s)
    wq, sw = fg.fp8_quant_128x128(w)
    torch.cuda.synchronize()
    qo, so = oracle.quant_128x128(bits(w))
    assert np.array_equal(to_np(wq), qo) and np.array_equal(to_np(sw), so)


@pytest.mark.parametrize("rows,cols", [(128, 128), (256, 384), (640, 1024), (1024, 7168)])
def test_quant_dual(rows, cols):
    """One read, both layouts: bit-identical to the oracle's 1x128 row
    quantisation and its transposed 128x1 quantisation."""
    x = _x(rows, cols, seed=rows + 3 * cols)
    q, s, qT, sT = fg.fp8_quant_1x128_dual(x)
    assert fg.device_status() == 0
    assert_quant_1x128(x, q, s)
    qo, so = oracle.quant_128x1_t(bits(x))
    assert np.array_equal(to_np(qT), qo)
    assert np.array_equal(to_np(sT)[:, :cols].view(np.uint32), so.view(np.uint32))


def test_quant_dual_timeout_is_reported_not_hung():
    """The dual quantiser's bounded wait on its TMA tile: a withheld copy
    (test hook) makes it run out, the launch reports FP8FG_ETIMEOUT, and the
    next launch is clean and bit-exact."""
    x = _x(1024, 1024, seed=3)
    fg.set_wait_limit_ns(50_000_000)
    try:
        fg.inject_skip_first_load(True)
        fg.fp8_quant_1x128_dual(x)
        assert fg.device_status() == 5  # FP8FG_ETIMEOUT
        q, s, qT, sT = fg.fp8_quant_1x128_dual(x)
        assert fg.device_status() == 0
    finally:
        fg.set_wait_limit_ns(2_000_000_000)
    assert_quant_1x128(x, q, s)
    qo, so = oracle.quant_128x1_t(bits(x))
    assert np.array_equal(to_np(qT), qo) and np.array_equal(to_np(sT)[:, :1024].view(np.uint32), so.view(np.uint32))


def test_quant_dual_pitched_outputs():
    base = _x(256, 640, seed=9)
    x = base[:, :512]
    q = torch.zeros((256, 528), dtype=torch.uint8, device=DEV)[:, :512]
    qT = torch.zeros((512, 272), dtype=torch.uint8, device=DEV)[:, :256]
    fg.fp8_quant_1x128_dual(x, q=q, qT=qT)
    torch.cuda.synchronize()
    qo, _ = oracle.quant_1x128(bits(x))
    assert np.array_equal(to_np(q), qo)
    qto, _ = oracle.quant_128x1_t(bits(x))
    assert np.array_equal(to_np(qT), qto)


@pytest.mark.parametrize("n_src,rows,cols", [(300, 1, 128), (300, 777, 384), (64, 1000, 7168)])
def test_quant_1x128_gather(n_src, rows, cols):
    """Rows quantised in row-index order (with repeats, as top-k routing
    makes them) equal the oracle's 1x128 quantisation of those rows."""
    x = _x(n_src, cols, seed=n_src + rows + cols)
    ri = np.random.default_rng(rows).integers(0, n_src, rows).astype(np.int32)
    q, s = fg.fp8_quant_1x128_gather(x, torch.from_numpy(ri).to(DEV))
    assert fg.device_status() == 0
    qo, so = oracle.quant_1x128(bits(x)[ri])
    assert np.array_equal(to_np(q), qo)
    assert np.array_equal(rows_scales(s, rows).view(np.uint32), so.view(np.uint32))


def test_quant_1x128_gather_bad_index_reported():
    x = _x(16, 256, seed=5)
    ri = np.array([3, 10 ** 6, 0], np.int32)
    q, s = fg.fp8_quant_1x128_gather(x, torch.from_numpy(ri).to(DEV))
    assert fg.device_status() == 6  # FP8FG_EDEVICE; the bad row reads source row 0
    qo, _ = oracle.quant_1x128(bits(x)[[3, 0, 0]])
    assert np.array_equal(to_np(q), qo)


def _routing(n_src, k, seed):
    """Destinations of k copies of every source row, grouped by expert the
    way top-k routing makes them: a random permutation of n_src*k rows."""
    perm = np.random.default_rng(seed).permutation(n_src * k).astype(np.int32)
    return perm.reshape(n_src, k)


@pytest.mark.parametrize("n_src,k,cols", [(1, 1, 128), (37, 8, 384), (300, 3, 7168), (4096, 8, 1024)])
@pytest.mark.parametrize("pow2", [False, True])
def test_quant_1x128_scatter(n_src, k, cols, pow2):
    """Every source row quantised once and written to its k destination rows
    equals the oracle's 1x128 quantisation of the gathered rows."""
    x = _x(n_src, cols, seed=n_src + k + cols)
    dest = _routing(n_src, k, seed=n_src * k)
    n_out = n_src * k
    q, s = fg.fp8_quant_1x128_scatter(x, torch.from_numpy(dest).to(DEV), n_out, pow2=pow2)
    assert fg.device_status() == 0
    src_of = np.empty(n_out, np.int64)
    src_of[dest.reshape(-1)] = np.repeat(np.arange(n_src), k)
    qo, so = oracle.quant_1x128(bits(x)[src_of], pow2=pow2)
    assert np.array_equal(to_np(q), qo)
    assert np.array_equal(rows_scales(s, n_out).view(np.uint32), so.view(np.uint32))


def test_quant_1x128_scatter_skips_and_reports():
    """Negative destinations are not written and leave their rows untouched;
    a destination past the output is reported and not written."""
    x = _x(8, 256, seed=7)
    dest = np.array([[0, -1], [3, 1], [-1, -1], [2, 50], [4, 5], [6, 7], [8, 9], [10, 11]], np.int32)
    n_out = 12
    q = torch.full((n_out, 256), 0xAB, dtype=torch.uint8, device=DEV)
    s = torch.full((2, 12), -1.0, dtype=torch.float32, device=DEV)
    fg.fp8_quant_1x128_scatter(x, torch.from_numpy(dest).to(DEV), n_out, q=q, scales=s)
    assert fg.device_status() == 6  # FP8FG_EDEVICE for the 50
    qo, so = oracle.quant_1x128(bits(x))
    qg, sg = to_np(q), to_np(s)
    for r in range(8):
        for d in dest[r]:
            if 0 <= d < n_out:
                assert np.array_equal(qg[d], qo[r])
                assert np.array_equal(sg[:, d], so[r])
    untouched = sorted(set(range(n_out)) - {int(d) for d in dest.reshape(-1) if 0 <= d < n_out})
    for d in untouched:
        assert np.all(qg[d] == 0xAB) and np.all(sg[:, d] == -1.0)


def test_quant_zero_size_is_noop():
    x = torch.empty(0, 256, dtype=torch.bfloat16, device=DEV)
    q, s = fg.fp8_quant_1x128(x)
    assert q.shape == (0, 256)
