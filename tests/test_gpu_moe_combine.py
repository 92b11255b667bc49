"""GPU parity of the MoE combine (fp8_moe_combine) and of the one-GPU MoE
layer forward (FP8 dispatch by scatter-quantisation, the grouped expert
GEMM, the combine), against the CPU oracle.

The combine is specified bit for bit (FP32 products and sums in slot order,
no fused multiply-add, then bf16 rounding), so the kernel's output is
compared exactly with the oracle's on the same bf16 expert rows."""
import numpy as np
import pytest
import torch

import oracle
from fp8_fine_grained_gb300 import ep, synth
from tests.gpu_util import assert_quant_1x128, bits, check_gemm, to_np

pytestmark = pytest.mark.gpu

fg = pytest.importorskip("fp8_fine_grained_gb300")
DEV = "cuda"


def _gen(seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    return g


def _case(T, k, rows, N, seed, skip_frac=0.1):
    g = _gen(seed)
    y = (torch.randn(rows, N, generator=g, device=DEV) * torch.exp(torch.randn(rows, 1, generator=g, device=DEV))
         ).to(torch.bfloat16)
    dest = torch.randint(0, rows, (T, k), generator=g, device=DEV, dtype=torch.int32)
    drop = torch.rand(T, k, generator=g, device=DEV) < skip_frac
    dest = torch.where(drop, torch.full_like(dest, -1), dest)
    w = torch.rand(T, k, generator=g, device=DEV)
    return y, dest, w


@pytest.mark.parametrize("T,k,rows,N", [(1, 1, 1, 8), (37, 8, 100, 136), (300, 3, 50, 2048), (64, 16, 1000, 512)])
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_combine_bit_exact(T, k, rows, N, out):
    y, dest, w = _case(T, k, rows, N, seed=T * 7 + k)
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    got = fg.fp8_moe_combine(y, dest, w, out_dtype=dt)
    assert fg.device_status() == 0
    ref = oracle.moe_combine(bits(y), to_np(dest), to_np(w), out_f32=out == "f32")
    g = to_np(got) if out == "f32" else bits(got)
    assert np.array_equal(g.view(np.uint32 if out == "f32" else np.uint16),
                          ref.view(np.uint32 if out == "f32" else np.uint16))


def test_combine_output_pitch_and_untouched_padding():
    y, dest, w = _case(20, 4, 30, 128, seed=5)
    out = torch.full((20, 160), 3.0, dtype=torch.bfloat16, device=DEV)
    fg.fp8_moe_combine(y, dest, w, out=out[:, :128])
    assert fg.device_status() == 0
    assert torch.all(out[:, 128:] == 3.0)
    ref = oracle.moe_combine(bits(y), to_np(dest), to_np(w))
    assert np.array_equal(bits(out[:, :128]), ref)


def test_combine_reports_a_row_out_of_range():
    y, dest, w = _case(8, 2, 10, 64, seed=6, skip_frac=0.0)
    bad = dest.clone()
    bad[3, 1] = 10 ** 6
    fg.fp8_moe_combine(y, bad, w)
    assert fg.device_status() == 6  # FP8FG_EDEVICE
    assert fg.device_status() == 0  # cleared


def test_combine_full_moe_size():
    """4096 tokens, top-8, 2048-wide expert rows (the MoE workload)."""
    y, dest, w = _case(4096, 8, 32768, 2048, seed=7, skip_frac=0.0)
    got = fg.fp8_moe_combine(y, dest, w)
    assert fg.device_status() == 0
    rows = np.unique(np.concatenate([np.random.default_rng(0).choice(4096, 64, replace=False), [0, 4095]]))
    ref = oracle.moe_combine(bits(y), to_np(dest)[rows], to_np(w)[rows])
    assert np.array_equal(bits(got)[rows], ref)


def _layer_inputs(seed, T=300, K=384, N=512, E=16, topk=4):
    g = _gen(seed)
    x = torch.randn(T, K, generator=g, device=DEV).to(torch.bfloat16)
    w = (torch.randn(E, N, K, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    logits = torch.randn(T, E, generator=g, device=DEV)
    ids = torch.topk(logits, topk, dim=1).indices.to(torch.int32)
    gate = torch.softmax(torch.gather(logits, 1, ids.long()), dim=1).float().contiguous()
    return x, w, ids.contiguous(), gate


def test_moe_layer_one_gpu_against_the_oracle():
    x, w, ids, gate = _layer_inputs(seed=11)
    E = w.shape[0]
    wq, sw = fg.fp8_quant_128x128(w)
    out = ep.moe_forward(x, ids, gate, wq, sw, E)
    assert fg.device_status() == 0
    # the same steps one by one: dispatch (scatter-quantise), expert GEMM, combine
    plan = ep.plan_dispatch(ids, E, 1)
    q_send, s_send = fg.fp8_quant_1x128_scatter(x, plan.dest, plan.n_send)
    off = torch.zeros(E + 1, dtype=torch.int32, device=DEV)
    off[1:] = torch.cumsum(plan.send_counts[0], 0).to(torch.int32)
    y = fg.fp8_grouped_gemm(q_send, s_send, None, off, wq, sw, plan.n_send)
    comb = fg.fp8_moe_combine(y, plan.dest, gate)
    assert fg.device_status() == 0
    assert torch.equal(out, comb)                      # moe_forward runs exactly these kernels
    # dispatch: the send rows are the tokens' 1x128 codes and scales, bit-exact
    xo, sxo = oracle.quant_1x128(bits(x))
    dest = to_np(plan.dest)
    tok = np.empty(plan.n_send, np.int64)
    for t in range(dest.shape[0]):
        for j in range(dest.shape[1]):
            tok[dest[t, j]] = t
    assert np.array_equal(to_np(q_send), xo[tok])
    assert np.array_equal(to_np(s_send)[:, :plan.n_send].T.view(np.uint32), sxo[tok].view(np.uint32))
    # expert GEMM within the GEMM tolerance
    wo, swo = to_np(wq), to_np(sw)
    c, _, t = oracle.grouped(xo, sxo, tok, to_np(off), wo, swo)
    check_gemm(to_np(y), c, t, True, "expert GEMM")
    # combine of the GPU's own expert rows: bit-exact
    assert np.array_equal(bits(out), oracle.moe_combine(bits(y), dest, to_np(gate)))
