"""The expert-parallel MoE forward (fp8_fine_grained_gb300.ep.moe_forward
with a process group) on the GPU kernels, two ranks in one process.

Two host threads play two ranks. Their exchanges go through an in-process
stand-in for torch.distributed's all_to_all_single that copies the splits
on the host after each side has synchronised its device work, so no
kernel waits on another. Each rank owns half of the experts. The test
checks that every rank's output equals, byte for byte, the single-GPU
layer (moe_forward without a process group, all experts local) on the
same tokens: each expert row is computed from the same codes and scales
and combined in the same slot order, whichever rank computed it. The
single-GPU layer is itself checked against the oracle in
tests/test_gpu_moe_combine.py."""
import threading

import numpy as np
import pytest
import torch

import oracle
from fp8_fine_grained_gb300 import ep
from tests.gpu_util import bits, check_gemm, to_np

pytestmark = pytest.mark.gpu

fg = pytest.importorskip("fp8_fine_grained_gb300")
DEV = "cuda"
WORLD, E, T, K, N, TOPK = 2, 16, 300, 384, 512, 4


class ThreadGroup:
    """all_to_all_single between threads of one process (host copies)."""

    def __init__(self, world):
        self.world = world
        self.barrier = threading.Barrier(world, timeout=120)
        self.slots = {}

    def rank_view(self, rank):
        group = self

        class View:
            def all_to_all_single(self, output, input, output_split_sizes=None, input_split_sizes=None):
                torch.cuda.synchronize()
                rows = input.shape[0]
                ins = input_split_sizes or [rows // group.world] * group.world
                outs = output_split_sizes or [output.shape[0] // group.world] * group.world
                host = input.detach().cpu()
                off = np.concatenate([[0], np.cumsum(ins)])
                for dst in range(group.world):
                    group.slots[(rank, dst)] = host[off[dst]:off[dst + 1]].clone()
                group.barrier.wait()
                parts = [group.slots[(src, rank)] for src in range(group.world)]
                assert [p.shape[0] for p in parts] == list(outs)
                output.copy_(torch.cat(parts).to(output.device))
                group.barrier.wait()
        return View()


def _problem(seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    w = (torch.randn(E, N, K, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
    wq, sw = fg.fp8_quant_128x128(w)
    ranks = []
    for r in range(WORLD):
        x = (torch.randn(T, K, generator=g, device=DEV) * torch.exp(torch.randn(K, generator=g, device=DEV))
             ).to(torch.bfloat16)
        logits = torch.randn(T, E, generator=g, device=DEV)
        ids = torch.topk(logits, TOPK, dim=1).indices.to(torch.int32)
        ids[5, 2] = -1                                   # an unused slot
        gate = torch.softmax(torch.gather(logits, 1, ids.clamp(min=0).long()), dim=1).float().contiguous()
        ranks.append((x, ids.contiguous(), gate))
    return wq, sw, ranks


def test_two_rank_forward_equals_the_single_gpu_layer():
    wq, sw, ranks = _problem(seed=77)
    group = ThreadGroup(WORLD)
    Er = E // WORLD
    out, errors = [None] * WORLD, []

    def run(r):
        try:
            x, ids, gate = ranks[r]
            out[r] = ep.moe_forward(x, ids, gate, wq[r * Er:(r + 1) * Er], sw[r * Er:(r + 1) * Er], E,
                                    pg=group.rank_view(r), world=WORLD)
            torch.cuda.synchronize()
        except BaseException as e:  # noqa: BLE001 - reported below
            errors.append(e)
            group.barrier.abort()

    threads = [threading.Thread(target=run, args=(r,)) for r in range(WORLD)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(300)
    assert not errors, errors
    assert fg.device_status() == 0
    for r in range(WORLD):
        x, ids, gate = ranks[r]
        single = ep.moe_forward(x, ids, gate, wq, sw, E)
        assert fg.device_status() == 0
        assert torch.equal(out[r], single), "rank %d" % r


def test_two_rank_expert_rows_against_the_oracle():
    """Rank 0's received rows through the grouped GEMM's row-index mode,
    within the GEMM tolerance of the oracle."""
    wq, sw, ranks = _problem(seed=78)
    Er = E // WORLD
    # what rank 0 receives: the rows every rank routes to experts 0..Er-1
    plans = [ep.plan_dispatch(ids, E, WORLD) for _, ids, _ in ranks]
    recv_counts = torch.stack([p.send_counts[0] for p in plans])
    lay = ep.receive_layout(recv_counts, DEV)
    q_recv, s_recv = [], []
    for (x, ids, _), p in zip(ranks, plans):
        q, s = fg.fp8_quant_1x128_scatter(x, p.dest, max(p.n_send, 1))
        n0 = int(p.send_counts[0].sum())
        q_recv.append(q[:n0])
        s_recv.append(s[:, :n0])
    q_recv = torch.cat(q_recv)
    s_cat = torch.cat(s_recv, dim=1)
    ld = (max(lay.n_recv, 1) + 3) // 4 * 4
    s_cols = torch.zeros((K // 128, ld), dtype=torch.float32, device=DEV)
    s_cols[:, :lay.n_recv] = s_cat
    y = fg.fp8_grouped_gemm(q_recv, s_cols, lay.row_index, lay.expert_offsets, wq[:Er], sw[:Er], lay.n_recv,
                            out_dtype=torch.float32)
    assert fg.device_status() == 0
    c, _, t = oracle.grouped(to_np(q_recv), to_np(s_cols)[:, :lay.n_recv].T.copy(), to_np(lay.row_index),
                             to_np(lay.expert_offsets), to_np(wq[:Er]), to_np(sw[:Er]))
    check_gemm(to_np(y), c, t, False, "expert rows of rank 0")
    # and the scatter-quantised rows are the tokens' own 1x128 codes
    x0 = ranks[0][0]
    xo, _ = oracle.quant_1x128(bits(x0))
    d0 = to_np(plans[0].dest)
    q0 = to_np(fg.fp8_quant_1x128_scatter(x0, plans[0].dest, plans[0].n_send)[0])
    for tk, j in ((0, 0), (5, 1), (T - 1, TOPK - 1)):
        assert np.array_equal(q0[d0[tk, j]], xo[tk])
