"""The MoE workload's inputs agree with one another (CPU, small sizes): the
per-token expert choices (topk_ids) are the experts the routing's row order
(row_index, expert_offsets) lists for each token, the dispatch plan built
from topk_ids reproduces the same expert offsets, and the gate weights are
a softmax over each token's chosen experts."""
import numpy as np
import torch

from fp8_fine_grained_gb300 import ep, synth


def _small(seed):
    return synth.moe(seed=seed, device="cpu", T=200, K=256, N=128, E=16, topk=4, make_weights=False)


def test_choices_match_the_row_order():
    mo = _small(1)
    T, k = mo.topk_ids.shape
    ri, off = mo.row_index.numpy(), mo.expert_offsets.numpy()
    per_token = [set() for _ in range(T)]
    for e in range(len(off) - 1):
        for r in range(off[e], off[e + 1]):
            per_token[ri[r]].add(e)
    for t in range(T):
        assert per_token[t] == set(mo.topk_ids[t].tolist())
    assert np.array_equal(mo.counts.numpy(), np.diff(off))


def test_dispatch_plan_reproduces_the_offsets():
    mo = _small(2)
    plan = ep.plan_dispatch(mo.topk_ids, 16, 1)
    assert plan.n_send == int(mo.expert_offsets[-1])
    assert np.array_equal(np.concatenate([[0], np.cumsum(plan.send_counts[0].numpy())]), mo.expert_offsets.numpy())
    # the plan's rows carry the same tokens as the routing's row order
    tok = np.empty(plan.n_send, np.int64)
    dest = plan.dest.numpy()
    for t in range(dest.shape[0]):
        for j in range(dest.shape[1]):
            tok[dest[t, j]] = t
    assert np.array_equal(tok, mo.row_index.numpy())


def test_gates_are_a_softmax_over_the_chosen_experts():
    mo = _small(3)
    g = mo.gates
    assert g.dtype == torch.float32 and g.shape == mo.topk_ids.shape
    assert torch.all(g > 0)
    assert torch.allclose(g.sum(1), torch.ones(g.shape[0]), atol=1e-6)
    # best-ranked expert first: gates are not required to be sorted (the
    # bias enters the ranking only), but each row's ids are distinct
    for row in mo.topk_ids.tolist():
        assert len(set(row)) == len(row)
