"""Expert-parallel FP8 dispatch and combine across two and four ranks
(gloo, CPU).

Each rank holds its own tokens and an equal share of the experts. The test
runs the protocol of fp8_fine_grained_gb300.ep (dispatch plan, the count
and row all-to-alls, the receive layout, the return exchange) with the CPU
oracle in place of the GPU kernels (1x128 quantisation, the expert GEMM, the combine),
and checks every token's combined output bit for bit against the same
layer computed in one process without expert parallelism: every expert row
is computed from the same codes and scales and combined in the same slot
order, so the exchanges must not change a single bit. Byte-exact checks of
the received FP8 rows and scales come first."""
import os

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from fp8_fine_grained_gb300 import ep

E, K, N, T, TOPK = 8, 256, 256, 20, 3


def _problem(rank, skewed=False):
    """Experts (same on every rank) and this rank's tokens and routing.
    skewed: rank 1 routes every token to its own experts (it sends rank 0
    nothing) and rank 0's token 7 uses no slot at all."""
    g = torch.Generator().manual_seed(1234)
    w = (torch.randn(E, N, K, generator=g) * 0.02).to(torch.bfloat16)
    wq, sw = [], []
    for e in range(E):
        q, s = oracle.quant_128x128(w[e].view(torch.int16).numpy().view(np.uint16))
        wq.append(q)
        sw.append(s)
    gt = torch.Generator().manual_seed(100 + rank)
    x = (torch.randn(T, K, generator=gt) * torch.exp(torch.randn(K, generator=gt))).to(torch.bfloat16)
    logits = torch.randn(T, E, generator=gt)
    if skewed and rank == 1:
        logits[:, :E // 2] = -1e9                       # only experts E/2.. (rank 1's own)
    topk = torch.topk(logits, TOPK, dim=1).indices.to(torch.int32)
    topk[3, 1] = -1                                     # one unused slot
    if skewed and rank == 0:
        topk[7, :] = -1                                 # a token routed nowhere
    gate = torch.softmax(torch.gather(logits, 1, topk.clamp(min=0).long()), dim=1).to(torch.float32)
    return np.stack(wq), np.stack(sw), x.view(torch.int16).numpy().view(np.uint16), topk, gate


def _expert_rows(q, s, wq_e, sw_e):
    """bf16 bits of one expert's output rows (the oracle's GEMM, rounded as
    the GPU GEMM's bf16 output is)."""
    c, _, _ = oracle.fprop(q, s, wq_e, sw_e, want_exact=False)
    return oracle.to_bf16_bits(c)


def _reference(wq, sw, xb, topk, gate):
    q, s = oracle.quant_1x128(xb)
    rows, dest = [], np.full(topk.shape, -1, np.int32)
    for t in range(T):
        for j in range(TOPK):
            e = int(topk[t, j])
            if e < 0:
                continue
            dest[t, j] = len(rows)
            rows.append(_expert_rows(q[t:t + 1], s[t:t + 1], wq[e], sw[e])[0])
    return oracle.moe_combine(np.stack(rows), dest, gate.numpy())


def _rank(rank, world, port, out, skewed=False):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wq, sw, xb, topk, gate = _problem(rank, skewed)
        Er = E // world
        plan = ep.plan_dispatch(topk, E, world)
        # dispatch: every token quantised once, its codes and scales copied to its k send rows
        q, s = oracle.quant_1x128(xb)
        q_send = np.zeros((plan.n_send, K), np.uint8)
        s_send = np.zeros((plan.n_send, K // 128), np.float32)
        for t in range(T):
            for j in range(TOPK):
                d = int(plan.dest[t, j])
                if d >= 0:
                    q_send[d], s_send[d] = q[t], s[t]
        recv_counts = ep.exchange_counts(plan.send_counts, dist)
        srows, rrows = ep.rank_rows(plan.send_counts), ep.rank_rows(recv_counts)
        q_recv = ep.exchange_rows(torch.from_numpy(q_send), srows, rrows, dist).numpy()
        s_recv = ep.exchange_rows(torch.from_numpy(s_send), srows, rrows, dist).numpy()
        lay = ep.receive_layout(recv_counts)
        ri = lay.row_index.numpy().astype(np.int64)
        off = lay.expert_offsets.numpy()
        # every received row is a token of some rank routed to one of my experts
        y = np.zeros((lay.n_recv, N), np.uint16)
        for el in range(Er):
            rows = ri[off[el]:off[el + 1]]
            if rows.size:
                e = rank * Er + el
                y[off[el]:off[el + 1]] = _expert_rows(q_recv[rows], s_recv[rows], wq[e], sw[e])
        y_recv = ep.to_receive_order(torch.from_numpy(y.view(np.int16)), lay.row_index, lay.n_recv)
        y_back = ep.exchange_rows(y_recv, rrows, srows, dist).numpy().view(np.uint16)
        got = oracle.moe_combine(y_back, plan.dest.numpy(), gate.numpy())
        ref = _reference(wq, sw, xb, topk, gate)
        out[rank] = {
            "combine_equal": bool(np.array_equal(got, ref)),
            "sent": srows, "received": rrows, "n_recv": lay.n_recv,
            "recv_rows_sorted_by_expert": bool(np.all(np.diff(off) >= 0)),
            "q_recv": q_recv, "s_recv": s_recv, "recv_counts": recv_counts.numpy(),
            "q": q, "s": s, "plan_dest": plan.dest.numpy(), "send_counts": plan.send_counts.numpy(),
            "out": got,
        }
    finally:
        dist.destroy_process_group()


def _run_two(port, skewed, world=2):
    oracle.build.build()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_rank, args=(r, world, port, out, skewed)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    return dict(out)


@pytest.fixture(scope="module")
def two_ranks():
    return _run_two(29500 + (os.getpid() % 1000), False)


def test_four_ranks():
    """Four ranks of two experts each: every token's output equals the
    single-process layer, and each rank receives exactly what the others
    route to its experts."""
    res = _run_two(31700 + (os.getpid() % 1000), False, world=4)
    for r in range(4):
        assert res[r]["combine_equal"], "rank %d" % r
        for src in range(4):
            assert np.array_equal(res[r]["recv_counts"][src], res[src]["send_counts"][r])
        assert res[r]["n_recv"] == sum(int(res[src]["send_counts"][r].sum()) for src in range(4))


def test_empty_splits_and_a_token_routed_nowhere():
    """Rank 1 sends rank 0 no row (zero-size splits in the all-to-alls) and
    rank 0 has a token whose slots are all unused (its output is zero)."""
    res = _run_two(30600 + (os.getpid() % 1000), True)
    assert res[1]["sent"][0] == 0 and res[0]["received"][1] == 0
    for r in range(2):
        assert res[r]["combine_equal"], "rank %d" % r
    assert np.all(res[0]["out"][7] == 0)


def test_every_token_output_matches_the_single_process_layer(two_ranks):
    for r in range(2):
        assert two_ranks[r]["combine_equal"], "rank %d" % r


def test_rows_and_scales_arrive_byte_exact(two_ranks):
    """Rank r receives, from each source s, exactly the codes and scales of
    the source's tokens routed to r's experts, in (expert, token, slot)
    order."""
    Er = E // 2
    for r in range(2):
        got_q, got_s = two_ranks[r]["q_recv"], two_ranks[r]["s_recv"]
        pos = 0
        for src in range(2):
            d = two_ranks[src]
            _, _, _, topk, _ = _problem(src)
            want = [(int(topk[t, j]), t, j) for t in range(T) for j in range(TOPK)
                    if r * Er <= int(topk[t, j]) < (r + 1) * Er]
            for e, t, j in sorted(want):
                assert np.array_equal(got_q[pos], d["q"][t]), (r, src, e, t, j)
                assert np.array_equal(got_s[pos].view(np.uint32), d["s"][t].view(np.uint32))
                pos += 1
        assert pos == two_ranks[r]["n_recv"]


def test_counts_are_consistent(two_ranks):
    for r in range(2):
        assert two_ranks[r]["sent"] == [int(v) for v in two_ranks[r]["send_counts"].sum(1)]
        for src in range(2):
            assert np.array_equal(two_ranks[r]["recv_counts"][src], two_ranks[src]["send_counts"][r])
    # one unused slot on each rank: 20 tokens x 3 slots - 1 rows sent per rank
    assert sum(two_ranks[0]["sent"]) == T * TOPK - 1 and sum(two_ranks[1]["sent"]) == T * TOPK - 1


def test_plan_orders_rows_by_expert_then_token():
    topk = torch.tensor([[3, 0], [0, 5], [-1, 3], [5, 0]], dtype=torch.int32)
    plan = ep.plan_dispatch(topk, 6, 2)
    # expert 0: (0,1) (1,0) (3,1); expert 3: (0,0) (2,1); expert 5: (1,1) (3,0)
    assert plan.dest.tolist() == [[3, 0], [1, 5], [-1, 4], [6, 2]]
    assert plan.send_counts.tolist() == [[3, 0, 0], [2, 0, 2]]
    assert plan.n_send == 7


def test_receive_layout_lists_rows_expert_by_expert():
    # two sources, two local experts: source 0 sent 2 rows of e0 and 1 of e1,
    # source 1 sent 1 row of e0 and 2 of e1
    lay = ep.receive_layout(torch.tensor([[2, 1], [1, 2]]))
    assert lay.row_index.tolist() == [0, 1, 3, 2, 4, 5]
    assert lay.expert_offsets.tolist() == [0, 3, 6]
    assert lay.n_recv == 6


@pytest.mark.parametrize("seed", range(6))
def test_plan_matches_a_brute_force_sort(seed):
    """dest lists every used (token, slot) exactly once, rows ordered by
    expert, then token, then slot; the counts per rank and local expert add
    up (random routings with unused slots, several world sizes)."""
    rng = np.random.default_rng(seed)
    world = [1, 2, 4, 8][seed % 4]
    E = world * int(rng.integers(1, 5))
    T, k = int(rng.integers(0, 40)), int(rng.integers(1, 6))
    ids = rng.integers(-1, E, (T, k)).astype(np.int32)
    plan = ep.plan_dispatch(torch.from_numpy(ids), E, world)
    order = sorted((int(ids[t, j]), t, j) for t in range(T) for j in range(k) if ids[t, j] >= 0)
    want = np.full((T, k), -1, np.int64)
    for row, (_, t, j) in enumerate(order):
        want[t, j] = row
    assert np.array_equal(plan.dest.numpy(), want)
    assert plan.n_send == len(order)
    counts = np.bincount([e for e, _, _ in order], minlength=E).reshape(world, E // world)
    assert np.array_equal(plan.send_counts.numpy(), counts)


@pytest.mark.parametrize("seed", range(6))
def test_receive_layout_matches_a_brute_force_walk(seed):
    """row_index walks the received rows expert by expert, sources
    ascending inside an expert, each source's rows in arrival order."""
    rng = np.random.default_rng(100 + seed)
    R, Er = int(rng.integers(1, 6)), int(rng.integers(1, 5))
    counts = rng.integers(0, 5, (R, Er))
    lay = ep.receive_layout(torch.from_numpy(counts))
    # arrival order: source by source, each source's rows expert by expert
    arrival = [(s, e) for s in range(R) for e in range(Er) for _ in range(counts[s, e])]
    want = [i for e in range(Er) for s in range(R) for i, a in enumerate(arrival) if a == (s, e)]
    assert lay.row_index.tolist() == want
    assert lay.n_recv == len(arrival)
    assert lay.expert_offsets.tolist() == [0] + np.cumsum(counts.sum(0)).tolist()
