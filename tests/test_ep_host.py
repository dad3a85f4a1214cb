"""Expert parallelism's host logic (sparse_expert_ffn_gb300/ep.py) on CPU.

The exchange plan is checked as plain functions. Then two or three gloo
ranks run the whole expert-parallel forward. Each rank owns an equal share
of the experts and routes tokens of its own (some ranks have none). The
oracle stands in for the library's kernels (route, gather, experts,
combine). Each rank's output must equal the oracle's layer over all experts
for its tokens. The collective calls are the ones the GPU path makes:
all_to_all_single of the count table and of the row blocks (over NCCL
there)."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from sparse_expert_ffn_gb300.ep import ExchangePlan, Steps, ep_forward


def test_plan_from_counts():
    counts = torch.tensor([3, 0, 2, 5, 0, 0, 1, 4], dtype=torch.int32)
    p = ExchangePlan.from_counts(counts, 2)
    assert p.experts_per_rank == 4
    assert p.send_rows == [10, 5]
    assert p.send_table.tolist() == [[3, 0, 2, 5], [0, 0, 1, 4]]
    with pytest.raises(ValueError):
        ExchangePlan.from_counts(torch.zeros(6, dtype=torch.int32), 4)


def test_local_ids_follow_sources_then_experts():
    p = ExchangePlan.from_counts(torch.zeros(6, dtype=torch.int32), 3)
    p.recv_table = torch.tensor([[1, 0], [0, 2], [2, 1]])
    assert p.recv_rows == [1, 2, 3]
    assert p.local_expert_ids().tolist() == [0, 1, 1, 0, 0, 1]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _layer(seed, E=8, d=32, f=48):
    rng = np.random.default_rng(seed)
    wr = rng.standard_normal((d, E)) / np.sqrt(d)
    wg = rng.standard_normal((E, d, f)) / np.sqrt(d)
    wu = rng.standard_normal((E, d, f)) / np.sqrt(d)
    wd = rng.standard_normal((E, f, d)) / np.sqrt(f)
    return wr, wg, wu, wd


def _rank_main(rank, world, port, T, k, E, out):
    import torch.distributed as dist
    import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wr, wg, wu, wd = _layer(5, E=E)
        E = wr.shape[1]
        El = E // world
        x = np.random.default_rng(100 + rank).standard_normal((T[rank], wr.shape[0]))
        # this rank's experts only, for the owner step
        mine = range(rank * El, (rank + 1) * El)

        def route(xt):
            l = oracle.router_logits(xt.numpy(), wr)
            idx = oracle.topk_select(l, k)
            g = oracle.softmax_selected(l, idx)
            counts, _, perm, _ = oracle.dispatch(idx, E)
            return (torch.from_numpy(idx.astype(np.int32)), torch.from_numpy(g),
                    torch.from_numpy(counts.astype(np.int32)), torch.from_numpy(perm.astype(np.int32)))

        def gather(xt, perm, kk):
            return xt[perm.long() // kk]

        def experts(rows, ids):
            outr = torch.zeros_like(rows)
            for e_local in range(El):
                sel = (ids == e_local).nonzero().flatten()
                if sel.numel():
                    e = mine[e_local]
                    outr[sel] = torch.from_numpy(
                        oracle.swiglu_expert(rows[sel].numpy(), wg[e], wu[e], wd[e]))
            return outr

        def combine(back, g, perm):
            inv = torch.empty_like(perm)
            inv[perm.long()] = torch.arange(perm.numel(), dtype=perm.dtype)
            y = torch.zeros((g.shape[0], back.shape[1]), dtype=back.dtype)
            for j in range(g.shape[1]):
                pos = inv.view(-1, g.shape[1])[:, j].long()
                y += g[:, j:j + 1] * back[pos]
            return y

        y = ep_forward(torch.from_numpy(x), Steps(route, gather, experts, combine), world)
        ref = oracle.moe_layer(x, wr, wg, wu, wd, k)["y"]
        assert tuple(y.shape) == ref.shape
        err = float(np.abs(y.numpy() - ref).max(initial=0.0))
        out[rank] = (err, float(np.abs(ref).max(initial=0.0)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("T,k,E", [((7, 11), 2, 8), ((5, 0), 2, 8), ((9, 0, 4), 3, 6),
                                   ((1, 6, 13), 1, 6)])
def test_gloo_ranks_match_the_whole_layer(T, k, E):
    world, port = len(T), _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, T, k, E, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        err, scale = res[rank]
        assert err <= 1e-12 * max(scale, 1.0), (rank, err)
