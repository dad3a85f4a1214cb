"""Expert parallelism on one GPU.

Two ranks' shares of one layer (each the full router and half of the 8
experts, sparse_expert_ffn_gb300.ep.ExpertParallelLayer) are driven from one
process: each routes and gathers its own tokens with the library, the
all-to-all exchanges are done by slicing on the device in the order the
collective delivers (sources in rank order, each source's rows in its expert
order), each owner runs its experts on the rows it receives
(colibri_forward_routed) and each source combines its returned rows
(colibri_combine_rows).  Every token of every rank is checked against the
oracle's layer over all experts, under the routing near-tie rule.  One more
test runs ExpertParallelLayer.forward through a one-rank NCCL group, the
collective calls included.  Ranks here never wait on one another inside a
kernel: each step is a separate, ordered library call."""

import os
import socket

import pytest
import torch

import synth
from parity import Case, check_output, check_routing
from sparse_expert_ffn_gb300.ep import ExchangePlan, ExpertParallelLayer

pytestmark = pytest.mark.gpu

SHAPE = synth.LayerShape("ep", 512, 1024, 8, 2, "bf16")


def _shares(case, world, max_tokens):
    dev = case.dev
    wr = synth.router_weight(case.shape, case.seed, 0, dev)
    wg, wu, wd = synth.expert_weights(case.shape, case.seed, 0, dev)
    El = case.shape.n_experts // world
    return [ExpertParallelLayer(wr, case.bias, wg[g * El:(g + 1) * El], wu[g * El:(g + 1) * El],
                                wd[g * El:(g + 1) * El], case.shape.top_k, case.shape.n_experts,
                                max_tokens, world=world)
            for g in range(world)]


def _emulated_forward(shares, xs):
    """ep_forward's steps for every rank, the exchanges by slicing."""
    G = len(shares)
    k = shares[0].k
    routed, rows, plans = [], [], []
    for g in range(G):
        idx, w, cnt, perm = shares[g].route(xs[g])
        routed.append((idx.clone(), w.clone(), cnt.clone(), perm.clone()))
        rows.append(shares[g].gather(xs[g], routed[g][3], k))
        plans.append(ExchangePlan.from_counts(routed[g][2], G))
    for g in range(G):                   # all-to-all of the count tables
        plans[g].recv_table = torch.stack([plans[s].send_table[g] for s in range(G)])
    send_off = [[sum(plans[s].send_rows[:g]) for g in range(G)] for s in range(G)]
    outs = []
    for g in range(G):                   # rows to their owners, experts run there
        recv = torch.cat([rows[s][send_off[s][g]:send_off[s][g] + plans[s].send_rows[g]]
                          for s in range(G)])
        outs.append(shares[g].experts(recv, plans[g].local_expert_ids().to(recv.device)))
    ys = []
    for s in range(G):                   # results back to their sources, combined
        back = []
        for g in range(G):
            off = sum(plans[g].recv_rows[:s])
            back.append(outs[g][off:off + plans[g].recv_rows[s]])
        ys.append(shares[s].combine(torch.cat(back), routed[s][1], routed[s][3]))
    torch.cuda.synchronize()
    return ys, routed


@pytest.mark.parametrize("T", [(37, 5), (64, 0), (1024, 700)])
def test_two_emulated_ranks_match_the_oracle(lib, T):
    case = Case(SHAPE, seed=21, max_tokens=sum(T))
    shares = _shares(case, 2, max(T))
    try:
        x_all, x64 = case.tokens(sum(T))
        xs = [x_all[:T[0]], x_all[T[0]:]]
        ys, routed = _emulated_forward(shares, xs)
        for g in range(2):
            assert shares[g].check() == 0
        lo = 0
        for g in range(2):
            n = T[g]
            assert tuple(ys[g].shape) == (n, SHAPE.d_model)
            if n:
                idx, w, cnt, perm = (t.cpu().numpy() for t in routed[g])
                r = {"topk_idx": idx, "topk_w": w, "counts": cnt, "perm": perm}
                l, near = check_routing(case, x64[lo:lo + n], r)
                assert near.sum() <= max(1, n // 50)
                check_output(case, x64[lo:lo + n], ys[g], r, l)
            lo += n
        ys2, _ = _emulated_forward(shares, xs)
        for a, b in zip(ys, ys2):
            assert torch.equal(a, b)
    finally:
        for s in shares:
            s.close()
        case.close()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_forward_through_a_one_rank_nccl_group(lib):
    import torch.distributed as dist
    if dist.is_initialized():
        pytest.skip("a process group is already initialised")
    case = Case(SHAPE, seed=22, max_tokens=300)
    os.environ.setdefault("NCCL_SOCKET_IFNAME", "lo")
    os.environ.setdefault("NCCL_NVLS_ENABLE", "0")
    torch.cuda.set_device(0)
    store = dist.TCPStore("127.0.0.1", _free_port(), 1, True)
    dist.init_process_group("nccl", store=store, rank=0, world_size=1)
    share = None
    try:
        share = _shares(case, 1, 300)[0]
        x, x64 = case.tokens(300)
        y = share.forward(x)
        torch.cuda.synchronize()
        assert share.check() == 0
        idx, w, cnt, perm = (t.cpu().numpy() for t in share.route(x))
        r = {"topk_idx": idx, "topk_w": w, "counts": cnt, "perm": perm}
        l, _ = check_routing(case, x64, r)
        check_output(case, x64, y, r, l)
        assert share.forward(x[:0]).shape == (0, SHAPE.d_model)
    finally:
        if share is not None:
            share.close()
        dist.destroy_process_group()
        case.close()
