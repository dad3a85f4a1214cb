"""The benchmark's multi-rank logic on CPU with the gloo backend (world size 2).

On a GPU node each rank runs its own replica of the layer on its own tokens
(token-parallel, weak scaling) and the ranks meet only for the timing barrier
and the max over ranks; these tests exercise that host logic without a GPU."""

import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times_ms, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    w, r, local = bench.dist_setup(None, backend="gloo")
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    slowest = bench.max_over_ranks(times_ms[rank], w, device="cpu")
    out[rank] = (slowest, bench.rank_seed(10, rank),
                 bench.job_throughput(w, 4096, 50, slowest))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_tokens():
    world, port = 2, _free_port()
    times = [100.0, 125.0]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, times, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        slowest, seed, value = res[rank]
        assert slowest == 125.0
        assert seed == 10 + rank                      # distinct replicas per rank
        assert value == pytest.approx(2 * 4096 * 50 / 0.125)


def test_single_rank_needs_no_process_group(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_setup(None, backend="gloo") == (1, 0, 0)
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(1, 16, 10, 20.0) == pytest.approx(8000.0)
