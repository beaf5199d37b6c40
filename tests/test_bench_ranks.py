"""Host logic of the multi-replica bench (torchrun, one process per GPU) on CPU with two
gloo ranks: each rank draws its own input seeds, the timing is the slowest rank's, and the
reported value is every rank's tokens over that time."""

import os
import socket

import pytest
import torch.multiprocessing as mp

import bench

K, W, T = 5, 3, 4


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      LOCAL_RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, _, w = bench.dist_info()
        slowest = bench.max_over_ranks(1.5 + r, w, "cpu")      # rank r "took" 1.5 + r s
        q.put((r, w, slowest, bench.rank_seed_base(r, K, W),
               bench.job_throughput(w, K, T, slowest)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_replicas_host_logic():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[0] for g in got] == [0, 1] and all(g[1] == 2 for g in got)
    assert all(g[2] == 2.5 for g in got)                       # both see the slowest rank
    seeds = [set(range(g[3], g[3] + K + W)) for g in got]
    assert not seeds[0] & seeds[1]                              # disjoint inputs
    assert all(g[4] == pytest.approx(2 * K * T / 2.5) for g in got)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.25, 1, "cpu") == 3.25
    assert bench.job_throughput(1, 10, 2048, 2.0) == 10240.0
    assert bench.rank_seed_base(0, K, W) == 0
