"""bench.py's replica aggregation on two gloo ranks (CPU): the process group
comes up from the torchrun environment, the step time is the max over ranks
and the barrier returns on every rank."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    import torch.distributed as dist
    r, w, lr = bench.dist_setup()
    assert (r, w, lr) == (rank, world, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    got = bench.reduce_max(1.5 + 2.0 * rank, w)
    out.put((rank, got))
    bench.barrier(w)
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_reduce_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    world, port = 2, _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(100)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    assert got == [(0, 3.5), (1, 3.5)]


def test_single_rank_needs_no_group(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    import bench
    assert bench.dist_setup() == (0, 1, 0)
    assert bench.reduce_max(2.25, 1) == 2.25
    bench.barrier(1)
