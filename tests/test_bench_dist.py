"""The multi-rank path of bench.py on CPU: two gloo ranks, as torchrun would
launch them (one process per rank, rendezvous on 127.0.0.1). Each rank
verifies its own batch, so the only collectives are the barrier and the
max-over-ranks of the elapsed time."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        # rank r took (r + 1) ms: the job's time is the slowest rank's
        slowest = bench.max_over_ranks(float(rank + 1), world)
        value = bench.job_throughput(world, 1000, slowest / 1e3)
        bench.barrier(world)
        q.put((rank, slowest, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_time_by_the_slowest_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    assert [g[0] for g in got] == [0, 1]
    # both ranks agree on the slowest rank's 2 ms, and the job's tokens/s
    # counts both ranks' tokens over it
    for _, slowest, value in got:
        assert slowest == 2.0
        assert value == pytest.approx(2 * 1000 / 2e-3)


def test_one_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(1, 1361, 0.5) == pytest.approx(2722.0)
