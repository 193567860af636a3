"""World-size-2 gloo check of bench.py's rank logic (CPU, no GPU): whole-job
throughput = units of all ranks / slowest rank's time."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r = bench.dist_init("gloo")
    units, secs, rate = bench.aggregate(1000.0 * (rank + 1), 2.0 + rank)
    bench.barrier()
    q.put((r, w, units, secs, rate, bench.dist_info()))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, world, units, secs, rate, info in results:
        assert world == 2 and info[0] == 2 and info[1] == rank
        assert units == 3000.0          # 1000 + 2000
        assert secs == 3.0              # slowest rank
        assert rate == pytest.approx(1000.0)


def test_single_process_is_identity():
    import bench
    assert bench.aggregate(5.0, 2.0) == (5.0, 2.0, 2.5)
