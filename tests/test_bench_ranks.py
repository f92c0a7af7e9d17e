"""The N > 1 path of bench.py (replicas, no data-path collective): whole-job
throughput sums the ranks' units and divides by the slowest rank's time.
Run as two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    units, secs = bench.aggregate(1000.0 * (rank + 1), 0.5 + rank, world)
    bench.barrier(world)
    q.put((rank, units, secs, bench.dist_env()))
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_sum_over_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, units, secs, env in out:
        assert units == 3000.0 and secs == 1.5
        assert env == (2, rank, rank)


def test_single_rank_aggregate_is_identity():
    import bench
    assert bench.aggregate(123.0, 2.0, 1) == (123.0, 2.0)
