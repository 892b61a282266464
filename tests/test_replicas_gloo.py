"""The N-GPU path of bench.py runs independent replicas of the layer (the path does not
shard); the only cross-rank logic is the aggregation: all ranks' tokens over the slowest
rank's time, and the barrier.  Checked here with two gloo ranks on the CPU."""

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


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, lr = bench.dist_setup()
    assert (w, r, lr) == (world, rank, rank)
    bench.barrier(world)
    # rank 0 processed 4096 tokens in 10 ms, rank 1 4096 tokens in 12.5 ms
    ms = 10.0 if rank == 0 else 12.5
    total, ms_max, value = bench.replica_throughput(world, 4096.0, ms)
    q.put((rank, total, ms_max, value))
    dist.destroy_process_group()


def test_two_rank_replica_aggregation():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, total, ms_max, value in res:
        assert total == 8192.0
        assert ms_max == 12.5
        assert value == pytest.approx(8192.0 / 0.0125)
