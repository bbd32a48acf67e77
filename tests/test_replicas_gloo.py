"""Multi-GPU runs are independent replicas (weak scaling, no data-path
collective); the only cross-rank steps are the benchmark's barrier and its
max-over-ranks time / sum-over-ranks work.  Checked here with two gloo ranks
on the CPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        t = bench.allreduce_max(dist, 1.0 + rank, "cpu")          # slowest rank's time
        rows = bench.allreduce_sum(dist, 17 * 20, "cpu")          # every rank's verified rows
        q.put((rank, t, rows, rows / t))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_replica_aggregation(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, rows, value in res:
        assert t == float(world)                     # max over ranks
        assert rows == 17 * 20 * world               # whole-job work
        assert value == rows / world
