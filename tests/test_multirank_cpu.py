"""The multi-rank path of the benchmark on CPU: two gloo ranks, each a
replica with its own units and time. The job's throughput is the sum of all
ranks' units over the slowest rank's time (weak scaling, no collective on the
data path; the only collectives are the barrier and these reductions)."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    units = 1000.0 * (rank + 1)          # rank 0: 1000 units, rank 1: 2000
    secs = 0.5 if rank == 0 else 2.0     # rank 1 is the slowest
    value, slowest = bench.aggregate(units, secs)
    assert bench.dist_env() == (rank, world, rank)
    dist.barrier()
    q.put((rank, value, slowest))
    dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, value, slowest in got:
        assert slowest == pytest.approx(2.0)
        assert value == pytest.approx(3000.0 / 2.0)


def test_single_process_is_identity():
    import bench
    assert bench.aggregate(10.0, 2.0) == (5.0, 2.0)
