"""The N > 1 path of bench.py on CPU: replicas only (the layer has no exchange step), so the only
cross-rank work is the timing aggregation: units summed over ranks, time = the slowest rank."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    assert bench.dist_env() == (rank, rank, world)
    units, secs = bench.aggregate(1000.0 * (rank + 1), 0.5 + rank, device=None)
    bench.barrier()
    q.put((rank, units, secs))
    dist.destroy_process_group()


def test_replica_aggregation_two_ranks_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    results = sorted(q.get(timeout=10) for _ in range(world))
    for rank, units, secs in results:
        assert units == 3000.0       # 1000 + 2000 units over both replicas
        assert secs == 1.5           # the slowest rank's time


def test_single_process_aggregation_is_identity():
    import bench
    assert bench.aggregate(123.0, 0.25) == (123.0, 0.25)
