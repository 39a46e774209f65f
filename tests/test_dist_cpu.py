"""Multi-process host logic of the benchmark on CPU (gloo, world size 2):
replicas exchange nothing on the data path; the timed interval is the max
over ranks and ranks meet at barriers around it."""
import os

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, ws, lr = bench.dist_env()
    bench.barrier(torch.device("cpu"))
    got = bench.reduce_max(10.0 * (rank + 1), torch.device("cpu"))
    bench.barrier(torch.device("cpu"))
    q.put((r, ws, lr, got))
    dist.destroy_process_group()


def test_reduce_max_and_barrier_gloo():
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 2, 0, 20.0), (1, 2, 1, 20.0)]


def test_single_process_reduce_is_identity():
    import bench
    assert bench.reduce_max(3.5) == 3.5
    assert bench.dist_env()[1] >= 1
