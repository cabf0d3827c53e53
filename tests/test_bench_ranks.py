"""Multi-rank bench logic on CPU (gloo, world size 2): independent replicas,
no data-path collective; the job time is the max over ranks and the value is
the total work over that time."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms_local = [10.0, 12.5][rank]
    ms, value = bench.aggregate(ms_local, 1e12, world, torch.device("cpu"))
    bench.barrier(world)
    q.put((rank, ms, value))
    dist.destroy_process_group()


def test_aggregate_two_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, value in res:
        assert ms == pytest.approx(12.5)
        assert value == pytest.approx(2 * 1e12 / 12.5e-3 / 1e12)


def test_aggregate_single_rank():
    import bench
    ms, value = bench.aggregate(8.0, 2e12, 1, torch.device("cpu"))
    assert ms == 8.0 and value == pytest.approx(250.0)
