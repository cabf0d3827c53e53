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


# ---------------------------------------------------------------- head sharding (strong scaling)
def test_kv_head_ranges_partition():
    from shared_prompt_exact_gb300.dualkv import kv_head_ranges
    for hkv in (1, 2, 3, 8):
        for parts in (1, 2, 3, 4, 8, 9):
            rs = kv_head_ranges(hkv, parts)
            assert len(rs) == parts and rs[0][0] == 0 and rs[-1][1] == hkv
            assert all(a[1] == b[0] for a, b in zip(rs, rs[1:]))
            sizes = [hi - lo for lo, hi in rs]
            assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 0
    with pytest.raises(ValueError):
        kv_head_ranges(0, 2)


def _strong_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms_local, flops_local = [(10.0, 3e12), (12.0, 1e12)][rank]
    q.put((rank,) + bench.aggregate_strong(ms_local, flops_local, world, torch.device("cpu")))
    dist.destroy_process_group()


def test_aggregate_strong_two_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_strong_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, ms, value in sorted(q.get(timeout=10) for _ in range(2)):
        assert ms == pytest.approx(12.0)
        assert value == pytest.approx(4e12 / 12e-3 / 1e12)


def _oracle_shard_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    from shared_prompt_exact_gb300 import workloads as wl
    from shared_prompt_exact_gb300.dualkv import kv_head_ranges
    w = wl.custom(40, [17, 0, 30], 6, 3, 64, 0, seed=99)
    qx, kx, vx, dox = wl.draw_inputs(w)
    gs = w.Hq // w.Hkv
    lo, hi = kv_head_ranges(w.Hkv, world)[rank]
    part = oracle.dualkv(w.P, w.N, w.offsets, (hi - lo) * gs, hi - lo, w.D, w.scale, w.window,
                         qx[:, lo * gs:hi * gs].contiguous(), kx[:, lo:hi].contiguous(), vx[:, lo:hi].contiguous(),
                         dox[:, lo * gs:hi * gs].contiguous())
    parts = [None] * world
    dist.all_gather_object(parts, {k: part[k] for k in ("out", "lse", "dq", "dk", "dv")})
    ok = True
    if rank == 0:
        import numpy as np
        full = oracle.dualkv(w.P, w.N, w.offsets, w.Hq, w.Hkv, w.D, w.scale, w.window, qx, kx, vx, dox)
        ok = (np.array_equal(np.concatenate([p["out"] for p in parts], axis=1), full["out"]) and
              np.array_equal(np.concatenate([p["lse"] for p in parts], axis=0), full["lse"]) and
              np.array_equal(np.concatenate([p["dq"] for p in parts], axis=1), full["dq"]) and
              np.array_equal(np.concatenate([p["dk"] for p in parts], axis=1), full["dk"]) and
              np.array_equal(np.concatenate([p["dv"] for p in parts], axis=1), full["dv"]))
    q.put((rank, ok))
    dist.destroy_process_group()


def test_head_sharded_oracle_matches_full_gloo():
    """Two ranks, each with a contiguous kv-head group (the split bench.py --shard heads
    uses), reproduce the full result exactly: heads never interact."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_oracle_shard_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    assert all(ok for _, ok in (q.get(timeout=10) for _ in range(2)))


def test_reference_arm_json_line():
    """bench.py --impl reference prints one JSON line with the contract's keys (CPU only:
    the reference arm times the fp64 oracle on the host cores)."""
    import contextlib
    import io
    import json
    import bench
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--config", "tiny", "--steps", "2", "--warmup", "1"])
    assert rc == 0
    lines = [ln for ln in buf.getvalue().splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "TFLOP/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] == "tiny"
