#!/usr/bin/env python
"""DualKV shared-prompt attention benchmark on GB300.

One step = one DualKV forward + backward (dualkv_fwd + dualkv_bwd) over one
packed micro-batch of the chosen workload (default: the Qwen3-8B GRPO-shaped
layer, P=6144, N=32, R=2048, Hq=32, Hkv=8, D=128, causal), inputs resident in
HBM.  The metric is useful TFLOP/s: forward 4*D*Hq*pairs + backward
10*D*Hq*pairs per step, where pairs counts attended (query, key) pairs of one
head with every packed query row counted once.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl dualkv|reference]

With N > 1 (launched by torch.distributed.run) every rank runs an independent
replica of the step on its own GPU (no collective on the data path), timing is
the max over ranks and the value is the total over ranks ("weak" scaling).
``--impl reference`` times the fp64 CPU oracle (the only reference this method
has) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from shared_prompt_exact_gb300 import workloads as wl  # noqa: E402

METRIC = "DualKV attn fwd+bwd useful TFLOP/s & % BF16 tensor peak, N=32 P=6144 R=2048"
UNIT = "TFLOP/s"

# algorithmic tensor-core FLOPs per attended pair per head (x D) of each kernel kind:
# forward S and PV; dK/dV recomputes S and dP and forms dV and dK; dQ recomputes S
# and dP and forms dQ
KERNEL_FLOPS_PER_PAIR = {"fwd": 4, "dkv": 8, "dq": 6}


def kernel_flops_per_pair(kind, D):
    return KERNEL_FLOPS_PER_PAIR.get(kind)


# ------------------------------------------------------------------ helpers
def useful_flops(pairs, D, Hq):
    return 4.0 * D * Hq * pairs, 10.0 * D * Hq * pairs


def layout_pairs(w):
    from shared_prompt_exact_gb300 import dualkv
    return dualkv.dualkv_pairs(w.P, w.N, w.offsets, w.window)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            m = json.load(f)
        return dict(bf16_burst=float(m["bf16_tflops"]), bf16_sustained=float(m["bf16_tflops_sustained"]),
                    hbm_gbs=float(m["hbm_gbs"]), source="measured")
    except Exception:
        return dict(bf16_burst=1900.0, bf16_sustained=1700.0, hbm_gbs=6800.0, source="fallback")


# source files each timed kernel kind is built from (its kernel, the shared device
# helpers, the work-list planner and the launch code)
_COMMON_SOURCES = ["ptx.cuh", "checks.cuh", "kernels.h", "plan.h", "plan.cpp", "api.cu"]
KERNEL_SOURCES = {"fwd": ["fwd.cu"] + _COMMON_SOURCES, "dkv": ["bwd.cu"] + _COMMON_SOURCES,
                  "dq": ["bwd.cu"] + _COMMON_SOURCES}


def source_digest(kernel=None):
    """Digest of the sources of `kernel` (a KERNEL_SOURCES key), or of every source."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "shared_prompt_exact_gb300", "csrc")
    names = KERNEL_SOURCES[kernel] if kernel else sorted(os.listdir(csrc))
    for name in names:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if taken on the kernel's current sources."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}_ncu.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    s = re.search(r"source_digest:\s*([0-9a-f]+)", text)
    if not m or not s or s.group(1) != source_digest(kernel if kernel in KERNEL_SOURCES else None):
        return None
    return float(m.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the GPU is under load."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.lines = []
        self.marks = []

    def start(self):
        sel = self._selector()
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200"] + sel, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _selector(self):
        try:
            uuid = str(torch.cuda.get_device_properties(self.dev).uuid)
            if uuid:
                return ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            pass
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis:
            return ["-i", vis.split(",")[self.dev]]
        return ["-i", str(self.dev)]

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        self.marks.append(time.time())

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()

    def summary(self, t0, t1):
        def parse(rows):
            sm, mx, reasons = [], [], set()
            names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
            for _, line in rows:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(nm)
            return sm, mx, reasons
        window = [r for r in self.lines if t0 <= r[0] <= t1]
        sm, mx, reasons = parse(window)
        scope = "timed region"
        if len(sm) < 3:
            sm, mx, reasons = parse([r for r in self.lines if r[0] >= t0])
            scope = "timed region and the measurement phases after it"
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "scope": "unavailable"}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "scope": scope}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x, world, device):
    if world <= 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, world, device):
    if world <= 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def aggregate_strong(ms_local, flops_local, world, device):
    """Whole-job throughput when the ranks split one step's work (head sharding):
    total work over the slowest rank's time."""
    ms = max_over_ranks(ms_local, world, device)
    return ms, sum_over_ranks(flops_local, world, device) / (ms * 1e-3) / 1e12


def aggregate(ms_local, flops_per_rank, world, device):
    """Whole-job throughput of `world` independent replicas: every rank does
    flops_per_rank per step; the job's step time is the slowest rank's."""
    ms = max_over_ranks(ms_local, world, device)
    return ms, world * flops_per_rank / (ms * 1e-3) / 1e12


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ oracle (CPU baseline / reference arm)
def oracle_sample(w, q, k, v, do, n_seg=1):
    """A bounded sample of the workload (about 10-20 s for the fp64 oracle on 16
    cores): the prompt, the first n_seg responses, the first q-head and its kv-head."""
    n_seg = min(n_seg, w.N)
    off = w.offsets[: n_seg + 1]
    T = w.P + off[-1]
    return dict(P=w.P, N=n_seg, off=off, Hq=1, Hkv=1, D=w.D, scale=w.scale, window=w.window,
                q=q[:T, :1].contiguous(), k=k[:T, :1].contiguous(), v=v[:T, :1].contiguous(),
                do=do[:T, :1].contiguous())


def time_oracle(s):
    import oracle
    from oracle import index as oindex
    pairs = oindex.pairs(s["P"], s["off"], s["window"])
    flops = 14.0 * s["D"] * s["Hq"] * pairs
    t0 = time.perf_counter()
    oracle.dualkv(s["P"], s["N"], s["off"], s["Hq"], s["Hkv"], s["D"], s["scale"], s["window"], s["q"], s["k"],
                  s["v"], s["do"])
    dt = time.perf_counter() - t0
    return flops, dt, oracle.num_threads()


def sample_text(w, s):
    return (f"{w.name}: prompt P={s['P']} with the first {s['N']} of {w.N} responses "
            f"(R_offsets {s['off']}), q-head 0 and kv-head 0, D={s['D']}, "
            f"fwd+bwd; useful FLOPs counted on the sample's packed pairs")


def run_reference(args, w):
    world, rank, local = dist_setup()
    if rank != 0:
        return 0
    q, k, v, do = wl.draw_inputs(w)
    s = oracle_sample(w, q, k, v, do, n_seg=args.oracle_segments)
    for _ in range(args.warmup):
        time_oracle(s)
    times = []
    flops = 0.0
    cores = 1
    for _ in range(args.steps):
        flops, dt, cores = time_oracle(s)
        times.append(dt)
    ms = 1e3 * sum(times) / len(times)
    value = flops / (ms * 1e-3) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "P": w.P, "N": w.N, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
                   "window": w.window, "sample": sample_text(w, s)},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample_text(w, s)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ tensor packing
def measure_packing(w, dev, stream, reps):
    """dualkv_pack / dualkv_unpack / dualkv_fold on hidden-size rows (Hq * D bf16)
    of the workload's layout; each call timed alone with CUDA events on the
    launching stream.  Algorithmic bytes: every source row the definition needs
    read once, every destination row written once."""
    from shared_prompt_exact_gb300 import dualkv
    E = w.Hq * w.D
    T, T_rep = w.T, w.T_replicated
    row = 2 * E
    gen = torch.Generator(device=dev).manual_seed(w.seed + 7)
    x_rep = torch.randn(T_rep, E, generator=gen, device=dev).to(torch.bfloat16)
    x_pk = torch.empty(T, E, dtype=torch.bfloat16, device=dev)
    ops = {
        "pack": (lambda: dualkv.dualkv_pack(x_rep, x_pk, w.P, w.N, w.offsets, stream), 2 * T * row),
        "unpack": (lambda: dualkv.dualkv_unpack(x_pk, x_rep, w.P, w.N, w.offsets, stream), (T + T_rep) * row),
        "fold": (lambda: dualkv.dualkv_fold(x_rep, x_pk, w.P, w.N, w.offsets, stream), (T_rep + T) * row),
    }
    hbm = peaks()
    res = {"row_elems": E, "packed_rows": T, "replicated_rows": T_rep,
           "l2": "no flush: each call moves more than L2 (%.2f GB replicated)" % (T_rep * row / 1e9)}
    for name, (fn, nbytes) in ops.items():
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / reps
        gbs = nbytes / (ms * 1e-3) / 1e9
        res[name] = {"ms": ms, "algorithmic_bytes": nbytes, "GB/s": gbs, "frac_hbm": gbs / hbm["hbm_gbs"],
                     "peak_source": hbm["source"] + " copy bandwidth"}
    dualkv.dualkv_check_status(stream)
    del x_rep, x_pk
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------------ other workloads, fresh layouts
def _timed_on(stream, dev, fn, reps):
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / reps


def measure_workload(name, dev, stream, steps, sampler):
    """fwd, bwd and fwd+bwd useful TFLOP/s of one workload (its own seeded inputs,
    resident in HBM) and the per-kernel times of its launches; each timed alone with
    CUDA events on the launching stream after two warm-up steps."""
    from shared_prompt_exact_gb300 import dualkv
    w = wl.WORKLOADS[name]
    q, k, v, do = (x.to(dev) for x in wl.draw_inputs(w))
    out = torch.empty_like(q)
    lse = torch.empty(w.Hq, w.T, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = dualkv.workspace_for(w.P, w.offsets, w.Hq, w.Hkv, w.D, w.window, dev)

    def fwd():
        dualkv.dualkv_fwd(q, k, v, w.P, w.N, w.offsets, w.Hq, w.Hkv, w.D, w.scale, w.window, out, lse, stream)

    def bwd():
        dualkv.dualkv_bwd(q, k, v, out, lse, do, w.P, w.N, w.offsets, w.Hq, w.Hkv, w.D, w.scale, w.window, dq, dk,
                          dv, ws, None, stream)

    def step():
        fwd()
        bwd()

    for _ in range(2):
        step()
    dualkv.dualkv_check_status(stream)
    # enough steps for the timed region to last about 0.6 s, so that the clock sampler
    # (every 200 ms) sees it
    reps = max(steps, min(200, int(math.ceil(600.0 / max(_timed_on(stream, dev, step, 1), 1e-3)))))
    t0 = time.time()
    ms_step = _timed_on(stream, dev, step, reps)
    t1 = time.time()
    ms_fwd = _timed_on(stream, dev, fwd, steps)
    ms_bwd = _timed_on(stream, dev, bwd, steps)
    dualkv.dualkv_profile_read()
    dualkv.dualkv_profile_enable(True)
    for _ in range(2):
        step()
    torch.cuda.synchronize(dev)
    kt = dualkv.dualkv_profile_read()
    dualkv.dualkv_profile_enable(False)
    dualkv.dualkv_check_status(stream)
    pairs = layout_pairs(w)
    f_fwd, f_bwd = useful_flops(pairs, w.D, w.Hq)
    pk = peaks()
    res = {
        "P": w.P, "N": w.N, "R": (w.R[0] if len(set(w.R)) == 1 else "ragged"), "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
        "window": w.window, "pairs_per_head": pairs, "rho": dualkv.dualkv_rho(w.P, w.N, w.offsets),
        "timed_steps": reps,
        "fwd": {"ms": ms_fwd, "tflops": f_fwd / (ms_fwd * 1e-3) / 1e12},
        "bwd": {"ms": ms_bwd, "tflops": f_bwd / (ms_bwd * 1e-3) / 1e12},
        "fwd_bwd": {"ms": ms_step, "tflops": (f_fwd + f_bwd) / (ms_step * 1e-3) / 1e12},
        "kernels_ms_per_step": {kk: ms / 2 for kk, (ms, n) in kt.items() if n},
        "clocks": sampler.summary(t0, t1),
    }
    res["pct_bf16_peak"] = {"measured_burst": res["fwd_bwd"]["tflops"] / pk["bf16_burst"],
                            "measured_sustained": res["fwd_bwd"]["tflops"] / pk["bf16_sustained"],
                            "nominal_2250": res["fwd_bwd"]["tflops"] / 2250.0}
    del q, k, v, do, out, lse, dq, dk, dv, ws
    torch.cuda.empty_cache()
    return res


def fresh_r_lists(n, N=32, lo=256, hi=4096, seed=20260518):
    """Per-step ragged response lengths, uniform on [lo, hi], one fixed-seed draw per step."""
    import numpy as np
    return [[int(x) for x in np.random.default_rng(seed + 1000 + i).integers(lo, hi + 1, N)] for i in range(n)]


def measure_fresh_layouts(base, dev, stream, steps):
    """The DAPO-like workload with a new ragged response list every step (a training
    loop repacks each micro-batch, so every call meets a layout it has not planned):
    plan building, its upload and the step all inside the timed region.  Compared
    with the same steps repeated on one layout (plans cached)."""
    from shared_prompt_exact_gb300 import dualkv
    lists = fresh_r_lists(steps, N=base.N)
    ws_ = [wl.custom(base.P, R, base.Hq, base.Hkv, base.D, base.window, seed=base.seed) for R in lists]
    Tmax = max(x.T for x in ws_)
    gen = torch.Generator(device=dev).manual_seed(base.seed)
    rnd = lambda *shape: torch.randn(*shape, generator=gen, device=dev).to(torch.bfloat16)  # noqa: E731
    q, k, v, do = rnd(Tmax, base.Hq, base.D), rnd(Tmax, base.Hkv, base.D), rnd(Tmax, base.Hkv, base.D), \
        rnd(Tmax, base.Hq, base.D)
    out = torch.empty_like(q)
    lse_all = torch.empty(base.Hq * Tmax, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_bytes = max(dualkv.dualkv_bwd_workspace_bytes(x.P, x.N, x.offsets, x.Hq, x.Hkv, x.D, x.window) for x in ws_)
    wsb = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)

    def step(x):
        T = x.T
        lse = lse_all[: x.Hq * T].view(x.Hq, T)
        dualkv.dualkv_fwd(q[:T], k[:T], v[:T], x.P, x.N, x.offsets, x.Hq, x.Hkv, x.D, x.scale, x.window, out[:T], lse,
                          stream)
        dualkv.dualkv_bwd(q[:T], k[:T], v[:T], out[:T], lse, do[:T], x.P, x.N, x.offsets, x.Hq, x.Hkv, x.D, x.scale,
                          x.window, dq[:T], dk[:T], dv[:T], wsb, None, stream)

    flops = sum(sum(useful_flops(layout_pairs(x), x.D, x.Hq)) for x in ws_)
    # fresh: drop every plan, warm up on three other layouts, then a layout not seen
    # before on each timed step
    warm = [wl.custom(base.P, R, base.Hq, base.Hkv, base.D, base.window, seed=base.seed)
            for R in fresh_r_lists(3, N=base.N, seed=base.seed + 777)]
    torch.cuda.synchronize(dev)
    dualkv.dualkv_release()
    for x in warm:
        step(x)
    it = iter(ws_)
    ms_fresh = _timed_on(stream, dev, lambda: step(next(it)), steps)
    # cached: the same sequence of layouts again, every plan now resident
    it = iter(ws_)
    ms_cached = _timed_on(stream, dev, lambda: step(next(it)), steps)
    dualkv.dualkv_check_status(stream)
    tf_fresh = flops / (ms_fresh * steps * 1e-3) / 1e12
    tf_cached = flops / (ms_cached * steps * 1e-3) / 1e12
    n_plans, cache_bytes = dualkv.dualkv_plan_cache_info()
    del q, k, v, do, out, lse_all, dq, dk, dv, wsb
    torch.cuda.empty_cache()
    return {"workload": f"{base.name} with a new R list each step (uniform [256, 4096], N={base.N})",
            "steps": steps, "ms_per_step_fresh": ms_fresh, "tflops_fresh": tf_fresh,
            "ms_per_step_cached": ms_cached, "tflops_cached": tf_cached,
            "fresh_over_cached_tflops": tf_fresh / tf_cached,
            "compared": "the same sequence of layouts, first unplanned, then with every plan cached",
            "plan_cache": {"resident_plans": n_plans, "device_bytes": cache_bytes}}


# ------------------------------------------------------------------ GPU arm
def run_dualkv(args, w):
    from shared_prompt_exact_gb300 import build as pbuild
    from shared_prompt_exact_gb300 import dualkv

    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pbuild.build()
    dualkv.load()

    q_h, k_h, v_h, do_h = wl.draw_inputs(w)
    q, k, v, do = (x.to(dev) for x in (q_h, k_h, v_h, do_h))
    T, Hq, Hkv, D = w.T, w.Hq, w.Hkv, w.D
    out = torch.empty_like(q)
    lse = torch.empty(Hq, T, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = dualkv.workspace_for(w.P, w.offsets, Hq, Hkv, D, w.window, dev)
    stream = torch.cuda.current_stream(dev)

    # --shard heads: every rank computes its own contiguous group of kv-heads of the
    # same micro-batch through the head-range entry points (the layout a
    # head-sharded sequence-parallel rank holds after its exchange); no collective
    shard = args.shard == "heads" and world > 1
    klo, khi = dualkv.kv_head_ranges(Hkv, world)[rank] if shard else (0, Hkv)
    head_frac = (khi - klo) / Hkv

    def run_fwd(q_, k_, v_, out_, lse_):
        if not shard:
            dualkv.dualkv_fwd(q_, k_, v_, w.P, w.N, w.offsets, Hq, Hkv, D, w.scale, w.window, out_, lse_, stream)
        elif khi > klo:
            dualkv.dualkv_fwd_heads(q_, k_, v_, w.P, w.N, w.offsets, Hq, Hkv, D, w.scale, w.window, klo, khi, out_,
                                    lse_, stream)

    def run_bwd(q_, k_, v_, out_, lse_, do_, dq_, dk_, dv_):
        if not shard:
            dualkv.dualkv_bwd(q_, k_, v_, out_, lse_, do_, w.P, w.N, w.offsets, Hq, Hkv, D, w.scale, w.window, dq_,
                              dk_, dv_, ws, None, stream)
        elif khi > klo:
            dualkv.dualkv_bwd_heads(q_, k_, v_, out_, lse_, do_, w.P, w.N, w.offsets, Hq, Hkv, D, w.scale, w.window,
                                    klo, khi, dq_, dk_, dv_, ws, None, stream)

    def fwd():
        run_fwd(q, k, v, out, lse)

    def bwd():
        run_bwd(q, k, v, out, lse, do, dq, dk, dv)

    def step():
        fwd()
        bwd()

    pairs = layout_pairs(w)
    f_fwd, f_bwd = useful_flops(pairs, D, Hq)
    f_step = f_fwd + f_bwd

    for _ in range(max(args.warmup, 1)):
        step()
    dualkv.dualkv_check_status(stream)

    sampler = ClockSampler(local)
    sampler.start()

    def timed(fn, reps):
        barrier(world)
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        return e0.elapsed_time(e1) / reps

    t_start = time.time()
    ms_step = timed(step, args.steps)
    t_end = time.time()
    if shard:
        ms_step, value = aggregate_strong(ms_step, f_step * head_frac, world, dev)
    else:
        ms_step, value = aggregate(ms_step, f_step, world, dev)
    ms_fwd = max_over_ranks(timed(fwd, args.steps), world, dev)
    ms_bwd = max_over_ranks(timed(bwd, args.steps), world, dev)
    dualkv.dualkv_check_status(stream)

    # per-kernel durations (events on the launching stream, recorded by the library)
    prof_steps = max(1, min(args.steps, 5))
    dualkv.dualkv_profile_read()
    dualkv.dualkv_profile_enable(True)
    for _ in range(prof_steps):
        step()
    torch.cuda.synchronize(dev)
    kt = dualkv.dualkv_profile_read()
    dualkv.dualkv_profile_enable(False)
    launches_per_step = sum(n for _, n in kt.values()) / prof_steps
    dom = max(kt, key=lambda kk: kt[kk][0])
    pk = peaks()
    roofline = None
    if kernel_flops_per_pair(dom, D) and kt[dom][1] > 0:
        per_launch_flops = kernel_flops_per_pair(dom, D) * D * Hq * pairs * head_frac
        avg_ms = kt[dom][0] / kt[dom][1]
        achieved = per_launch_flops / (avg_ms * 1e-3) / 1e12
        roofline = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": pk["bf16_burst"],
                    "unit": "TFLOP/s", "frac": achieved / pk["bf16_burst"],
                    "traffic": ncu_traffic(dom, w.name),
                    "peak_source": pk["source"] + " bf16 burst (each launch lasts milliseconds, inside a step of "
                                   "tens of milliseconds)",
                    "frac_of_sustained": achieved / pk["bf16_sustained"],
                    "avg_launch_ms": avg_ms, "algorithmic_flops_per_launch": per_launch_flops}
    kernels = {kk: {"ms_per_launch": (ms / n if n else None), "launches": n} for kk, (ms, n) in kt.items()}

    # the same step as W head-range calls of Hkv / W kv-heads each (the per-rank
    # share of a W-way head split), run back to back on this GPU
    head_groups = {}
    for W in (() if shard else (2, Hkv)):
        if W < 2 or Hkv % W:
            continue
        ranges = [(i * Hkv // W, (i + 1) * Hkv // W) for i in range(W)]

        def hstep(ranges=ranges):
            for lo, hi in ranges:
                dualkv.dualkv_fwd_heads(q, k, v, w.P, w.N, w.offsets, Hq, Hkv, D, w.scale, w.window, lo, hi, out,
                                        lse, stream)
                dualkv.dualkv_bwd_heads(q, k, v, out, lse, do, w.P, w.N, w.offsets, Hq, Hkv, D, w.scale, w.window,
                                        lo, hi, dq, dk, dv, ws, None, stream)

        hstep()
        ms_h = max_over_ranks(timed(hstep, max(1, min(args.steps, 5))), world, dev)
        head_groups[f"{W}x{Hkv // W}kv"] = {"ms_per_step": ms_h, "tflops": f_step / (ms_h * 1e-3) / 1e12,
                                             "ms_per_group": ms_h / W}
    dualkv.dualkv_check_status(stream)

    # end to end through the C ABI with host buffers: every step uploads its q, k, v, dO
    # from pinned host memory and downloads out, lse, dq, dk, dv.  As in a training
    # loop that prefetches its next micro-batch, device buffers are double-buffered:
    # uploads run on their own stream (dO's overlaps the forward, the next step's
    # overlap this step's backward), downloads on another (out and lse overlap the
    # backward).  Every copy lies inside the timed region.
    e2e = None
    if not args.no_e2e:
        pin = lambda x: x.pin_memory()  # noqa: E731
        hq, hk, hv, hdo = (pin(x) for x in (q_h, k_h, v_h, do_h))
        ho, hl, hdq, hdk, hdv = (torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in (out, lse, dq, dk, dv))
        h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, hdo))
        d2h = sum(x.numel() * x.element_size() for x in (ho, hl, hdq, hdk, hdv))
        up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        dins = [(q, k, v, do)] + [tuple(torch.empty_like(x) for x in (q, k, v, do))]
        douts = [(out, lse, dq, dk, dv)] + [tuple(torch.empty_like(x) for x in (out, lse, dq, dk, dv))]
        in_free, out_free = [None, None], [None, None]

        def e2e_step(i):
            bsel = i & 1
            qd, kd, vd, dod = dins[bsel]
            od, ld, dqd, dkd, dvd = douts[bsel]
            with torch.cuda.stream(up):
                if in_free[bsel] is not None:
                    up.wait_event(in_free[bsel])
                qd.copy_(hq, non_blocking=True)
                kd.copy_(hk, non_blocking=True)
                vd.copy_(hv, non_blocking=True)
                e_qkv = torch.cuda.Event()
                e_qkv.record(up)
                dod.copy_(hdo, non_blocking=True)
                e_do = torch.cuda.Event()
                e_do.record(up)
            stream.wait_event(e_qkv)
            if out_free[bsel] is not None:
                stream.wait_event(out_free[bsel])
            run_fwd(qd, kd, vd, od, ld)
            e_fwd = torch.cuda.Event()
            e_fwd.record(stream)
            stream.wait_event(e_do)
            run_bwd(qd, kd, vd, od, ld, dod, dqd, dkd, dvd)
            e_bwd = torch.cuda.Event()
            e_bwd.record(stream)
            in_free[bsel] = e_bwd
            with torch.cuda.stream(down):
                down.wait_event(e_fwd)
                ho.copy_(od, non_blocking=True)
                hl.copy_(ld, non_blocking=True)
                down.wait_event(e_bwd)
                hdq.copy_(dqd, non_blocking=True)
                hdk.copy_(dkd, non_blocking=True)
                hdv.copy_(dvd, non_blocking=True)
                e_out = torch.cuda.Event()
                e_out.record(down)
                out_free[bsel] = e_out

        def timed_e2e(reps):
            barrier(world)
            torch.cuda.synchronize(dev)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            up.wait_event(e0)
            down.wait_event(e0)
            for i in range(reps):
                e2e_step(i)
            stream.wait_stream(up)
            stream.wait_stream(down)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            barrier(world)
            return e0.elapsed_time(e1) / reps

        e2e_step(0)
        e2e_step(1)
        torch.cuda.synchronize(dev)
        ms_e2e = max_over_ranks(timed_e2e(max(2, min(args.steps, 10))), world, dev)
        dualkv.dualkv_check_status(stream)
        job_flops = f_step if shard else world * f_step
        e2e = {"value": job_flops / (ms_e2e * 1e-3) / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e,
               "pipelining": "double-buffered device inputs/outputs; uploads and downloads on their own streams"}
        dins.clear()
        douts.clear()

    # the same kernels on the replicated layout (prompt copied into every sequence)
    replicated = None
    if not args.no_replicated and not shard:
        wr = w.replicated()
        del out, dq
        torch.cuda.empty_cache()
        qr, kr, vr, dor = (wl.replicate_rows(w, x) for x in (q, k, v, do))
        outr = torch.empty_like(qr)
        lser = torch.empty(Hq, wr.T, dtype=torch.float32, device=dev)
        dqr, dkr, dvr = torch.empty_like(qr), torch.empty_like(kr), torch.empty_like(vr)
        wsr = dualkv.workspace_for(wr.P, wr.offsets, Hq, Hkv, D, wr.window, dev)

        def rstep():
            dualkv.dualkv_fwd(qr, kr, vr, wr.P, wr.N, wr.offsets, Hq, Hkv, D, wr.scale, wr.window, outr, lser, stream)
            dualkv.dualkv_bwd(qr, kr, vr, outr, lser, dor, wr.P, wr.N, wr.offsets, Hq, Hkv, D, wr.scale, wr.window,
                              dqr, dkr, dvr, wsr, None, stream)

        rstep()
        ms_rep = max_over_ranks(timed(rstep, max(1, min(args.steps, 5))), world, dev)
        dualkv.dualkv_check_status(stream)
        pairs_r = layout_pairs(wr)
        fr = sum(useful_flops(pairs_r, D, Hq))
        replicated = {"ms_per_step": ms_rep, "tflops_own_pairs": fr / (ms_rep * 1e-3) / 1e12,
                      "tflops_effective": f_step / (ms_rep * 1e-3) / 1e12, "pairs_per_head": pairs_r,
                      "speedup_packed_over_replicated": ms_rep / ms_step}
        del qr, kr, vr, dor, outr, dqr, dkr, dvr, wsr

    packing = None
    if not args.no_pack:
        packing = measure_packing(w, dev, stream, max(3, min(args.steps, 10)))

    # every other workload of the benchmark's configuration list, measured the same way
    others = {}
    if not args.no_configs and not shard:
        for name in ("qwen16", "dapo32", "gemma_global", "gemma_window"):
            if name != w.name:
                others[name] = measure_workload(name, dev, stream, max(3, min(args.steps, 5)), sampler)

    fresh = None
    if not args.no_fresh_layouts and not shard:
        fresh = measure_fresh_layouts(wl.WORKLOADS["dapo32"], dev, stream, max(4, min(args.steps, 10)))

    sampler.stop()
    clocks = sampler.summary(t_start, t_end)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        s = oracle_sample(w, q_h, k_h, v_h, do_h, n_seg=args.oracle_segments)
        flops_s, dt, cores = time_oracle(s)
        cpu = {"value": flops_s / dt / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": sample_text(w, s), "seconds": dt}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "strong" if shard else "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "P": w.P, "N": w.N, "R": (w.R[0] if len(set(w.R)) == 1 else "ragged"),
                       "Hq": Hq, "Hkv": Hkv, "D": D, "window": w.window, "packed_tokens": T,
                       "replicated_tokens": w.T_replicated, "pairs_per_head": pairs,
                       "l2": "no flush: inputs larger than L2 (q+k+v+dO = %.2f GB)" % (
                           sum(x.numel() * x.element_size() for x in (q, k, v, do)) / 1e9),
                       "parallelism": (f"kv-head groups x{world}" if shard else f"replicas x{world}")},
            "pct_bf16_peak": {"measured_burst": value / world / pk["bf16_burst"],  # per GPU
                              "measured_sustained": value / world / pk["bf16_sustained"],
                              "nominal_2250": value / world / 2250.0},
            "fwd": {"ms": ms_fwd, "tflops": f_fwd / (ms_fwd * 1e-3) / 1e12},
            "bwd": {"ms": ms_bwd, "tflops": f_bwd / (ms_bwd * 1e-3) / 1e12},
            "rho": dualkv.dualkv_rho(w.P, w.N, w.offsets),
            "kernels": kernels,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "replicated": replicated,
            "tensor_packing": packing,
            "head_groups": head_groups,
            "other_workloads": others,
            "fresh_layouts": fresh,
            "gpu_launches": int(round(launches_per_step * args.steps)),
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------------------ layer stacks
def run_layers(args, w):
    """A stack of attention layers over one packed micro-batch: `--layers` is a
    pattern of S (sliding window `--slide-window`) and G (global) layers.  One
    step = dualkv_fwd_layers over the stack + dualkv_bwd_layers in reverse layer
    order; the metric is the stack's useful TFLOP/s."""
    from shared_prompt_exact_gb300 import build as pbuild
    from shared_prompt_exact_gb300 import dualkv

    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pbuild.build()
    dualkv.load()
    windows = [args.slide_window if c == "S" else 0 for c in args.layers]
    n = len(windows)
    T, Hq, Hkv, D = w.T, w.Hq, w.Hkv, w.D
    gen = torch.Generator(device=dev).manual_seed(w.seed)
    rnd = lambda *shape: torch.randn(*shape, generator=gen, device=dev).to(torch.bfloat16)  # noqa: E731
    qs = [rnd(T, Hq, D) for _ in range(n)]
    ks = [rnd(T, Hkv, D) for _ in range(n)]
    vs = [rnd(T, Hkv, D) for _ in range(n)]
    dos = [rnd(T, Hq, D) for _ in range(n)]
    outs = [torch.empty_like(x) for x in qs]
    lses = [torch.empty(Hq, T, dtype=torch.float32, device=dev) for _ in range(n)]
    dqs, dks, dvs = ([torch.empty_like(x) for x in xs] for xs in (qs, ks, vs))
    nbytes = dualkv.dualkv_bwd_layers_workspace_bytes(windows, w.P, w.N, w.offsets, Hq, Hkv, D)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    r = lambda xs: xs[::-1]  # noqa: E731

    def step():
        dualkv.dualkv_fwd_layers(qs, ks, vs, windows, w.P, w.N, w.offsets, Hq, Hkv, D, w.scale, outs, lses, stream)
        dualkv.dualkv_bwd_layers(r(qs), r(ks), r(vs), r(outs), r(lses), r(dos), r(windows), w.P, w.N, w.offsets, Hq,
                                 Hkv, D, w.scale, r(dqs), r(dks), r(dvs), ws, None, stream)

    flops = 0.0
    per_window = {}
    for W in windows:
        pairs = dualkv.dualkv_pairs(w.P, w.N, w.offsets, W)
        flops += sum(useful_flops(pairs, D, Hq))
        per_window[str(W)] = pairs
    for _ in range(max(args.warmup, 1)):
        step()
    dualkv.dualkv_check_status(stream)
    sampler = ClockSampler(local)
    sampler.start()
    barrier(world)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start = time.time()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    t_end = time.time()
    ms, value = aggregate(e0.elapsed_time(e1) / args.steps, flops, world, dev)
    dualkv.dualkv_profile_read()
    dualkv.dualkv_profile_enable(True)
    step()
    torch.cuda.synchronize(dev)
    kt = dualkv.dualkv_profile_read()
    dualkv.dualkv_profile_enable(False)
    dualkv.dualkv_check_status(stream)
    sampler.stop()
    pk = peaks()
    if rank == 0:
        line = {
            "metric": "DualKV layer stack fwd+bwd useful TFLOP/s", "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"{w.name}-stack-{args.layers}", "layers": args.layers, "windows": windows,
                       "P": w.P, "N": w.N, "R": list(sorted(set(w.R))), "Hq": Hq, "Hkv": Hkv, "D": D,
                       "pairs_per_head": per_window,
                       "l2": "no flush: every layer's inputs are larger than L2"},
            "pct_bf16_peak": {"measured_sustained": value / world / pk["bf16_sustained"]},
            "kernels": {kk: {"ms_per_launch": (t / c if c else None), "launches": c} for kk, (t, c) in kt.items()},
            "gpu_launches": int(sum(c for _, c in kt.values()) * args.steps),
            "clocks": sampler.summary(t_start, t_end),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("dualkv", "reference"), default="dualkv")
    ap.add_argument("--config", default="grpo32", choices=sorted(wl.WORKLOADS))
    ap.add_argument("--oracle-segments", type=int, default=1)
    ap.add_argument("--heads", default=None,
                    help="Hq,Hkv override: a smaller case of the same layout for ncu captures")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-replicated", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-pack", action="store_true", help="skip the pack/unpack/fold measurement")
    ap.add_argument("--no-configs", action="store_true", help="skip the blocks of the other four workloads")
    ap.add_argument("--no-fresh-layouts", action="store_true",
                    help="skip the block with a new ragged layout every step")
    ap.add_argument("--shard", choices=("replicas", "heads"), default="replicas",
                    help="N > 1: independent replicas (weak scaling) or one micro-batch split by kv-head group "
                         "(strong scaling)")
    ap.add_argument("--layers", default=None,
                    help="time a layer stack instead: a pattern of S (sliding) and G (global) layers, e.g. SSSSSG")
    ap.add_argument("--slide-window", type=int, default=1024, help="window of the S layers of --layers")
    args = ap.parse_args(argv)
    w = wl.WORKLOADS[args.config]
    if args.heads:
        hq, hkv = (int(x) for x in args.heads.split(","))
        w = dataclasses.replace(w, name=f"{w.name}-h{hq}x{hkv}", Hq=hq, Hkv=hkv)
    if args.layers:
        if set(args.layers) - {"S", "G"}:
            ap.error("--layers takes a pattern of S and G")
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "--layers times the GPU path only"}))
            return 0
        return run_layers(args, w)
    if args.impl == "reference":
        return run_reference(args, w)
    return run_dualkv(args, w)


if __name__ == "__main__":
    sys.exit(main())
