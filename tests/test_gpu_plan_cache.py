"""The plan cache under a changing layout: a training loop repacks every
micro-batch, so the response offsets differ from call to call.  Over 100
distinct layouts the cache keeps at most its capacity of plans, its device
memory stops growing once the pool of released buffers is warm, and every
call still computes the right result (checked against the fp64 oracle on a few
of them and, for all, against a second run on a layout already evicted)."""
import numpy as np
import pytest
import torch

import oracle
from parity_checks import check_full
from shared_prompt_exact_gb300 import build as pbuild
from shared_prompt_exact_gb300 import dualkv
from shared_prompt_exact_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

CAPACITY = 32


def _layout(i):
    rng = np.random.default_rng(1000 + i)
    R = [int(x) for x in rng.integers(0, 200, 4)]
    return wl.custom(96 + int(rng.integers(0, 64)), R, 2, 1, 64, 0, seed=2000 + i)


def test_cache_stays_bounded_and_correct_over_100_layouts():
    pbuild.build()
    dualkv.dualkv_release()
    first = {}
    bytes_after = {}
    for i in range(100):
        w = _layout(i)
        q, k, v, do = wl.draw_inputs(w)
        qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
        out, lse = dualkv.forward(qd, kd, vd, w.P, w.offsets, w.window, w.scale)
        dq, dk, dv = dualkv.backward(qd, kd, vd, out, lse, dod, w.P, w.offsets, w.window, w.scale)
        if i in (0, 57, 99):
            dualkv.dualkv_check_status()
            ref = oracle.dualkv(w.P, w.N, w.offsets, w.Hq, w.Hkv, w.D, w.scale, w.window, q, k, v, do)
            check_full(dict(out=out, lse=lse, dq=dq, dk=dk, dv=dv), ref)
        if i < 8:
            first[i] = (w, (qd, kd, vd, dod), [t.clone() for t in (out, lse, dq, dk, dv)])
        n, nbytes = dualkv.dualkv_plan_cache_info()
        assert n <= CAPACITY
        bytes_after[i] = nbytes
    dualkv.dualkv_check_status()
    assert dualkv.dualkv_plan_cache_info()[0] == CAPACITY
    # the pool is warm after the first evictions: no growth over the last 40 layouts
    assert bytes_after[99] <= bytes_after[59]
    # layouts evicted long ago are planned again and give bitwise the same results
    for i, (w, (qd, kd, vd, dod), want) in first.items():
        out, lse = dualkv.forward(qd, kd, vd, w.P, w.offsets, w.window, w.scale)
        dq, dk, dv = dualkv.backward(qd, kd, vd, out, lse, dod, w.P, w.offsets, w.window, w.scale)
        for a, b in zip((out, lse, dq, dk, dv), want):
            assert torch.equal(a, b), i
    dualkv.dualkv_check_status()
