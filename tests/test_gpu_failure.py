"""Failure detection without a GPU fault: a bounded device wait on a barrier
that nothing completes gives up after its limit, the host reads the timeout
from the status word, and the context keeps working afterwards."""
import time

import pytest
import torch

from shared_prompt_exact_gb300 import build as pbuild
from shared_prompt_exact_gb300 import dualkv
from shared_prompt_exact_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    pbuild.build()
    dualkv.dualkv_check_status()  # clear
    t0 = time.time()
    dualkv.dualkv_selftest_timeout(50_000_000)  # 50 ms
    with pytest.raises(dualkv.DualKVError) as ei:
        dualkv.dualkv_check_status()
    assert ei.value.code == dualkv.DUALKV_ERR_DEVICE
    assert time.time() - t0 < 30
    # status was cleared and the context still runs kernels correctly
    dualkv.dualkv_check_status()
    w = wl.WORKLOADS["tiny"]
    q, k, v, _ = wl.draw_inputs(w, with_dout=False)
    out, lse = dualkv.forward(q.cuda(), k.cuda(), v.cuda(), w.P, w.offsets)
    dualkv.dualkv_check_status()
    assert torch.isfinite(out.float()).all()


KERNEL_CASES = [
    (0, "forward: a K/V tile never loaded"),
    (1, "dK/dV: a query block one barrier arrival short"),
    (2, "forward: a work item past the last row"),
    (3, "dQ: a work item past the last row, emptied by the preprocess"),
    (4, "D = 512 P / dS pass: a K/V tile never loaded"),
]


@pytest.mark.parametrize("which,what", KERNEL_CASES,
                         ids=["fwd-timeout", "dkv-timeout", "fwd-bounds", "dq-bounds", "pds512-timeout"])
def test_production_kernel_failure_paths(which, what):
    # the real kernels' failure handling: the bounded waits (50 ms here) run out, or
    # the range check skips the bad entry; the kernel drains, frees its tensor memory
    # and returns, the host reads the status, and the next launches are correct
    import numpy as np

    import oracle
    from parity_checks import check_full

    pbuild.build()
    dualkv.dualkv_check_status()  # clear
    t0 = time.time()
    dualkv.dualkv_selftest_kernel(which, 50_000_000)
    with pytest.raises(dualkv.DualKVError) as ei:
        dualkv.dualkv_check_status()
    assert ei.value.code == dualkv.DUALKV_ERR_DEVICE, what
    assert time.time() - t0 < 30
    dualkv.dualkv_check_status()  # the status word was cleared
    w = wl.custom(128, [128, 128], 1, 1, 128, 0, seed=9)
    q, k, v, do = wl.draw_inputs(w)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    out, lse = dualkv.forward(qd, kd, vd, w.P, w.offsets, w.window, w.scale)
    dq, dk, dv = dualkv.backward(qd, kd, vd, out, lse, dod, w.P, w.offsets, w.window, w.scale)
    dualkv.dualkv_check_status()
    ref = oracle.dualkv(w.P, w.N, w.offsets, w.Hq, w.Hkv, w.D, w.scale, w.window, q, k, v, do)
    check_full(dict(out=out, lse=lse, dq=dq, dk=dk, dv=dv), ref)
    assert np.isfinite(out.float().cpu().numpy()).all()
