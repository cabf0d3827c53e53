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
