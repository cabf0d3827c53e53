"""dualkv_bwd_noalloc: the backward pass for callers that cannot allocate
device memory (its scratch is a fixed array inside the library).  Two calls in
a row must reproduce what dualkv_bwd computes with a caller-provided
workspace, within the parity tolerance the other GPU tests use (normwise
relative 2e-2 on dQ, dK, dV); a layout too large for the fixed scratch must be
refused.  This file is collected last on purpose."""
import numpy as np
import pytest
import torch

from shared_prompt_exact_gb300 import build as pbuild
from shared_prompt_exact_gb300 import dualkv
from shared_prompt_exact_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

G_REL = 2e-2


def relF(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


@pytest.mark.parametrize("layout", [
    ("tiny", None),
    ("split-prompt-tiles", (128, [512] * 16, 4, 1, 64, 0)),  # exercises the split partials in the scratch
    ("ragged-window-gqa", (300, [200, 0, 129, 1, 64], 4, 2, 128, 70)),
])
def test_noalloc_backward_matches_workspace_backward_twice(layout):
    pbuild.build()
    name, c = layout
    w = wl.WORKLOADS["tiny"] if c is None else wl.custom(*c, seed=77)
    q, k, v, do = (x.cuda() for x in wl.draw_inputs(w))
    out, lse = dualkv.forward(q, k, v, w.P, w.offsets, w.window, w.scale)
    ref = dualkv.backward(q, k, v, out, lse, do, w.P, w.offsets, w.window, w.scale)
    dualkv.dualkv_check_status()
    for _ in range(2):
        dq = torch.full_like(q, float("nan"))
        dk = torch.full_like(k, float("nan"))
        dv = torch.full_like(v, float("nan"))
        dualkv.dualkv_bwd_noalloc(q, k, v, out, lse, do, w.P, w.N, w.offsets, w.Hq, w.Hkv, w.D, w.scale, w.window,
                                  dq, dk, dv)
        for got, want in zip((dq, dk, dv), ref):
            assert torch.isfinite(got.float()).all()
            assert relF(got, want) <= G_REL


def test_noalloc_refuses_layouts_beyond_the_fixed_scratch():
    pbuild.build()
    # Delta + lse2 alone need 8 * Hq * T bytes = 64 MiB here, twice the scratch
    w = wl.custom(0, [1 << 16], 128, 128, 64, 0)
    t = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    f = torch.empty(16, dtype=torch.float32, device="cuda")
    with pytest.raises(dualkv.DualKVError) as ei:
        dualkv.dualkv_bwd_noalloc(t, t, t, t, f, t, w.P, w.N, w.offsets, w.Hq, w.Hkv, w.D, w.scale, 0, t, t, t)
    assert ei.value.code == dualkv.DUALKV_ERR_WORKSPACE
