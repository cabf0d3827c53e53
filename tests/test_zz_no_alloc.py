"""dualkv_bwd_noalloc: the backward pass for callers that cannot allocate device
memory -- a runtime that hands all device memory to its own pool at start-up
and fails any later cudaMalloc, or a host binding that owns no device
allocator.  Its scratch is a fixed array inside the library.

It runs the same kernels on the same work lists as dualkv_bwd, so its dQ, dK
and dV must be bitwise those of dualkv_bwd with a caller-provided workspace,
on two calls in a row, even when the scratch still holds another layout's
contents; one case is also compared with the fp64 oracle.  A layout too large
for the fixed scratch and a head dimension it does not serve must be refused.
This file is collected last on purpose."""
import ctypes

import pytest
import torch

import oracle
from parity_checks import check_full
from shared_prompt_exact_gb300 import build as pbuild
from shared_prompt_exact_gb300 import dualkv
from shared_prompt_exact_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16)


def _noalloc(w, q, k, v, out, lse, do, fill=float("nan")):
    dq = torch.full_like(q, fill)
    dk = torch.full_like(k, fill)
    dv = torch.full_like(v, fill)
    dualkv.dualkv_bwd_noalloc(q, k, v, out, lse, do, w.P, w.N, w.offsets, w.Hq, w.Hkv, w.D, w.scale, w.window,
                              dq, dk, dv)
    return dq, dk, dv


def _inputs(w):
    host = wl.draw_inputs(w)
    q, k, v, do = (x.cuda() for x in host)
    out, lse = dualkv.forward(q, k, v, w.P, w.offsets, w.window, w.scale)
    return host, (q, k, v, out, lse, do)


def _leave_foreign_scratch():
    """One call on another, larger layout (split prompt tiles, D = 128) so that every
    region of the scratch the next call uses first holds that call's values."""
    w = wl.custom(256, [384] * 24, 4, 1, 128, 0, seed=4242)
    _, (q, k, v, out, lse, do) = _inputs(w)
    _noalloc(w, q, k, v, out, lse, do)


LAYOUTS = [
    ("tiny", None),
    ("split-prompt-tiles", (128, [512] * 16, 4, 1, 64, 0)),  # exercises the split partials in the scratch
    ("ragged-window-gqa", (300, [200, 0, 129, 1, 64], 4, 2, 128, 70)),
]


@pytest.mark.parametrize("layout", LAYOUTS, ids=[c[0] for c in LAYOUTS])
def test_noalloc_backward_is_bitwise_the_workspace_backward_twice(layout):
    pbuild.build()
    name, c = layout
    w = wl.WORKLOADS["tiny"] if c is None else wl.custom(*c, seed=77)
    _, (q, k, v, out, lse, do) = _inputs(w)
    ref = dualkv.backward(q, k, v, out, lse, do, w.P, w.offsets, w.window, w.scale)
    dualkv.dualkv_check_status()
    _leave_foreign_scratch()
    for _ in range(2):
        got = _noalloc(w, q, k, v, out, lse, do)
        for g, want in zip(got, ref):
            assert torch.equal(_bits(g), _bits(want))


def test_noalloc_backward_matches_the_oracle():
    pbuild.build()
    w = wl.custom(300, [200, 0, 129, 1, 64], 4, 2, 128, 70, seed=78)
    (hq, hk, hv, hdo), (q, k, v, out, lse, do) = _inputs(w)
    _leave_foreign_scratch()
    dq, dk, dv = _noalloc(w, q, k, v, out, lse, do)
    ref = oracle.dualkv(w.P, w.N, w.offsets, w.Hq, w.Hkv, w.D, w.scale, w.window, hq, hk, hv, hdo)
    check_full(dict(out=out, lse=lse, dq=dq, dk=dk, dv=dv), ref)


def test_noalloc_refuses_layouts_beyond_the_fixed_scratch():
    pbuild.build()
    # Delta + lse2 alone need 8 * Hq * T bytes = 64 MiB here, twice the scratch; the
    # call goes straight to the C ABI (the binding would first refuse these
    # deliberately undersized tensors), which refuses it before touching them
    w = wl.custom(0, [1 << 16], 128, 128, 64, 0)
    t = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    f = torch.empty(16, dtype=torch.float32, device="cuda")
    p, pf = ctypes.c_void_p(t.data_ptr()), ctypes.c_void_p(f.data_ptr())
    off = (ctypes.c_int32 * 2)(*w.offsets)
    rc = dualkv.load().dualkv_bwd_noalloc(p, p, p, p, pf, p, w.P, w.N, off, w.Hq, w.Hkv, w.D, w.scale, 0, p, p, p,
                                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == dualkv.DUALKV_ERR_WORKSPACE
