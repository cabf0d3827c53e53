"""GPU tests of the layer-stack entry points dualkv_fwd_layers / dualkv_bwd_layers.

A stack of sliding-window and global layers over one packed micro-batch must
match the fp64 oracle layer by layer (each layer with its own window), give
bitwise what separate dualkv_fwd / dualkv_bwd calls give, and launch nothing
when any layer's arguments are bad.
"""
import pytest
import torch

import oracle
from parity_checks import check_full
from shared_prompt_exact_gb300 import build as pbuild
from shared_prompt_exact_gb300 import dualkv
from shared_prompt_exact_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pbuild.build()
    dualkv.load()


def _bits(t):
    return t.view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32)


def _layers(w, windows, host=None):
    """Device inputs (q, k, v, dO) of each layer; with a list `host`, also their CPU copies."""
    layers = []
    for i, W in enumerate(windows):
        wi = wl.custom(w.P, w.R, w.Hq, w.Hkv, w.D, W, seed=w.seed + 101 * i)
        xs = wl.draw_inputs(wi)
        if host is not None:
            host.append(xs)
        layers.append(tuple(x.cuda() for x in xs))
    return layers


CASES = [
    # name, P, R, Hq, Hkv, D, windows (0 = global)
    ("d512-sgs", 300, [200, 129, 70], 4, 2, 512, [100, 0, 100]),
    ("d128-mixed", 257, [130, 0, 64, 3], 4, 1, 128, [0, 64, 0, 1]),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_stack_equals_single_layer_calls(case, o_error_log):
    name, P, R, Hq, Hkv, D, windows = case
    w = wl.custom(P, R, Hq, Hkv, D, 0, seed=77)
    host = []
    layers = _layers(w, windows, host)
    n = len(windows)
    qs, ks, vs, dos = ([x[i] for x in layers] for i in range(4))
    outs = [torch.full_like(q, float("nan")) for q in qs]
    lses = [torch.full((Hq, w.T), float("nan"), device="cuda") for _ in range(n)]
    dualkv.dualkv_fwd_layers(qs, ks, vs, windows, P, w.N, w.offsets, Hq, Hkv, D, w.scale, outs, lses)
    nbytes = dualkv.dualkv_bwd_layers_workspace_bytes(windows, P, w.N, w.offsets, Hq, Hkv, D)
    assert nbytes == max(dualkv.dualkv_bwd_workspace_bytes(P, w.N, w.offsets, Hq, Hkv, D, W) for W in windows)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    dqs, dks, dvs = ([torch.full_like(x, float("nan")) for x in xs] for xs in (qs, ks, vs))
    # backward in model order: last layer first
    rev = lambda xs: xs[::-1]  # noqa: E731
    dualkv.dualkv_bwd_layers(rev(qs), rev(ks), rev(vs), rev(outs), rev(lses), rev(dos), rev(windows), P, w.N,
                             w.offsets, Hq, Hkv, D, w.scale, rev(dqs), rev(dks), rev(dvs), ws)
    dualkv.dualkv_check_status()
    for l in range(n):
        # each layer of the stack against the fp64 oracle of that layer (its own window)
        hq, hk, hv, hdo = host[l]
        ref = oracle.dualkv(P, w.N, w.offsets, Hq, Hkv, D, w.scale, windows[l], hq, hk, hv, hdo)
        got = dict(out=outs[l], lse=lses[l], dq=dqs[l], dk=dks[l], dv=dvs[l])
        o_error_log(f"{name} layer {l} (window {windows[l]})", check_full(got, ref))
        out, lse = dualkv.forward(qs[l], ks[l], vs[l], P, w.offsets, windows[l], w.scale)
        dq, dk, dv = dualkv.backward(qs[l], ks[l], vs[l], out, lse, dos[l], P, w.offsets, windows[l], w.scale)
        for key, a, b in (("out", outs[l], out), ("lse", lses[l], lse), ("dq", dqs[l], dq), ("dk", dks[l], dk),
                          ("dv", dvs[l], dv)):
            assert torch.equal(_bits(a), _bits(b)), (l, key)


def test_stack_checks_every_layer_before_launching():
    w = wl.custom(64, [32, 40], 2, 2, 64, 0, seed=5)
    windows = [0, 16]
    layers = _layers(w, windows)
    qs, ks, vs, dos = ([x[i] for x in layers] for i in range(4))
    outs = [torch.full_like(q, float("nan")) for q in qs]
    lses = [torch.full((w.Hq, w.T), float("nan"), device="cuda") for _ in windows]
    # the last layer's output is misaligned: nothing may run, not even layer 0
    bad = torch.empty(outs[1].numel() + 8, dtype=torch.bfloat16, device="cuda")[1:1 + outs[1].numel()]
    bad = bad.view(outs[1].shape)
    with pytest.raises(dualkv.DualKVError) as e:
        dualkv.dualkv_fwd_layers(qs, ks, vs, windows, w.P, w.N, w.offsets, w.Hq, w.Hkv, w.D, w.scale,
                                 [outs[0], bad], lses)
    assert e.value.code == dualkv.DUALKV_ERR_ALIGN
    torch.cuda.synchronize()
    assert torch.isnan(outs[0].float()).all() and torch.isnan(lses[0]).all()
    # a workspace smaller than the largest window needs is refused
    dualkv.dualkv_fwd_layers(qs, ks, vs, windows, w.P, w.N, w.offsets, w.Hq, w.Hkv, w.D, w.scale, outs, lses)
    nbytes = dualkv.dualkv_bwd_layers_workspace_bytes(windows, w.P, w.N, w.offsets, w.Hq, w.Hkv, w.D)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    grads = [[torch.empty_like(x) for x in xs] for xs in (qs, ks, vs)]
    with pytest.raises(dualkv.DualKVError) as e:
        dualkv.dualkv_bwd_layers(qs, ks, vs, outs, lses, dos, windows, w.P, w.N, w.offsets, w.Hq, w.Hkv, w.D,
                                 w.scale, *grads, ws, nbytes - 256)
    assert e.value.code == dualkv.DUALKV_ERR_WORKSPACE
    dualkv.dualkv_bwd_layers(qs, ks, vs, outs, lses, dos, windows, w.P, w.N, w.offsets, w.Hq, w.Hkv, w.D, w.scale,
                             *grads, ws)
    dualkv.dualkv_check_status()
