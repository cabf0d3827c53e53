"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances (GPU output widened to fp64, compared over the compared slice):
  O     max-abs <= 1e-2 beyond the output's own bf16 rounding (half an ulp of the
        exact value; above |O| = 4 that half ulp alone exceeds 1e-2), and
        normwise relative <= 5e-3
  LSE   max-abs <= 1e-3
  dQ/dK/dV  normwise relative <= 2e-2 each
Small and medium layouts are compared on every row and head.  The full-size
workloads are compared on sampled rows / keys of two GQA groups (the oracle
computes each sampled output by the definition), on conservation properties
that hold at any size, and against the same kernels run on the replicated
layout (P = 0, one sequence per response) folded on the host.
"""
import math
import zlib

import numpy as np
import pytest
import torch

import oracle
from shared_prompt_exact_gb300 import build as pbuild
from shared_prompt_exact_gb300 import dualkv
from shared_prompt_exact_gb300 import workloads as wl
from parity_checks import G_REL, LSE_ABS, O_ABS, O_REL, assert_o_close, check_full, relF

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pbuild.build()
    dualkv.load()


def run_gpu(w, q, k, v, do, backward=True):
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out, lse = dualkv.forward(qd, kd, vd, w.P, w.offsets, w.window, w.scale)
    res = dict(out=out, lse=lse)
    if backward:
        dod = do.cuda()
        dq, dk, dv = dualkv.backward(qd, kd, vd, out, lse, dod, w.P, w.offsets, w.window, w.scale)
        res.update(dq=dq, dk=dk, dv=dv)
    dualkv.dualkv_check_status()
    return res


SMALL = [
    # name, P, R, Hq, Hkv, D, window
    ("tiny-config", 64, [32] * 4, 2, 2, 64, 0),
    ("ragged-gqa", 300, [200, 0, 129, 1, 64], 4, 2, 128, 0),
    ("aligned", 128, [128, 128], 2, 2, 128, 0),
    ("no-prompt", 0, [257, 3], 2, 1, 64, 0),
    ("one-seg-p1", 1, [130], 2, 2, 128, 0),
    ("window-boundary", 129, [127, 129], 4, 1, 128, 64),
    ("empty-segments", 127, [0, 5, 0], 2, 2, 128, 0),
    ("gqa4-window", 400, [33] * 6, 8, 2, 128, 150),
    ("split-prompt-tiles", 128, [512] * 16, 4, 1, 64, 0),
    ("long-prompt-d128", 1000, [100, 300, 7], 2, 1, 128, 0),
    ("d512-ragged-gqa", 300, [200, 0, 129, 70], 4, 2, 512, 0),
    ("d512-window", 300, [200, 129, 70], 2, 1, 512, 100),
    # D = 512 global with more than 512 (q-head, 64-row) entries per prompt key tile
    # (38 query tiles x 8 heads x 2 halves), so the dK/dV GEMMs split the prompt
    # tiles and the fixed-order reduction runs
    ("d512-split-prompt-tiles", 200, [100] * 36, 8, 1, 512, 0),
    # an odd group size: the P / dS pass cannot pair q-heads and runs one CTA per tile
    ("d512-group3-window", 260, [150, 0, 90], 3, 1, 512, 64),
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_parity_small(case, o_error_log):
    name, P, R, Hq, Hkv, D, W = case
    w = wl.WORKLOADS["tiny"] if name == "tiny-config" else wl.custom(P, R, Hq, Hkv, D, W, seed=zlib.crc32(name.encode()) % 100000)
    q, k, v, do = wl.draw_inputs(w)
    g = run_gpu(w, q, k, v, do)
    ref = oracle.dualkv(w.P, w.N, w.offsets, w.Hq, w.Hkv, w.D, w.scale, w.window, q, k, v, do)
    assert ref["prompt_invariant"] == 1
    o_error_log(name, check_full(g, ref))


def test_window_one_attends_only_itself():
    # W = 1: P_ii = 1, so O = v exactly, LSE = scale q.k, dV = sum of the group's dO,
    # and dS = 0 makes dQ and dK vanish (only rounding of Delta remains)
    w = wl.custom(200, [70, 300], 4, 2, 64, 1, seed=11)
    q, k, v, do = wl.draw_inputs(w)
    g = run_gpu(w, q, k, v, do)
    gs = w.Hq // w.Hkv
    out = g["out"].cpu()
    for h in range(w.Hq):
        assert torch.equal(out[:, h], v[:, h // gs])
    lse_ref = (q.double() * k.double().repeat_interleave(gs, dim=1)).sum(-1).T * w.scale
    assert float((g["lse"].cpu().double() - lse_ref).abs().max()) <= LSE_ABS
    dv_ref = do.double().reshape(w.T, w.Hkv, gs, w.D).sum(2)
    assert relF(g["dv"].double().cpu().numpy(), dv_ref.numpy()) <= G_REL
    scale_ref = float(dv_ref.norm())
    assert float(g["dq"].double().norm()) <= G_REL * scale_ref
    assert float(g["dk"].double().norm()) <= G_REL * scale_ref


def test_determinism_bitwise():
    w = wl.custom(128, [512] * 16, 4, 1, 64, 0, seed=7)  # includes split prompt key tiles
    q, k, v, do = wl.draw_inputs(w)
    a = run_gpu(w, q, k, v, do)
    b = run_gpu(w, q, k, v, do)
    for key in ("out", "lse", "dq", "dk", "dv"):
        assert torch.equal(a[key], b[key]), key


def test_outputs_fully_overwritten():
    w = wl.custom(70, [40, 90], 2, 2, 128, 0, seed=3)
    q, k, v, do = wl.draw_inputs(w)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    outs = []
    for fill in (0.0, float("nan")):
        out = torch.full_like(qd, fill)
        lse = torch.full((w.Hq, w.T), fill, device="cuda")
        dualkv.dualkv_fwd(qd, kd, vd, w.P, w.N, w.offsets, w.Hq, w.Hkv, w.D, w.scale, 0, out, lse)
        dq, dk, dv = (torch.full_like(x, fill) for x in (qd, kd, vd))
        ws = dualkv.workspace_for(w.P, w.offsets, w.Hq, w.Hkv, w.D)
        ws.fill_(255)
        dualkv.dualkv_bwd(qd, kd, vd, out, lse, dod, w.P, w.N, w.offsets, w.Hq, w.Hkv, w.D, w.scale, 0, dq, dk, dv, ws)
        dualkv.dualkv_check_status()
        outs.append((out, lse, dq, dk, dv))
    for a, b in zip(*outs):
        assert torch.equal(a, b)


# ------------------------------------------------------------------ full size
FULL_D128 = ["qwen16", "grpo32", "dapo32"]


def sample_rows(w, rng, n_random=24):
    """(uniform random rows, boundary rows).  The uniform sample estimates the
    normwise error of the whole tensor; boundary rows (first prompt rows, segment
    starts / middles / ends) are edge cases checked on the tensor's scale."""
    off = w.offsets
    edge = {0, 1, w.P // 2, w.P - 1} if w.P > 0 else set()
    for n in (0, w.N // 2, w.N - 1):
        a, b = w.P + off[n], w.P + off[n + 1]
        if b > a:
            edge |= {a, (a + b) // 2, b - 1}
    uni = sorted(set(int(x) for x in rng.integers(0, w.T, n_random)))
    return uni, sorted(r for r in edge if 0 <= r < w.T)


def sample_response_keys(w, rng, n_random=6, late_only=False):
    """Response keys: segment starts / middles / ends and random ones, or (late_only)
    only keys near segment ends, which few queries attend (keeps the oracle cheap)."""
    off = w.offsets
    keys = set()
    for n in (0, w.N // 2, w.N - 1):
        a, b = w.P + off[n], w.P + off[n + 1]
        if b > a:
            keys |= {b - 1, max(a, b - 2), max(a, b - 65)} if late_only else {a, b - 1, (a + b) // 2}
    if not late_only:
        keys |= set(int(x) for x in rng.integers(w.P, w.T, n_random))
    return sorted(keys)


def attended_keys(w, row):
    off = w.offsets
    if row < w.P:
        pos = row
    else:
        n = max(i for i in range(w.N) if w.P + off[i] <= row and off[i + 1] > off[i])
        pos = w.P + row - (w.P + off[n])
    return pos + 1 if w.window <= 0 else min(pos + 1, w.window)


def groups_to_check(w, rng):
    return sorted({int(rng.integers(0, w.Hkv)), w.Hkv - 1})


def prompt_keys_of(w):
    """Prompt keys checked element by element at full size: the last keys of the
    prompt (attended by every segment's queries and a few prompt rows) and one
    mid-prompt key (also attended by half of the prompt's queries).  Each carries the
    fold over all N segments."""
    if w.P <= 0:
        return set()
    return {k for k in (w.P - 1, w.P - 2, w.P - 64, w.P - 129, w.P // 2 + 7) if 0 <= k < w.P}


def check_sampled(w, q, k, v, do, g, prompt_keys=False, late_keys_only=False, o_log=None):
    """Sampled query rows of two GQA groups and sampled keys against the oracle.  With
    prompt_keys, the last group's keys include prompt_keys_of(w) (one group only: each
    prompt key needs every response row of every segment from the oracle)."""
    rng = np.random.default_rng(w.seed)
    out = g["out"].cpu()
    lse = g["lse"].cpu()
    dq = g["dq"].cpu()
    dk = g["dk"].cpu()
    dv = g["dv"].cpu()
    gs = w.Hq // w.Hkv
    uni, edge = sample_rows(w, rng)
    rows = uni + edge
    nu = len(uni)
    raw_o = 0.0
    for grp in groups_to_check(w, rng):
        for h in range(grp * gs, grp * gs + gs):
            o_r, l_r, dq_r = oracle.query_rows(w.P, w.N, w.offsets, w.Hq, w.Hkv, w.D, w.scale, w.window, h, rows,
                                               q, k, v, do)
            raw_o = max(raw_o, assert_o_close(out[rows, h].double().numpy(), o_r))
            assert np.max(np.abs(lse[h, rows].double().numpy() - l_r)) <= LSE_ABS
            dq_g = dq[rows, h].double().numpy()
            assert relF(dq_g[:nu], dq_r[:nu]) <= G_REL
            rms_row = np.linalg.norm(dq_r[:nu]) / math.sqrt(nu)
            for i in range(nu, len(rows)):
                # a row attending only a handful of keys (the first prompt rows) carries the
                # inherent error of Delta computed on the bf16 output, |dDelta| ~ 2^-9 |dO o O|,
                # which is of the order of its own tiny-key dQ; such rows are compared in the
                # small full-oracle cases instead
                if attended_keys(w, rows[i]) < 64:
                    continue
                assert np.linalg.norm(dq_g[i] - dq_r[i]) <= G_REL * max(rms_row, np.linalg.norm(dq_r[i])), rows[i]
        keys = set(sample_response_keys(w, rng, late_only=late_keys_only))
        pkeys = sorted(prompt_keys_of(w)) if (prompt_keys and grp == w.Hkv - 1) else []
        keys = sorted(keys | set(pkeys))
        dk_r, dv_r = oracle.key_rows(w.P, w.N, w.offsets, w.Hq, w.Hkv, w.D, w.scale, w.window, grp, keys,
                                     q, k, v, do)
        assert relF(dk[keys, grp].double().numpy(), dk_r) <= G_REL
        assert relF(dv[keys, grp].double().numpy(), dv_r) <= G_REL
        if pkeys:
            # the prompt keys on their own as well: their fold over all N segments is the
            # part of dK/dV that packing changes
            sel = [keys.index(kk) for kk in pkeys]
            assert relF(dk[pkeys, grp].double().numpy(), dk_r[sel]) <= G_REL
            assert relF(dv[pkeys, grp].double().numpy(), dv_r[sel]) <= G_REL
    if o_log is not None:
        o_log(w.name + " (sampled rows)", raw_o)


def check_conservation(w, do, g):
    # sum_j dV_j = sum over the group's heads and all packed rows of dO_i  (rows of P sum to 1)
    # sum_j dK_j = 0                                                          (rows of dS sum to 0)
    gs = w.Hq // w.Hkv
    dv = g["dv"].double()
    dk = g["dk"].double()
    dod = do.cuda().double()
    for grp in range(w.Hkv):
        want = dod[:, grp * gs:(grp + 1) * gs].sum(dim=(0, 1))
        got = dv[:, grp].sum(dim=0)
        assert float((got - want).norm() / want.norm()) <= G_REL
        s = dk[:, grp].sum(dim=0)
        assert float(s.norm()) <= 1e-2 * float(dk[:, grp].norm()) * math.sqrt(w.D)


def fold_replicated(w, x_rep):
    """Sum replicated prompt rows over replicas; response rows map 1:1 (x_rep on GPU)."""
    off = w.offsets
    out = torch.zeros((w.T,) + tuple(x_rep.shape[1:]), dtype=torch.float32, device=x_rep.device)
    pos = 0
    for n in range(w.N):
        Rn = off[n + 1] - off[n]
        out[: w.P] += x_rep[pos: pos + w.P].float()
        out[w.P + off[n]: w.P + off[n + 1]] = x_rep[pos + w.P: pos + w.P + Rn].float()
        pos += w.P + Rn
    return out


def check_packed_vs_replicated(w, q, k, v, do, g):
    wr = w.replicated()
    qr, kr, vr = (wl.replicate_rows(w, x.cuda()) for x in (q, k, v))
    dor = wl.replicate_rows(w, do.cuda()).clone()
    pos = 0
    off = w.offsets
    for n in range(w.N):  # prompt upstream gradient carried by replica 0 only
        if n > 0:
            dor[pos: pos + w.P] = 0
        pos += w.P + off[n + 1] - off[n]
    out_r, lse_r = dualkv.forward(qr, kr, vr, wr.P, wr.offsets, wr.window, wr.scale)
    dq_r, dk_r, dv_r = dualkv.backward(qr, kr, vr, out_r, lse_r, dor, wr.P, wr.offsets, wr.window, wr.scale)
    dualkv.dualkv_check_status()
    # forward: every replica's rows equal the packed rows
    out_p = wl.replicate_rows(w, g["out"]).float()
    assert float((out_r.float() - out_p).norm() / out_p.norm()) <= O_REL
    assert float((out_r.float() - out_p).abs().max()) <= O_ABS
    for name, rep in (("dq", dq_r), ("dk", dk_r), ("dv", dv_r)):
        folded = fold_replicated(w, rep)
        got = g[name].float()
        assert float((got - folded).norm() / folded.norm()) <= G_REL, name


@pytest.mark.parametrize("name", FULL_D128)
def test_parity_full_size_sampled(name, o_error_log):
    w = wl.WORKLOADS[name]
    q, k, v, do = wl.draw_inputs(w)
    g = run_gpu(w, q, k, v, do)
    check_sampled(w, q, k, v, do, g, prompt_keys=True, o_log=o_error_log)
    check_conservation(w, do, g)
    check_packed_vs_replicated(w, q, k, v, do, g)


# Head dimension 512 (Gemma-style slice, global and sliding window 1024).  The
# global configuration's replicated run would need ~100 GB of P/dS blocks, so
# packed-vs-replicated is checked on the window configuration only; its
# prompt keys are cheap for the oracle there (few queries fall in the window).
@pytest.mark.parametrize("name", ["gemma_global", "gemma_window"])
def test_parity_full_size_d512(name, o_error_log):
    w = wl.WORKLOADS[name]
    q, k, v, do = wl.draw_inputs(w)
    g = run_gpu(w, q, k, v, do)
    windowed = w.window > 0
    check_sampled(w, q, k, v, do, g, prompt_keys=windowed, late_keys_only=not windowed, o_log=o_error_log)
    check_conservation(w, do, g)
    if windowed:
        check_packed_vs_replicated(w, q, k, v, do, g)
