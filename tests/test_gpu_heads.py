"""GPU tests of the head-range entry points dualkv_fwd_heads / dualkv_bwd_heads.

A range call must write exactly the heads of its kv-head group (and their
q-heads), bit for bit what the full call writes there, must leave every other
head of every output untouched, and must not read the other heads of the
inputs: here those heads are NaN in the range calls' inputs.  Disjoint ranges
together then equal the full call, which the parity tests compare with the
oracle; one range is also compared with the oracle directly.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
from shared_prompt_exact_gb300 import build as pbuild
from shared_prompt_exact_gb300 import dualkv
from shared_prompt_exact_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pbuild.build()
    dualkv.load()


def _bits(t):
    return t.contiguous().view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32)


def _nan_outside(t, lo, hi, head_dim):
    """Copy of t with every head outside [lo, hi) along head_dim set to NaN."""
    x = t.clone()
    idx = [h for h in range(t.shape[head_dim]) if not lo <= h < hi]
    if idx:
        x.index_fill_(head_dim, torch.tensor(idx, device=t.device), float("nan"))
    return x


CASES = [
    # name, P, R, Hq, Hkv, D, window, kv-head ranges (disjoint, covering 0..Hkv)
    ("gqa2-d128", 300, [200, 0, 129, 1, 64], 8, 4, 128, 0, [(0, 1), (1, 3), (3, 4)]),
    ("window-d64", 129, [127, 129], 4, 2, 64, 64, [(1, 2), (0, 1)]),
    ("split-prompt-tiles", 128, [512] * 16, 4, 2, 64, 0, [(0, 1), (1, 2)]),
    ("d512", 300, [200, 129, 70], 4, 2, 512, 0, [(1, 2), (0, 1)]),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_head_ranges_equal_full_call(case):
    name, P, R, Hq, Hkv, D, W, ranges = case
    w = wl.custom(P, R, Hq, Hkv, D, W, seed=zlib.crc32(name.encode()) % 100000)
    gs = Hq // Hkv
    q, k, v, do = (x.cuda() for x in wl.draw_inputs(w))
    out, lse = dualkv.forward(q, k, v, w.P, w.offsets, w.window, w.scale)
    dq, dk, dv = dualkv.backward(q, k, v, out, lse, do, w.P, w.offsets, w.window, w.scale)
    ws = dualkv.workspace_for(w.P, w.offsets, Hq, Hkv, D, w.window)

    nan = lambda t: torch.full_like(t, float("nan"))  # noqa: E731
    r_out, r_lse, r_dq, r_dk, r_dv = nan(out), nan(lse), nan(dq), nan(dk), nan(dv)
    done_q, done_kv = set(), set()
    for lo, hi in ranges:
        qlo, qhi = lo * gs, hi * gs
        # inputs outside the group are NaN: the call must not read them
        q_r, do_r = _nan_outside(q, qlo, qhi, 1), _nan_outside(do, qlo, qhi, 1)
        k_r, v_r = _nan_outside(k, lo, hi, 1), _nan_outside(v, lo, hi, 1)
        o_r, l_r = _nan_outside(out, qlo, qhi, 1), _nan_outside(lse, qlo, qhi, 0)
        dualkv.dualkv_fwd_heads(q_r, k_r, v_r, w.P, w.N, w.offsets, Hq, Hkv, D, w.scale, w.window, lo, hi,
                                r_out, r_lse)
        dualkv.dualkv_bwd_heads(q_r, k_r, v_r, o_r, l_r, do_r, w.P, w.N, w.offsets, Hq, Hkv, D, w.scale, w.window,
                                lo, hi, r_dq, r_dk, r_dv, ws)
        dualkv.dualkv_check_status()
        done_q |= set(range(qlo, qhi))
        done_kv |= set(range(lo, hi))
        for h in range(Hq):
            if h in done_q:
                assert torch.equal(_bits(r_out[:, h]), _bits(out[:, h])), ("out", h)
                assert torch.equal(_bits(r_lse[h]), _bits(lse[h])), ("lse", h)
                assert torch.equal(_bits(r_dq[:, h]), _bits(dq[:, h])), ("dq", h)
            else:
                assert torch.isnan(r_out[:, h].float()).all() and torch.isnan(r_lse[h]).all(), ("touched", h)
                assert torch.isnan(r_dq[:, h].float()).all(), ("touched dq", h)
        for g in range(Hkv):
            if g in done_kv:
                assert torch.equal(_bits(r_dk[:, g]), _bits(dk[:, g])), ("dk", g)
                assert torch.equal(_bits(r_dv[:, g]), _bits(dv[:, g])), ("dv", g)
            else:
                assert torch.isnan(r_dk[:, g].float()).all() and torch.isnan(r_dv[:, g].float()).all(), ("dkv", g)


def test_head_range_against_oracle():
    """One kv-head group of a GQA layout against the oracle run on that group alone."""
    w = wl.custom(260, [90, 0, 200], 6, 3, 128, 0, seed=4242)
    lo, hi, gs = 1, 2, 2
    q, k, v, do = wl.draw_inputs(w)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    out = torch.zeros_like(qd)
    lse = torch.zeros(w.Hq, w.T, dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.zeros_like(qd), torch.zeros_like(kd), torch.zeros_like(vd)
    ws = dualkv.workspace_for(w.P, w.offsets, w.Hq, w.Hkv, w.D, w.window)
    dualkv.dualkv_fwd_heads(qd, kd, vd, w.P, w.N, w.offsets, w.Hq, w.Hkv, w.D, w.scale, w.window, lo, hi, out, lse)
    dualkv.dualkv_bwd_heads(qd, kd, vd, out, lse, dod, w.P, w.N, w.offsets, w.Hq, w.Hkv, w.D, w.scale, w.window,
                            lo, hi, dq, dk, dv, ws)
    dualkv.dualkv_check_status()
    qs = slice(lo * gs, hi * gs)
    ref = oracle.dualkv(w.P, w.N, w.offsets, gs, 1, w.D, w.scale, w.window, q[:, qs].contiguous(),
                        k[:, lo:hi].contiguous(), v[:, lo:hi].contiguous(), do[:, qs].contiguous())
    got_o = out[:, qs].double().cpu().numpy()
    excess = np.abs(got_o - ref["out"]) - np.ldexp(1.0, (np.floor(np.log2(np.maximum(np.abs(ref["out"]), 2.0 ** -126))) - 8).astype(np.int64))
    assert np.max(excess) <= 1e-2
    assert np.max(np.abs(lse[qs].double().cpu().numpy() - ref["lse"])) <= 1e-3
    for key, t in (("dq", dq[:, qs]), ("dk", dk[:, lo:hi]), ("dv", dv[:, lo:hi])):
        got = t.double().cpu().numpy()
        rel = np.linalg.norm(got - ref[key]) / np.linalg.norm(ref[key])
        assert rel <= 2e-2, (key, rel)
    # heads outside the group were not written
    assert float(out[:, : lo * gs].abs().max()) == 0.0 and float(dk[:, hi:].abs().max()) == 0.0


def test_head_range_rejects_bad_ranges():
    w = wl.custom(64, [32, 32], 4, 2, 64, 0, seed=1)
    q, k, v, _ = (x.cuda() for x in wl.draw_inputs(w))
    out = torch.empty_like(q)
    lse = torch.empty(w.Hq, w.T, dtype=torch.float32, device="cuda")
    for lo, hi in ((1, 1), (-1, 1), (0, 3), (2, 1)):
        with pytest.raises(dualkv.DualKVError) as e:
            dualkv.dualkv_fwd_heads(q, k, v, w.P, w.N, w.offsets, w.Hq, w.Hkv, w.D, w.scale, 0, lo, hi, out, lse)
        assert e.value.code == dualkv.DUALKV_ERR_INVALID
