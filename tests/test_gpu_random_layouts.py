"""GPU parity on seeded random layouts: every output of the CUDA path against the
fp64 oracle, on layouts drawn at random (prompt length, number and lengths of the
responses including empty ones, GQA ratio, head dimension, window).  The drawn
cases cover combinations the hand-picked cases of test_gpu_parity.py do not: odd
group sizes, P = 0, windows shorter and longer than the prompt, single responses,
all-empty tails, and D = 512 with GQA.  Tolerances as in test_gpu_parity.py.
"""
import numpy as np
import pytest

import oracle
from shared_prompt_exact_gb300 import build as pbuild
from shared_prompt_exact_gb300 import dualkv
from shared_prompt_exact_gb300 import workloads as wl
from parity_checks import check_full

pytestmark = pytest.mark.gpu

N_CASES = 18


def draw_case(i):
    """Layout i of the sweep (fixed seed per index)."""
    rng = np.random.default_rng(20261203 + i)
    D = int(rng.choice([64, 128, 512], p=[0.4, 0.4, 0.2]))
    Hkv = int(rng.integers(1, 3))
    gs = int(rng.integers(1, 5))
    if D == 512:
        Hkv, gs = 1, int(rng.integers(1, 4))
    N = int(rng.integers(1, 7))
    cap = 160 if D == 512 else 300
    R = [int(x) if rng.random() > 0.15 else 0 for x in rng.integers(1, cap, size=N)]
    P = 0 if rng.random() < 0.1 else int(rng.integers(1, 2 * cap))
    if sum(R) + P == 0:
        R[0] = 1
    W = 0 if rng.random() < 0.5 else int(rng.integers(1, 2 * cap))
    return P, R, gs * Hkv, Hkv, D, W


CASES = [draw_case(i) for i in range(N_CASES)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pbuild.build()
    dualkv.load()


@pytest.mark.parametrize("idx", range(N_CASES), ids=[f"rand{i}-D{c[4]}-g{c[2] // c[3]}-W{c[5]}" for i, c in enumerate(CASES)])
def test_random_layout_matches_oracle(idx, o_error_log):
    P, R, Hq, Hkv, D, W = CASES[idx]
    w = wl.custom(P, R, Hq, Hkv, D, W, seed=1000 + idx)
    q, k, v, do = wl.draw_inputs(w)
    qd, kd, vd, dod = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    out, lse = dualkv.forward(qd, kd, vd, w.P, w.offsets, w.window, w.scale)
    dq, dk, dv = dualkv.backward(qd, kd, vd, out, lse, dod, w.P, w.offsets, w.window, w.scale)
    dualkv.dualkv_check_status()
    g = dict(out=out, lse=lse, dq=dq, dk=dk, dv=dv)
    ref = oracle.dualkv(w.P, w.N, w.offsets, w.Hq, w.Hkv, w.D, w.scale, w.window, q, k, v, do)
    assert ref["prompt_invariant"] == 1
    o_error_log(f"rand{idx} P={P} R={R} {Hq}/{Hkv} D={D} W={W}", check_full(g, ref))
