"""Pins of the fp64 oracle against things other than itself.

DualKV paper, abstract: the packed computation gives exactly what ordinary
attention gives on the replicated sequences.  The oracle writes that definition out (replicated causal
attention + analytic backward + fold).  These tests tie it to:
  * an independent dense packed-mask formulation (oracle.brute);
  * torch float64 autograd through the library's scaled_dot_product_attention
    on the replicated sequences;
  * central finite differences of L = sum(O * dO);
  * invariants (replica invariance of prompt rows, dO-split linearity,
    key-shift invariance which holds only when every row of dS sums to zero);
  * closed forms (equal keys -> uniform weights; constant values).
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import brute
from oracle import index as oindex


def rand_case(seed, P, R, Hq, Hkv, D, window=0, scale=None):
    rng = np.random.default_rng(seed)
    off = [0]
    for r in R:
        off.append(off[-1] + r)
    T = P + off[-1]
    # bf16-representable values so the widened inputs are exact on both sides
    q = torch.tensor(rng.standard_normal((T, Hq, D))).to(torch.bfloat16).double().numpy()
    k = torch.tensor(rng.standard_normal((T, Hkv, D))).to(torch.bfloat16).double().numpy()
    v = torch.tensor(rng.standard_normal((T, Hkv, D))).to(torch.bfloat16).double().numpy()
    do = torch.tensor(rng.standard_normal((T, Hq, D))).to(torch.bfloat16).double().numpy()
    sc = scale if scale is not None else 1.0 / math.sqrt(D)
    return dict(P=P, N=len(R), off=off, Hq=Hq, Hkv=Hkv, D=D, scale=sc, window=window, q=q, k=k, v=v, do=do)


def run_oracle(c, **kw):
    return oracle.dualkv(c["P"], c["N"], c["off"], c["Hq"], c["Hkv"], c["D"], c["scale"], c["window"],
                         c["q"], c["k"], c["v"], c["do"], **kw)


def rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


CASES = [
    # (seed, P, R list, Hq, Hkv, D, window)
    (1, 5, [3, 4], 2, 2, 4, 0),
    (2, 7, [0, 5, 1], 4, 2, 8, 0),          # empty segment, GQA 2:1
    (3, 0, [6, 3, 4], 2, 1, 8, 0),          # no prompt
    (4, 9, [4], 3, 3, 5, 0),                # N = 1
    (5, 11, [6, 2, 7], 4, 1, 6, 4),         # window crossing the prompt/response boundary
    (6, 6, [5, 5], 2, 2, 3, 1),             # window 1: self only
    (7, 1, [1, 0, 2], 2, 2, 4, 0),          # P = 1
    (8, 10, [4, 6], 2, 1, 8, 100),          # window wider than any sequence
]


@pytest.mark.parametrize("case", CASES)
def test_oracle_matches_dense_packed_bruteforce(case):
    seed, P, R, Hq, Hkv, D, W = case
    c = rand_case(seed, P, R, Hq, Hkv, D, W)
    o = run_oracle(c)
    b = brute.dualkv_dense(P, c["off"], Hq, Hkv, D, c["scale"], W, c["q"], c["k"], c["v"], c["do"])
    assert o["prompt_invariant"] == 1
    for key in ("out", "lse", "dq", "dk", "dv"):
        err = np.max(np.abs(o[key] - b[key])) / max(np.max(np.abs(b[key])), 1e-30)
        assert err <= 1e-12, (key, err)


def test_brute_mask_structure():
    # prompt row 2 sees prompt keys 0..2; response row r of segment n sees all
    # prompt keys and own-segment keys up to itself, never another segment's.
    P, off = 3, [0, 2, 4]
    m = brute.packed_mask(P, off)
    assert m[2].tolist() == [True, True, True, False, False, False, False]
    assert m[3].tolist() == [True, True, True, True, False, False, False]
    assert m[6].tolist() == [True, True, True, False, False, True, True]
    mw = brute.packed_mask(P, off, window=2)
    assert mw[6].tolist() == [False, False, False, False, False, True, True]
    assert mw[5].tolist() == [False, False, True, False, False, True, False]


def torch_replicated_reference(c, dout_mode=0):
    """torch float64 SDPA + autograd on the replicated sequences, folded by index_add."""
    P, N, off, Hq, Hkv, D, W = c["P"], c["N"], c["off"], c["Hq"], c["Hkv"], c["D"], c["window"]
    T = P + off[-1]
    q = torch.tensor(c["q"], requires_grad=True)
    k = torch.tensor(c["k"], requires_grad=True)
    v = torch.tensor(c["v"], requires_grad=True)
    do = torch.tensor(c["do"])
    grp = Hq // Hkv
    loss = 0.0
    out = torch.zeros(T, Hq, D, dtype=torch.float64)
    for n in range(N):
        rows = list(range(P)) + list(range(P + off[n], P + off[n + 1]))
        L = len(rows)
        idx = torch.tensor(rows)
        qn = q[idx].transpose(0, 1)  # [Hq, L, D]
        kn = k[idx].transpose(0, 1).repeat_interleave(grp, dim=0)
        vn = v[idx].transpose(0, 1).repeat_interleave(grp, dim=0)
        pos = torch.arange(L)
        mask = pos[None, :] <= pos[:, None]
        if W > 0:
            mask &= (pos[:, None] - pos[None, :]) < W
        on = F.scaled_dot_product_attention(qn, kn, vn, attn_mask=mask, scale=c["scale"])
        on = on.transpose(0, 1)  # [L, Hq, D]
        dn = do[idx].clone()
        if dout_mode == 0:
            if n > 0:
                dn[:P] = 0.0
        else:
            dn[:P] = dn[:P] / N
        loss = loss + (on * dn).sum()
        if n == 0:
            out[:P] = on[:P].detach()
        out[P + off[n]: P + off[n + 1]] = on[P:].detach()
    loss.backward()
    return dict(out=out.numpy(), dq=q.grad.numpy(), dk=k.grad.numpy(), dv=v.grad.numpy())


@pytest.mark.parametrize("case", CASES[:6])
def test_oracle_matches_torch_float64_autograd(case):
    seed, P, R, Hq, Hkv, D, W = case
    c = rand_case(seed + 100, P, R, Hq, Hkv, D, W)
    o = run_oracle(c)
    t = torch_replicated_reference(c)
    for key in ("out", "dq", "dk", "dv"):
        assert rel(o[key], t[key]) <= 1e-12, key


def test_finite_differences_of_loss():
    # L = sum(O * dO) over packed outputs; dL/dx must match the oracle's
    # gradients, including prompt k/v rows (which carry the fold over replicas).
    c = rand_case(11, 5, [3, 0, 4], 4, 2, 4, 0)
    o = run_oracle(c)
    rng = np.random.default_rng(0)
    eps = 1e-6

    def loss(cc):
        r = oracle.dualkv(cc["P"], cc["N"], cc["off"], cc["Hq"], cc["Hkv"], cc["D"], cc["scale"],
                          cc["window"], cc["q"], cc["k"], cc["v"], None, forward_only=True)
        return float(np.sum(r["out"] * cc["do"]))

    checked = 0
    for name, grad in (("q", o["dq"]), ("k", o["dk"]), ("v", o["dv"])):
        shp = c[name].shape
        coords = [tuple(rng.integers(0, s) for s in shp) for _ in range(25)]
        # always include prompt rows for k and v
        if name in ("k", "v"):
            coords += [(0, 0, 1), (2, 1, 3), (4, 1, 0)]
        for co in coords:
            cp = dict(c); cm = dict(c)
            cp[name] = c[name].copy(); cm[name] = c[name].copy()
            cp[name][co] += eps
            cm[name][co] -= eps
            fd = (loss(cp) - loss(cm)) / (2 * eps)
            assert abs(fd - grad[co]) <= 1e-6 * max(1.0, abs(grad[co])), (name, co, fd, grad[co])
            checked += 1
    assert checked >= 80


def test_invariant_dout_split_linearity():
    c = rand_case(12, 8, [5, 3, 6], 4, 2, 8, 0)
    a = run_oracle(c, dout_mode=0)
    b = run_oracle(c, dout_mode=1)
    for key in ("dq", "dk", "dv"):
        assert rel(a[key], b[key]) <= 1e-12, key
    t = torch_replicated_reference(c, dout_mode=1)
    for key in ("dq", "dk", "dv"):
        assert rel(b[key], t[key]) <= 1e-12, key


def test_invariant_prompt_rows_identical_across_replicas():
    c = rand_case(13, 12, [4, 7, 1, 0], 2, 2, 8, 5)
    o = run_oracle(c)
    assert o["prompt_invariant"] == 1
    # prompt outputs do not depend on any response row
    c2 = dict(c)
    for name in ("q", "k", "v"):
        c2[name] = c[name].copy()
        c2[name][c["P"]:] = 7.0
    o2 = run_oracle(c2)
    assert np.array_equal(o["out"][: c["P"]], o2["out"][: c["P"]])
    assert np.array_equal(o["lse"][:, : c["P"]], o2["lse"][:, : c["P"]])


def test_invariant_key_shift():
    # Adding one vector c to every key shifts S_ij by scale*q_i.c for all j:
    # softmax weights, O and dV unchanged, LSE shifts by scale*q_i.c, and dQ is
    # unchanged only because each row of dS sums to zero.
    c = rand_case(14, 6, [4, 5], 2, 2, 4, 0)
    o = run_oracle(c)
    shift = np.array([0.5, -1.0, 0.25, 2.0])
    c2 = dict(c)
    c2["k"] = c["k"] + shift[None, None, :]
    o2 = run_oracle(c2)
    assert rel(o2["out"], o["out"]) <= 1e-12
    assert rel(o2["dv"], o["dv"]) <= 1e-12
    assert rel(o2["dq"], o["dq"]) <= 1e-11
    qs = np.einsum("thd,d->ht", c["q"], shift) * c["scale"]
    assert np.max(np.abs(o2["lse"] - o["lse"] - qs)) <= 1e-12


def test_closed_form_equal_keys():
    # all keys equal: uniform weights over the allowed set A_i;
    # O_i = mean of allowed v, LSE_i = ln|A_i| + scale q_i.k
    c = rand_case(15, 6, [3, 4], 2, 1, 4, 3)
    c["k"][:] = c["k"][0:1]
    o = run_oracle(c)
    mask = brute.packed_mask(c["P"], c["off"], c["window"])
    for h in range(2):
        for i in range(mask.shape[0]):
            allowed = np.nonzero(mask[i])[0]
            np.testing.assert_allclose(o["out"][i, h], c["v"][allowed, 0].mean(axis=0), rtol=0, atol=1e-13)
            want = math.log(len(allowed)) + c["scale"] * float(c["q"][i, h] @ c["k"][0, 0])
            assert abs(o["lse"][h, i] - want) <= 1e-12


def test_closed_form_constant_values():
    # v_j = const: O = const, dQ = dK = 0, dV_j = sum_i P_ij dO_i
    c = rand_case(16, 5, [4, 2], 2, 2, 4, 0)
    c["v"][:] = np.array([1.0, -2.0, 0.5, 3.0])
    o = run_oracle(c)
    assert np.max(np.abs(o["out"] - np.array([1.0, -2.0, 0.5, 3.0]))) <= 1e-13
    assert np.max(np.abs(o["dq"])) <= 1e-13
    assert np.max(np.abs(o["dk"])) <= 1e-13
    b = brute.dualkv_dense(c["P"], c["off"], 2, 2, 4, c["scale"], 0, c["q"], c["k"], c["v"], c["do"])
    assert rel(o["dv"], b["dv"]) <= 1e-12


def test_special_case_gqa_equals_repeated_heads():
    c = rand_case(17, 6, [3, 5], 4, 2, 4, 0)
    g = run_oracle(c)
    m = dict(c)
    m["k"] = np.repeat(c["k"], 2, axis=1)
    m["v"] = np.repeat(c["v"], 2, axis=1)
    m["Hkv"] = 4
    r = run_oracle(m)
    assert rel(g["out"], r["out"]) <= 1e-14
    assert rel(g["dq"], r["dq"]) <= 1e-14
    assert rel(g["dk"], r["dk"].reshape(-1, 2, 2, 4).sum(axis=2)) <= 1e-13
    assert rel(g["dv"], r["dv"].reshape(-1, 2, 2, 4).sum(axis=2)) <= 1e-13


def test_special_case_no_prompt_is_independent_sequences():
    c = rand_case(18, 0, [4, 6], 2, 2, 4, 0)
    o = run_oracle(c)
    for n, (a, b) in enumerate([(0, 4), (4, 10)]):
        sub = dict(c)
        sub["off"] = [0, b - a]
        sub["N"] = 1
        for name in ("q", "k", "v", "do"):
            sub[name] = c[name][a:b]
        s = run_oracle(sub)
        for key in ("out", "dq", "dk", "dv"):
            assert np.array_equal(o[key][a:b], s[key]), key


def test_special_case_wide_window_equals_global():
    c = rand_case(19, 7, [5, 3], 2, 2, 4, 0)
    g = run_oracle(c)
    c["window"] = 12
    w = run_oracle(c)
    for key in ("out", "lse", "dq", "dk", "dv"):
        assert np.array_equal(g[key], w[key]), key


def test_sampled_rows_match_full_oracle():
    c = rand_case(20, 9, [5, 0, 7, 3], 4, 2, 8, 6)
    o = run_oracle(c)
    rows = [0, 3, 8, 9, 13, 16, 20, 23]
    for h in (0, 3):
        orow, lrow, dqrow = oracle.query_rows(c["P"], c["N"], c["off"], 4, 2, 8, c["scale"], 6, h, rows,
                                              c["q"], c["k"], c["v"], c["do"])
        assert np.max(np.abs(orow - o["out"][rows, h])) <= 1e-13
        assert np.max(np.abs(lrow - o["lse"][h, rows])) <= 1e-13
        assert np.max(np.abs(dqrow - o["dq"][rows, h])) <= 1e-12
    keys = [0, 4, 8, 9, 15, 23]
    for g in (0, 1):
        dk, dv = oracle.key_rows(c["P"], c["N"], c["off"], 4, 2, 8, c["scale"], 6, g, keys,
                                 c["q"], c["k"], c["v"], c["do"])
        assert np.max(np.abs(dk - o["dk"][keys, g])) <= 1e-12
        assert np.max(np.abs(dv - o["dv"][keys, g])) <= 1e-12


def test_sampled_prompt_keys_match_full_oracle_under_both_dout_splits():
    # key_rows skips the prompt rows of replicas >= 1 when only replica 0 carries the
    # prompt's upstream gradient; both splits must give the full oracle's folded dK/dV
    c = rand_case(21, 10, [6, 3, 0, 8], 4, 1, 8, 0)
    keys = [0, 1, 5, 9, 10, 17, 26]
    for mode in (0, 1):
        o = run_oracle(c, dout_mode=mode)
        dk, dv = oracle.key_rows(c["P"], c["N"], c["off"], 4, 1, 8, c["scale"], 0, 0, keys,
                                 c["q"], c["k"], c["v"], c["do"], dout_mode=mode)
        assert np.max(np.abs(dk - o["dk"][keys, 0])) <= 1e-12
        assert np.max(np.abs(dv - o["dv"][keys, 0])) <= 1e-12


def test_index_oracle_small_layout():
    seg, pos, cu, r2p = oindex.build_index(3, [0, 2, 2, 3])
    assert seg == [-1, -1, -1, 0, 0, 2]
    assert pos == [0, 1, 2, 3, 4, 3]
    assert cu == [0, 5, 8, 12]
    assert r2p == [0, 1, 2, 3, 4, 0, 1, 2, 0, 1, 2, 5]


def test_pairs_closed_form():
    # causal pair count: P(P+1)/2 + sum_n [R_n P + R_n(R_n+1)/2]
    for P, R in ((5, [3, 0, 4]), (0, [2, 2]), (7, [1])):
        off = [0]
        for r in R:
            off.append(off[-1] + r)
        want = P * (P + 1) // 2 + sum(r * P + r * (r + 1) // 2 for r in R)
        assert oindex.pairs(P, off) == want
        assert oindex.pairs(P, off) == int(brute.packed_mask(P, off).sum())
    off = [0, 4, 9]
    assert oindex.pairs(6, off, window=3) == int(brute.packed_mask(6, off, 3).sum())


def test_pairs_replicated_counts_the_replicated_mask():
    # the replicated layout is N independent sequences of P + R_n tokens, i.e. a
    # packed layout with no prompt whose segments are those sequences; its pair
    # count is that mask's population and, for global causal attention, the sum of
    # the sequences' triangles L_n (L_n + 1) / 2
    for P, R, W in ((5, [3, 0, 4], 0), (0, [2, 2], 0), (7, [1], 0), (6, [4, 5], 3), (4, [0, 6, 2], 1),
                    (9, [3, 3], 100)):
        off = [0]
        for r in R:
            off.append(off[-1] + r)
        rep_off = [0]
        for r in R:
            rep_off.append(rep_off[-1] + P + r)
        got = oindex.pairs_replicated(P, off, W)
        assert got == int(brute.packed_mask(0, rep_off, W).sum())
        if W <= 0:
            assert got == sum((P + r) * (P + r + 1) // 2 for r in R)
        # replicating never removes a pair: every packed pair appears at least once
        assert got >= oindex.pairs(P, off, W)
        if len(R) == 1:
            assert got == oindex.pairs(P, off, W)
