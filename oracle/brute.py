"""Dense packed-mask brute force -- TEST INFRASTRUCTURE (see ``oracle/__init__``).

A second, independent fp64 formulation used to pin the C oracle on tiny
inputs.  Where the C oracle unpacks into N replicated sequences and folds,
this one works on the packed rows directly: it writes out the T x T mask that
DualKV implies (paper abstract: prompt queries attend causally within the
prompt; response queries of segment n attend to the prompt and causally to
their own segment), then runs dense softmax attention and the textbook
analytic softmax-attention backward with numpy matrix products.
"""
from __future__ import annotations

import numpy as np


def packed_mask(P, off, window=0):
    """Boolean [T, T] mask: mask[i, j] is True when packed query i attends packed key j."""
    N = len(off) - 1
    T = P + off[N]
    seg = np.full(T, -1)
    pos = np.arange(T)
    for n in range(N):
        a, b = P + off[n], P + off[n + 1]
        seg[a:b] = n
        pos[a:b] = P + np.arange(b - a)
    same_seq = (seg[None, :] == -1) | (seg[None, :] == seg[:, None])
    causal = pos[None, :] <= pos[:, None]
    mask = same_seq & causal
    if window > 0:
        mask &= (pos[:, None] - pos[None, :]) < window
    return mask


def dualkv_dense(P, off, Hq, Hkv, D, scale, window, q, k, v, dout=None):
    """Packed forward (out [T,Hq,D], lse [Hq,T]) and, with dout, gradients
    dq [T,Hq,D], dk, dv [T,Hkv,D]; all fp64."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    T = q.shape[0]
    mask = packed_mask(P, off, window)
    grp = Hq // Hkv
    out = np.zeros((T, Hq, D))
    lse = np.zeros((Hq, T))
    dq = np.zeros((T, Hq, D)) if dout is not None else None
    dk = np.zeros((T, Hkv, D)) if dout is not None else None
    dv = np.zeros((T, Hkv, D)) if dout is not None else None
    for h in range(Hq):
        g = h // grp
        Q, K, V = q[:, h, :], k[:, g, :], v[:, g, :]
        S = scale * (Q @ K.T)
        S = np.where(mask, S, -np.inf)
        m = S.max(axis=1, keepdims=True)
        E = np.exp(S - m)
        lsum = E.sum(axis=1, keepdims=True)
        A = E / lsum
        O = A @ V
        out[:, h, :] = O
        lse[h] = (m + np.log(lsum))[:, 0]
        if dout is not None:
            dO = np.asarray(dout, dtype=np.float64)[:, h, :]
            dV = A.T @ dO
            dA = dO @ V.T
            delta = np.sum(dO * O, axis=1, keepdims=True)
            dS = A * (dA - delta)
            dq[:, h, :] = scale * (dS @ K)
            dk[:, g, :] += scale * (dS.T @ Q)
            dv[:, g, :] += dV
    return dict(out=out, lse=lse, dq=dq, dk=dk, dv=dv)
