"""Tensor packing oracle -- TEST INFRASTRUCTURE (see ``oracle/__init__``).

Plain numpy definitions of the three tensor-level moves between the
replicated and the packed micro-batch layout.  They carry the token reduction
of shared-prompt packing past attention: per-token layers then run on P+NR
rows instead of N(P+R) (DualKV paper, abstract: once the data pipeline stores
the prompt once, every per-token layer of the model, not only attention,
works on the smaller row count).

All three are written through ``rep2pack`` of ``oracle.index`` (the packed row
of every replicated row):

* ``pack``   packed row t takes the first replicated row that maps to it,
  i.e. replica 0 for a prompt row;
* ``unpack`` replicated row x takes packed row rep2pack[x];
* ``fold``   packed row t is the fp64 sum of every replicated row that maps
  to it, visited in replicated order -- the transpose of ``unpack`` and hence
  the gradient of the packed rows given the gradient of the replicated ones.

Pinned by ``tests/test_pack_oracle.py``: a hand-derived worked layout,
the adjoint identity <unpack x, g> = <x, fold g> in exact arithmetic, the
round trips, the N = 1 and P = 0 reductions, and the fold of ones (prompt
rows count N, response rows 1).
"""
from __future__ import annotations

import numpy as np

from .index import build_index


def _rep2pack(P, off):
    return np.asarray(build_index(P, list(off))[3], dtype=np.int64)


def packed_rows(P, off):
    return P + off[-1]


def replicated_rows(P, off):
    return (len(off) - 1) * P + off[-1]


def pack(x_rep, P, off):
    """x_rep [T_rep, ...] -> [T, ...]; each packed row from its first replicated row."""
    r2p = _rep2pack(P, off)
    x_rep = np.asarray(x_rep)
    assert x_rep.shape[0] == len(r2p)
    out = np.zeros((packed_rows(P, off),) + x_rep.shape[1:], dtype=x_rep.dtype)
    seen = np.zeros(packed_rows(P, off), dtype=bool)
    for x, t in enumerate(r2p):
        if not seen[t]:
            out[t] = x_rep[x]
            seen[t] = True
    assert seen.all()
    return out


def unpack(x_packed, P, off):
    """x_packed [T, ...] -> [T_rep, ...]; replicated row x is packed row rep2pack[x]."""
    r2p = _rep2pack(P, off)
    x_packed = np.asarray(x_packed)
    assert x_packed.shape[0] == packed_rows(P, off)
    return x_packed[r2p]


def fold(g_rep, P, off):
    """g_rep [T_rep, ...] -> fp64 [T, ...]; sum over the replicated rows of each packed row."""
    r2p = _rep2pack(P, off)
    g_rep = np.asarray(g_rep, dtype=np.float64)
    assert g_rep.shape[0] == len(r2p)
    out = np.zeros((packed_rows(P, off),) + g_rep.shape[1:], dtype=np.float64)
    for x, t in enumerate(r2p):
        out[t] += g_rep[x]
    return out
