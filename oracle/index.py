"""Packing-index oracle -- TEST INFRASTRUCTURE (see ``oracle/__init__``).

Plain Python restatement of the packed micro-batch layout of DualKV (paper
abstract: the data pipeline stores the N(P+R) tokens of N replicated sequences
as P+NR rows, the prompt only once):
packed rows are [prompt 0..P-1][segment 0][segment 1]...[segment N-1], where
segment n holds rows P+off[n] .. P+off[n+1]-1.  The replicated layout is the
N sequences prompt ++ segment n laid end to end.
"""
from __future__ import annotations


def build_index(P, off):
    """Return (seg_id, pos_id, cu_seqlens_rep, rep2pack) as Python int lists.

    seg_id[t]   -1 for a prompt row, else the segment that holds packed row t.
    pos_id[t]   position of packed row t in its replicated sequence (prompt row
                j -> j; row r of a segment -> P + r).
    cu_seqlens_rep[n]  start of replicated sequence n (N+1 entries).
    rep2pack[x] packed row of replicated row x.
    """
    N = len(off) - 1
    seg_id, pos_id = [], []
    for j in range(P):
        seg_id.append(-1)
        pos_id.append(j)
    for n in range(N):
        for r in range(off[n + 1] - off[n]):
            seg_id.append(n)
            pos_id.append(P + r)
    cu = [0]
    rep2pack = []
    for n in range(N):
        length = P + off[n + 1] - off[n]
        cu.append(cu[-1] + length)
        for p in range(length):
            rep2pack.append(p if p < P else P + off[n] + (p - P))
    return seg_id, pos_id, cu, rep2pack


def rho(P, off):
    """Token-reduction factor: replicated tokens over packed tokens.

    The abstract defines rho = N(P+R)/(P+NR) for equal lengths; with ragged
    lengths the same ratio reads sum_n (P+R_n) / (P + sum_n R_n).
    """
    N = len(off) - 1
    return (N * P + off[N]) / (P + off[N])


def allowed_count(pos, window):
    """Number of keys a query at replicated position ``pos`` attends."""
    return pos + 1 if window <= 0 else min(pos + 1, window)


def pairs(P, off, window=0):
    """Attended (query, key) pairs of one head in the packed layout: every
    packed query row counted once (prompt rows once, not N times)."""
    N = len(off) - 1
    total = sum(allowed_count(j, window) for j in range(P))
    for n in range(N):
        for r in range(off[n + 1] - off[n]):
            total += allowed_count(P + r, window)
    return total


def pairs_replicated(P, off, window=0):
    """Attended pairs of one head in the replicated layout."""
    N = len(off) - 1
    total = 0
    for n in range(N):
        for pos in range(P + off[n + 1] - off[n]):
            total += allowed_count(pos, window)
    return total
