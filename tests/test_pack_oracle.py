"""Pins of the tensor packing oracle (``oracle.pack``) -- CPU only.

The packed layout of DualKV (paper abstract: N(P+R) replicated tokens repacked
into P+NR) fixes pack, unpack and fold completely; these tests check the
oracle against values worked out by hand from that layout, against the
adjoint identity that makes fold the gradient of unpack, and against the
special cases where the layouts coincide.
"""
import numpy as np
import pytest

from oracle import pack as opk


def test_worked_layout_ragged():
    # P = 2, segments of 1 and 2 responses.  Replicated rows:
    #   seq 0: p0 p1 a0        seq 1: p0 p1 b0 b1      (7 rows)
    # packed rows: p0 p1 a0 b0 b1                      (5 rows)
    P, off = 2, [0, 1, 3]
    x_rep = np.array([[10], [11], [12], [20], [21], [22], [23]], dtype=np.float64)
    assert opk.pack(x_rep, P, off).ravel().tolist() == [10, 11, 12, 22, 23]
    assert opk.fold(x_rep, P, off).ravel().tolist() == [30, 32, 12, 22, 23]
    x_packed = np.array([[1], [2], [3], [4], [5]], dtype=np.float64)
    assert opk.unpack(x_packed, P, off).ravel().tolist() == [1, 2, 3, 1, 2, 4, 5]


def test_worked_layout_empty_segments():
    # P = 1, N = 3 with segments 0 and 2 empty: replicated seq 0 = [p0],
    # seq 1 = [p0 b0 b1], seq 2 = [p0]; packed rows p0 b0 b1.
    P, off = 1, [0, 0, 2, 2]
    x_rep = np.array([[1], [2], [3], [4], [5]], dtype=np.float64)
    assert opk.pack(x_rep, P, off).ravel().tolist() == [1, 3, 4]
    assert opk.fold(x_rep, P, off).ravel().tolist() == [8, 3, 4]
    assert opk.unpack(np.array([[7], [8], [9]]), P, off).ravel().tolist() == [7, 7, 8, 9, 7]


LAYOUTS = [(3, [0, 2, 2, 5]), (4, [0, 1]), (0, [0, 3, 4]), (5, [0, 0, 0, 1]), (7, [0, 4, 9, 9, 10, 16])]


@pytest.mark.parametrize("P,off", LAYOUTS)
def test_fold_is_adjoint_of_unpack(P, off):
    # integers keep every product and sum exact in fp64
    rng = np.random.default_rng(11 + P)
    T, T_rep = opk.packed_rows(P, off), opk.replicated_rows(P, off)
    x = rng.integers(-50, 50, size=(T, 3)).astype(np.float64)
    g = rng.integers(-50, 50, size=(T_rep, 3)).astype(np.float64)
    assert float(np.sum(opk.unpack(x, P, off) * g)) == float(np.sum(x * opk.fold(g, P, off)))


@pytest.mark.parametrize("P,off", LAYOUTS)
def test_round_trips(P, off):
    rng = np.random.default_rng(5 + P)
    T = opk.packed_rows(P, off)
    x = rng.standard_normal((T, 2))
    np.testing.assert_array_equal(opk.pack(opk.unpack(x, P, off), P, off), x)
    # every replicated prompt copy of unpack(x) agrees, so fold counts it N times
    N = len(off) - 1
    folded = opk.fold(opk.unpack(x, P, off), P, off)
    np.testing.assert_array_equal(folded[:P], N * x[:P])
    np.testing.assert_array_equal(folded[P:], x[P:])


def test_prompt_rows_come_from_replica_zero():
    # replicas that disagree: pack must take sequence 0's copy, not the last one
    P, off = 3, [0, 1, 2, 3]
    T_rep = opk.replicated_rows(P, off)
    x_rep = np.arange(T_rep, dtype=np.float64)[:, None]
    packed = opk.pack(x_rep, P, off).ravel().tolist()
    assert packed[:P] == [0, 1, 2]
    # response rows: seq n's response sits at n*P + off[n] + P
    assert packed[P:] == [3, 3 + 4, 3 + 8]


@pytest.mark.parametrize("off", [[0, 5], [0, 1]])
def test_single_segment_is_identity(off):
    # N = 1: the replicated and packed layouts coincide
    P = 4
    x = np.random.default_rng(3).standard_normal((P + off[-1], 5))
    np.testing.assert_array_equal(opk.pack(x, P, off), x)
    np.testing.assert_array_equal(opk.unpack(x, P, off), x)
    np.testing.assert_array_equal(opk.fold(x, P, off), x)


def test_no_prompt_is_identity():
    # P = 0: segments are laid end to end in both layouts
    off = [0, 2, 2, 6]
    x = np.random.default_rng(4).standard_normal((6, 3))
    for f in (opk.pack, opk.unpack, opk.fold):
        np.testing.assert_array_equal(f(x, 0, off), x)


def test_fold_of_ones_counts_replicas():
    P, off = 6, [0, 3, 3, 8, 10]
    N = len(off) - 1
    f = opk.fold(np.ones((opk.replicated_rows(P, off), 1)), P, off).ravel()
    assert f[:P].tolist() == [N] * P
    assert f[P:].tolist() == [1] * off[-1]
