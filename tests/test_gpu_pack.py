"""GPU parity of dualkv_pack / dualkv_unpack / dualkv_fold against ``oracle.pack``.

Copies (pack, unpack, the response rows of fold) must be bit-exact.  A folded
prompt row is the fp32 sum of N bf16 values rounded once to bf16; against the
fp64 oracle it may differ by the final rounding (half a bf16 ulp, at most
2^-8 of the magnitude) plus the fp32 accumulation error (at most
N * 2^-24 * sum |g|, doubled for margin).  The header also fixes the order of
that sum (replica 0 first), so the prompt rows are additionally compared
bit-exactly with a sequential fp32 sum done on the host.
"""
import numpy as np
import pytest
import torch

from oracle import pack as opk
from shared_prompt_exact_gb300 import dualkv as dk
from shared_prompt_exact_gb300.workloads import WORKLOADS

pytestmark = pytest.mark.gpu


def _u16(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def _check_fold(got, g_rep, P, off):
    """got: bf16 CUDA [T, E]; g_rep: bf16 CPU tensor [T_rep, E]."""
    N = len(off) - 1
    exact = opk.fold(_f64(g_rep), P, off)
    absum = opk.fold(np.abs(_f64(g_rep)), P, off)
    err = np.abs(_f64(got) - exact)
    tol = 2.0 ** -8 * np.abs(exact) + 2 * N * 2.0 ** -24 * absum
    assert np.all(err <= tol), f"fold: worst excess {float(np.max(err - tol)):.3e}"
    # response rows are copies
    np.testing.assert_array_equal(_u16(got[P:]), opk.pack(_u16(g_rep), P, off)[P:])
    # prompt rows: the documented fp32 sum in replica order, one rounding
    if P > 0:
        g32 = g_rep.float().numpy()
        acc = np.zeros((P, g32.shape[1]), dtype=np.float32)
        for n in range(N):
            start = n * P + off[n]
            acc = acc + g32[start:start + P]
        want = torch.from_numpy(acc).to(torch.bfloat16)
        np.testing.assert_array_equal(_u16(got[:P]), _u16(want))


CASES = [
    ("ragged", 37, [0, 5, 5, 19, 20, 44], 24),
    ("one-vector-rows", 16, [0, 3, 9], 8),
    ("wide-rows", 130, [0, 64, 200, 201], 4096),
    ("no-prompt", 0, [0, 7, 7, 12], 40),
    ("single-segment", 50, [0, 70], 136),
    ("prompt-only-replicas", 9, [0, 0, 0, 0], 16),
    ("odd-chunks", 21, [0, 2, 30, 31], 8 * 45),
]


@pytest.mark.parametrize("name,P,off,E", CASES, ids=[c[0] for c in CASES])
def test_pack_unpack_fold_small(name, P, off, E):
    N = len(off) - 1
    T, T_rep = opk.packed_rows(P, off), opk.replicated_rows(P, off)
    gen = torch.Generator().manual_seed(1000 + P + E)
    x_rep = torch.randn(T_rep, E, generator=gen).to(torch.bfloat16)
    x_packed = torch.randn(T, E, generator=gen).to(torch.bfloat16)
    g_rep = torch.randn(T_rep, E, generator=gen).to(torch.bfloat16)
    dev = torch.device("cuda")

    out = torch.full((T, E), float("nan"), dtype=torch.bfloat16, device=dev)
    dk.dualkv_pack(x_rep.to(dev), out, P, N, off)
    np.testing.assert_array_equal(_u16(out), opk.pack(_u16(x_rep), P, off))

    out_rep = torch.full((T_rep, E), float("nan"), dtype=torch.bfloat16, device=dev)
    dk.dualkv_unpack(x_packed.to(dev), out_rep, P, N, off)
    np.testing.assert_array_equal(_u16(out_rep), opk.unpack(_u16(x_packed), P, off))

    got = torch.full((T, E), float("nan"), dtype=torch.bfloat16, device=dev)
    dk.dualkv_fold(g_rep.to(dev), got, P, N, off)
    torch.cuda.synchronize()
    _check_fold(got, g_rep, P, off)


def test_pack_rejects_bad_arguments():
    dev = torch.device("cuda")
    P, off = 4, [0, 2, 3]
    T, T_rep = opk.packed_rows(P, off), opk.replicated_rows(P, off)
    lib = dk.load()
    src = torch.zeros(T_rep, 16, dtype=torch.bfloat16, device=dev)
    dst = torch.zeros(T, 16, dtype=torch.bfloat16, device=dev)
    off_c = dk._offsets(off)
    s = dk._stream(None)
    vp = dk._ptr
    assert lib.dualkv_pack(vp(src), vp(dst), P, 2, off_c, 12, s) == dk.DUALKV_ERR_INVALID  # not whole vectors
    assert lib.dualkv_pack(vp(src), vp(dst), P, 2, off_c, 0, s) == dk.DUALKV_ERR_INVALID
    assert lib.dualkv_pack(vp(src), vp(src), P, 2, off_c, 16, s) == dk.DUALKV_ERR_INVALID  # overlap
    assert lib.dualkv_pack(vp(src), vp(dst), -1, 2, off_c, 16, s) == dk.DUALKV_ERR_INVALID
    assert lib.dualkv_pack(vp(src), None, P, 2, off_c, 16, s) == dk.DUALKV_ERR_INVALID
    odd = torch.zeros(T * 16 + 8, dtype=torch.bfloat16, device=dev)[1:]
    assert lib.dualkv_fold(vp(src), vp(odd), P, 2, off_c, 16, s) == dk.DUALKV_ERR_ALIGN
    with pytest.raises(ValueError):
        dk.dualkv_pack(src, dst[:-1], P, 2, off)


@pytest.mark.parametrize("wl_name", ["grpo32", "dapo32"])
def test_pack_full_size_sampled_columns(wl_name):
    """Hidden-size rows (Hq * D) of the full workload; every row is checked on a
    sample of 16-byte column vectors (first, last and two seeded ones), which the
    oracle computes from the same columns of the input."""
    wl = WORKLOADS[wl_name]
    P, off, N = wl.P, list(wl.offsets), wl.N
    E = wl.Hq * wl.D
    T, T_rep = opk.packed_rows(P, off), opk.replicated_rows(P, off)
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev).manual_seed(wl.seed)
    x_rep = torch.randn(T_rep, E, generator=gen, device=dev).to(torch.bfloat16)
    x_packed = torch.randn(T, E, generator=gen, device=dev).to(torch.bfloat16)
    rng = np.random.default_rng(wl.seed)
    vecs = sorted({0, E // 8 - 1, *rng.integers(1, E // 8 - 1, size=2).tolist()})
    cols = torch.tensor([8 * v + e for v in vecs for e in range(8)], device=dev)

    out = torch.empty(T, E, dtype=torch.bfloat16, device=dev)
    dk.dualkv_pack(x_rep, out, P, N, off)
    np.testing.assert_array_equal(_u16(out[:, cols]), opk.pack(_u16(x_rep[:, cols]), P, off))

    out_rep = torch.empty(T_rep, E, dtype=torch.bfloat16, device=dev)
    dk.dualkv_unpack(x_packed, out_rep, P, N, off)
    np.testing.assert_array_equal(_u16(out_rep[:, cols]), opk.unpack(_u16(x_packed[:, cols]), P, off))

    dk.dualkv_fold(x_rep, out, P, N, off)
    torch.cuda.synchronize()
    _check_fold(out[:, cols], x_rep[:, cols].cpu(), P, off)
