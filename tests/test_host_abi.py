"""Host-side checks of libdualkv.so: it loads, exports every symbol the header
declares, its packing-index builder matches the oracle's bit for bit, and its
argument validation rejects bad calls before touching a GPU."""
import ctypes
import os
import re

import pytest

from oracle import index as oindex
from shared_prompt_exact_gb300 import build as pbuild
from shared_prompt_exact_gb300 import dualkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    pbuild.build()
    return dualkv.load()


def header_symbols():
    text = open(os.path.join(ROOT, "include", "dualkv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dualkv_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    syms = header_symbols()
    assert len(syms) >= 9
    assert sorted(dualkv.EXPORTS) == syms
    for s in syms:
        assert hasattr(lib, s), s


LAYOUTS = [
    (64, [0, 32, 64, 96, 128]),
    (5, [0, 3, 3, 7]),
    (0, [0, 4, 10]),
    (1, [0, 0]),
    (300, [0, 200, 200, 329, 330, 394]),
]


@pytest.mark.parametrize("P,off", LAYOUTS)
def test_index_builder_bit_exact(lib, P, off):
    N = len(off) - 1
    seg, pos, cu, r2p = dualkv.dualkv_build_index(P, N, off)
    oseg, opos, ocu, or2p = oindex.build_index(P, off)
    assert seg.tolist() == oseg
    assert pos.tolist() == opos
    assert cu.tolist() == ocu
    assert r2p.tolist() == or2p


@pytest.mark.parametrize("P,off", LAYOUTS)
def test_rho_and_pairs(lib, P, off):
    N = len(off) - 1
    assert dualkv.dualkv_rho(P, N, off) == pytest.approx(oindex.rho(P, off), rel=1e-15)
    for w in (0, 1, 3, 64, 10000):
        assert dualkv.dualkv_pairs(P, N, off, w) == oindex.pairs(P, off, w)


def test_rho_matches_paper_formula(lib):
    # equal lengths: rho = N(P+R)/(P+NR)
    for P, N, R in ((6144, 32, 2048), (8192, 16, 1024), (16384, 16, 3072), (64, 4, 32)):
        off = [n * R for n in range(N + 1)]
        assert dualkv.dualkv_rho(P, N, off) == pytest.approx(N * (P + R) / (P + N * R), rel=1e-15)


def test_index_builder_rejects_bad_offsets(lib):
    i32 = ctypes.c_int32
    bad = (i32 * 3)(0, 5, 4)
    assert lib.dualkv_build_index(3, 2, bad, None, None, None, None) == dualkv.DUALKV_ERR_INVALID
    bad0 = (i32 * 2)(1, 4)
    assert lib.dualkv_build_index(3, 1, bad0, None, None, None, None) == dualkv.DUALKV_ERR_INVALID


def _fwd_rc(lib, P, off, Hq, Hkv, D, ptr=0x10000, scale=0.125):
    N = len(off) - 1
    arr = (ctypes.c_int32 * len(off))(*off)
    p = ctypes.c_void_p(ptr)
    return lib.dualkv_fwd(p, p, p, P, N, arr, Hq, Hkv, D, scale, 0, p, p, None)


def test_validation_before_any_device_work(lib):
    # every case below is rejected by host checks; no pointer is dereferenced
    assert _fwd_rc(lib, 4, [0, 2], 4, 3, 128) == dualkv.DUALKV_ERR_INVALID          # Hq % Hkv
    assert _fwd_rc(lib, 4, [0, 2], 4, 2, 96) == dualkv.DUALKV_ERR_INVALID           # D
    assert _fwd_rc(lib, -1, [0, 2], 4, 2, 128) == dualkv.DUALKV_ERR_INVALID         # P
    assert _fwd_rc(lib, 4, [0, 3, 2], 4, 2, 128) == dualkv.DUALKV_ERR_INVALID       # offsets
    assert _fwd_rc(lib, 4, [0, 2], 4, 2, 128, scale=0.0) == dualkv.DUALKV_ERR_INVALID
    assert _fwd_rc(lib, 4, [0, 2], 4, 2, 128, ptr=0x10008) == dualkv.DUALKV_ERR_ALIGN
    assert lib.dualkv_bwd_workspace_bytes(4, 1, (ctypes.c_int32 * 2)(0, 2), 4, 3, 128, 0) == 0


def test_error_strings(lib):
    for code in range(0, 8):
        assert isinstance(dualkv.error_string(code), str) and dualkv.error_string(code)


def test_binding_refuses_cpu_tensors(lib):
    import torch
    x = torch.zeros(4, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        dualkv.dualkv_fwd(x, x, x, 2, 1, [0, 2], 2, 2, 64, 0.125, 0, x, torch.zeros(2, 4), None)


def test_selftest_rejects_out_of_range_limit(lib):
    assert lib.dualkv_selftest_timeout(10, None) == dualkv.DUALKV_ERR_INVALID
    assert lib.dualkv_selftest_timeout(100 * 10**9, None) == dualkv.DUALKV_ERR_INVALID
