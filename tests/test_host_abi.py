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


def test_binding_checks_shapes_before_the_c_call(lib):
    # meta tensors carry shapes and dtypes but no memory: a shape that does not fit the
    # layout (T = P + R_offsets[N] rows) is refused before any pointer is passed on
    import torch
    P, off, Hq, Hkv, D = 6, [0, 3, 5], 4, 2, 64
    T = P + off[-1]

    def t(*shape, dt=torch.bfloat16):
        return torch.empty(*shape, dtype=dt, device="meta")

    q, kv, lse = t(T, Hq, D), t(T, Hkv, D), t(Hq, T, dt=torch.float32)
    bad = {"q": t(T - 1, Hq, D), "k": t(T, Hq, D), "v": t(T, Hkv, D // 2), "out": t(T, Hq * D), "lse": t(T, Hq)}
    args = dict(q=q, k=kv, v=kv, out=q, lse=lse)
    for name, b in bad.items():
        a = dict(args, **{name: b})
        with pytest.raises(ValueError, match="shape"):
            dualkv.dualkv_fwd(a["q"], a["k"], a["v"], P, 2, off, Hq, Hkv, D, 0.125, 0, a["out"], a["lse"])
    with pytest.raises(ValueError, match="shape"):
        dualkv.dualkv_bwd(q, kv, kv, q, lse, q, P, 2, off, Hq, Hkv, D, 0.125, 0, q, t(T + 1, Hkv, D), kv, None, 0)
    with pytest.raises(ValueError, match="shape"):
        dualkv.dualkv_bwd_noalloc(q, kv, kv, q, lse, t(T, Hq, 2 * D), P, 2, off, Hq, Hkv, D, 0.125, 0, q, kv, kv)
    with pytest.raises(ValueError, match="shape"):
        dualkv.dualkv_fwd_layers([q, q], [kv, kv], [kv, t(1, Hkv, D)], [0, 0], P, 2, off, Hq, Hkv, D, 0.125, [q, q],
                                 [lse, lse])
    with pytest.raises(ValueError, match="R_offsets"):
        dualkv.dualkv_fwd(q, kv, kv, P, 3, off, Hq, Hkv, D, 0.125, 0, q, lse)
    # right shapes: refused next for not being CUDA tensors, still before the C call
    with pytest.raises(ValueError, match="CUDA"):
        dualkv.dualkv_fwd(q, kv, kv, P, 2, off, Hq, Hkv, D, 0.125, 0, q, lse)


def test_noalloc_refuses_head_dim_512_before_any_device_work(lib):
    off = (ctypes.c_int32 * 2)(0, 2)
    p = ctypes.c_void_p(0x10000)
    assert lib.dualkv_bwd_noalloc(p, p, p, p, p, p, 4, 1, off, 4, 2, 512, 0.125, 0, p, p, p, None) == \
        dualkv.DUALKV_ERR_UNSUPPORTED
    assert lib.dualkv_bwd_noalloc(p, p, p, p, p, p, 4, 1, off, 4, 2, 96, 0.125, 0, p, p, p, None) == \
        dualkv.DUALKV_ERR_INVALID


def test_selftest_rejects_out_of_range_limit(lib):
    assert lib.dualkv_selftest_timeout(10, None) == dualkv.DUALKV_ERR_INVALID
    assert lib.dualkv_selftest_timeout(100 * 10**9, None) == dualkv.DUALKV_ERR_INVALID
    assert lib.dualkv_selftest_kernel(0, 10, None) == dualkv.DUALKV_ERR_INVALID
    assert lib.dualkv_selftest_kernel(5, 50_000_000, None) == dualkv.DUALKV_ERR_INVALID
    assert lib.dualkv_selftest_kernel(-1, 50_000_000, None) == dualkv.DUALKV_ERR_INVALID


def test_plan_cache_evicts_least_recently_used(tmp_path):
    # the cache class is host-only C++: compile a small driver against it and run it
    import shutil
    import subprocess
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    exe = str(tmp_path / "lru")
    subprocess.run([cxx, "-std=c++17", "-O1", "-Wall", "-I", os.path.join(ROOT, "shared_prompt_exact_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "plan_cache_lru.cpp"), "-o", exe], check=True)
    res = subprocess.run([exe], capture_output=True, text=True)
    assert res.returncode == 0 and res.stdout.strip() == "ok", res.stdout + res.stderr


def test_head_range_validation_before_any_device_work(lib):
    off = (ctypes.c_int32 * 2)(0, 2)
    p, bad = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x10008)
    # kv-head range must satisfy 0 <= begin < end <= Hkv
    for lo, hi in ((1, 1), (-1, 1), (0, 3), (2, 1)):
        assert lib.dualkv_fwd_heads(p, p, p, 4, 1, off, 4, 2, 128, 0.125, 0, lo, hi, p, p, None) == \
            dualkv.DUALKV_ERR_INVALID
        assert lib.dualkv_bwd_heads(p, p, p, p, p, p, 4, 1, off, 4, 2, 128, 0.125, 0, lo, hi, p, p, p, p, 1 << 20,
                                    None) == dualkv.DUALKV_ERR_INVALID
    assert lib.dualkv_fwd_heads(p, p, p, 4, 1, off, 4, 2, 128, 0.125, 0, 0, 1, bad, p, None) == dualkv.DUALKV_ERR_ALIGN


def test_layer_stack_validation_before_any_device_work(lib):
    off = (ctypes.c_int32 * 2)(0, 2)
    n = 2
    good = (ctypes.c_void_p * n)(0x10000, 0x20000)
    mixed = (ctypes.c_void_p * n)(0x10000, 0x20008)  # the second layer's pointer is misaligned
    win = (ctypes.c_int32 * n)(0, 64)
    assert lib.dualkv_fwd_layers(0, good, good, good, win, 4, 1, off, 4, 2, 128, 0.125, good, good, None) == \
        dualkv.DUALKV_ERR_INVALID
    assert lib.dualkv_fwd_layers(n, None, good, good, win, 4, 1, off, 4, 2, 128, 0.125, good, good, None) == \
        dualkv.DUALKV_ERR_INVALID
    assert lib.dualkv_fwd_layers(n, good, good, good, win, 4, 1, off, 4, 3, 128, 0.125, good, good, None) == \
        dualkv.DUALKV_ERR_INVALID
    assert lib.dualkv_fwd_layers(n, good, good, mixed, win, 4, 1, off, 4, 2, 128, 0.125, good, good, None) == \
        dualkv.DUALKV_ERR_ALIGN
    assert lib.dualkv_bwd_layers_workspace_bytes(0, win, 4, 1, off, 4, 2, 128) == 0
    assert lib.dualkv_bwd_layers_workspace_bytes(n, None, 4, 1, off, 4, 2, 128) == 0
    # the stack needs what its most demanding window needs
    single = [lib.dualkv_bwd_workspace_bytes(4, 1, off, 4, 2, 128, w) for w in (0, 64)]
    assert lib.dualkv_bwd_layers_workspace_bytes(n, win, 4, 1, off, 4, 2, 128) == max(single) > 0


def test_pack_validation_before_any_device_work(lib):
    off = (ctypes.c_int32 * 3)(0, 2, 3)   # P = 4, N = 2: T = 7, T_rep = 11 rows
    src, dst = ctypes.c_void_p(0x100000), ctypes.c_void_p(0x200000)
    assert lib.dualkv_pack(src, dst, 4, 2, off, 12, None) == dualkv.DUALKV_ERR_INVALID    # not whole 16-byte vectors
    assert lib.dualkv_pack(src, dst, 4, 2, off, 0, None) == dualkv.DUALKV_ERR_INVALID
    assert lib.dualkv_pack(src, dst, -1, 2, off, 16, None) == dualkv.DUALKV_ERR_INVALID
    assert lib.dualkv_unpack(src, None, 4, 2, off, 16, None) == dualkv.DUALKV_ERR_INVALID
    # source and destination ranges overlap (11 replicated rows of 32 bytes from 0x100000)
    assert lib.dualkv_fold(src, ctypes.c_void_p(0x100000 + 5 * 32), 4, 2, off, 16, None) == dualkv.DUALKV_ERR_INVALID
    assert lib.dualkv_pack(ctypes.c_void_p(0x100008), dst, 4, 2, off, 16, None) == dualkv.DUALKV_ERR_ALIGN
    bad_off = (ctypes.c_int32 * 3)(0, 3, 2)
    assert lib.dualkv_pack(src, dst, 4, 2, bad_off, 16, None) == dualkv.DUALKV_ERR_INVALID
