"""fp64 CPU oracle for DualKV shared-prompt attention -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA product path never imports,
links or calls it, and it imports nothing from the product package.

Contents
--------
* ``dualkv_oracle.c`` (loaded here through ctypes): the plain definition --
  standard causal attention on the N replicated sequences, its analytic
  backward, and the fold of replicated prompt gradients by summation
  (DualKV paper, abstract: the packed result is exactly that of ordinary
  attention on the replicated sequences).
* ``brute``: an independent dense numpy formulation over the *packed* rows with
  an explicit T x T mask, used to pin the C oracle on tiny inputs.
* ``index``: an independent pure-Python packing-index builder (seg-id, pos-id,
  replicated cu_seqlens, replicated->packed row map), the token-reduction
  factor rho and the attended-pair count.

Parity status: every function here is pinned by the ``-m "not gpu"`` tests
(brute force, torch float64 autograd, finite differences, invariants and
closed forms); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_SRC = os.path.join(_HERE, "dualkv_oracle.c")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (portable flags: runs on x86_64 and aarch64)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i32p = ctypes.POINTER(ctypes.c_int32)
            i64p = ctypes.POINTER(ctypes.c_int64)
            f64p = ctypes.POINTER(ctypes.c_double)
            ci, cd = ctypes.c_int, ctypes.c_double
            lib.oracle_dualkv.argtypes = [ci, ci, i32p, ci, ci, ci, cd, ci, ci, ci, f64p, f64p, f64p,
                                          f64p, ci, f64p, f64p, f64p, f64p, f64p,
                                          ctypes.POINTER(ctypes.c_int)]
            lib.oracle_dualkv.restype = ci
            lib.oracle_query_rows.argtypes = [ci, ci, i32p, ci, ci, ci, cd, ci, ci, i64p, ci, f64p,
                                              f64p, f64p, f64p, ci, f64p, f64p, f64p]
            lib.oracle_query_rows.restype = ci
            lib.oracle_key_rows.argtypes = [ci, ci, i32p, ci, ci, ci, cd, ci, ci, i64p, ci, f64p,
                                            f64p, f64p, f64p, ci, f64p, f64p]
            lib.oracle_key_rows.restype = ci
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = ci
            _lib = lib
    return _lib


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor (bf16 widens exactly to fp64)
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a, typ=ctypes.c_double):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(typ))


def _offsets(off):
    return np.ascontiguousarray(np.asarray(off, dtype=np.int32))


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def dualkv(P, N, off, Hq, Hkv, D, scale, window, q, k, v, dout=None, heads=None, dout_mode=0,
           forward_only=False):
    """Full oracle over packed inputs. Returns dict with out, lse, dq, dk, dv (fp64
    arrays in packed layout; rows of heads outside ``heads`` are zero) and
    ``prompt_invariant`` (1 when all replicas' prompt outputs are identical)."""
    lib = _load()
    off = _offsets(off)
    T = P + int(off[N])
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    q = q.reshape(T, Hq, D); k = k.reshape(T, Hkv, D); v = v.reshape(T, Hkv, D)
    h_lo, h_hi = (0, Hq) if heads is None else heads
    out = np.zeros((T, Hq, D)); lse = np.zeros((Hq, T))
    bwd = (dout is not None) and not forward_only
    dq = np.zeros((T, Hq, D)) if bwd else None
    dk = np.zeros((T, Hkv, D)) if bwd else None
    dv = np.zeros((T, Hkv, D)) if bwd else None
    inv = ctypes.c_int(-1)
    rc = lib.oracle_dualkv(P, N, _ptr(off, ctypes.c_int32), Hq, Hkv, D, float(scale), int(window),
                           h_lo, h_hi, _ptr(q), _ptr(k), _ptr(v), _ptr(dout.reshape(T, Hq, D) if bwd else None),
                           int(dout_mode), _ptr(out), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
                           ctypes.byref(inv))
    if rc != 0:
        raise RuntimeError(f"oracle_dualkv failed with code {rc}")
    return dict(out=out, lse=lse, dq=dq, dk=dk, dv=dv, prompt_invariant=inv.value)


def query_rows(P, N, off, Hq, Hkv, D, scale, window, h, rows, q, k, v, dout=None, dout_mode=0):
    """O [n,D], LSE [n], dQ [n,D] (or None) of packed query rows ``rows`` for q-head h."""
    lib = _load()
    off = _offsets(off)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    n = len(rows)
    o = np.zeros((n, D)); lse = np.zeros(n)
    dq = np.zeros((n, D)) if dout is not None else None
    rc = lib.oracle_query_rows(P, N, _ptr(off, ctypes.c_int32), Hq, Hkv, D, float(scale), int(window),
                               int(h), _ptr(rows, ctypes.c_int64), n, _ptr(q), _ptr(k), _ptr(v),
                               _ptr(dout), int(dout_mode), _ptr(o), _ptr(lse), _ptr(dq))
    if rc != 0:
        raise RuntimeError(f"oracle_query_rows failed with code {rc}")
    return o, lse, dq


def key_rows(P, N, off, Hq, Hkv, D, scale, window, g, keys, q, k, v, dout, dout_mode=0):
    """dK [n,D], dV [n,D] of packed key rows ``keys`` for kv-head g."""
    lib = _load()
    off = _offsets(off)
    keys = np.ascontiguousarray(np.asarray(keys, dtype=np.int64))
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    n = len(keys)
    dk = np.zeros((n, D)); dv = np.zeros((n, D))
    rc = lib.oracle_key_rows(P, N, _ptr(off, ctypes.c_int32), Hq, Hkv, D, float(scale), int(window),
                             int(g), _ptr(keys, ctypes.c_int64), n, _ptr(q), _ptr(k), _ptr(v), _ptr(dout),
                             int(dout_mode), _ptr(dk), _ptr(dv))
    if rc != 0:
        raise RuntimeError(f"oracle_key_rows failed with code {rc}")
    return dk, dv
