"""ctypes binding of libdualkv.so (declared in include/dualkv.h).

Argument marshalling only: every step of the attention path runs in the
library's CUDA kernels.  The functions keep the C names and signatures
(tensors in place of raw pointers); ``forward``/``backward`` add buffer
allocation on top.  If the library is missing, loading raises: there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdualkv.so")

DUALKV_OK = 0
DUALKV_ERR_INVALID = 1
DUALKV_ERR_ALIGN = 2
DUALKV_ERR_WORKSPACE = 3
DUALKV_ERR_CUDA = 4
DUALKV_ERR_DEVICE = 5
DUALKV_ERR_UNSUPPORTED = 6

# every symbol the header declares
EXPORTS = ("dualkv_fwd", "dualkv_bwd_workspace_bytes", "dualkv_bwd", "dualkv_build_index", "dualkv_rho",
           "dualkv_pairs", "dualkv_check_status", "dualkv_error_string", "dualkv_profile_enable",
           "dualkv_profile_read", "dualkv_selftest_timeout", "dualkv_bwd_noalloc", "dualkv_release",
           "dualkv_pack", "dualkv_unpack", "dualkv_fold", "dualkv_fwd_heads", "dualkv_bwd_heads",
           "dualkv_fwd_layers", "dualkv_bwd_layers", "dualkv_bwd_layers_workspace_bytes",
           "dualkv_selftest_kernel", "dualkv_plan_cache_info")
NOALLOC_SCRATCH_BYTES = 32 << 20
KERNEL_KINDS = ("fwd", "prep", "dkv", "reduce", "dq", "pack")

_lock = threading.Lock()
_lib = None


class DualKVError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {error_string(code)} (code {code})")


def load(path: Optional[str] = None):
    """Load libdualkv.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build it with shared_prompt_exact_gb300.build.build()")
        lib = ctypes.CDLL(p)
        vp, ci, cf = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        i32p = ctypes.POINTER(ctypes.c_int32)
        lib.dualkv_fwd.argtypes = [vp, vp, vp, ci, ci, i32p, ci, ci, ci, cf, ci, vp, vp, vp]
        lib.dualkv_fwd.restype = ci
        lib.dualkv_bwd_workspace_bytes.argtypes = [ci, ci, i32p, ci, ci, ci, ci]
        lib.dualkv_bwd_workspace_bytes.restype = ctypes.c_size_t
        lib.dualkv_bwd.argtypes = [vp, vp, vp, vp, vp, vp, ci, ci, i32p, ci, ci, ci, cf, ci, vp, vp, vp, vp,
                                   ctypes.c_size_t, vp]
        lib.dualkv_bwd.restype = ci
        lib.dualkv_fwd_heads.argtypes = [vp, vp, vp, ci, ci, i32p, ci, ci, ci, cf, ci, ci, ci, vp, vp, vp]
        lib.dualkv_fwd_heads.restype = ci
        lib.dualkv_bwd_heads.argtypes = [vp, vp, vp, vp, vp, vp, ci, ci, i32p, ci, ci, ci, cf, ci, ci, ci, vp, vp,
                                         vp, vp, ctypes.c_size_t, vp]
        lib.dualkv_bwd_heads.restype = ci
        lib.dualkv_build_index.argtypes = [ci, ci, i32p, i32p, i32p, i32p, i32p]
        lib.dualkv_build_index.restype = ci
        lib.dualkv_rho.argtypes = [ci, ci, i32p]
        lib.dualkv_rho.restype = ctypes.c_double
        lib.dualkv_pairs.argtypes = [ci, ci, i32p, ci]
        lib.dualkv_pairs.restype = ctypes.c_int64
        lib.dualkv_check_status.argtypes = [vp]
        lib.dualkv_check_status.restype = ci
        lib.dualkv_error_string.argtypes = [ci]
        lib.dualkv_error_string.restype = ctypes.c_char_p
        lib.dualkv_profile_enable.argtypes = [ci]
        lib.dualkv_profile_enable.restype = ci
        lib.dualkv_profile_read.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64)]
        lib.dualkv_profile_read.restype = ci
        lib.dualkv_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, ci, ci, i32p, ci, ci, ci, cf, ci, vp, vp, vp, vp]
        lib.dualkv_bwd_noalloc.restype = ci
        lib.dualkv_selftest_timeout.argtypes = [ctypes.c_uint64, vp]
        lib.dualkv_selftest_timeout.restype = ci
        lib.dualkv_selftest_kernel.argtypes = [ci, ctypes.c_uint64, vp]
        lib.dualkv_selftest_kernel.restype = ci
        lib.dualkv_plan_cache_info.argtypes = [ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int64)]
        lib.dualkv_plan_cache_info.restype = ci
        for name in ("dualkv_pack", "dualkv_unpack", "dualkv_fold"):
            getattr(lib, name).argtypes = [vp, vp, ci, ci, i32p, ci, vp]
            getattr(lib, name).restype = ci
        lib.dualkv_bwd_layers_workspace_bytes.argtypes = [ci, i32p, ci, ci, i32p, ci, ci, ci]
        lib.dualkv_bwd_layers_workspace_bytes.restype = ctypes.c_size_t
        lib.dualkv_fwd_layers.argtypes = [ci, vp, vp, vp, i32p, ci, ci, i32p, ci, ci, ci, cf, vp, vp, vp]
        lib.dualkv_fwd_layers.restype = ci
        lib.dualkv_bwd_layers.argtypes = [ci, vp, vp, vp, vp, vp, vp, i32p, ci, ci, i32p, ci, ci, ci, cf, vp, vp, vp,
                                          vp, ctypes.c_size_t, vp]
        lib.dualkv_bwd_layers.restype = ci
        lib.dualkv_release.argtypes = []
        lib.dualkv_release.restype = None
        _lib = lib
        return lib


def error_string(code: int) -> str:
    return load().dualkv_error_string(int(code)).decode()


def _offsets(R_offsets: Sequence[int]):
    arr = (ctypes.c_int32 * len(R_offsets))(*[int(x) for x in R_offsets])
    return arr


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check_dev(name, t, dtype):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _check_shapes(where, P, N, R_offsets, Hq, Hkv, D, **tensors):
    """Every attention tensor must have exactly its layout's shape: q, out, dout, dq
    (T, Hq, D); k, v, dk, dv (T, Hkv, D); lse (Hq, T), with T = P + R_offsets[N].  The
    library builds its TMA views from these sizes, so an undersized tensor would be read
    or written past its end; the check runs before anything reaches the C ABI."""
    N = int(N)
    if N < 1 or len(R_offsets) != N + 1:
        raise ValueError(f"{where}: R_offsets must hold N + 1 = {N + 1} entries, got {len(R_offsets)}")
    T = int(P) + int(R_offsets[N])
    want = {"q": (T, Hq, D), "out": (T, Hq, D), "dout": (T, Hq, D), "dq": (T, Hq, D),
            "k": (T, Hkv, D), "v": (T, Hkv, D), "dk": (T, Hkv, D), "dv": (T, Hkv, D), "lse": (Hq, T)}
    for name, t in tensors.items():
        shape = tuple(int(x) for x in want[name.split("[")[0]])
        if not isinstance(t, torch.Tensor):
            raise ValueError(f"{where}: {name} must be a tensor")
        if tuple(t.shape) != shape:
            raise ValueError(f"{where}: {name} must have shape {shape} for this layout, got {tuple(t.shape)}")


def _raise(code, where):
    if code != DUALKV_OK:
        raise DualKVError(code, where)


def dualkv_fwd(q, k, v, P, N, R_offsets, Hq, Hkv, D, scale, window, out, lse, stream=None) -> None:
    _check_shapes("dualkv_fwd", P, N, R_offsets, Hq, Hkv, D, q=q, k=k, v=v, out=out, lse=lse)
    for name, t, dt in (("q", q, torch.bfloat16), ("k", k, torch.bfloat16), ("v", v, torch.bfloat16),
                        ("out", out, torch.bfloat16), ("lse", lse, torch.float32)):
        _check_dev(name, t, dt)
    off = _offsets(R_offsets)
    rc = load().dualkv_fwd(_ptr(q), _ptr(k), _ptr(v), int(P), int(N), off, int(Hq), int(Hkv), int(D),
                           float(scale), int(window), _ptr(out), _ptr(lse), _stream(stream))
    _raise(rc, "dualkv_fwd")


def dualkv_bwd_workspace_bytes(P, N, R_offsets, Hq, Hkv, D, window) -> int:
    return int(load().dualkv_bwd_workspace_bytes(int(P), int(N), _offsets(R_offsets), int(Hq), int(Hkv), int(D),
                                                  int(window)))


def dualkv_bwd(q, k, v, out, lse, dout, P, N, R_offsets, Hq, Hkv, D, scale, window, dq, dk, dv, workspace,
               workspace_bytes=None, stream=None) -> None:
    _check_shapes("dualkv_bwd", P, N, R_offsets, Hq, Hkv, D, q=q, k=k, v=v, out=out, lse=lse, dout=dout, dq=dq,
                  dk=dk, dv=dv)
    for name, t, dt in (("q", q, torch.bfloat16), ("k", k, torch.bfloat16), ("v", v, torch.bfloat16),
                        ("out", out, torch.bfloat16), ("lse", lse, torch.float32), ("dout", dout, torch.bfloat16),
                        ("dq", dq, torch.bfloat16), ("dk", dk, torch.bfloat16), ("dv", dv, torch.bfloat16)):
        _check_dev(name, t, dt)
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    rc = load().dualkv_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), int(P), int(N),
                           _offsets(R_offsets), int(Hq), int(Hkv), int(D), float(scale), int(window), _ptr(dq),
                           _ptr(dk), _ptr(dv), _ptr(workspace), int(workspace_bytes), _stream(stream))
    _raise(rc, "dualkv_bwd")


def dualkv_fwd_heads(q, k, v, P, N, R_offsets, Hq, Hkv, D, scale, window, kv_head_begin, kv_head_end, out, lse,
                     stream=None) -> None:
    """dualkv_fwd restricted to kv-heads [kv_head_begin, kv_head_end) and their q-heads."""
    _check_shapes("dualkv_fwd_heads", P, N, R_offsets, Hq, Hkv, D, q=q, k=k, v=v, out=out, lse=lse)
    for name, t, dt in (("q", q, torch.bfloat16), ("k", k, torch.bfloat16), ("v", v, torch.bfloat16),
                        ("out", out, torch.bfloat16), ("lse", lse, torch.float32)):
        _check_dev(name, t, dt)
    rc = load().dualkv_fwd_heads(_ptr(q), _ptr(k), _ptr(v), int(P), int(N), _offsets(R_offsets), int(Hq), int(Hkv),
                                 int(D), float(scale), int(window), int(kv_head_begin), int(kv_head_end), _ptr(out),
                                 _ptr(lse), _stream(stream))
    _raise(rc, "dualkv_fwd_heads")


def dualkv_bwd_heads(q, k, v, out, lse, dout, P, N, R_offsets, Hq, Hkv, D, scale, window, kv_head_begin,
                     kv_head_end, dq, dk, dv, workspace, workspace_bytes=None, stream=None) -> None:
    """dualkv_bwd restricted to kv-heads [kv_head_begin, kv_head_end) and their q-heads."""
    _check_shapes("dualkv_bwd_heads", P, N, R_offsets, Hq, Hkv, D, q=q, k=k, v=v, out=out, lse=lse, dout=dout,
                  dq=dq, dk=dk, dv=dv)
    for name, t, dt in (("q", q, torch.bfloat16), ("k", k, torch.bfloat16), ("v", v, torch.bfloat16),
                        ("out", out, torch.bfloat16), ("lse", lse, torch.float32), ("dout", dout, torch.bfloat16),
                        ("dq", dq, torch.bfloat16), ("dk", dk, torch.bfloat16), ("dv", dv, torch.bfloat16)):
        _check_dev(name, t, dt)
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    rc = load().dualkv_bwd_heads(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), int(P), int(N),
                                 _offsets(R_offsets), int(Hq), int(Hkv), int(D), float(scale), int(window),
                                 int(kv_head_begin), int(kv_head_end), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
                                 int(workspace_bytes), _stream(stream))
    _raise(rc, "dualkv_bwd_heads")


def _check_layer_shapes(where, n, P, N, R_offsets, Hq, Hkv, D, **stacks):
    for name, ts in stacks.items():
        if len(ts) != n:
            raise ValueError(f"{where}: {name}: expected {n} tensors, got {len(ts)}")
        for i, t in enumerate(ts):
            _check_shapes(where, P, N, R_offsets, Hq, Hkv, D, **{f"{name}[{i}]": t})


def _ptr_array(name, tensors, n, dtype):
    if len(tensors) != n:
        raise ValueError(f"{name}: expected {n} tensors, got {len(tensors)}")
    for i, t in enumerate(tensors):
        _check_dev(f"{name}[{i}]", t, dtype)
    return (ctypes.c_void_p * n)(*[t.data_ptr() for t in tensors])


def dualkv_bwd_layers_workspace_bytes(windows, P, N, R_offsets, Hq, Hkv, D) -> int:
    n = len(windows)
    return int(load().dualkv_bwd_layers_workspace_bytes(n, (ctypes.c_int32 * n)(*[int(x) for x in windows]), int(P),
                                                         int(N), _offsets(R_offsets), int(Hq), int(Hkv), int(D)))


def dualkv_fwd_layers(qs, ks, vs, windows, P, N, R_offsets, Hq, Hkv, D, scale, outs, lses, stream=None) -> None:
    """Forward of a layer stack: layer l uses qs[l], ks[l], vs[l] and windows[l]."""
    n = len(windows)
    _check_layer_shapes("dualkv_fwd_layers", n, P, N, R_offsets, Hq, Hkv, D, q=qs, k=ks, v=vs, out=outs, lse=lses)
    bf = torch.bfloat16
    rc = load().dualkv_fwd_layers(n, _ptr_array("q", qs, n, bf), _ptr_array("k", ks, n, bf), _ptr_array("v", vs, n, bf),
                                  (ctypes.c_int32 * n)(*[int(x) for x in windows]), int(P), int(N),
                                  _offsets(R_offsets), int(Hq), int(Hkv), int(D), float(scale),
                                  _ptr_array("out", outs, n, bf), _ptr_array("lse", lses, n, torch.float32),
                                  _stream(stream))
    _raise(rc, "dualkv_fwd_layers")


def dualkv_bwd_layers(qs, ks, vs, outs, lses, douts, windows, P, N, R_offsets, Hq, Hkv, D, scale, dqs, dks, dvs,
                      workspace, workspace_bytes=None, stream=None) -> None:
    """Backward of a layer stack, layers in the order given, one shared workspace."""
    n = len(windows)
    _check_layer_shapes("dualkv_bwd_layers", n, P, N, R_offsets, Hq, Hkv, D, q=qs, k=ks, v=vs, out=outs, lse=lses,
                        dout=douts, dq=dqs, dk=dks, dv=dvs)
    bf = torch.bfloat16
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    rc = load().dualkv_bwd_layers(n, _ptr_array("q", qs, n, bf), _ptr_array("k", ks, n, bf), _ptr_array("v", vs, n, bf),
                                  _ptr_array("out", outs, n, bf), _ptr_array("lse", lses, n, torch.float32),
                                  _ptr_array("dout", douts, n, bf), (ctypes.c_int32 * n)(*[int(x) for x in windows]),
                                  int(P), int(N), _offsets(R_offsets), int(Hq), int(Hkv), int(D), float(scale),
                                  _ptr_array("dq", dqs, n, bf), _ptr_array("dk", dks, n, bf),
                                  _ptr_array("dv", dvs, n, bf), _ptr(workspace), int(workspace_bytes),
                                  _stream(stream))
    _raise(rc, "dualkv_bwd_layers")


def kv_head_ranges(Hkv: int, parts: int):
    """Contiguous kv-head groups [lo, hi) for `parts` ranks (sizes differ by at most one;
    a rank gets an empty range when parts > Hkv)."""
    Hkv, parts = int(Hkv), int(parts)
    if Hkv < 1 or parts < 1:
        raise ValueError("Hkv and parts must be positive")
    base, extra = divmod(Hkv, parts)
    out, lo = [], 0
    for r in range(parts):
        hi = lo + base + (1 if r < extra else 0)
        out.append((lo, hi))
        lo = hi
    return out


def dualkv_bwd_noalloc(q, k, v, out, lse, dout, P, N, R_offsets, Hq, Hkv, D, scale, window, dq, dk, dv,
                       stream=None) -> None:
    """dualkv_bwd without a workspace: for callers that cannot allocate device
    memory.  Its scratch is a fixed array inside the library (NOALLOC_SCRATCH_BYTES
    per GPU); calls overlapping on the GPU race on it.  Returns once the pass has
    finished on `stream`."""
    _check_shapes("dualkv_bwd_noalloc", P, N, R_offsets, Hq, Hkv, D, q=q, k=k, v=v, out=out, lse=lse, dout=dout,
                  dq=dq, dk=dk, dv=dv)
    for name, t, dt in (("q", q, torch.bfloat16), ("k", k, torch.bfloat16), ("v", v, torch.bfloat16),
                        ("out", out, torch.bfloat16), ("lse", lse, torch.float32), ("dout", dout, torch.bfloat16),
                        ("dq", dq, torch.bfloat16), ("dk", dk, torch.bfloat16), ("dv", dv, torch.bfloat16)):
        _check_dev(name, t, dt)
    rc = load().dualkv_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), int(P), int(N),
                                   _offsets(R_offsets), int(Hq), int(Hkv), int(D), float(scale), int(window),
                                   _ptr(dq), _ptr(dk), _ptr(dv), _stream(stream))
    _raise(rc, "dualkv_bwd_noalloc")


def _pack_call(fn, name, src, dst, P, N, R_offsets, stream):
    for nm, t in (("src", src), ("dst", dst)):
        _check_dev(nm, t, torch.bfloat16)
        if t.dim() < 2:
            raise ValueError(f"{name}: {nm} must have a row dimension and at least one more")
    T = int(P) + int(R_offsets[N])
    T_rep = int(N) * int(P) + int(R_offsets[N])
    rows_src, rows_dst = (T, T_rep) if name == "dualkv_unpack" else (T_rep, T)
    if src.shape[0] != rows_src or dst.shape[0] != rows_dst:
        raise ValueError(f"{name}: expected {rows_src} source and {rows_dst} destination rows, "
                         f"got {src.shape[0]} and {dst.shape[0]}")
    row_elems = src.numel() // rows_src
    if dst.numel() // rows_dst != row_elems:
        raise ValueError(f"{name}: src and dst rows must have the same number of elements")
    rc = fn(_ptr(src), _ptr(dst), int(P), int(N), _offsets(R_offsets), int(row_elems), _stream(stream))
    _raise(rc, name)


def dualkv_pack(x_rep, x_packed, P, N, R_offsets, stream=None) -> None:
    """x_rep [N*P + R_offsets[N], ...] -> x_packed [P + R_offsets[N], ...] (prompt rows from replica 0)."""
    _pack_call(load().dualkv_pack, "dualkv_pack", x_rep, x_packed, P, N, R_offsets, stream)


def dualkv_unpack(x_packed, x_rep, P, N, R_offsets, stream=None) -> None:
    """x_packed [T, ...] -> x_rep [T_rep, ...] (prompt rows copied into every replica)."""
    _pack_call(load().dualkv_unpack, "dualkv_unpack", x_packed, x_rep, P, N, R_offsets, stream)


def dualkv_fold(g_rep, g_packed, P, N, R_offsets, stream=None) -> None:
    """g_rep [T_rep, ...] -> g_packed [T, ...]: prompt rows summed over the N replicas (fp32, in order)."""
    _pack_call(load().dualkv_fold, "dualkv_fold", g_rep, g_packed, P, N, R_offsets, stream)


def dualkv_build_index(P, N, R_offsets):
    """Host index builder: returns (seg_id, pos_id, cu_seqlens_rep, rep2pack) as int32 CPU tensors."""
    T = int(P) + int(R_offsets[N])
    n_rep = int(N) * int(P) + int(R_offsets[N])
    seg = torch.empty(T, dtype=torch.int32)
    pos = torch.empty(T, dtype=torch.int32)
    cu = torch.empty(int(N) + 1, dtype=torch.int32)
    r2p = torch.empty(max(n_rep, 1), dtype=torch.int32)
    i32p = ctypes.POINTER(ctypes.c_int32)
    rc = load().dualkv_build_index(int(P), int(N), _offsets(R_offsets),
                                   ctypes.cast(seg.data_ptr(), i32p), ctypes.cast(pos.data_ptr(), i32p),
                                   ctypes.cast(cu.data_ptr(), i32p), ctypes.cast(r2p.data_ptr(), i32p))
    _raise(rc, "dualkv_build_index")
    return seg, pos, cu, r2p[:n_rep]


def dualkv_rho(P, N, R_offsets) -> float:
    return float(load().dualkv_rho(int(P), int(N), _offsets(R_offsets)))


def dualkv_pairs(P, N, R_offsets, window=0) -> int:
    return int(load().dualkv_pairs(int(P), int(N), _offsets(R_offsets), int(window)))


def dualkv_check_status(stream=None) -> None:
    _raise(load().dualkv_check_status(_stream(stream)), "dualkv_check_status")


def dualkv_profile_enable(on: bool) -> None:
    _raise(load().dualkv_profile_enable(1 if on else 0), "dualkv_profile_enable")


def dualkv_profile_read():
    """{kernel kind: (total ms, launches)} of the launches timed since the last read."""
    n = len(KERNEL_KINDS)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int64 * n)()
    _raise(load().dualkv_profile_read(ms, cnt), "dualkv_profile_read")
    return {KERNEL_KINDS[i]: (float(ms[i]), int(cnt[i])) for i in range(n)}


def dualkv_selftest_timeout(limit_ns: int, stream=None) -> None:
    _raise(load().dualkv_selftest_timeout(int(limit_ns), _stream(stream)), "dualkv_selftest_timeout")


def dualkv_selftest_kernel(which: int, limit_ns: int, stream=None) -> None:
    """Runs a production kernel on a tiny internal layout with its failure path
    forced (0: forward, a K/V tile never loaded; 1: dK/dV, a query block one
    barrier arrival short; 2: forward, a work item past the last row; 3: dQ, a
    work item past the last row; 4: the D = 512 P / dS pass, a K/V tile never
    loaded) and every wait limited to limit_ns.  dualkv_check_status() then raises DUALKV_ERR_DEVICE."""
    _raise(load().dualkv_selftest_kernel(int(which), int(limit_ns), _stream(stream)), "dualkv_selftest_kernel")


def dualkv_plan_cache_info():
    """(resident plans, device bytes held by the plan cache, resident and pooled)."""
    n = ctypes.c_int(0)
    b = ctypes.c_int64(0)
    _raise(load().dualkv_plan_cache_info(ctypes.byref(n), ctypes.byref(b)), "dualkv_plan_cache_info")
    return int(n.value), int(b.value)


def dualkv_release() -> None:
    load().dualkv_release()


# ------------------------------------------------------------------ convenience
def forward(q, k, v, P, R_offsets, window=0, scale=None, stream=None):
    """Allocate out/lse and run dualkv_fwd. q [T,Hq,D], k/v [T,Hkv,D] bf16 CUDA."""
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    N = len(R_offsets) - 1
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    out = torch.empty_like(q)
    lse = torch.empty(Hq, T, dtype=torch.float32, device=q.device)
    dualkv_fwd(q, k, v, P, N, R_offsets, Hq, Hkv, D, scale, window, out, lse, stream)
    return out, lse


def workspace_for(P, R_offsets, Hq, Hkv, D, window=0, device="cuda"):
    nbytes = dualkv_bwd_workspace_bytes(P, len(R_offsets) - 1, R_offsets, Hq, Hkv, D, window)
    if nbytes == 0:
        raise DualKVError(DUALKV_ERR_INVALID, "dualkv_bwd_workspace_bytes")
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def backward(q, k, v, out, lse, dout, P, R_offsets, window=0, scale=None, workspace=None, stream=None):
    """Allocate dq/dk/dv (and workspace if not given) and run dualkv_bwd."""
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    N = len(R_offsets) - 1
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    if workspace is None:
        workspace = workspace_for(P, R_offsets, Hq, Hkv, D, window, q.device)
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    dualkv_bwd(q, k, v, out, lse, dout, P, N, R_offsets, Hq, Hkv, D, scale, window, dq, dk, dv, workspace,
               None, stream)
    return dq, dk, dv
