"""fp64 CPU oracle of the routed MoE FFN layer -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
leg of ``bench.py`` may import this package.  The CUDA library never does.

The arithmetic lives in ``moe_oracle.cpp`` (plain C++17, double precision);
this module compiles it with g++ and wraps its C entry points with ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cpp")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")

ACT_F32, ACT_BF16 = 0, 1
W_F32, W_INT4_G32 = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle (g++ -O2, OpenMP) next to its source."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["g++", "-std=c++17", "-O2", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", _LIB + ".tmp"]
        subprocess.check_call(cmd)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _act(x):
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        return x, ACT_BF16
    if x.dtype == np.float32:
        return x, ACT_F32
    raise TypeError(f"activations must be bf16 bits (uint16) or float32, got {x.dtype}")


def nthreads_default() -> int:
    return os.cpu_count() or 1


def widen(x) -> np.ndarray:
    x, dt = _act(x)
    out = np.empty(x.shape, dtype=np.float64)
    lib().orc_widen(ctypes.c_size_t(x.size), _p(x), dt, _p(out))
    return out


def f16_to_double(h) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float64)
    lib().orc_f16_to_double(ctypes.c_size_t(h.size), _p(h), _p(out))
    return out


def dequant(q, s, rows: int, cols: int) -> np.ndarray:
    q = np.ascontiguousarray(q)
    wfmt = W_F32 if q.dtype == np.float32 else W_INT4_G32
    s = None if s is None else np.ascontiguousarray(s, dtype=np.uint16)
    out = np.empty((rows, cols), dtype=np.float64)
    rc = lib().orc_dequant(rows, cols, wfmt, _p(q), _p(s), _p(out))
    if rc:
        raise ValueError("orc_dequant failed")
    return out


def route(x, Wr, bias, K: int, nthreads: int = 0):
    """Returns (logits [T,E], idx [T,K] int32, w [T,K] float64, gap [T])."""
    x, dt = _act(x)
    T, d = x.shape
    Wr = np.ascontiguousarray(Wr, dtype=np.float32)
    E = Wr.shape[0]
    bias = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    logits = np.empty((T, E), np.float64)
    idx = np.empty((T, K), np.int32)
    w = np.empty((T, K), np.float64)
    gap = np.empty(T, np.float64)
    rc = lib().orc_route(T, d, E, K, _p(x), dt, _p(Wr), _p(bias), _p(logits), _p(idx), _p(w), _p(gap),
                         nthreads)
    if rc:
        raise ValueError("orc_route failed")
    return logits, idx, w, gap


def weights_for(logits, idx) -> np.ndarray:
    logits = np.ascontiguousarray(logits, dtype=np.float64)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    T, E = logits.shape
    K = idx.shape[1]
    w = np.empty((T, K), np.float64)
    lib().orc_weights_for(T, E, K, _p(logits), _p(idx), _p(w))
    return w


def dispatch(idx, E: int):
    """Returns (counts [E], offs [E+1], perm [T*K], active [n_active])."""
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    T, K = idx.shape
    counts = np.empty(E, np.int32)
    offs = np.empty(E + 1, np.int32)
    perm = np.empty(T * K, np.int32)
    active = np.empty(E, np.int32)
    n_active = ctypes.c_int32(0)
    rc = lib().orc_dispatch(T, K, E, _p(idx), _p(counts), _p(offs), _p(perm), _p(active),
                            ctypes.byref(n_active))
    if rc:
        raise ValueError("orc_dispatch failed")
    return counts, offs, perm, active[: n_active.value].copy()


def _wfmt(planes) -> int:
    return W_F32 if planes["gu_q"].dtype == np.float32 else W_INT4_G32


def expert(planes, x_vec) -> np.ndarray:
    gu = np.ascontiguousarray(planes["gu_q"])
    dn = np.ascontiguousarray(planes["dn_q"])
    f2, dcols = gu.shape
    wfmt = _wfmt(planes)
    d = dcols if wfmt == W_F32 else dcols * 2
    f = f2 // 2
    gs = None if planes["gu_s"] is None else np.ascontiguousarray(planes["gu_s"])
    ds = None if planes["dn_s"] is None else np.ascontiguousarray(planes["dn_s"])
    x = np.ascontiguousarray(x_vec, dtype=np.float64)
    y = np.empty(d, np.float64)
    lib().orc_expert(d, f, wfmt, _p(gu), _p(gs), _p(dn), _p(ds), _p(x), _p(y))
    return y


def layer(x, Wr, bias, experts: dict, E: int, K: int, shared=None, idx=None, nthreads: int = 0):
    """y [T,d] float64 for the layer.  `experts` maps expert index -> planes (only the used ones
    are needed).  Returns (y, idx_used, w_used)."""
    x, dt = _act(x)
    T, d = x.shape
    any_e = next(iter(experts.values())) if experts else shared
    wfmt = _wfmt(any_e)
    f = any_e["gu_q"].shape[0] // 2
    Wr = np.ascontiguousarray(Wr, dtype=np.float32)
    bias = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    keep = []

    def table(name):
        arr = (ctypes.c_void_p * E)()
        for e, pl in experts.items():
            if not 0 <= e < E:
                raise ValueError(f"expert index {e} outside [0, {E})")
            if pl[name] is not None:
                a = np.ascontiguousarray(pl[name])
                keep.append(a)
                arr[e] = a.ctypes.data
        return arr

    gu, gs, dn, ds = table("gu_q"), table("gu_s"), table("dn_q"), table("dn_s")
    sh = {}
    if shared is not None:
        for name in ("gu_q", "gu_s", "dn_q", "dn_s"):
            sh[name] = None if shared[name] is None else np.ascontiguousarray(shared[name])
    idx_in = None if idx is None else np.ascontiguousarray(idx, dtype=np.int32)
    idx_out = np.empty((T, K), np.int32)
    w_out = np.empty((T, K), np.float64)
    y = np.empty((T, d), np.float64)
    rc = lib().orc_layer(T, d, f, E, K, wfmt, 1 if shared is not None else 0, _p(x), dt, _p(Wr), _p(bias),
                         gu, gs, dn, ds,
                         _p(sh.get("gu_q")), _p(sh.get("gu_s")), _p(sh.get("dn_q")), _p(sh.get("dn_s")),
                         _p(idx_in), _p(idx_out), _p(w_out), _p(y), nthreads)
    if rc:
        raise ValueError(f"orc_layer failed ({rc}): an expert used by the routing was not provided")
    return y, idx_out, w_out


def rmsnorm(x, eps: float) -> np.ndarray:
    x, dt = _act(x)
    T, d = x.shape
    out = np.empty((T, d), np.float64)
    lib().orc_rmsnorm(T, d, _p(x), dt, ctypes.c_double(eps), _p(out))
    return out
