"""Float64 CPU oracle for fused linear attention (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package.  The product path (the CUDA library and its Python binding)
never does.  The arithmetic lives in ``la_oracle.c`` (plain C, float64, recurrent
definition with hand-derived gradients); this module only compiles it with gcc and
marshals numpy arrays into it.

Parity: pinned.  The pins live in ``tests/test_oracle_pins.py`` (quadratic brute-force
definition, autograd of that definition, central finite differences, closed forms,
symmetries, the grouped-query expand/reduce rule) and ``tests/golden/`` (hand-derived
worked examples).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "la_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libla_oracle.so")

PHI = {"elu+1": 0, "relu": 1, "identity": 2}

_lock = threading.Lock()
_lib = None


def compile_source(src: str, out: str, extra_flags: list[str] | None = None) -> str:
    """Compile a C oracle source into a shared library with gcc (OpenMP on)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           src, "-o", out + ".tmp", "-lm"] + (extra_flags or [])
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


def build(force: bool = False) -> str:
    """Build ``libla_oracle.so`` next to this file if it is missing or stale."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        compile_source(_SRC, _LIB_PATH)
    return _LIB_PATH


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    dp = ctypes.POINTER(ctypes.c_double)
    i = ctypes.c_int
    lib.la_oracle_fwd.argtypes = [dp, dp, dp, dp, i, i, i, i, i, i, i, ctypes.c_double, dp, dp]
    lib.la_oracle_fwd.restype = None
    lib.la_oracle_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, i, i, i, i, i, i, i,
                                  ctypes.c_double, dp, dp]
    lib.la_oracle_bwd.restype = ctypes.c_int
    lib.la_oracle_fwd_v.argtypes = [dp, dp, dp, dp, i, i, i, i, i, i, i, i, ctypes.c_double, dp, dp]
    lib.la_oracle_fwd_v.restype = None
    lib.la_oracle_bwd_v.argtypes = [dp, dp, dp, dp, dp, dp, dp, i, i, i, i, i, i, i, i,
                                    ctypes.c_double, dp, dp]
    lib.la_oracle_bwd_v.restype = ctypes.c_int
    lib.la_oracle_num_threads.argtypes = []
    lib.la_oracle_num_threads.restype = ctypes.c_int
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the oracle library (building it first when needed).  ``path`` selects
    another build of an oracle source, e.g. a deliberately broken copy in a test."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def num_threads() -> int:
    return load().la_oracle_num_threads()


def _f64(x) -> np.ndarray:
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: widen exactly, on the CPU
        import torch
        x = x.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _check(q, k, v, cos_weight, sin_weight):
    """Shapes: q [B, Hq, N, D], k [B, Hkv, N, D], v [B, Hkv, N, Dv] (Dv may differ from D)."""
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be [B, H, N, D]")
    B, Hq, N, D = q.shape
    Bk, Hkv, Nk, Dk = k.shape
    if (Bk, Nk, Dk) != (B, N, D) or v.shape[:3] != k.shape[:3] or v.shape[3] < 1:
        raise ValueError("q, k, v shapes disagree")
    if Hkv <= 0 or Hq % Hkv != 0:
        raise ValueError("query heads must be a multiple of key/value heads")
    if (cos_weight is None) != (sin_weight is None):
        raise ValueError("give both position weights or neither")
    if cos_weight is not None and (cos_weight.shape != (N,) or sin_weight.shape != (N,)):
        raise ValueError("position weights must have length N")
    return B, Hq, Hkv, N, D, v.shape[3]


def fwd(q, k, v, is_causal: bool = False, phi: str = "elu+1", eps: float = 1e-6,
        cos_weight=None, sin_weight=None, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """Oracle forward: ``out`` as float64 [B, Hq, N, Dv]."""
    q, k, v, cw, sw = (_f64(x) for x in (q, k, v, cos_weight, sin_weight))
    B, Hq, Hkv, N, D, Dv = _check(q, k, v, cw, sw)
    out = np.empty((B, Hq, N, Dv), dtype=np.float64)
    (lib or load()).la_oracle_fwd_v(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, Hq, Hkv, N, D, Dv,
                                    int(bool(is_causal)), PHI[phi], float(eps), _ptr(cw), _ptr(sw))
    return out


def bwd(q, k, v, grad_out, is_causal: bool = False, phi: str = "elu+1", eps: float = 1e-6,
        cos_weight=None, sin_weight=None, lib: ctypes.CDLL | None = None):
    """Oracle backward: ``(dq, dk, dv)`` as float64; dk, dv have the key/value shape."""
    q, k, v, g, cw, sw = (_f64(x) for x in (q, k, v, grad_out, cos_weight, sin_weight))
    B, Hq, Hkv, N, D, Dv = _check(q, k, v, cw, sw)
    if g.shape != (B, Hq, N, Dv):
        raise ValueError("grad_out must have the shape of out ([B, Hq, N, Dv])")
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    rc = (lib or load()).la_oracle_bwd_v(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(dq), _ptr(dk),
                                         _ptr(dv), B, Hq, Hkv, N, D, Dv, int(bool(is_causal)), PHI[phi],
                                         float(eps), _ptr(cw), _ptr(sw))
    if rc != 0:
        raise MemoryError("oracle could not allocate its scratch arrays")
    return dq, dk, dv
