"""ctypes front end of the fp64 KDA oracle (``kda_oracle.c``).

TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's
CPU-baseline leg may import this module; the library path never does.  It
shares no code with the CUDA path: it compiles its own C file with gcc and
computes the recurrence token by token in fp64 (see the header of
``kda_oracle.c`` for the five steps and the passages they follow).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compiles the oracle C file into a shared library and returns its path."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def load(path: str | None = None) -> ctypes.CDLL:
    """Loads (building first if needed) the oracle library."""
    global _lib
    with _lock:
        if path is not None:
            lib = ctypes.CDLL(path)
        elif _lib is not None:
            return _lib
        else:
            lib = ctypes.CDLL(build())
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int32)
        i32 = ctypes.c_int32
        lib.kda_oracle_run.restype = ctypes.c_int
        lib.kda_oracle_run.argtypes = [dp, dp, dp, dp, dp, ip, i32, i32, i32, i32,
                                       dp, dp, dp, i32, ip, dp, i32]
        if path is None:
            _lib = lib
        return lib


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a, ctype):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctype))


def run(q, k, v, g, beta, cu_seqlens, S0=None, snap_t=None, threads: int | None = None, lib=None):
    """Token-by-token KDA recurrence in fp64.

    Shapes: q, k, g ``[T, H, dk]``; v ``[T, H, dv]``; beta ``[T, H]``;
    cu_seqlens ``[N + 1]``; S0 ``[N, H, dk, dv]`` or None (zeros).
    Returns ``(o [T, H, dv], S_final [N, H, dk, dv], S_snap)`` where S_snap
    is ``[len(snap_t), N, H, dk, dv]`` (NaN where a sequence is shorter than
    the requested count) or None.
    """
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    T, H, dk = q.shape
    dv = v.shape[2]
    N = cu.shape[0] - 1
    assert k.shape == (T, H, dk) and g.shape == (T, H, dk)
    assert v.shape == (T, H, dv) and beta.shape == (T, H)
    s0 = None if S0 is None else _f64(S0)
    if s0 is not None:
        assert s0.shape == (N, H, dk, dv)
    o = np.zeros((T, H, dv), dtype=np.float64)
    S_final = np.zeros((N, H, dk, dv), dtype=np.float64)
    n_snap = 0
    snaps = None
    snap_arr = None
    if snap_t is not None and len(snap_t) > 0:
        snap_arr = np.ascontiguousarray(np.asarray(snap_t, dtype=np.int32))
        n_snap = snap_arr.shape[0]
        snaps = np.full((n_snap, N, H, dk, dv), np.nan, dtype=np.float64)
    lib = lib or load()
    rc = lib.kda_oracle_run(_ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double), _ptr(v, ctypes.c_double),
                            _ptr(g, ctypes.c_double), _ptr(beta, ctypes.c_double), _ptr(cu, ctypes.c_int32),
                            N, H, dk, dv, _ptr(s0, ctypes.c_double), _ptr(o, ctypes.c_double),
                            _ptr(S_final, ctypes.c_double), n_snap, _ptr(snap_arr, ctypes.c_int32),
                            _ptr(snaps, ctypes.c_double), int(threads or default_threads()))
    if rc != 0:
        raise ValueError("kda_oracle_run failed with code %d" % rc)
    return o, S_final, snaps


def rel_err(x, ref) -> float:
    """max|x - ref| / max|ref| (the tolerance metric of the parity contract)."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    denom = float(np.max(np.abs(ref))) if ref.size else 0.0
    num = float(np.max(np.abs(x - ref))) if ref.size else 0.0
    if denom == 0.0:
        return num
    return num / denom
