"""fp64 CPU oracle for the selective-scan linear recurrence.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The GPU library
never imports it and shares no code with it.

Contents
--------
``diag_scan`` / ``ssd_scan``
    The definition: a strictly sequential fp64 recurrence written in plain C
    (``ssm_oracle.c``), following ``selective_scan_seq`` and the shape API of
    "scan output is different between sequential and parallel versions"
    (mamba.py issue 26), and the bidirectional reading of "Some questions of
    Bi-Mamba2 and Hydra" (Bi-Mamba2 issue 1): a forward and a backward SSM
    with shared weights, summed, plus D x once.
``forms``
    Second and third forms of the same result (Blelloch up-sweep/down-sweep,
    chunkwise with carry, chunked SSD), used only to cross-check the
    definition, exactly as the pages compare their sequential, parallel and
    chunkwise forms.

Inputs are numpy arrays (any float dtype; they are upcast exactly to fp64).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_libs = {}


def compile_source(src: str, out: str) -> str:
    """Compile an oracle C source into a shared library with gcc (-O2, IEEE math)."""
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile ``ssm_oracle.c`` into ``liboracle.so``."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        compile_source(_SRC, _LIB)
    return _LIB


def _load(path: str | None = None):
    key = path or _LIB
    if key not in _libs:
        if path is None:
            build()
        lib = ctypes.CDLL(key)
        dp = ctypes.POINTER(ctypes.c_double)
        i64 = ctypes.c_int64
        lib.oracle_diag_scan_range.argtypes = [dp] * 7 + [i64] * 6 + [ctypes.c_int]
        lib.oracle_diag_scan_range.restype = None
        lib.oracle_ssd_scan_range.argtypes = [dp] * 7 + [i64] * 5 + [ctypes.c_int, i64, i64, ctypes.c_int]
        lib.oracle_ssd_scan_range.restype = None
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = ctypes.c_int
        _libs[key] = lib
    return _libs[key]


def max_threads() -> int:
    """Threads the OpenMP runtime will use by default (all host cores)."""
    return _load().oracle_max_threads()


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor -> numpy, exact upcast
        a = a.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def diag_scan(x, delta, A, B, C, D=None, nthreads: int = 0, channels=None, library=None):
    """Sequential diagonal selective scan in fp64.

    x, delta: (Bs, L, ED); A: (ED, N); B, C: (Bs, L, N); D: (ED) or None.
    Returns y: (Bs, L, ED) fp64.  ``channels=(c0, c1)`` computes only the
    flattened (b, e) channels in [c0, c1) (the rest of y is NaN); used to time
    a bounded sample.  ``library`` selects another compiled copy of the oracle
    (the tests use it to show that planted mistakes are caught).
    """
    x, delta, A, B, C, D = map(_f64, (x, delta, A, B, C, D))
    Bs, L, ED = x.shape
    N = A.shape[1]
    assert delta.shape == x.shape and A.shape == (ED, N)
    assert B.shape == (Bs, L, N) and C.shape == (Bs, L, N)
    assert D is None or D.shape == (ED,)
    y = np.full((Bs, L, ED), np.nan) if channels else np.zeros((Bs, L, ED))
    c0, c1 = channels if channels else (0, Bs * ED)
    _load(library).oracle_diag_scan_range(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                   _ptr(y), Bs, L, ED, N, c0, c1, nthreads)
    return y


def ssd_scan(x, dt, A_head, B, C, D=None, bidirectional: bool = False,
             nthreads: int = 0, units=None, library=None):
    """Sequential scalar-per-head (SSD) scan in fp64, optionally bidirectional.

    x: (Bs, L, H, P); dt: (Bs, L, H); A_head: (H); B, C: (Bs, L, N) or
    (Bs, L, 1, N) (one group shared by all heads); D: (H) or None.
    Returns y: (Bs, L, H, P) fp64.  ``units=(u0, u1)`` computes only the
    flattened (b, h) pairs in [u0, u1) (the rest of y is NaN).
    """
    x, dt, A_head, B, C, D = map(_f64, (x, dt, A_head, B, C, D))
    Bs, L, H, P = x.shape
    if B.ndim == 4:
        assert B.shape[2] == 1 and C.shape[2] == 1, "one group of B, C shared by all heads"
        B = np.ascontiguousarray(B[:, :, 0, :])
        C = np.ascontiguousarray(C[:, :, 0, :])
    N = B.shape[-1]
    assert dt.shape == (Bs, L, H) and A_head.shape == (H,)
    assert B.shape == (Bs, L, N) and C.shape == (Bs, L, N)
    assert D is None or D.shape == (H,)
    y = np.full((Bs, L, H, P), np.nan) if units else np.zeros((Bs, L, H, P))
    u0, u1 = units if units else (0, Bs * H)
    _load(library).oracle_ssd_scan_range(_ptr(x), _ptr(dt), _ptr(A_head), _ptr(B), _ptr(C), _ptr(D),
                                  _ptr(y), Bs, L, H, P, N, int(bool(bidirectional)), u0, u1, nthreads)
    return y
