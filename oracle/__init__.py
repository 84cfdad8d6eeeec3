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
        dbl = ctypes.c_double
        lib.oracle_diag_scan_ex_range.argtypes = ([dp] * 7 + [i64] * 4 + [dp, ctypes.c_int, ctypes.c_int,
                                                  dbl, dbl, dp, dp, dp, i64, i64, ctypes.c_int])
        lib.oracle_diag_scan_ex_range.restype = None
        lib.oracle_ssd_scan_ex_range.argtypes = ([dp] * 7 + [i64] * 6 + [ctypes.c_int, dp, ctypes.c_int,
                                                 ctypes.c_int, dbl, dbl, dp, dp, dp, i64, i64,
                                                 ctypes.c_int])
        lib.oracle_ssd_scan_ex_range.restype = None
        lib.oracle_diag_scan_bwd_range.argtypes = [dp] * 13 + [i64] * 6 + [ctypes.c_int]
        lib.oracle_diag_scan_bwd_range.restype = None
        lib.oracle_ssd_scan_bwd.argtypes = [dp] * 13 + [i64] * 6 + [ctypes.c_int, ctypes.c_int]
        lib.oracle_ssd_scan_bwd.restype = None
        lib.oracle_ssd_scan_bwd_ex.argtypes = ([dp] * 13 + [i64] * 6 + [ctypes.c_int, dp, ctypes.c_int,
                                               ctypes.c_int, dbl, dbl, dp, dp, dp, dp, dp,
                                               ctypes.c_int])
        lib.oracle_ssd_scan_bwd_ex.restype = None
        lib.oracle_diag_scan_bwd_ex.argtypes = ([dp] * 13 + [i64] * 4 + [dp, ctypes.c_int, ctypes.c_int,
                                                dbl, dbl, dp, dp, dp, dp, dp, ctypes.c_int])
        lib.oracle_diag_scan_bwd_ex.restype = None
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


def _limit(dt_limit):
    if dt_limit is None:
        return 0, 0.0, 0.0
    lo, hi = dt_limit
    return 1, float(lo), float(hi)


def diag_scan(x, delta, A, B, C, D=None, nthreads: int = 0, channels=None, library=None,
              dt_bias=None, dt_softplus: bool = False, dt_limit=None, z=None, h0=None,
              return_final_state: bool = False):
    """Sequential diagonal selective scan in fp64.

    x, delta: (Bs, L, ED); A: (ED, N); B, C: (Bs, L, N); D: (ED) or None.
    Returns y: (Bs, L, ED) fp64.  ``channels=(c0, c1)`` computes only the
    flattened (b, e) channels in [c0, c1) (the rest of y is NaN); used to time
    a bounded sample.  ``library`` selects another compiled copy of the oracle
    (the tests use it to show that planted mistakes are caught).

    Options (argument list of the chunked scan in "Some questions of
    Bi-Mamba2 and Hydra"): ``dt_bias`` (ED) is added to delta, then
    ``dt_softplus`` applies log(1 + exp(.)), then ``dt_limit=(lo, hi)`` clamps;
    ``z`` (Bs, L, ED) gates the output with silu(z); ``h0`` (Bs, ED, N) is the
    initial state; ``return_final_state`` also returns h_{L-1} (Bs, ED, N).
    """
    x, delta, A, B, C, D, dt_bias, z, h0 = map(_f64, (x, delta, A, B, C, D, dt_bias, z, h0))
    Bs, L, ED = x.shape
    N = A.shape[1]
    assert delta.shape == x.shape and A.shape == (ED, N)
    assert B.shape == (Bs, L, N) and C.shape == (Bs, L, N)
    assert D is None or D.shape == (ED,)
    assert dt_bias is None or dt_bias.shape == (ED,)
    assert z is None or z.shape == x.shape
    assert h0 is None or h0.shape == (Bs, ED, N)
    y = np.full((Bs, L, ED), np.nan) if channels else np.zeros((Bs, L, ED))
    hf = np.zeros((Bs, ED, N)) if return_final_state else None
    c0, c1 = channels if channels else (0, Bs * ED)
    lim, lo, hi = _limit(dt_limit)
    _load(library).oracle_diag_scan_ex_range(
        _ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(y), Bs, L, ED, N,
        _ptr(dt_bias), int(bool(dt_softplus)), lim, lo, hi, _ptr(z), _ptr(h0), _ptr(hf), c0, c1,
        nthreads)
    return (y, hf) if return_final_state else y


def diag_scan_bwd(x, delta, A, B, C, D, dy, nthreads: int = 0, library=None):
    """Gradients of the diagonal scan in fp64 (reverse mode written out by hand).

    Same inputs as ``diag_scan`` plus dy (Bs, L, ED), the gradient of the loss
    with respect to y.  Returns dict(dx, ddelta, dA, dB, dC, dD) shaped like
    x, delta, A, B, C, D (dD is None when D is None).
    """
    x, delta, A, B, C, D, dy = map(_f64, (x, delta, A, B, C, D, dy))
    Bs, L, ED = x.shape
    N = A.shape[1]
    assert delta.shape == x.shape and dy.shape == x.shape and A.shape == (ED, N)
    assert B.shape == (Bs, L, N) and C.shape == (Bs, L, N)
    out = dict(dx=np.zeros((Bs, L, ED)), ddelta=np.zeros((Bs, L, ED)), dA=np.zeros((ED, N)),
               dB=np.zeros((Bs, L, N)), dC=np.zeros((Bs, L, N)),
               dD=None if D is None else np.zeros(ED))
    _load(library).oracle_diag_scan_bwd_range(
        _ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(dy), _ptr(out["dx"]),
        _ptr(out["ddelta"]), _ptr(out["dA"]), _ptr(out["dB"]), _ptr(out["dC"]), _ptr(out["dD"]),
        Bs, L, ED, N, 0, Bs * ED, nthreads)
    return out


def diag_scan_bwd_ex(x, delta, A, B, C, D, dy, dt_bias=None, dt_softplus: bool = False,
                     dt_limit=None, z=None, h0=None, nthreads: int = 0, library=None):
    """Gradients of the diagonal scan with its options, in fp64.

    Inputs as in ``diag_scan`` with the options (``delta`` before the
    optional bias, softplus and clamp; gate ``z``; initial state ``h0``)
    plus dy.  Returns the keys of ``diag_scan_bwd`` and dz (like x),
    ddt_bias (ED), dh0 (Bs, ED, N) -- each None when its option is off;
    ddelta is the gradient with respect to the delta given.
    """
    x, delta, A, B, C, D, dy, dt_bias, z, h0 = map(
        _f64, (x, delta, A, B, C, D, dy, dt_bias, z, h0))
    Bs, L, ED = x.shape
    N = A.shape[1]
    assert delta.shape == x.shape and dy.shape == x.shape and A.shape == (ED, N)
    assert B.shape == (Bs, L, N) and C.shape == (Bs, L, N)
    assert dt_bias is None or dt_bias.shape == (ED,)
    assert z is None or z.shape == x.shape
    assert h0 is None or h0.shape == (Bs, ED, N)
    out = dict(dx=np.zeros((Bs, L, ED)), ddelta=np.zeros((Bs, L, ED)), dA=np.zeros((ED, N)),
               dB=np.zeros((Bs, L, N)), dC=np.zeros((Bs, L, N)),
               dD=None if D is None else np.zeros(ED),
               dz=None if z is None else np.zeros((Bs, L, ED)),
               ddt_bias=None if dt_bias is None else np.zeros(ED),
               dh0=None if h0 is None else np.zeros((Bs, ED, N)))
    lim, lo, hi = _limit(dt_limit)
    _load(library).oracle_diag_scan_bwd_ex(
        _ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(dy), _ptr(out["dx"]),
        _ptr(out["ddelta"]), _ptr(out["dA"]), _ptr(out["dB"]), _ptr(out["dC"]), _ptr(out["dD"]),
        Bs, L, ED, N, _ptr(dt_bias), int(bool(dt_softplus)), lim, lo, hi, _ptr(z), _ptr(h0),
        _ptr(out["dz"]), _ptr(out["ddt_bias"]), _ptr(out["dh0"]), nthreads)
    return out


def ssd_scan(x, dt, A_head, B, C, D=None, bidirectional: bool = False,
             nthreads: int = 0, units=None, library=None, dt_bias=None,
             dt_softplus: bool = False, dt_limit=None, z=None, h0=None,
             return_final_state: bool = False):
    """Sequential scalar-per-head (SSD) scan in fp64, optionally bidirectional.

    x: (Bs, L, H, P); dt: (Bs, L, H); A_head: (H); B, C: (Bs, L, N) (one
    group shared by all heads) or (Bs, L, G, N) with G dividing H (head h
    reads group h // (H // G)); D: (H) or None.
    Returns y: (Bs, L, H, P) fp64.  ``units=(u0, u1)`` computes only the
    flattened (b, h) pairs in [u0, u1) (the rest of y is NaN).
    Options as in ``diag_scan``, per head: ``dt_bias`` (H), ``z`` (Bs, L, H, P),
    ``h0`` and the final state (Bs, H, P, N) -- state I/O for a single
    direction only.
    """
    x, dt, A_head, B, C, D, dt_bias, z, h0 = map(_f64, (x, dt, A_head, B, C, D, dt_bias, z, h0))
    Bs, L, H, P = x.shape
    if B.ndim == 3:
        B, C = B[:, :, None, :], C[:, :, None, :]
    G, N = B.shape[2], B.shape[3]
    assert G >= 1 and H % G == 0, "heads must split evenly into the groups of B, C"
    assert dt.shape == (Bs, L, H) and A_head.shape == (H,)
    assert B.shape == (Bs, L, G, N) and C.shape == (Bs, L, G, N)
    B, C = np.ascontiguousarray(B), np.ascontiguousarray(C)
    assert D is None or D.shape == (H,)
    assert dt_bias is None or dt_bias.shape == (H,)
    assert z is None or z.shape == x.shape
    assert h0 is None or h0.shape == (Bs, H, P, N)
    if bidirectional and (h0 is not None or return_final_state):
        raise ValueError("state input/output is defined for a single direction only")
    y = np.full((Bs, L, H, P), np.nan) if units else np.zeros((Bs, L, H, P))
    hf = np.zeros((Bs, H, P, N)) if return_final_state else None
    u0, u1 = units if units else (0, Bs * H)
    lim, lo, hi = _limit(dt_limit)
    _load(library).oracle_ssd_scan_ex_range(
        _ptr(x), _ptr(dt), _ptr(A_head), _ptr(B), _ptr(C), _ptr(D), _ptr(y), Bs, L, H, P, N, G,
        int(bool(bidirectional)), _ptr(dt_bias), int(bool(dt_softplus)), lim, lo, hi, _ptr(z),
        _ptr(h0), _ptr(hf), u0, u1, nthreads)
    return (y, hf) if return_final_state else y


def ssd_scan_bwd(x, dt, A_head, B, C, D, dy, bidirectional: bool = False, nthreads: int = 0,
                 library=None):
    """Gradients of the SSD scan in fp64 (reverse mode written out by hand).

    Same inputs as ``ssd_scan`` (no options) plus dy (Bs, L, H, P), the
    gradient of the loss with respect to y.  Returns dict(dx, ddt, dA, dB, dC,
    dD) shaped like x, dt, A_head, B, C (as given: (Bs, L, N) or
    (Bs, L, G, N)), D (dD is None when D is None).
    """
    x, dt, A_head, B, C, D, dy = map(_f64, (x, dt, A_head, B, C, D, dy))
    Bs, L, H, P = x.shape
    shape_bc = B.shape
    if B.ndim == 3:
        B, C = B[:, :, None, :], C[:, :, None, :]
    G, N = B.shape[2], B.shape[3]
    assert G >= 1 and H % G == 0, "heads must split evenly into the groups of B, C"
    assert dt.shape == (Bs, L, H) and A_head.shape == (H,) and dy.shape == x.shape
    assert B.shape == (Bs, L, G, N) and C.shape == (Bs, L, G, N)
    B, C = np.ascontiguousarray(B), np.ascontiguousarray(C)
    assert D is None or D.shape == (H,)
    out = dict(dx=np.zeros((Bs, L, H, P)), ddt=np.zeros((Bs, L, H)), dA=np.zeros(H),
               dB=np.zeros((Bs, L, G, N)), dC=np.zeros((Bs, L, G, N)),
               dD=None if D is None else np.zeros(H))
    _load(library).oracle_ssd_scan_bwd(
        _ptr(x), _ptr(dt), _ptr(A_head), _ptr(B), _ptr(C), _ptr(D), _ptr(dy), _ptr(out["dx"]),
        _ptr(out["ddt"]), _ptr(out["dA"]), _ptr(out["dB"]), _ptr(out["dC"]), _ptr(out["dD"]),
        Bs, L, H, P, N, G, int(bool(bidirectional)), nthreads)
    out["dB"] = out["dB"].reshape(shape_bc)
    out["dC"] = out["dC"].reshape(shape_bc)
    return out


def ssd_scan_bwd_ex(x, dt, A_head, B, C, D, dy, bidirectional: bool = False, dt_bias=None,
                    dt_softplus: bool = False, dt_limit=None, z=None, h0=None, nthreads: int = 0,
                    library=None):
    """Gradients of the SSD scan with its options, in fp64.

    Inputs as in ``ssd_scan`` with the options (``dt`` before the optional
    bias, softplus and clamp; gate ``z``; initial state ``h0``, single
    direction only) plus dy.  Returns the keys of ``ssd_scan_bwd`` and
    dz (like x), ddt_bias (H), dh0 (Bs, H, P, N) -- each None when its option
    is off; ddt is the gradient with respect to the dt given.
    """
    x, dt, A_head, B, C, D, dy, dt_bias, z, h0 = map(
        _f64, (x, dt, A_head, B, C, D, dy, dt_bias, z, h0))
    Bs, L, H, P = x.shape
    shape_bc = B.shape
    if B.ndim == 3:
        B, C = B[:, :, None, :], C[:, :, None, :]
    G, N = B.shape[2], B.shape[3]
    assert G >= 1 and H % G == 0, "heads must split evenly into the groups of B, C"
    assert dt.shape == (Bs, L, H) and A_head.shape == (H,) and dy.shape == x.shape
    assert B.shape == (Bs, L, G, N) and C.shape == (Bs, L, G, N)
    B, C = np.ascontiguousarray(B), np.ascontiguousarray(C)
    assert D is None or D.shape == (H,)
    assert dt_bias is None or dt_bias.shape == (H,)
    assert z is None or z.shape == x.shape
    assert h0 is None or h0.shape == (Bs, H, P, N)
    if bidirectional and h0 is not None:
        raise ValueError("state input is defined for a single direction only")
    out = dict(dx=np.zeros((Bs, L, H, P)), ddt=np.zeros((Bs, L, H)), dA=np.zeros(H),
               dB=np.zeros((Bs, L, G, N)), dC=np.zeros((Bs, L, G, N)),
               dD=None if D is None else np.zeros(H),
               dz=None if z is None else np.zeros((Bs, L, H, P)),
               ddt_bias=None if dt_bias is None else np.zeros(H),
               dh0=None if h0 is None else np.zeros((Bs, H, P, N)))
    lim, lo, hi = _limit(dt_limit)
    _load(library).oracle_ssd_scan_bwd_ex(
        _ptr(x), _ptr(dt), _ptr(A_head), _ptr(B), _ptr(C), _ptr(D), _ptr(dy), _ptr(out["dx"]),
        _ptr(out["ddt"]), _ptr(out["dA"]), _ptr(out["dB"]), _ptr(out["dC"]), _ptr(out["dD"]),
        Bs, L, H, P, N, G, int(bool(bidirectional)), _ptr(dt_bias), int(bool(dt_softplus)), lim,
        lo, hi, _ptr(z), _ptr(h0), _ptr(out["dz"]), _ptr(out["ddt_bias"]), _ptr(out["dh0"]),
        nthreads)
    out["dB"] = out["dB"].reshape(shape_bc)
    out["dC"] = out["dC"].reshape(shape_bc)
    return out
