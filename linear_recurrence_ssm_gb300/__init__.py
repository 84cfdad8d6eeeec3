"""GB300-native selective-scan linear recurrence: a thin Python binding of
libssmscan.so (C ABI declared in include/ssm_scan.h).

Every call marshals torch CUDA tensors into raw device pointers plus the
current CUDA stream and calls the C entry point of the same name; all of the
computation runs in the library's sm_103a kernels.  There is no fallback: if
the library is missing or fails to load, importing a function raises.

Functions
---------
ssm_scan_fwd(x, delta, A, B, C, D=None, y=None, **options)
    Diagonal-A selective scan (shape API of selective_scan in "scan output is
    different between sequential and parallel versions", mamba.py issue 26).
    x, delta: (Bs, L, ED); A: (ED, N) fp32; B, C: (Bs, L, N); D: (ED) fp32.
    fp32 inputs call the C ``ssm_scan_fwd``; bf16 inputs call
    ``ssm_scan_fwd_bf16``.  Returns y (Bs, L, ED) fp32.
ssd_chunk_scan_fwd(x, dt, A_head, B, C, D=None, chunk=256, bidirectional=False, y=None, **options)
    Chunked scalar-decay scan ("Some questions of Bi-Mamba2 and Hydra",
    Bi-Mamba2 issue 1).  x: (Bs, L, H, P) bf16 or fp32; dt: (Bs, L, H), same type;
    A_head: (H) fp32; B, C: (Bs, L, N) or (Bs, L, G, N) bf16 (head h reads
    group h // (H // G)); D: (H) fp32.  Returns y (Bs, L, H, P) fp32.

Options (either function; any of them selects the ``*_ex`` C entry point):
``dt_bias`` (ED or H, fp32), ``dt_softplus``, ``dt_limit=(lo, hi)``, ``z``
(shaped and typed like x), ``h0`` (fp32 initial state, (Bs, ED, N) or
(Bs, H, P, N)) and ``return_final_state`` (the call then returns
``(y, h_final)``).
"""
from __future__ import annotations

import ctypes
import os

from . import _build

__all__ = ["ssm_scan_fwd", "ssm_scan_fwd_bf16", "ssd_chunk_scan_fwd", "ssm_check_device_errors",
           "ssm_scan_fwd_plan", "ssm_scan_bwd", "ssd_chunk_scan_bwd", "ScanOptions",
           "SsmError", "library", "build", "status_string", "STATUS"]

STATUS = {
    0: "SSM_OK", 1: "SSM_ERR_INVALID_ARG", 2: "SSM_ERR_UNSUPPORTED", 3: "SSM_ERR_ALIGNMENT",
    4: "SSM_ERR_CUDA", 5: "SSM_ERR_DEVICE_TIMEOUT", 6: "SSM_ERR_NO_DEVICE",
}

# Every symbol include/ssm_scan.h declares, with its ctypes signature.
_VP = ctypes.c_void_p
_I64 = ctypes.c_int64
SIGNATURES = {
    "ssm_scan_fwd": ([_VP] * 7 + [_I64] * 4 + [_VP], ctypes.c_int),
    "ssm_scan_fwd_bf16": ([_VP] * 7 + [_I64] * 4 + [_VP], ctypes.c_int),
    "ssd_chunk_scan_fwd": ([_VP] * 7 + [_I64] * 6 + [ctypes.c_int, _VP], ctypes.c_int),
    "ssd_chunk_scan_fwd_noalloc": ([_VP] * 7 + [_I64] * 6 + [ctypes.c_int, _VP], ctypes.c_int),
    "ssm_scan_fwd_plan": ([_I64] * 4 + [ctypes.c_int] + [ctypes.POINTER(ctypes.c_int32)] * 3,
                          ctypes.c_int),
    "ssm_scan_fwd_ex": ([_VP] * 7 + [_I64] * 4 + [ctypes.c_int, _VP, _VP], ctypes.c_int),
    "ssm_scan_bwd": ([_VP] * 13 + [_I64] * 4 + [ctypes.c_int, _VP], ctypes.c_int),
    "ssd_chunk_scan_bwd": ([_VP] * 13 + [_I64] * 6 + [ctypes.c_int, ctypes.c_int, _VP], ctypes.c_int),
    "ssm_scan_bwd_ex": ([_VP] * 16 + [_I64] * 4 + [ctypes.c_int, _VP, _VP], ctypes.c_int),
    "ssd_chunk_scan_bwd_ex": ([_VP] * 16 + [_I64] * 5 + [ctypes.c_int, ctypes.c_int, _VP, _VP],
                              ctypes.c_int),
    "ssd_chunk_scan_fwd_ex": ([_VP] * 7 + [_I64] * 6 + [ctypes.c_int, ctypes.c_int, _VP, _VP],
                              ctypes.c_int),
    "ssm_check_device_errors": ([_VP], ctypes.c_int),
    "ssm_selftest_wait_timeout": ([_VP], ctypes.c_int),
    "ssm_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "ssm_version": ([], ctypes.c_int),
}

_lib = None


class ScanOptions(ctypes.Structure):
    """ssm_scan_options_t of include/ssm_scan.h."""
    _fields_ = [("dt_bias", _VP), ("dt_softplus", ctypes.c_int32), ("dt_limit", ctypes.c_int32),
                ("dt_min", ctypes.c_float), ("dt_max", ctypes.c_float), ("z", _VP),
                ("h0", _VP), ("h_final", _VP), ("ngroups", ctypes.c_int32)]


_OPTION_KEYS = ("dt_bias", "dt_softplus", "dt_limit", "z", "h0", "return_final_state")


def _options(x, channels, state_shape, dev, dt_bias=None, dt_softplus=False, dt_limit=None,
             z=None, h0=None, return_final_state=False, ngroups=1):
    """Validate the options and build (ScanOptions, h_final tensor or None, keep-alive list)."""
    import torch
    o = ScanOptions()
    keep = []
    if dt_bias is not None:
        _check(dt_bias, "dt_bias", (torch.float32,), dev, (1,))
        if dt_bias.shape[0] != channels:
            raise ValueError("dt_bias must have %d entries" % channels)
        o.dt_bias = dt_bias.data_ptr()
        keep.append(dt_bias)
    o.dt_softplus = 1 if dt_softplus else 0
    if dt_limit is not None:
        o.dt_limit = 1
        o.dt_min, o.dt_max = float(dt_limit[0]), float(dt_limit[1])
    if z is not None:
        _check(z, "z", (x.dtype,), dev)
        if z.shape != x.shape:
            raise ValueError("z must have the shape of x")
        o.z = z.data_ptr()
        keep.append(z)
    if h0 is not None:
        _check(h0, "h0", (torch.float32,), dev)
        if tuple(h0.shape) != tuple(state_shape):
            raise ValueError("h0 must have shape %s" % (tuple(state_shape),))
        o.h0 = h0.data_ptr()
        keep.append(h0)
    o.ngroups = int(ngroups)
    hf = None
    if return_final_state:
        hf = torch.empty(state_shape, dtype=torch.float32, device=dev)
        o.h_final = hf.data_ptr()
    return o, hf, keep


class SsmError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__("%s failed: %s" % (fn, status_string(status)))


def build(force: bool = False) -> str:
    """Compile libssmscan.so in-tree (nvcc, sm_103a)."""
    return _build.build(force=force)


def library() -> ctypes.CDLL:
    """The loaded C library (built first if its sources are newer)."""
    global _lib
    if _lib is None:
        path = _build.LIB_PATH
        if _build.needs_build():
            _build.build()
        if not os.path.exists(path):
            raise RuntimeError("libssmscan.so is missing and could not be built")
        lib = ctypes.CDLL(path)
        for name, (argtypes, restype) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = argtypes
            fn.restype = restype
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    return library().ssm_status_string(int(status)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(dev):
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _check(t, name, dtypes, dev, ndim=None):
    import torch
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.device != dev:
        raise ValueError("%s is on %s, expected %s" % (name, t.device, dev))
    if t.dtype not in dtypes:
        raise TypeError("%s has dtype %s, expected one of %s" % (name, t.dtype, dtypes))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if ndim is not None and t.dim() not in ndim:
        raise ValueError("%s must have %s dims, got %d" % (name, ndim, t.dim()))


def ssm_scan_fwd(x, delta, A, B, C, D=None, y=None, **options):
    """Diagonal selective scan on the current CUDA stream; returns y (fp32),
    or (y, h_final) with ``return_final_state=True``."""
    import torch
    dev = x.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    ins = (torch.float32, torch.bfloat16)
    for t, n in ((x, "x"), (delta, "delta"), (B, "B"), (C, "C")):
        _check(t, n, (x.dtype,) if x.dtype in ins else ins, dev, (3,))
    _check(A, "A", (torch.float32,), dev, (2,))
    _check(D, "D", (torch.float32,), dev, (1,))
    Bs, L, ED = x.shape
    N = A.shape[1]
    if delta.shape != x.shape or tuple(A.shape) != (ED, N) or tuple(B.shape) != (Bs, L, N) \
            or tuple(C.shape) != (Bs, L, N) or (D is not None and tuple(D.shape) != (ED,)):
        raise ValueError("shape mismatch: x, delta (Bs,L,ED); A (ED,N); B, C (Bs,L,N); D (ED)")
    if y is None:
        y = torch.empty((Bs, L, ED), dtype=torch.float32, device=dev)
    _check(y, "y", (torch.float32,), dev, (3,))
    bad = set(options) - set(_OPTION_KEYS)
    if bad:
        raise TypeError("unknown options: %s" % sorted(bad))
    if options:
        o, hf, keep = _options(x, ED, (Bs, ED, N), dev, **options)
        st = library().ssm_scan_fwd_ex(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                                       _ptr(y), Bs, L, ED, N, int(x.dtype == torch.bfloat16),
                                       ctypes.byref(o), _stream(dev))
        if st != 0:
            raise SsmError("ssm_scan_fwd_ex", st)
        return (y, hf) if options.get("return_final_state") else y
    name = "ssm_scan_fwd" if x.dtype == torch.float32 else "ssm_scan_fwd_bf16"
    fn = getattr(library(), name)
    st = fn(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(y),
            Bs, L, ED, N, _stream(dev))
    if st != 0:
        raise SsmError(name, st)
    return y


def ssm_scan_fwd_bf16(x, delta, A, B, C, D=None, y=None, **options):
    """Same as ``ssm_scan_fwd`` but requires bf16 x, delta, B, C."""
    import torch
    if x.dtype != torch.bfloat16:
        raise TypeError("ssm_scan_fwd_bf16 takes bf16 x, delta, B, C")
    return ssm_scan_fwd(x, delta, A, B, C, D, y, **options)


def ssd_chunk_scan_fwd(x, dt, A_head, B, C, D=None, chunk: int = 256,
                       bidirectional: bool = False, y=None, **options):
    """Chunked scalar-decay scan on the current CUDA stream; returns y (fp32),
    or (y, h_final) with ``return_final_state=True``."""
    import torch
    dev = x.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    if x.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("x must be bf16 or fp32")
    bf = (x.dtype,)
    _check(x, "x", bf, dev, (4,))
    _check(dt, "dt", bf, dev, (3,))
    _check(B, "B", bf, dev, (3, 4))
    _check(C, "C", bf, dev, (3, 4))
    _check(A_head, "A_head", (torch.float32,), dev, (1,))
    _check(D, "D", (torch.float32,), dev, (1,))
    Bs, L, H, P = x.shape
    G = B.shape[2] if B.dim() == 4 else 1
    if B.dim() == 4 and (C.dim() != 4 or C.shape[2] != G or H % G != 0):
        raise ValueError("B, C must be (Bs, L, G, N) with G dividing H")
    N = B.shape[-1]
    if tuple(dt.shape) != (Bs, L, H) or tuple(A_head.shape) != (H,) \
            or B.shape[0] != Bs or B.shape[1] != L or tuple(C.shape) != tuple(B.shape) \
            or (D is not None and tuple(D.shape) != (H,)):
        raise ValueError("shape mismatch: x (Bs,L,H,P); dt (Bs,L,H); A_head (H); B, C (Bs,L,[G,]N)")
    if y is None:
        y = torch.empty((Bs, L, H, P), dtype=torch.float32, device=dev)
    _check(y, "y", (torch.float32,), dev, (4,))
    bad = set(options) - set(_OPTION_KEYS)
    if bad:
        raise TypeError("unknown options: %s" % sorted(bad))
    if G > 1:
        options = dict(options, ngroups=G)
    if options or x.dtype != torch.bfloat16:
        o, hf, keep = _options(x, H, (Bs, H, P, N), dev, **options)
        st = library().ssd_chunk_scan_fwd_ex(_ptr(x), _ptr(dt), _ptr(A_head), _ptr(B), _ptr(C),
                                             _ptr(D), _ptr(y), Bs, L, H, P, N, int(chunk),
                                             int(bool(bidirectional)),
                                             int(x.dtype == torch.bfloat16), ctypes.byref(o),
                                             _stream(dev))
        if st != 0:
            raise SsmError("ssd_chunk_scan_fwd_ex", st)
        return (y, hf) if options.get("return_final_state") else y
    st = library().ssd_chunk_scan_fwd(_ptr(x), _ptr(dt), _ptr(A_head), _ptr(B), _ptr(C), _ptr(D),
                                      _ptr(y), Bs, L, H, P, N, int(chunk), int(bool(bidirectional)),
                                      _stream(dev))
    if st != 0:
        raise SsmError("ssd_chunk_scan_fwd", st)
    return y


def ssm_scan_bwd(x, delta, A, B, C, D, dy, **options):
    """Gradients of the diagonal scan for the upstream gradient dy (fp32,
    shaped like y): dict(dx, ddelta, dA, dB, dC, dD) as fp32 tensors (dD is
    None when D is None).  With the forward scan's options (dt_bias,
    dt_softplus, dt_limit, z, h0) the dict also holds dz, ddt_bias and dh0
    (None when the matching option is off), and ddelta is the gradient with
    respect to delta before the options."""
    import torch
    dev = x.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    ins = (torch.float32, torch.bfloat16)
    for t, n in ((x, "x"), (delta, "delta"), (B, "B"), (C, "C")):
        _check(t, n, (x.dtype,) if x.dtype in ins else ins, dev, (3,))
    _check(A, "A", (torch.float32,), dev, (2,))
    _check(D, "D", (torch.float32,), dev, (1,))
    _check(dy, "dy", (torch.float32,), dev, (3,))
    Bs, L, ED = x.shape
    N = A.shape[1]
    if delta.shape != x.shape or dy.shape != x.shape or tuple(A.shape) != (ED, N) \
            or tuple(B.shape) != (Bs, L, N) or tuple(C.shape) != (Bs, L, N):
        raise ValueError("shape mismatch: x, delta, dy (Bs,L,ED); A (ED,N); B, C (Bs,L,N)")
    f32 = dict(dtype=torch.float32, device=dev)
    g = dict(dx=torch.empty((Bs, L, ED), **f32), ddelta=torch.empty((Bs, L, ED), **f32),
             dA=torch.empty((ED, N), **f32), dB=torch.empty((Bs, L, N), **f32),
             dC=torch.empty((Bs, L, N), **f32), dD=None if D is None else torch.empty(ED, **f32))
    bad = set(options) - (set(_OPTION_KEYS) - {"return_final_state"})
    if bad:
        raise TypeError("unknown options: %s" % sorted(bad))
    if options:
        o, _, keep = _options(x, ED, (Bs, ED, N), dev, **options)
        g["dz"] = torch.empty((Bs, L, ED), **f32) if options.get("z") is not None else None
        g["ddt_bias"] = torch.empty(ED, **f32) if options.get("dt_bias") is not None else None
        g["dh0"] = torch.empty((Bs, ED, N), **f32) if options.get("h0") is not None else None
        st = library().ssm_scan_bwd_ex(
            _ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(dy), _ptr(g["dx"]),
            _ptr(g["ddelta"]), _ptr(g["dA"]), _ptr(g["dB"]), _ptr(g["dC"]), _ptr(g["dD"]),
            _ptr(g["dz"]), _ptr(g["ddt_bias"]), _ptr(g["dh0"]), Bs, L, ED, N,
            int(x.dtype == torch.bfloat16), ctypes.byref(o), _stream(dev))
        if st != 0:
            raise SsmError("ssm_scan_bwd_ex", st)
        return g
    st = library().ssm_scan_bwd(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(dy),
                                _ptr(g["dx"]), _ptr(g["ddelta"]), _ptr(g["dA"]), _ptr(g["dB"]),
                                _ptr(g["dC"]), _ptr(g["dD"]), Bs, L, ED, N,
                                int(x.dtype == torch.bfloat16), _stream(dev))
    if st != 0:
        raise SsmError("ssm_scan_bwd", st)
    return g


def ssd_chunk_scan_bwd(x, dt, A_head, B, C, D, dy, bidirectional: bool = False, **options):
    """Gradients of the chunked scan for the upstream gradient dy (fp32,
    shaped like y): dict(dx, ddt, dA, dB, dC, dD) as fp32 tensors (dB, dC
    shaped like B, C; dD is None when D is None).  With the forward scan's
    options (dt_bias, dt_softplus, dt_limit, z, h0) the dict also holds dz,
    ddt_bias and dh0 (None when the matching option is off), and ddt is the
    gradient with respect to dt before the options."""
    import torch
    dev = x.device
    if dev.type != "cuda":
        raise ValueError("inputs must be CUDA tensors")
    ins = (torch.float32, torch.bfloat16)
    _check(x, "x", ins, dev, (4,))
    _check(dt, "dt", (x.dtype,), dev, (3,))
    _check(B, "B", (x.dtype,), dev, (3, 4))
    _check(C, "C", (x.dtype,), dev, (3, 4))
    _check(A_head, "A_head", (torch.float32,), dev, (1,))
    _check(D, "D", (torch.float32,), dev, (1,))
    _check(dy, "dy", (torch.float32,), dev, (4,))
    Bs, L, H, P = x.shape
    G = 1 if B.dim() == 3 else B.shape[2]
    N = B.shape[-1]
    bc = (Bs, L, N) if B.dim() == 3 else (Bs, L, G, N)
    if tuple(dt.shape) != (Bs, L, H) or tuple(A_head.shape) != (H,) or dy.shape != x.shape \
            or tuple(B.shape) != bc or tuple(C.shape) != bc:
        raise ValueError("shape mismatch: x, dy (Bs,L,H,P); dt (Bs,L,H); A_head (H); "
                         "B, C (Bs,L,N) or (Bs,L,G,N)")
    f32 = dict(dtype=torch.float32, device=dev)
    g = dict(dx=torch.empty((Bs, L, H, P), **f32), ddt=torch.empty((Bs, L, H), **f32),
             dA=torch.empty(H, **f32), dB=torch.empty(bc, **f32), dC=torch.empty(bc, **f32),
             dD=None if D is None else torch.empty(H, **f32))
    bad = set(options) - (set(_OPTION_KEYS) - {"return_final_state"})
    if bad:
        raise TypeError("unknown options: %s" % sorted(bad))
    if options:
        o, _, keep = _options(x, H, (Bs, H, P, N), dev, ngroups=G, **options)
        g["dz"] = torch.empty((Bs, L, H, P), **f32) if options.get("z") is not None else None
        g["ddt_bias"] = torch.empty(H, **f32) if options.get("dt_bias") is not None else None
        g["dh0"] = torch.empty((Bs, H, P, N), **f32) if options.get("h0") is not None else None
        st = library().ssd_chunk_scan_bwd_ex(
            _ptr(x), _ptr(dt), _ptr(A_head), _ptr(B), _ptr(C), _ptr(D), _ptr(dy), _ptr(g["dx"]),
            _ptr(g["ddt"]), _ptr(g["dA"]), _ptr(g["dB"]), _ptr(g["dC"]), _ptr(g["dD"]),
            _ptr(g["dz"]), _ptr(g["ddt_bias"]), _ptr(g["dh0"]), Bs, L, H, P, N,
            int(bool(bidirectional)), int(x.dtype == torch.bfloat16), ctypes.byref(o),
            _stream(dev))
        if st != 0:
            raise SsmError("ssd_chunk_scan_bwd_ex", st)
        return g
    st = library().ssd_chunk_scan_bwd(
        _ptr(x), _ptr(dt), _ptr(A_head), _ptr(B), _ptr(C), _ptr(D), _ptr(dy), _ptr(g["dx"]),
        _ptr(g["ddt"]), _ptr(g["dA"]), _ptr(g["dB"]), _ptr(g["dC"]), _ptr(g["dD"]),
        Bs, L, H, P, N, G, int(bool(bidirectional)), int(x.dtype == torch.bfloat16), _stream(dev))
    if st != 0:
        raise SsmError("ssd_chunk_scan_bwd", st)
    return g


def ssm_scan_fwd_plan(Bs: int, L: int, ED: int, N: int, bf16: bool = True):
    """(states per thread, lanes per channel, time segments) the diagonal scan
    uses for this shape on the current device; time segments > 1 means two
    kernel launches per call."""
    s, g, k = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    st = library().ssm_scan_fwd_plan(Bs, L, ED, N, int(bool(bf16)), ctypes.byref(s),
                                     ctypes.byref(g), ctypes.byref(k))
    if st != 0:
        raise SsmError("ssm_scan_fwd_plan", st)
    return s.value, g.value, k.value


def ssm_check_device_errors(device=None) -> None:
    """Synchronise the current stream and raise SsmError if a kernel of the
    library abandoned its work after a bounded device wait ran out."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    st = library().ssm_check_device_errors(_stream(dev))
    if st != 0:
        raise SsmError("ssm_check_device_errors", st)
