"""Host-side checks of the C ABI (CPU only: no kernel is launched).

The library must load, export every function include/ssm_scan.h declares,
and reject bad arguments with status codes before touching any device.
"""
import ctypes
import os
import re

import pytest

import linear_recurrence_ssm_gb300 as lrs

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "ssm_scan.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = "\n".join(l for l in text.splitlines() if not l.lstrip().startswith("#"))
    return sorted(set(re.findall(r"SSM_API\s+[^;(]*?\b([a-z_][a-z0-9_]*)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("ssm_scan_fwd", "ssm_scan_fwd_bf16", "ssd_chunk_scan_fwd", "ssm_status_string",
              "ssm_version", "ssm_check_device_errors"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = lrs.library()
    for name in declared_functions():
        assert hasattr(lib, name), "missing export " + name
    assert set(declared_functions()) == set(lrs.SIGNATURES)


def test_status_strings():
    for code, name in lrs.STATUS.items():
        assert lrs.status_string(code).startswith(name)
    assert "unknown" in lrs.status_string(99)


P = ctypes.c_void_p(0x10000)       # never dereferenced: validation fails first
P_ODD = ctypes.c_void_p(0x10001)


def diag(fn="ssm_scan_fwd", ptrs=None, Bs=2, L=8, ED=4, N=16):
    p = ptrs or [P] * 7
    return getattr(lrs.library(), fn)(*p, Bs, L, ED, N, None)


def ssd(ptrs=None, Bs=1, L=8, H=2, P_=64, N=64, chunk=128, bidir=0):
    p = ptrs or [P] * 7
    return lrs.library().ssd_chunk_scan_fwd(*p, Bs, L, H, P_, N, chunk, bidir, None)


@pytest.mark.parametrize("fn", ["ssm_scan_fwd", "ssm_scan_fwd_bf16"])
def test_diag_rejects_bad_arguments(fn):
    for i in (0, 1, 2, 3, 4, 6):          # every pointer but D is required
        ptrs = [P] * 7
        ptrs[i] = None
        assert diag(fn, ptrs) == 1
    assert diag(fn, Bs=0) == 1
    assert diag(fn, L=0) == 1
    assert diag(fn, ED=-3) == 1
    assert diag(fn, N=0) == 1
    assert diag(fn, Bs=2 ** 40, L=2 ** 40) == 1      # element count overflows int64
    assert diag(fn, N=257) == 2
    ptrs = [P] * 7
    ptrs[6] = P_ODD                       # y not 4-byte aligned
    assert diag(fn, ptrs) == 3


def test_ssd_rejects_bad_arguments():
    ptrs = [P] * 7
    ptrs[0] = None
    assert ssd(ptrs) == 1
    assert ssd(L=0) == 1
    assert ssd(chunk=0) == 1
    assert ssd(P_=48) == 2
    assert ssd(P_=512) == 2
    assert ssd(P_=8) == 2
    assert ssd(N=48) == 2
    assert ssd(N=8) == 2
    assert ssd(N=512) == 2
    assert ssd(chunk=96) == 2
    ptrs = [P] * 7
    ptrs[3] = P_ODD                       # B not 16-byte aligned
    assert ssd(ptrs) == 3


def test_noalloc_rejects_scratch_beyond_its_fixed_size():
    lib = lrs.library()
    # bidirectional, Bs*H*ceil(L/128)*P*N*2 = 1 GiB > SSM_NOALLOC_SCRATCH_BYTES: rejected up front
    assert lib.ssd_chunk_scan_fwd_noalloc(*([P] * 7), 64, 4096, 32, 64, 128, 256, 1, None) == 2
    ptrs = [P] * 7
    ptrs[4] = None
    assert lib.ssd_chunk_scan_fwd_noalloc(*ptrs, 1, 8, 2, 64, 64, 128, 1, None) == 1


def test_valid_call_without_device_reports_no_device():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    assert diag() == 6
    assert ssd() == 6
    assert lrs.library().ssm_check_device_errors(None) == 6
    # the same large call without the reverse scan needs no scratch: passes the size check
    assert lrs.library().ssd_chunk_scan_fwd_noalloc(*([P] * 7), 64, 4096, 32, 64, 128, 256, 0,
                                                    None) == 6


def _opts(**kw):
    o = lrs.ScanOptions()
    for k, v in kw.items():
        setattr(o, k, v)
    return o


def test_option_entry_points_reject_bad_arguments():
    lib = lrs.library()
    ptrs = [P] * 7
    ptrs[1] = None
    assert lib.ssm_scan_fwd_ex(*ptrs, 1, 8, 8, 4, 1, ctypes.byref(_opts()), None) == 1
    # misaligned option pointers
    assert lib.ssm_scan_fwd_ex(*([P] * 7), 1, 8, 8, 4, 1, ctypes.byref(_opts(z=P_ODD)), None) == 3
    assert lib.ssm_scan_fwd_ex(*([P] * 7), 1, 8, 8, 4, 0,
                               ctypes.byref(_opts(h_final=0x10002)), None) == 3
    assert lib.ssd_chunk_scan_fwd_ex(*([P] * 7), 1, 8, 2, 64, 64, 128, 0, 1,
                                     ctypes.byref(_opts(z=0x10008)), None) == 3
    # state input/output is defined for a single direction only
    assert lib.ssd_chunk_scan_fwd_ex(*([P] * 7), 1, 8, 2, 64, 64, 128, 1, 1,
                                     ctypes.byref(_opts(h0=P)), None) == 2
    assert lib.ssd_chunk_scan_fwd_ex(*([P] * 7), 1, 8, 2, 64, 64, 128, 1, 1,
                                     ctypes.byref(_opts(h_final=P)), None) == 2
    assert lib.ssd_chunk_scan_fwd_ex(*([P] * 7), 1, 8, 2, 48, 64, 128, 0, 1,
                                     ctypes.byref(_opts()), None) == 2


def test_option_calls_without_device_report_no_device():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    lib = lrs.library()
    o = _opts(dt_softplus=1, z=P, h0=P, h_final=P)
    assert lib.ssm_scan_fwd_ex(*([P] * 7), 1, 8, 8, 4, 1, ctypes.byref(o), None) == 6
    assert lib.ssd_chunk_scan_fwd_ex(*([P] * 7), 1, 8, 2, 64, 64, 128, 0, 1, ctypes.byref(o), None) == 6
    # a NULL options pointer is the plain call
    assert lib.ssd_chunk_scan_fwd_ex(*([P] * 7), 1, 8, 2, 64, 64, 128, 1, 1, None, None) == 6


def test_groups_are_validated():
    lib = lrs.library()
    # ngroups must divide H
    assert lib.ssd_chunk_scan_fwd_ex(*([P] * 7), 1, 8, 6, 64, 64, 128, 0, 1,
                                     ctypes.byref(_opts(ngroups=4)), None) == 1
    assert lib.ssd_chunk_scan_fwd_ex(*([P] * 7), 1, 8, 6, 64, 64, 128, 0, 1,
                                     ctypes.byref(_opts(ngroups=-1)), None) == 1
    # groups belong to the SSD scan only
    assert lib.ssm_scan_fwd_ex(*([P] * 7), 1, 8, 8, 4, 1, ctypes.byref(_opts(ngroups=2)), None) == 2


def test_backward_rejects_bad_arguments():
    lib = lrs.library()
    p13 = [P] * 13
    assert lib.ssm_scan_bwd(*p13, 1, 8, 8, 257, 0, None) == 2      # N > 256
    bad = list(p13)
    bad[6] = None                                                  # dy
    assert lib.ssm_scan_bwd(*bad, 1, 8, 8, 4, 0, None) == 1
    bad = list(p13)
    bad[8] = P_ODD                                                 # ddelta misaligned
    assert lib.ssm_scan_bwd(*bad, 1, 8, 8, 4, 0, None) == 3


def test_ssd_backward_rejects_bad_arguments():
    lib = lrs.library()
    p13 = [P] * 13
    # (Bs, L, H, P, N, ngroups, bidirectional, input_bf16)
    assert lib.ssd_chunk_scan_bwd(*p13, 1, 8, 2, 48, 64, 1, 0, 1, None) == 2     # P = 48
    assert lib.ssd_chunk_scan_bwd(*p13, 1, 8, 2, 64, 16, 1, 0, 1, None) == 2     # N = 16
    assert lib.ssd_chunk_scan_bwd(*p13, 1, 8, 2, 128, 128, 1, 0, 1, None) == 2   # P * N > 8192
    assert lib.ssd_chunk_scan_bwd(*p13, 1, 8, 3, 64, 64, 2, 0, 1, None) == 2     # H % G != 0
    assert lib.ssd_chunk_scan_bwd(*p13, 1, 8, 2, 64, 64, 0, 0, 1, None) == 1     # no groups
    assert lib.ssd_chunk_scan_bwd(*p13, 0, 8, 2, 64, 64, 1, 0, 1, None) == 1     # Bs = 0
    bad = list(p13)
    bad[6] = None                                                                 # dy
    assert lib.ssd_chunk_scan_bwd(*bad, 1, 8, 2, 64, 64, 1, 0, 1, None) == 1
    bad = list(p13)
    bad[8] = P_ODD                                                                # ddt misaligned
    assert lib.ssd_chunk_scan_bwd(*bad, 1, 8, 2, 64, 64, 1, 0, 1, None) == 3
    # a valid call reaches the device check (no GPU here, or a real launch there)
    assert lib.ssd_chunk_scan_bwd(*([None] * 13), 1, 8, 2, 64, 64, 1, 0, 1, None) == 1


def _declarations():
    """name -> list of parameter declarations, for every SSM_API function."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    out = {}
    for m in re.finditer(r"SSM_API\s+[^;(]*?\b([a-z_][a-z0-9_]*)\s*\(([^)]*)\)\s*;", text):
        params = [p.strip() for p in m.group(2).split(",") if p.strip() and p.strip() != "void"]
        out[m.group(1)] = params
    return out


def test_binding_signatures_match_the_header():
    """Each binding's ctypes argument list has the header's parameter count
    and, parameter by parameter, its kind: pointer, 64-bit or 32-bit integer,
    float (a 32-bit integer where an int64_t is declared passes garbage high
    bits)."""
    decls = _declarations()
    for name, (argtypes, _) in lrs.SIGNATURES.items():
        assert name in decls, name
        params = decls[name]
        assert len(argtypes) == len(params), (name, len(argtypes), len(params))
        for decl, at in zip(params, argtypes):
            if "*" in decl:
                assert at in (ctypes.c_void_p, ctypes.c_char_p) or hasattr(at, "_type_") and \
                    issubclass(at, ctypes._Pointer), (name, decl, at)
            elif "int64_t" in decl:
                assert at is ctypes.c_int64, (name, decl, at)
            elif re.search(r"\bint(32_t)?\b|\bssm_status_t\b", decl):   # the enum is an int
                assert at in (ctypes.c_int, ctypes.c_int32), (name, decl, at)
            elif "float" in decl:
                assert at is ctypes.c_float, (name, decl, at)
            else:
                raise AssertionError("unclassified parameter %r of %s" % (decl, name))
