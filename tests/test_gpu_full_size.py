"""Parity at the benchmark sizes for the widened paths: every scan option
on (the benchmark's option mode), the diagonal scan's gradients and the
chunked scan's gradients.

The GPU runs the whole workload in the launch configuration the benchmark
times; the fp64 oracle recomputes a spread-out sample of channels / heads
one by one (the option inputs follow the benchmark's recipe: seed + 7,
dt_limit = (1e-4, 100)).  For the gradients the sample is whole channels e
over all batch rows, so that the per-channel sums dA[e, :] and dD[e] are
complete; dB and dC (sums over all channels) are covered at small sizes in
test_gpu_backward.  The chunked scan's gradients are compared whole: the
oracle computes every head (seconds at these sizes).  Tolerance: 2e-2 * max|ref| of each compared quantity
(bf16 inputs).
"""
import numpy as np
import pytest
import torch

import linear_recurrence_ssm_gb300 as lrs
import oracle
import workloads

pytestmark = pytest.mark.gpu

TOL = 2e-2
LIMIT = (1e-4, 100.0)


def _close(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got)), what + " has non-finite values"
    scale = float(np.max(np.abs(ref)))
    err = float(np.max(np.abs(got - ref)))
    assert err <= TOL * scale, "%s: max abs err %.3e > %.3e (scale %.3e)" % (what, err, TOL * scale, scale)


def _options(w):
    s = w.shape
    if w.kind == "diag":
        return workloads.option_inputs((s["Bs"], s["L"], s["ED"]), (s["Bs"], s["L"], s["ED"]),
                                       s["ED"], (s["Bs"], s["ED"], s["N"]), w.dtype, w.seed + 7)
    state = (1,) if s["bidirectional"] else (s["Bs"], s["H"], s["P"], s["N"])
    return workloads.option_inputs((s["Bs"], s["L"], s["H"], s["P"]), (s["Bs"], s["L"], s["H"]),
                                   s["H"], state, w.dtype, w.seed + 7)


def test_diag_options_at_benchmark_size(cuda_device):
    w = workloads.BY_NAME["diag_bf16_Bs8_L2048_ED1536_N16"]
    s = w.shape
    Bs, ED = s["Bs"], s["ED"]
    inp = workloads.workload_inputs(w)
    o = _options(w)
    d = lambda t: t.to(cuda_device)
    y, hf = lrs.ssm_scan_fwd(d(inp["x"]), d(o["delta_raw"]), d(inp["A"]), d(inp["B"]), d(inp["C"]),
                             d(inp["D"]), dt_bias=d(o["dt_bias"]), dt_softplus=True, dt_limit=LIMIT,
                             z=d(o["z"]), h0=d(o["h0"]), return_final_state=True)
    torch.cuda.synchronize()
    y, hf = y.cpu().double().numpy(), hf.cpu().double().numpy()
    rng = np.random.default_rng(1)
    chans = sorted(set([0, Bs * ED - 1, ED - 1, ED] + list(rng.integers(0, Bs * ED, 40))))
    for c in chans:
        b, e = divmod(int(c), ED)
        one = dict(x=inp["x"][b:b + 1, :, e:e + 1], delta=o["delta_raw"][b:b + 1, :, e:e + 1],
                   A=inp["A"][e:e + 1], B=inp["B"][b:b + 1], C=inp["C"][b:b + 1], D=inp["D"][e:e + 1])
        ry, rh = oracle.diag_scan(**one, dt_bias=o["dt_bias"][e:e + 1], dt_softplus=True,
                                  dt_limit=LIMIT, z=o["z"][b:b + 1, :, e:e + 1],
                                  h0=o["h0"][b:b + 1, e:e + 1], return_final_state=True)
        _close(y[b, :, e], ry[0, :, 0], "y (b=%d, e=%d)" % (b, e))
        _close(hf[b, e], rh[0, 0], "h_final (b=%d, e=%d)" % (b, e))


@pytest.mark.parametrize("name", ["ssd_bf16_Bs4_L4096_H32_P64_N128_Q256",
                                  "bissd_bf16_Bs32_L400_H8_P64_N64_Q128"])
def test_ssd_options_at_benchmark_size(cuda_device, name):
    w = workloads.BY_NAME[name]
    s = w.shape
    Bs, H, bidir = s["Bs"], s["H"], s["bidirectional"]
    inp = workloads.workload_inputs(w)
    o = _options(w)
    d = lambda t: t.to(cuda_device)
    st = {} if bidir else dict(h0=d(o["h0"]), return_final_state=True)
    out = lrs.ssd_chunk_scan_fwd(d(inp["x"]), d(o["delta_raw"]), d(inp["A_head"]), d(inp["B"]),
                                 d(inp["C"]), d(inp["D"]), chunk=s["chunk"], bidirectional=bidir,
                                 dt_bias=d(o["dt_bias"]), dt_softplus=True, dt_limit=LIMIT,
                                 z=d(o["z"]), **st)
    torch.cuda.synchronize()
    y, hf = (out, None) if bidir else out
    y = y.cpu().double().numpy()
    hf = None if hf is None else hf.cpu().double().numpy()
    for b, h in [(0, 0), (Bs - 1, H - 1), (Bs // 2, H // 3), (1 % Bs, H - 2)]:
        one = dict(x=inp["x"][b:b + 1, :, h:h + 1], dt=o["delta_raw"][b:b + 1, :, h:h + 1],
                   A_head=inp["A_head"][h:h + 1], B=inp["B"][b:b + 1], C=inp["C"][b:b + 1],
                   D=inp["D"][h:h + 1])
        kw = dict(dt_bias=o["dt_bias"][h:h + 1], dt_softplus=True, dt_limit=LIMIT,
                  z=o["z"][b:b + 1, :, h:h + 1], bidirectional=bidir)
        if bidir:
            ry = oracle.ssd_scan(**one, **kw)
        else:
            ry, rh = oracle.ssd_scan(**one, **kw, h0=o["h0"][b:b + 1, h:h + 1], return_final_state=True)
            _close(hf[b, h], rh[0, 0], "h_final (b=%d, h=%d)" % (b, h))
        _close(y[b, :, h], ry[0, :, 0], "y (b=%d, h=%d)" % (b, h))
    lrs.ssm_check_device_errors()


def test_gradients_at_benchmark_size(cuda_device):
    w = workloads.BY_NAME["diag_bf16_Bs8_L2048_ED1536_N16"]
    s = w.shape
    ED = s["ED"]
    inp = workloads.workload_inputs(w)
    dy = workloads.grad_output((s["Bs"], s["L"], ED), seed=w.seed + 11)
    got = lrs.ssm_scan_bwd(**{k: v.to(cuda_device) for k, v in inp.items()}, dy=dy.to(cuda_device))
    torch.cuda.synchronize()
    got = {k: v.cpu().double().numpy() for k, v in got.items() if k in ("dx", "ddelta", "dA", "dD")}
    for e in (0, 1, 37, ED // 2, ED - 1):
        ch = dict(x=inp["x"][:, :, e:e + 1], delta=inp["delta"][:, :, e:e + 1], A=inp["A"][e:e + 1],
                  B=inp["B"], C=inp["C"], D=inp["D"][e:e + 1])
        ref = oracle.diag_scan_bwd(**ch, dy=dy[:, :, e:e + 1])
        _close(got["dx"][:, :, e], ref["dx"][:, :, 0], "dx (e=%d)" % e)
        _close(got["ddelta"][:, :, e], ref["ddelta"][:, :, 0], "ddelta (e=%d)" % e)
        _close(got["dA"][e], ref["dA"][0], "dA (e=%d)" % e)
        _close(got["dD"][e:e + 1], ref["dD"], "dD (e=%d)" % e)


@pytest.mark.parametrize("name", ["ssd_bf16_Bs4_L4096_H32_P64_N128_Q256",
                                  "bissd_bf16_Bs32_L400_H8_P64_N64_Q128"])
def test_ssd_gradients_at_benchmark_size(cuda_device, name):
    w = workloads.BY_NAME[name]
    s = w.shape
    bidir = s["bidirectional"]
    inp = workloads.workload_inputs(w)
    dy = workloads.grad_output((s["Bs"], s["L"], s["H"], s["P"]), seed=w.seed + 11)
    got = lrs.ssd_chunk_scan_bwd(**{k: v.to(cuda_device) for k, v in inp.items()},
                                 dy=dy.to(cuda_device), bidirectional=bidir)
    torch.cuda.synchronize()
    got = {k: v.cpu().double().numpy() for k, v in got.items()}
    ref = oracle.ssd_scan_bwd(**inp, dy=dy, bidirectional=bidir)
    for k in ("dx", "ddt", "dA", "dB", "dC", "dD"):
        assert got[k].shape == ref[k].shape, k
        _close(got[k], ref[k], k)
    lrs.ssm_check_device_errors()
