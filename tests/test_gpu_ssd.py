"""GPU parity of the chunked scalar-decay (SSD) scan, one and two directions,
against the fp64 oracle on the same bf16-rounded inputs.

Tolerance: max|y - y_ref| <= 2e-2 * max|y_ref| (bf16 inputs, bf16 tensor-core
operands with fp32 accumulation and fp32 state).
"""
import ctypes

import numpy as np
import pytest
import torch

import linear_recurrence_ssm_gb300 as lrs
import oracle
import workloads

pytestmark = pytest.mark.gpu

TOL = 2e-2


def _dev(inp, dev):
    return {k: (v.to(dev) if v is not None else None) for k, v in inp.items()}


def _check(y, ref):
    y = y.double().cpu().numpy()
    assert np.all(np.isfinite(y))
    scale = float(np.max(np.abs(ref)))
    err = float(np.max(np.abs(y - ref)))
    assert err <= TOL * scale, "max abs err %.3e > %.3e (scale %.3e)" % (err, TOL * scale, scale)
    return err / scale


@pytest.mark.parametrize("bidir", [False, True])
@pytest.mark.parametrize("Bs,L,H,N,chunk", [
    (1, 128, 1, 64, 128),     # exactly one tile
    (2, 300, 3, 64, 128),     # ragged last tile
    (1, 1, 2, 128, 256),      # L = 1
    (2, 257, 2, 128, 256),    # one row into a third tile
    (1, 400, 2, 64, 64),
    (1, 640, 1, 128, 128),    # five tiles
])
def test_ssd_matches_oracle(cuda_device, Bs, L, H, N, chunk, bidir):
    inp = workloads.ssd_inputs(Bs, L, H, 64, N, "bf16", seed=L + H + N + int(bidir))
    ref = oracle.ssd_scan(**inp, bidirectional=bidir)
    y = lrs.ssd_chunk_scan_fwd(**_dev(inp, cuda_device), chunk=chunk, bidirectional=bidir)
    _check(y, ref)
    lrs.ssm_check_device_errors()


def test_ssd_without_D(cuda_device):
    inp = workloads.ssd_inputs(2, 200, 2, 64, 64, "bf16", seed=21, with_D=False)
    ref = oracle.ssd_scan(**inp)
    y = lrs.ssd_chunk_scan_fwd(**_dev(inp, cuda_device), chunk=128)
    _check(y, ref)


def test_chunk_lengths_agree(cuda_device):
    inp = _dev(workloads.ssd_inputs(1, 300, 2, 64, 128, "bf16", seed=5), cuda_device)
    ys = [lrs.ssd_chunk_scan_fwd(**inp, chunk=q) for q in (64, 128, 256)]
    for y in ys[1:]:
        assert torch.allclose(y, ys[0], rtol=0, atol=1e-3 * ys[0].abs().max().item())


def test_bidirectional_reversal_equivariance(cuda_device):
    inp = workloads.ssd_inputs(2, 333, 2, 64, 64, "bf16", seed=8)
    flip = {k: (v.flip(1).contiguous() if k in ("x", "dt", "B", "C") else v) for k, v in inp.items()}
    y = lrs.ssd_chunk_scan_fwd(**_dev(inp, cuda_device), chunk=128, bidirectional=True)
    yf = lrs.ssd_chunk_scan_fwd(**_dev(flip, cuda_device), chunk=128, bidirectional=True)
    scale = y.abs().max().item()
    assert (yf.flip(1) - y).abs().max().item() <= TOL * scale


@pytest.mark.parametrize("name", ["ssd_bf16_Bs4_L4096_H32_P64_N128_Q256",
                                  "bissd_bf16_Bs32_L400_H8_P64_N64_Q128"])
def test_benchmark_shape_whole_output(cuda_device, name):
    """Full benchmark size in the benchmark's launch configuration; the whole
    y against the oracle on the same inputs."""
    w = workloads.BY_NAME[name]
    s = w.shape
    inp = workloads.workload_inputs(w)
    y = lrs.ssd_chunk_scan_fwd(**_dev(inp, cuda_device), chunk=s["chunk"],
                               bidirectional=s["bidirectional"])
    _check(y, oracle.ssd_scan(**inp, bidirectional=s["bidirectional"]))
    lrs.ssm_check_device_errors()


def test_bidirectional_benchmark_shape_repeats_bitwise(cuda_device):
    """Twenty calls at the bidirectional benchmark size give the same bits,
    and that y matches the oracle: the reverse entering states handed from one
    part of the computation to the next are the same on every call."""
    w = workloads.BY_NAME["bissd_bf16_Bs32_L400_H8_P64_N64_Q128"]
    s = w.shape
    inp = workloads.workload_inputs(w)
    dev_inp = _dev(inp, cuda_device)
    first = lrs.ssd_chunk_scan_fwd(**dev_inp, chunk=s["chunk"], bidirectional=True)
    torch.cuda.synchronize()
    for _ in range(19):
        y = torch.full_like(first, float("nan"))
        lrs.ssd_chunk_scan_fwd(**dev_inp, chunk=s["chunk"], bidirectional=True, y=y)
        torch.cuda.synchronize()
        assert torch.equal(y, first)
    _check(first, oracle.ssd_scan(**inp, bidirectional=True))
    lrs.ssm_check_device_errors()


def test_deterministic_and_guard_bands(cuda_device):
    inp = _dev(workloads.ssd_inputs(2, 260, 3, 64, 64, "bf16", seed=9), cuda_device)
    Bs, L, H, P = inp["x"].shape
    n = Bs * L * H * P
    guard = 4096
    buf = torch.full((n + 2 * guard,), float("nan"), device=cuda_device)
    y1 = buf[guard:guard + n].view(Bs, L, H, P)
    lrs.ssd_chunk_scan_fwd(**inp, chunk=128, bidirectional=True, y=y1)
    y2 = lrs.ssd_chunk_scan_fwd(**inp, chunk=128, bidirectional=True)
    torch.cuda.synchronize()
    assert torch.isnan(buf[:guard]).all() and torch.isnan(buf[guard + n:]).all()
    assert torch.equal(y1, y2)


def test_runs_on_caller_stream(cuda_device):
    inp = _dev(workloads.ssd_inputs(1, 256, 2, 64, 128, "bf16", seed=3), cuda_device)
    ref = lrs.ssd_chunk_scan_fwd(**inp, chunk=128, bidirectional=True)
    s = torch.cuda.Stream(cuda_device)
    with torch.cuda.stream(s):
        y = lrs.ssd_chunk_scan_fwd(**inp, chunk=128, bidirectional=True)
    s.synchronize()
    assert torch.equal(y, ref)


def test_bounded_wait_reports_timeout(cuda_device):
    """A bounded wait that cannot complete gives up, the error word records it,
    the check reports it once and the context stays usable."""
    lib = lrs.library()
    stream = ctypes.c_void_p(torch.cuda.current_stream(cuda_device).cuda_stream)
    assert lib.ssm_check_device_errors(stream) == 0
    assert lib.ssm_selftest_wait_timeout(stream) == 0
    assert lib.ssm_check_device_errors(stream) == 5      # SSM_ERR_DEVICE_TIMEOUT
    assert lib.ssm_check_device_errors(stream) == 0      # cleared
    inp = workloads.ssd_inputs(1, 200, 2, 64, 64, "bf16", seed=3)
    y = lrs.ssd_chunk_scan_fwd(**{k: v.to(cuda_device) for k, v in inp.items()})
    torch.cuda.synchronize()
    _check(y, oracle.ssd_scan(**inp))


@pytest.mark.parametrize("L", [1, 2, 127, 129, 384, 511, 512, 513])
@pytest.mark.parametrize("groups", [1, 2])
def test_short_bidirectional_boundaries(cuda_device, L, groups):
    """The bidirectional scan with N = 64 runs as two passes over independent
    tiles for up to four 128-row tiles (L <= 512) and on the single-role
    kernel beyond: both sides of that boundary, one and two rows into a
    tile, and groups of B, C, against the oracle."""
    Bs, H = 2, 4
    inp = workloads.ssd_inputs(Bs, L, H, 64, 64, "bf16", seed=L + 7 * groups, groups=groups)
    ref = oracle.ssd_scan(**inp, bidirectional=True)
    y = lrs.ssd_chunk_scan_fwd(**_dev(inp, cuda_device), chunk=128, bidirectional=True)
    _check(y, ref)


def test_short_bidirectional_many_tiles_per_cta(cuda_device):
    """4096 tiles of 128 rows on the persistent output pass: each CTA walks
    about 27 tiles, so every barrier phase and double buffer of the two
    passes wraps many times (the benchmark size gives about 7).  Sequences are
    independent, so batch rows from both ends (the first and the last CTAs'
    tiles) are checked against the oracle run on those rows alone."""
    Bs, L, H, N = 128, 512, 8, 64
    inp = workloads.ssd_inputs(Bs, L, H, 64, N, "bf16", seed=31)
    y = lrs.ssd_chunk_scan_fwd(**_dev(inp, cuda_device), chunk=128, bidirectional=True)
    for rows in (slice(0, 3), slice(Bs // 2, Bs // 2 + 2), slice(Bs - 3, Bs)):
        sub = {k: (v[rows] if v is not None and v.dim() > 1 else v) for k, v in inp.items()}
        _check(y[rows], oracle.ssd_scan(**sub, bidirectional=True))
