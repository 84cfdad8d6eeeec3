"""GPU parity of the scan options against the fp64 oracle.

The options are the remaining arguments of the chunked scan in "Some
questions of Bi-Mamba2 and Hydra" (Bi-Mamba2 issue 1): dt_bias, dt_softplus,
dt_limit, the silu output gate z, an initial state and the returned final
state.  Every case runs the C-ABI ``*_ex`` entry points (through the binding)
and the oracle on the same seeded, bf16-rounded inputs.  Tolerances as for
the plain scans: 1e-4 * max(1, max|ref|) for fp32 inputs, 2e-2 * max|ref|
for bf16 inputs / tensor-core paths; the final states use the same rule
relative to their own scale.
"""
import numpy as np
import pytest
import torch

import linear_recurrence_ssm_gb300 as lrs
import oracle
import workloads

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}
LIMIT = (0.05, 2.0)


def _close(got, ref, dtype, what):
    g = got.double().cpu().numpy()
    assert np.all(np.isfinite(g)), what + " has non-finite values"
    scale = float(np.max(np.abs(ref)))
    bound = TOL[dtype] * (max(1.0, scale) if dtype == "f32" else scale)
    err = float(np.max(np.abs(g - ref)))
    assert err <= bound, "%s: max abs err %.3e > bound %.3e (scale %.3e)" % (what, err, bound, scale)


def _diag_case(Bs, L, ED, N, dtype, seed):
    inp = workloads.diag_inputs(Bs, L, ED, N, dtype, seed=seed)
    opt = workloads.option_inputs((Bs, L, ED), (Bs, L, ED), ED, (Bs, ED, N), dtype, seed + 1)
    inp["delta"] = opt["delta_raw"]
    return inp, opt


def _dev(d, dev):
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("Bs,L,ED,N", [
    (2, 64, 64, 16),
    (3, 100, 200, 16),    # several time and channel tiles, ragged tails
    (2, 31, 70, 16),      # unvectorised loads for bf16
    (1, 45, 24, 5),       # padded states
    (1, 600, 128, 16),    # split into time segments (carry pass)
    (2, 3000, 128, 7),
    (2, 50, 64, 40),      # more than 16 states (padded to 64)
])
def test_diag_all_options(cuda_device, dtype, Bs, L, ED, N):
    inp, opt = _diag_case(Bs, L, ED, N, dtype, seed=L + ED + N)
    ref, href = oracle.diag_scan(**inp, dt_bias=opt["dt_bias"], dt_softplus=True, dt_limit=LIMIT,
                                 z=opt["z"], h0=opt["h0"], return_final_state=True)
    d = _dev(inp, cuda_device)
    y, hf = lrs.ssm_scan_fwd(**d, dt_bias=opt["dt_bias"].to(cuda_device), dt_softplus=True,
                             dt_limit=LIMIT, z=opt["z"].to(cuda_device),
                             h0=opt["h0"].to(cuda_device), return_final_state=True)
    torch.cuda.synchronize()
    _close(y, ref, dtype, "y")
    _close(hf, href, dtype, "h_final")


@pytest.mark.parametrize("option", ["dt_bias", "dt_softplus", "dt_limit", "z", "h0", "final"])
def test_diag_each_option_alone(cuda_device, option):
    Bs, L, ED, N = 2, 700, 96, 12          # time-split shape
    inp, opt = _diag_case(Bs, L, ED, N, "bf16", seed=77)
    if option in ("z", "h0", "final"):
        inp["delta"] = workloads.diag_inputs(Bs, L, ED, N, "bf16", seed=77)["delta"]
    kw = {"dt_bias": dict(dt_bias=opt["dt_bias"], dt_softplus=True),
          "dt_softplus": dict(dt_softplus=True),
          "dt_limit": dict(dt_softplus=True, dt_limit=LIMIT),
          "z": dict(z=opt["z"]),
          "h0": dict(h0=opt["h0"]),
          "final": dict(return_final_state=True)}[option]
    ref = oracle.diag_scan(**inp, **kw)
    out = lrs.ssm_scan_fwd(**_dev(inp, cuda_device), **_dev(kw, cuda_device))
    torch.cuda.synchronize()
    if option == "final":
        _close(out[0], ref[0], "bf16", "y")
        _close(out[1], ref[1], "bf16", "h_final")
    else:
        _close(out, ref, "bf16", "y")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_diag_streaming_in_two_calls(cuda_device, dtype):
    """Two calls chained through the final / initial state equal one call."""
    Bs, L, ED, N, cut = 2, 900, 64, 16, 352
    inp = workloads.diag_inputs(Bs, L, ED, N, dtype, seed=5)
    d = _dev(inp, cuda_device)
    y_full, h_full = lrs.ssm_scan_fwd(**d, return_final_state=True)
    part = lambda sl: {k: (v[:, sl].contiguous() if k in ("x", "delta", "B", "C") else v)
                       for k, v in d.items()}
    ya, ha = lrs.ssm_scan_fwd(**part(slice(0, cut)), return_final_state=True)
    yb, hb = lrs.ssm_scan_fwd(**part(slice(cut, None)), h0=ha, return_final_state=True)
    torch.cuda.synchronize()
    ref, href = oracle.diag_scan(**inp, return_final_state=True)
    _close(torch.cat([ya, yb], dim=1), ref, dtype, "y (two calls)")
    _close(hb, href, dtype, "h_final (two calls)")
    _close(y_full, ref, dtype, "y (one call)")


def _ssd_case(Bs, L, H, N, seed):
    inp = workloads.ssd_inputs(Bs, L, H, 64, N, "bf16", seed=seed)
    opt = workloads.option_inputs((Bs, L, H, 64), (Bs, L, H), H, (Bs, H, 64, N), "bf16", seed + 1)
    inp["dt"] = opt["delta_raw"]
    return inp, opt


@pytest.mark.parametrize("Bs,L,H,N", [
    (2, 300, 3, 64),
    (1, 1000, 2, 128),
    (2, 129, 2, 64),      # one row into the second tile
    (1, 77, 4, 128),      # a single ragged tile
])
def test_ssd_all_options(cuda_device, Bs, L, H, N):
    inp, opt = _ssd_case(Bs, L, H, N, seed=L + H + N)
    ref, href = oracle.ssd_scan(**inp, dt_bias=opt["dt_bias"], dt_softplus=True, dt_limit=LIMIT,
                                z=opt["z"], h0=opt["h0"], return_final_state=True)
    y, hf = lrs.ssd_chunk_scan_fwd(**_dev(inp, cuda_device), chunk=128,
                                   dt_bias=opt["dt_bias"].to(cuda_device), dt_softplus=True,
                                   dt_limit=LIMIT, z=opt["z"].to(cuda_device),
                                   h0=opt["h0"].to(cuda_device), return_final_state=True)
    torch.cuda.synchronize()
    _close(y, ref, "bf16", "y")
    _close(hf, href, "bf16", "h_final")


@pytest.mark.parametrize("Bs,L,H,N", [(2, 300, 3, 64), (1, 400, 2, 128)])
def test_ssd_bidirectional_with_dt_options_and_gate(cuda_device, Bs, L, H, N):
    inp, opt = _ssd_case(Bs, L, H, N, seed=3 * L + N)
    ref = oracle.ssd_scan(**inp, bidirectional=True, dt_bias=opt["dt_bias"], dt_softplus=True,
                          dt_limit=LIMIT, z=opt["z"])
    y = lrs.ssd_chunk_scan_fwd(**_dev(inp, cuda_device), chunk=128, bidirectional=True,
                               dt_bias=opt["dt_bias"].to(cuda_device), dt_softplus=True,
                               dt_limit=LIMIT, z=opt["z"].to(cuda_device))
    torch.cuda.synchronize()
    _close(y, ref, "bf16", "y")


def test_ssd_streaming_in_two_calls(cuda_device):
    Bs, L, H, N, cut = 2, 700, 2, 128, 256
    inp = workloads.ssd_inputs(Bs, L, H, 64, N, "bf16", seed=9)
    d = _dev(inp, cuda_device)
    part = lambda sl: {k: (v[:, sl].contiguous() if k in ("x", "dt", "B", "C") else v)
                       for k, v in d.items()}
    ya, ha = lrs.ssd_chunk_scan_fwd(**part(slice(0, cut)), return_final_state=True)
    yb, hb = lrs.ssd_chunk_scan_fwd(**part(slice(cut, None)), h0=ha, return_final_state=True)
    torch.cuda.synchronize()
    ref, href = oracle.ssd_scan(**inp, return_final_state=True)
    _close(torch.cat([ya, yb], dim=1), ref, "bf16", "y (two calls)")
    _close(hb, href, "bf16", "h_final (two calls)")


def test_ssd_state_io_rejected_when_bidirectional(cuda_device):
    inp, opt = _ssd_case(1, 64, 1, 64, seed=1)
    with pytest.raises(lrs.SsmError):
        lrs.ssd_chunk_scan_fwd(**_dev(inp, cuda_device), bidirectional=True,
                               h0=opt["h0"].to(cuda_device))


def test_plain_entry_points_unchanged_by_empty_options(cuda_device):
    """Options that turn nothing on (dt_softplus=False alone) run the plain
    kernels: the same bits as the plain call."""
    inp = workloads.diag_inputs(2, 300, 64, 16, "bf16", seed=4)
    d = _dev(inp, cuda_device)
    y0 = lrs.ssm_scan_fwd(**d)
    y1 = lrs.ssm_scan_fwd(**d, dt_softplus=False)
    s = workloads.ssd_inputs(1, 300, 2, 64, 64, "bf16", seed=4)
    ds = _dev(s, cuda_device)
    z0 = lrs.ssd_chunk_scan_fwd(**ds)
    z1 = lrs.ssd_chunk_scan_fwd(**ds, dt_softplus=False)
    torch.cuda.synchronize()
    for a, b in ((y0, y1), (z0, z1)):
        assert torch.equal(a, b)


@pytest.mark.parametrize("Bs,L,H,N,G,bidir", [
    (2, 300, 4, 64, 2, False),
    (1, 700, 6, 128, 3, False),
    (2, 260, 4, 64, 4, True),     # one group per head
    (1, 400, 8, 128, 2, True),
])
def test_ssd_groups_of_B_C(cuda_device, Bs, L, H, N, G, bidir):
    inp = workloads.ssd_inputs(Bs, L, H, 64, N, "bf16", seed=L + G, groups=G)
    ref = oracle.ssd_scan(**inp, bidirectional=bidir)
    y = lrs.ssd_chunk_scan_fwd(**_dev(inp, cuda_device), chunk=128, bidirectional=bidir)
    torch.cuda.synchronize()
    _close(y, ref, "bf16", "y")


def test_ssd_groups_with_options(cuda_device):
    Bs, L, H, N, G = 2, 333, 4, 64, 2
    inp = workloads.ssd_inputs(Bs, L, H, 64, N, "bf16", seed=61, groups=G)
    opt = workloads.option_inputs((Bs, L, H, 64), (Bs, L, H), H, (Bs, H, 64, N), "bf16", 62)
    inp["dt"] = opt["delta_raw"]
    ref, href = oracle.ssd_scan(**inp, dt_bias=opt["dt_bias"], dt_softplus=True, z=opt["z"],
                                h0=opt["h0"], return_final_state=True)
    y, hf = lrs.ssd_chunk_scan_fwd(**_dev(inp, cuda_device), chunk=128,
                                   dt_bias=opt["dt_bias"].to(cuda_device), dt_softplus=True,
                                   z=opt["z"].to(cuda_device), h0=opt["h0"].to(cuda_device),
                                   return_final_state=True)
    torch.cuda.synchronize()
    _close(y, ref, "bf16", "y")
    _close(hf, href, "bf16", "h_final")


@pytest.mark.parametrize("Bs,L,H,N,chunk,bidir,calls", [
    (4, 4096, 32, 128, 256, False, 800),   # the SSD benchmark shape
    (32, 400, 8, 64, 128, True, 2000),     # the short bidirectional benchmark shape
])
def test_ssd_repeated_calls_with_options_stay_exact(cuda_device, Bs, L, H, N, chunk, bidir, calls):
    """Back-to-back calls at a benchmark shape, with every option the
    direction allows: no kernel gives up a bounded wait, and every call
    writes the same bits.  The hand-offs between a kernel's warp roles must
    not depend on how far one role runs ahead of another (a parity wait that
    could alias showed up as an abandoned wait about once in 2000 calls)."""
    inp, opt = _ssd_case(Bs, L, H, N, seed=5)
    d = _dev(inp, cuda_device)
    kw = dict(chunk=chunk, bidirectional=bidir, dt_bias=opt["dt_bias"].to(cuda_device),
              dt_softplus=True, dt_limit=LIMIT, z=opt["z"].to(cuda_device))
    if not bidir:
        kw.update(h0=opt["h0"].to(cuda_device))
    y = torch.empty(Bs, L, H, 64, dtype=torch.float32, device=cuda_device)
    lrs.ssd_chunk_scan_fwd(**d, y=y, **kw)
    y0 = y.clone()
    for i in range(calls):
        if i % 100 == 0:
            y.fill_(float("nan"))   # a call that wrote nothing cannot pass
        lrs.ssd_chunk_scan_fwd(**d, y=y, **kw)
        if i % 100 == 99:
            assert torch.equal(y, y0), "call %d differs from the first" % i
    lrs.ssm_check_device_errors(cuda_device)
    assert torch.equal(y, y0)
    assert bool(torch.isfinite(y0).all())
