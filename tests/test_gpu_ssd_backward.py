"""GPU parity of the chunked scan's gradients against the fp64 oracle.

``ssd_chunk_scan_bwd`` (C ABI, through the binding) and
``oracle.ssd_scan_bwd`` (hand-written reverse mode, pinned by finite
differences) run on the same seeded, bf16-rounded inputs and upstream
gradient.  Every gradient satisfies the scans' tolerance rule relative to its
own scale: max|g - g_ref| <= 1e-4 * max(1, max|g_ref|) for fp32 inputs,
2e-2 * max|g_ref| for bf16 inputs.  A reference that is exactly zero (dA for
a one-step sequence: no earlier state) gives that relative rule no scale;
there max|g| <= 1e-6 (the chunked form's dA is a difference of two equal
terms at L = 1 and keeps their rounding residue, ~1e-9).
"""
import numpy as np
import pytest
import torch

import linear_recurrence_ssm_gb300 as lrs
import oracle
import workloads

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}


def _close(got, ref, dtype, what):
    g = got.double().cpu().numpy()
    assert np.all(np.isfinite(g)), what + " has non-finite values"
    scale = float(np.max(np.abs(ref)))
    bound = TOL[dtype] * (max(1.0, scale) if dtype == "f32" else scale)
    if scale == 0.0:
        bound = 1e-6
    err = float(np.max(np.abs(g - ref)))
    assert err <= bound, "%s: max abs err %.3e > bound %.3e (scale %.3e)" % (what, err, bound, scale)


@pytest.mark.parametrize("Bs,L,H,P,N,G,bidir,dtype", [
    (2, 50, 2, 16, 32, 1, False, "f32"),
    (1, 70, 2, 32, 64, 1, True, "f32"),
    (2, 40, 4, 64, 128, 2, False, "bf16"),   # groups: dB, dC sum over a group's heads
    (1, 33, 2, 64, 64, 1, True, "bf16"),
    (1, 20, 4, 128, 64, 2, True, "f32"),
    (1, 25, 1, 32, 256, 1, False, "bf16"),
    (1, 1, 2, 16, 32, 1, True, "f32"),       # L = 1
])
def test_gradients_match_oracle(cuda_device, Bs, L, H, P, N, G, bidir, dtype):
    inp = workloads.ssd_inputs(Bs, L, H, P, N, dtype, seed=L + P + N + G, groups=G)
    if G == 1:       # the one-group layout (Bs, L, N) as the forward scan also takes it
        inp["B"], inp["C"] = inp["B"][:, :, 0].contiguous(), inp["C"][:, :, 0].contiguous()
    dy = workloads.grad_output((Bs, L, H, P), seed=L + 3)
    ref = oracle.ssd_scan_bwd(**inp, dy=dy, bidirectional=bidir)
    dev = {k: v.to(cuda_device) for k, v in inp.items()}
    got = lrs.ssd_chunk_scan_bwd(**dev, dy=dy.to(cuda_device), bidirectional=bidir)
    torch.cuda.synchronize()
    for k in ("dx", "ddt", "dA", "dB", "dC", "dD"):
        assert tuple(got[k].shape) == ref[k].shape, k
        _close(got[k], ref[k], dtype, k)
    lrs.ssm_check_device_errors()


def test_gradients_without_D(cuda_device):
    inp = workloads.ssd_inputs(1, 30, 2, 32, 64, "f32", seed=5, with_D=False)
    dy = workloads.grad_output((1, 30, 2, 32), seed=6)
    ref = oracle.ssd_scan_bwd(**inp, dy=dy)
    got = lrs.ssd_chunk_scan_bwd(**{k: (v.to(cuda_device) if v is not None else None)
                                    for k, v in inp.items()}, dy=dy.to(cuda_device))
    torch.cuda.synchronize()
    assert got["dD"] is None
    for k in ("dx", "ddt", "dA", "dB", "dC"):
        _close(got[k], ref[k], "f32", k)


def test_unsupported_size_is_rejected(cuda_device):
    inp = workloads.ssd_inputs(1, 8, 2, 128, 128, "f32", seed=1)
    dy = workloads.grad_output((1, 8, 2, 128), seed=2)
    with pytest.raises(lrs.SsmError):
        lrs.ssd_chunk_scan_bwd(**{k: v.to(cuda_device) for k, v in inp.items()},
                               dy=dy.to(cuda_device))


@pytest.mark.parametrize("L", [1, 63, 64, 65, 129, 200])
@pytest.mark.parametrize("N,G,bidir,dtype", [
    (64, 1, True, "bf16"),
    (128, 2, False, "f32"),
    (128, 1, True, "f32"),
])
def test_chunked_form_around_chunk_lengths(cuda_device, L, N, G, bidir, dtype):
    """P = 64 and N = 64 or 128 take the chunked form (64-step chunks): one
    step, one step short of and past a chunk, ragged last chunks, with
    groups, both directions and fp32 or bf16 inputs."""
    Bs, H, P = 2, 4, 64
    inp = workloads.ssd_inputs(Bs, L, H, P, N, dtype, seed=7 * L + N + G, groups=G)
    dy = workloads.grad_output((Bs, L, H, P), seed=L + 11)
    ref = oracle.ssd_scan_bwd(**inp, dy=dy, bidirectional=bidir)
    dev = {k: v.to(cuda_device) for k, v in inp.items()}
    got = lrs.ssd_chunk_scan_bwd(**dev, dy=dy.to(cuda_device), bidirectional=bidir)
    torch.cuda.synchronize()
    for k in ("dx", "ddt", "dA", "dB", "dC", "dD"):
        _close(got[k], ref[k], dtype, k)
    lrs.ssm_check_device_errors()
