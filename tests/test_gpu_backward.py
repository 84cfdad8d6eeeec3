"""GPU parity of the diagonal scan's gradients against the fp64 oracle.

``ssm_scan_bwd`` (C ABI, through the binding) and ``oracle.diag_scan_bwd``
(hand-written reverse mode, pinned by finite differences) run on the same
seeded, bf16-rounded inputs and upstream gradient.  Every gradient must
satisfy the scans' tolerance rule relative to its own scale:
max|g - g_ref| <= 1e-4 * max(1, max|g_ref|) for fp32 inputs, 2e-2 * max|g_ref|
for bf16 inputs (all arithmetic is fp32 in both cases; the bf16 bound is the
one of the bf16 scan configurations).
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
    err = float(np.max(np.abs(g - ref)))
    assert err <= bound, "%s: max abs err %.3e > bound %.3e (scale %.3e)" % (what, err, bound, scale)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("Bs,L,ED,N", [
    (2, 64, 64, 16),
    (3, 100, 200, 16),    # several segments and channel tiles, ragged tails
    (1, 1, 8, 16),        # L = 1
    (1, 45, 24, 5),       # padded states
    (2, 33, 70, 16),
    (1, 600, 128, 16),    # long sequence
    (2, 70, 96, 17),      # two groups of states, the second of one state
    (2, 50, 64, 32),      # two full groups
    (1, 90, 40, 40),      # three groups, the last ragged
    (1, 20, 16, 256),     # the largest state count: 16 groups
])
def test_gradients_match_oracle(cuda_device, dtype, Bs, L, ED, N):
    inp = workloads.diag_inputs(Bs, L, ED, N, dtype, seed=2 * L + ED + N)
    dy = workloads.grad_output((Bs, L, ED), seed=L + 1)
    ref = oracle.diag_scan_bwd(**inp, dy=dy)
    dev = {k: v.to(cuda_device) for k, v in inp.items()}
    got = lrs.ssm_scan_bwd(**dev, dy=dy.to(cuda_device))
    torch.cuda.synchronize()
    for k in ("dx", "ddelta", "dA", "dB", "dC", "dD"):
        _close(got[k], ref[k], dtype, k)


def test_gradients_without_D(cuda_device):
    inp = workloads.diag_inputs(2, 80, 64, 16, "bf16", seed=3, with_D=False)
    dy = workloads.grad_output((2, 80, 64), seed=4)
    ref = oracle.diag_scan_bwd(**inp, dy=dy)
    got = lrs.ssm_scan_bwd(**{k: (v.to(cuda_device) if v is not None else None)
                             for k, v in inp.items()}, dy=dy.to(cuda_device))
    torch.cuda.synchronize()
    assert got["dD"] is None
    for k in ("dx", "ddelta", "dA", "dB", "dC"):
        _close(got[k], ref[k], "bf16", k)


def test_unsupported_state_count(cuda_device):
    inp = workloads.diag_inputs(1, 16, 8, 257, "f32", seed=1)
    dy = workloads.grad_output((1, 16, 8), seed=2)
    with pytest.raises(lrs.SsmError):
        lrs.ssm_scan_bwd(**{k: v.to(cuda_device) for k, v in inp.items()}, dy=dy.to(cuda_device))


@pytest.mark.parametrize("a_scale", [1e-3, -1e-3])
def test_split_checkpoints_with_slow_or_growing_decay(cuda_device, a_scale):
    """A shape the forward splits into time segments (few channels, a long
    sequence): the checkpointing pass runs split, and the carry pass adds the
    carried state to the later segments' checkpoints.  With |A| tiny the
    carried part never decays below the cut-off (positive A: the cut-off is
    off), so every checkpoint of a later segment is corrected."""
    Bs, L, ED, N = 1, 1200, 64, 16
    inp = workloads.diag_inputs(Bs, L, ED, N, "f32", seed=41)
    inp["A"] = a_scale * torch.rand(ED, N, generator=torch.Generator().manual_seed(3))
    dy = workloads.grad_output((Bs, L, ED), seed=42)
    ref = oracle.diag_scan_bwd(**inp, dy=dy)
    dev = {k: v.to(cuda_device) for k, v in inp.items()}
    got = lrs.ssm_scan_bwd(**dev, dy=dy.to(cuda_device))
    torch.cuda.synchronize()
    for k in ("dx", "ddelta", "dA", "dB", "dC", "dD"):
        _close(got[k], ref[k], "f32", k)
    lrs.ssm_check_device_errors()
