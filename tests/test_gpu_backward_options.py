"""GPU parity of the diagonal scan's gradients with its options.

``ssm_scan_bwd`` with the forward scan's options (delta bias, softplus,
clamp, the silu gate z, the initial state h0) calls ``ssm_scan_bwd_ex``
through the C ABI; ``oracle.diag_scan_bwd_ex`` (fp64, pinned by finite
differences) runs on the same seeded, bf16-rounded inputs.  Every gradient --
dz, ddt_bias and dh0 among them -- satisfies the scans' tolerance rule
relative to its own scale: max|g - g_ref| <= 1e-4 * max(1, max|g_ref|) for
fp32 inputs, 2e-2 * max|g_ref| for bf16 inputs.
"""
import numpy as np
import pytest
import torch

import linear_recurrence_ssm_gb300 as lrs
import oracle
import workloads

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}
KEYS = ("dx", "ddelta", "dA", "dB", "dC", "dD", "dz", "ddt_bias", "dh0")


def _close(got, ref, dtype, what):
    g = got.double().cpu().numpy()
    assert np.all(np.isfinite(g)), what + " has non-finite values"
    scale = float(np.max(np.abs(ref)))
    bound = TOL[dtype] * (max(1.0, scale) if dtype == "f32" else scale)
    err = float(np.max(np.abs(g - ref)))
    assert err <= bound, "%s: max abs err %.3e > bound %.3e (scale %.3e)" % (what, err, bound, scale)


def _run(Bs, L, ED, N, dtype, opts, seed):
    inp = workloads.diag_inputs(Bs, L, ED, N, dtype, seed=seed)
    o = workloads.option_inputs((Bs, L, ED), (Bs, L, ED), ED, (Bs, ED, N), dtype, seed + 1)
    kw = {}
    if "bias" in opts:
        kw["dt_bias"] = o["dt_bias"]
    if "softplus" in opts:
        kw["dt_softplus"] = True
    if "limit" in opts:
        kw["dt_limit"] = (0.05, 2.0)
    if "z" in opts:
        kw["z"] = o["z"]
    if "h0" in opts:
        kw["h0"] = o["h0"]
    if opts & {"bias", "softplus", "limit"}:
        inp["delta"] = o["delta_raw"]        # delta before the options
    dy = workloads.grad_output((Bs, L, ED), seed=seed + 2)
    ref = oracle.diag_scan_bwd_ex(**inp, dy=dy, **kw)
    dev = lambda t: t.to("cuda:0") if isinstance(t, torch.Tensor) else t
    got = lrs.ssm_scan_bwd(**{k: dev(v) for k, v in inp.items()}, dy=dev(dy),
                           **{k: dev(v) for k, v in kw.items()})
    torch.cuda.synchronize()
    for k in KEYS:
        if ref.get(k) is None:
            assert got.get(k) is None, k
            continue
        assert tuple(got[k].shape) == ref[k].shape, k
        _close(got[k], ref[k], dtype, k)
    lrs.ssm_check_device_errors()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("opts", [
    {"bias", "softplus", "limit", "z", "h0"},
    {"bias", "softplus"},
    {"limit"},
    {"z"},
    {"h0"},
])
def test_option_gradients_match_oracle(cuda_device, dtype, opts):
    _run(2, 70, 96, 16, dtype, opts, seed=len(opts) * 5 + (dtype == "bf16"))


@pytest.mark.parametrize("Bs,L,ED,N", [
    (1, 1, 8, 16),        # L = 1
    (1, 45, 24, 5),       # padded states
    (2, 600, 130, 16),    # long sequence (split into time segments), ragged channel tile
    (2, 60, 48, 40),      # three groups of states, the last ragged
])
def test_option_gradients_shapes(cuda_device, Bs, L, ED, N):
    _run(Bs, L, ED, N, "f32", {"bias", "softplus", "z", "h0"}, seed=L + ED + N)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_option_gradients_many_states(cuda_device, dtype):
    _run(1, 40, 32, 64, dtype, {"bias", "softplus", "limit", "z", "h0"}, seed=91)
