"""GPU parity of the chunked scan's gradients with its options.

``ssd_chunk_scan_bwd`` with the forward scan's options (dt bias, softplus,
clamp, the silu gate z, the initial state h0) calls ``ssd_chunk_scan_bwd_ex``
through the C ABI; ``oracle.ssd_scan_bwd_ex`` (fp64, pinned by finite
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
KEYS = ("dx", "ddt", "dA", "dB", "dC", "dD", "dz", "ddt_bias", "dh0")


def _close(got, ref, dtype, what):
    g = got.double().cpu().numpy()
    assert np.all(np.isfinite(g)), what + " has non-finite values"
    scale = float(np.max(np.abs(ref)))
    bound = TOL[dtype] * (max(1.0, scale) if dtype == "f32" else scale)
    err = float(np.max(np.abs(g - ref)))
    assert err <= bound, "%s: max abs err %.3e > bound %.3e (scale %.3e)" % (what, err, bound, scale)


def _run(Bs, L, H, P, N, G, bidir, dtype, opts, seed):
    inp = workloads.ssd_inputs(Bs, L, H, P, N, dtype, seed=seed, groups=G)
    if G == 1:
        inp["B"], inp["C"] = inp["B"][:, :, 0].contiguous(), inp["C"][:, :, 0].contiguous()
    o = workloads.option_inputs((Bs, L, H, P), (Bs, L, H), H, (Bs, H, P, N), dtype, seed + 1)
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
        inp["dt"] = o["delta_raw"]          # dt before the options
    dy = workloads.grad_output((Bs, L, H, P), seed=seed + 2)
    ref = oracle.ssd_scan_bwd_ex(**inp, dy=dy, bidirectional=bidir, **kw)
    dev = lambda t: t.to("cuda:0") if isinstance(t, torch.Tensor) else t
    got = lrs.ssd_chunk_scan_bwd(**{k: dev(v) for k, v in inp.items()}, dy=dev(dy),
                                 bidirectional=bidir, **{k: dev(v) for k, v in kw.items()})
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
    _run(2, 45, 3, 32, 64, 1, False, dtype, opts, seed=len(opts) * 7 + (dtype == "bf16"))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_option_gradients_bidirectional_and_groups(cuda_device, dtype):
    # the bidirectional scan takes every option but the initial state
    _run(1, 60, 4, 64, 64, 2, True, dtype, {"bias", "softplus", "limit", "z"}, seed=31)


@pytest.mark.parametrize("Bs,L,H,P,N", [
    (1, 1, 2, 16, 32),       # L = 1
    (1, 37, 2, 128, 64),     # the largest state the gradients take
    (2, 40, 2, 16, 256),
])
def test_option_gradients_shapes(cuda_device, Bs, L, H, P, N):
    _run(Bs, L, H, P, N, 1, False, "f32", {"bias", "softplus", "z", "h0"}, seed=L + P + N)


def test_h_final_is_refused(cuda_device):
    inp = workloads.ssd_inputs(1, 8, 2, 16, 32, "f32", seed=1)
    dy = workloads.grad_output((1, 8, 2, 16), seed=2)
    with pytest.raises(TypeError):
        lrs.ssd_chunk_scan_bwd(**{k: v.cuda() for k, v in inp.items()}, dy=dy.cuda(),
                               return_final_state=True)
