"""GPU parity of the chunked scan's CUDA-core path against the fp64 oracle.

Shapes and input types outside the tensor-core kernel (bf16, P = 64,
N in {64, 128}) run on the CUDA-core kernel: P and N in {16, 32, 64, 128,
256} and fp32 inputs.  P = 256 (and P = 128 with N = 256) is cut into row
slices owned by separate CTAs; N = 16 leaves half of each warp's lanes idle.  Tolerances as for
the scans: 1e-4 * max(1, max|ref|) for fp32 inputs, 2e-2 * max|ref| for bf16.
"""
import numpy as np
import pytest
import torch

import linear_recurrence_ssm_gb300 as lrs
import oracle
import workloads

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}


def _close(got, ref, dtype, what="y"):
    g = got.double().cpu().numpy()
    assert np.all(np.isfinite(g)), what + " has non-finite values"
    scale = float(np.max(np.abs(ref)))
    bound = TOL[dtype] * (max(1.0, scale) if dtype == "f32" else scale)
    err = float(np.max(np.abs(g - ref)))
    assert err <= bound, "%s: max abs err %.3e > bound %.3e (scale %.3e)" % (what, err, bound, scale)


def _dev(d, dev):
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("bidir", [False, True])
@pytest.mark.parametrize("Bs,L,H,P,N", [
    (2, 70, 3, 16, 32),
    (1, 200, 2, 32, 64),
    (2, 33, 2, 64, 32),
    (1, 150, 2, 128, 128),
    (1, 90, 1, 64, 256),
    (2, 17, 2, 16, 256),
    (1, 300, 2, 64, 128),     # the tensor-core shape, fp32 inputs take this path
    (2, 90, 2, 64, 16),       # N = 16
    (1, 70, 2, 256, 16),      # two 128-row slices, N = 16
    (1, 100, 2, 256, 64),
    (1, 130, 1, 128, 256),    # two 64-row slices
    (1, 60, 1, 256, 256),     # four 64-row slices, largest state
])
def test_general_path_matches_oracle(cuda_device, dtype, bidir, Bs, L, H, P, N):
    if dtype == "bf16" and P == 64 and N in (64, 128):
        pytest.skip("the tensor-core kernel's shape (covered by test_gpu_ssd)")
    inp = workloads.ssd_inputs(Bs, L, H, P, N, dtype, seed=L + P + N + bidir)
    ref = oracle.ssd_scan(**inp, bidirectional=bidir)
    y = lrs.ssd_chunk_scan_fwd(**_dev(inp, cuda_device), chunk=128, bidirectional=bidir)
    torch.cuda.synchronize()
    _close(y, ref, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_general_path_with_options_and_groups(cuda_device, dtype):
    Bs, L, H, P, N, G = 2, 180, 4, 32, 64, 2
    inp = workloads.ssd_inputs(Bs, L, H, P, N, dtype, seed=11, groups=G)
    opt = workloads.option_inputs((Bs, L, H, P), (Bs, L, H), H, (Bs, H, P, N), dtype, 12)
    inp["dt"] = opt["delta_raw"]
    ref, href = oracle.ssd_scan(**inp, dt_bias=opt["dt_bias"], dt_softplus=True,
                                dt_limit=(0.05, 2.0), z=opt["z"], h0=opt["h0"],
                                return_final_state=True)
    y, hf = lrs.ssd_chunk_scan_fwd(**_dev(inp, cuda_device), dt_bias=opt["dt_bias"].to(cuda_device),
                                   dt_softplus=True, dt_limit=(0.05, 2.0),
                                   z=opt["z"].to(cuda_device), h0=opt["h0"].to(cuda_device),
                                   return_final_state=True)
    torch.cuda.synchronize()
    _close(y, ref, dtype)
    _close(hf, href, dtype, "h_final")


@pytest.mark.parametrize("P,N", [(256, 16), (256, 256)])
def test_general_path_row_slices_with_state_io(cuda_device, P, N):
    """Initial and final states indexed by the slice's rows."""
    Bs, L, H = 1, 75, 2
    inp = workloads.ssd_inputs(Bs, L, H, P, N, "f32", seed=P + N)
    opt = workloads.option_inputs((Bs, L, H, P), (Bs, L, H), H, (Bs, H, P, N), "f32", P + N + 1)
    ref, href = oracle.ssd_scan(**inp, h0=opt["h0"], return_final_state=True)
    y, hf = lrs.ssd_chunk_scan_fwd(**_dev(inp, cuda_device), h0=opt["h0"].to(cuda_device),
                                   return_final_state=True)
    torch.cuda.synchronize()
    _close(y, ref, "f32")
    _close(hf, href, "f32", "h_final")


def test_general_path_bidirectional_gate(cuda_device):
    Bs, L, H, P, N = 1, 140, 2, 16, 128
    inp = workloads.ssd_inputs(Bs, L, H, P, N, "f32", seed=21)
    opt = workloads.option_inputs((Bs, L, H, P), (Bs, L, H), H, (Bs, H, P, N), "f32", 22)
    ref = oracle.ssd_scan(**inp, bidirectional=True, z=opt["z"])
    y = lrs.ssd_chunk_scan_fwd(**_dev(inp, cuda_device), bidirectional=True,
                               z=opt["z"].to(cuda_device))
    torch.cuda.synchronize()
    _close(y, ref, "f32")


def test_fp32_inputs_at_the_ssd_workload_size_sampled(cuda_device):
    """fp32 inputs at the SSD workload's size, checked on sampled heads."""
    w = workloads.BY_NAME["ssd_bf16_Bs4_L4096_H32_P64_N128_Q256"]
    s = w.shape
    inp = workloads.ssd_inputs(s["Bs"], s["L"], s["H"], s["P"], s["N"], "f32", seed=w.seed)
    y = lrs.ssd_chunk_scan_fwd(**_dev(inp, cuda_device), chunk=s["chunk"]).cpu().double().numpy()
    ref = oracle.ssd_scan(**inp, units=(5, 7))
    for u in (5, 6):
        b, h = divmod(u, s["H"])
        _close(torch.from_numpy(y[b, :, h]), ref[b, :, h], "f32", "y head %d" % u)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("Bs,L,H,P,N", [
    (4, 37, 80, 128, 64),    # 320 (b, h): 128-row slices, 16 rows per warp
    (2, 50, 160, 64, 128),   # 320 (b, h): 64-row slices, 8 rows per warp
    (2, 45, 160, 32, 32),    # 320 (b, h): 32-row slices, 4 rows per warp
])
def test_general_path_wide_slices(cuda_device, dtype, Bs, L, H, P, N):
    """Shapes with enough (b, h) pairs that the rows are not cut below the
    register limit, so each warp holds 4 to 16 rows of the state."""
    if dtype == "bf16" and P == 64 and N in (64, 128):
        pytest.skip("the tensor-core kernel's shape")
    inp = workloads.ssd_inputs(Bs, L, H, P, N, dtype, seed=L + P)
    for bidir in (False, True):
        ref = oracle.ssd_scan(**inp, bidirectional=bidir)
        y = lrs.ssd_chunk_scan_fwd(**_dev(inp, cuda_device), chunk=128, bidirectional=bidir)
        torch.cuda.synchronize()
        _close(y, ref, dtype)
