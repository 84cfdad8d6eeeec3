"""GPU parity of the diagonal selective scan against the fp64 oracle.

Every case runs the CUDA path through the C ABI (via the thin binding) on
seeded inputs and compares with the oracle run on the same (bf16-rounded)
values.  Tolerances: max|y - y_ref| <= 1e-4 * max(1, max|y_ref|) for fp32
inputs, <= 2e-2 * max|y_ref| for bf16 inputs.
"""
import numpy as np
import pytest
import torch

import linear_recurrence_ssm_gb300 as lrs
import oracle
import workloads

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-4
TOL_BF16 = 2e-2


def _to_dev(inp, dev):
    return {k: (v.to(dev) if v is not None else None) for k, v in inp.items()}


def _err(y, ref):
    return float(np.max(np.abs(y - ref)))


def _check(y_gpu, ref, dtype):
    y = y_gpu.double().cpu().numpy()
    assert np.all(np.isfinite(y))
    scale = float(np.max(np.abs(ref)))
    if dtype == "f32":
        bound = TOL_F32 * max(1.0, scale)
    else:
        bound = TOL_BF16 * scale
    err = _err(y, ref)
    assert err <= bound, "max abs err %.3e > bound %.3e (scale %.3e)" % (err, bound, scale)
    return err / max(scale, 1e-30)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("Bs,L,ED,N", [
    (2, 64, 64, 16),      # the fp32 benchmark shape
    (3, 100, 200, 16),    # several time tiles and channel tiles, ragged tails
    (1, 1, 8, 16),        # L = 1
    (2, 33, 128, 1),      # one state
    (1, 45, 24, 5),       # N not a multiple of 4 (padded states)
    (2, 40, 72, 17),      # N just above 16
    (1, 70, 136, 32),
    (1, 50, 40, 64),
    (2, 45, 40, 100),     # 128 padded states: 8 lanes per channel
    (1, 70, 24, 128),
    (2, 37, 20, 200),     # 256 padded states: 16 lanes per channel, 8 channels per CTA
    (1, 40, 16, 256),     # largest N
    (2, 31, 70, 16),      # ED*esize not a multiple of 16 (unvectorised loads for bf16)
    (1, 29, 3, 7),        # tiny odd shapes
])
def test_diag_matches_oracle(cuda_device, dtype, Bs, L, ED, N):
    inp = workloads.diag_inputs(Bs, L, ED, N, dtype, seed=Bs * 1000 + L + ED + N)
    ref = oracle.diag_scan(**inp)
    y = lrs.ssm_scan_fwd(**_to_dev(inp, cuda_device))
    torch.cuda.synchronize()
    _check(y, ref, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("Bs,L,ED,N", [
    (1, 4000, 256, 16),   # long sequence, few channels: split into time segments
    (2, 3000, 128, 7),
    (3, 700, 96, 12),
    (1, 600, 128, 16),
])
def test_time_split_matches_oracle(cuda_device, dtype, Bs, L, ED, N):
    inp = workloads.diag_inputs(Bs, L, ED, N, dtype, seed=L + ED)
    ref = oracle.diag_scan(**inp)
    y = lrs.ssm_scan_fwd(**_to_dev(inp, cuda_device))
    torch.cuda.synchronize()
    _check(y, ref, dtype)


def test_time_split_without_monotone_decay(cuda_device):
    # Some delta < 0 and some A > 0: the carried state's contribution can grow
    # again, so the second pass must not stop early.
    inp = workloads.diag_inputs(1, 900, 128, 16, "f32", seed=77)
    g = torch.Generator().manual_seed(1)
    inp["delta"] = (inp["delta"] - 0.05 * torch.rand(inp["delta"].shape, generator=g)).contiguous()
    inp["A"] = (0.1 * inp["A"]).contiguous()
    inp["A"][:, 0] = 0.002
    ref = oracle.diag_scan(**inp)
    y = lrs.ssm_scan_fwd(**_to_dev(inp, cuda_device))
    torch.cuda.synchronize()
    _check(y, ref, "f32")


def test_cumsum_worked_example_on_gpu(cuda_device):
    # a = 1, b = x = [1..8]: the scan is the page's cumsum, exact in fp32.
    x = torch.arange(1, 9, dtype=torch.float32).reshape(1, 8, 1)
    ones = torch.ones(1, 8, 1)
    y = lrs.ssm_scan_fwd(x.to(cuda_device), ones.to(cuda_device),
                         torch.zeros(1, 1, device=cuda_device), ones.to(cuda_device),
                         ones.to(cuda_device), None)
    assert y.cpu().flatten().tolist() == [1, 3, 6, 10, 15, 21, 28, 36]


def test_no_D_and_zero_input(cuda_device):
    inp = workloads.diag_inputs(2, 40, 64, 16, "bf16", seed=5, with_D=False)
    inp["x"] = torch.zeros_like(inp["x"])
    y = lrs.ssm_scan_fwd(**_to_dev(inp, cuda_device))
    assert torch.count_nonzero(y).item() == 0


@pytest.mark.parametrize("name", ["diag_bf16_Bs8_L2048_ED1536_N16",
                                  "diag_bf16_Bs16_L1000_ED2560_N16"])
def test_benchmark_shape_whole_output(cuda_device, name):
    """Full benchmark size in the launch configuration the benchmark times;
    the whole y against the oracle on the same inputs."""
    w = workloads.BY_NAME[name]
    inp = workloads.workload_inputs(w)
    y = lrs.ssm_scan_fwd(**_to_dev(inp, cuda_device)).cpu().double().numpy()
    ref = oracle.diag_scan(**inp)
    assert np.all(np.isfinite(y))
    err = float(np.max(np.abs(y - ref)))
    assert err <= TOL_BF16 * float(np.max(np.abs(ref))), err


def test_deterministic_and_guard_bands(cuda_device):
    inp = _to_dev(workloads.diag_inputs(2, 77, 96, 16, "bf16", seed=9), cuda_device)
    Bs, L, ED = inp["x"].shape
    n = Bs * L * ED
    guard = 4096
    buf = torch.full((n + 2 * guard,), float("nan"), device=cuda_device)
    y1 = buf[guard:guard + n].view(Bs, L, ED)
    lrs.ssm_scan_fwd(**inp, y=y1)
    y2 = lrs.ssm_scan_fwd(**inp)
    torch.cuda.synchronize()
    assert torch.isnan(buf[:guard]).all() and torch.isnan(buf[guard + n:]).all()
    assert torch.equal(y1, y2)


def test_runs_on_caller_stream(cuda_device):
    inp = _to_dev(workloads.diag_inputs(1, 64, 128, 16, "bf16", seed=3), cuda_device)
    ref = lrs.ssm_scan_fwd(**inp)
    s = torch.cuda.Stream(cuda_device)
    with torch.cuda.stream(s):
        y = lrs.ssm_scan_fwd(**inp)
    s.synchronize()
    assert torch.equal(y, ref)


def test_bad_dtype_is_rejected(cuda_device):
    inp = _to_dev(workloads.diag_inputs(1, 8, 8, 16, "f32", seed=1), cuda_device)
    inp["x"] = inp["x"].half()
    with pytest.raises(TypeError):
        lrs.ssm_scan_fwd(**inp)
