"""The allocation-free entry point ssd_chunk_scan_fwd_noalloc (GPU).

Some callers cannot allocate device memory at all (all device memory is owned
by their own allocator, or the call sits where the memory pool must not be
touched).  For them the library keeps the bidirectional scan's scratch in a
fixed array of its own.  This test calls that entry point through the C ABI,
twice in a row on the same inputs, and checks each result against the
regular entry point ssd_chunk_scan_fwd and against the fp64 oracle, within
the tolerance the other GPU tests use (2e-2 of the largest output
magnitude).  It lives in a file of its
own, collected last, and passes alone in a fresh process or after the rest.
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


def _call_noalloc(inp, y, chunk, bidir):
    Bs, L, H, P = inp["x"].shape
    N = inp["B"].shape[-1]
    p = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lrs.library().ssd_chunk_scan_fwd_noalloc(
        p(inp["x"]), p(inp["dt"]), p(inp["A_head"]), p(inp["B"]), p(inp["C"]), p(inp["D"]), p(y),
        Bs, L, H, P, N, chunk, int(bidir), stream)


@pytest.mark.parametrize("Bs,L,H,N,chunk", [
    (32, 400, 8, 64, 128),    # the bidirectional benchmark shape: 8 MiB of scratch
    (2, 300, 3, 128, 256),
])
def test_noalloc_matches_regular_entry_point(Bs, L, H, N, chunk):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda:0")
    host = workloads.ssd_inputs(Bs, L, H, 64, N, "bf16", seed=Bs + L)
    inp = {k: (v.to(dev) if v is not None else None) for k, v in host.items()}
    ref = lrs.ssd_chunk_scan_fwd(**inp, chunk=chunk, bidirectional=True)
    scale = ref.abs().max().item()
    y_oracle = oracle.ssd_scan(**host, bidirectional=True)
    oscale = float(np.max(np.abs(y_oracle)))
    for _ in range(2):
        y = torch.full_like(ref, float("nan"))
        assert _call_noalloc(inp, y, chunk, True) == 0
        torch.cuda.synchronize()
        assert torch.isfinite(y).all()
        assert (y - ref).abs().max().item() <= TOL * scale
        err = float(np.max(np.abs(y.double().cpu().numpy() - y_oracle)))
        assert err <= TOL * oscale, (err, TOL * oscale)
    lrs.ssm_check_device_errors()
