"""Seeded synthetic inputs for the selective-scan workloads.

This module only draws random numbers; it holds none of the scan's arithmetic.
Both the GPU tests/benchmark and the CPU oracle take their inputs from here.

Value recipes (per the workload definitions of the diagonal and chunked scans):

* diagonal scan: x, B, C ~ N(0, 1); delta = softplus(N(0, 1) - 1);
  A[e, n] = -(n + 1) * exp(0.1 * N(0, 1)); D ~ N(0, 1).
* chunked scalar-decay scan: x ~ N(0, 1); dt = softplus(N(0, 1) - 2);
  A_head = -exp(U(0, log 16)); B, C ~ N(0, 1) / sqrt(N), shape (Bs, L, 1, N),
  one group shared by all heads; D ~ N(0, 1).

All draws are fp32 from one ``torch.Generator`` seeded with ``seed``, in the
order x, delta (or dt), A, B, C, D, then cast (round-to-nearest-even) to the
requested input dtype.  A and D always stay fp32.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch
import torch.nn.functional as F


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str            # "diag" or "ssd"
    dtype: str           # "f32" or "bf16" (x, delta/dt, B, C)
    shape: dict = field(default_factory=dict)
    seed: int = 0

    @property
    def element_steps(self) -> int:
        s = self.shape
        if self.kind == "diag":
            return s["Bs"] * s["L"] * s["ED"] * s["N"]
        dirs = 2 if s.get("bidirectional") else 1
        return s["Bs"] * s["L"] * s["H"] * s["P"] * s["N"] * dirs

    @property
    def algorithmic_bytes(self) -> int:
        """Inputs read once plus y (fp32) written once."""
        s = self.shape
        ib = 4 if self.dtype == "f32" else 2
        if self.kind == "diag":
            Bs, L, ED, N = s["Bs"], s["L"], s["ED"], s["N"]
            return (2 * Bs * L * ED * ib + 2 * Bs * L * N * ib + ED * N * 4 + ED * 4
                    + Bs * L * ED * 4)
        Bs, L, H, P, N = s["Bs"], s["L"], s["H"], s["P"], s["N"]
        G = s.get("groups", 1)
        return (Bs * L * H * P * ib + Bs * L * H * ib + 2 * Bs * L * G * N * ib + H * 4 + H * 4
                + Bs * L * H * P * 4)


# The five workloads of the method's benchmark table.
WORKLOADS = [
    Workload("diag_f32_Bs2_L64_ED64_N16", "diag", "f32",
             dict(Bs=2, L=64, ED=64, N=16), seed=0),
    Workload("diag_bf16_Bs8_L2048_ED1536_N16", "diag", "bf16",
             dict(Bs=8, L=2048, ED=1536, N=16), seed=1),
    Workload("diag_bf16_Bs16_L1000_ED2560_N16", "diag", "bf16",
             dict(Bs=16, L=1000, ED=2560, N=16), seed=2),
    Workload("ssd_bf16_Bs4_L4096_H32_P64_N128_Q256", "ssd", "bf16",
             dict(Bs=4, L=4096, H=32, P=64, N=128, chunk=256, bidirectional=False), seed=3),
    Workload("bissd_bf16_Bs32_L400_H8_P64_N64_Q128", "ssd", "bf16",
             dict(Bs=32, L=400, H=8, P=64, N=64, chunk=128, bidirectional=True), seed=4),
    # The widened paths at the chunked scan's benchmark shape (not in the
    # method's table): fp32 inputs, and eight groups of B, C (four heads each).
    Workload("ssd_f32_Bs4_L4096_H32_P64_N128_Q256", "ssd", "f32",
             dict(Bs=4, L=4096, H=32, P=64, N=128, chunk=256, bidirectional=False), seed=5),
    Workload("ssd_bf16_Bs4_L4096_H32_G8_P64_N128_Q256", "ssd", "bf16",
             dict(Bs=4, L=4096, H=32, P=64, N=128, chunk=256, bidirectional=False, groups=8),
             seed=6),
]
BY_NAME = {w.name: w for w in WORKLOADS}


def _cast(t: torch.Tensor, dtype: str) -> torch.Tensor:
    if dtype == "f32":
        return t.contiguous()
    if dtype == "bf16":
        return t.to(torch.bfloat16).contiguous()
    raise ValueError(dtype)


def diag_inputs(Bs: int, L: int, ED: int, N: int, dtype: str = "f32", seed: int = 0,
                with_D: bool = True):
    """Inputs of the diagonal scan on the CPU: dict(x, delta, A, B, C, D)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = torch.randn(Bs, L, ED, generator=g)
    delta = F.softplus(torch.randn(Bs, L, ED, generator=g) - 1.0)
    A = -(torch.arange(N, dtype=torch.float32) + 1.0)[None, :] * torch.exp(
        0.1 * torch.randn(ED, N, generator=g))
    B = torch.randn(Bs, L, N, generator=g)
    C = torch.randn(Bs, L, N, generator=g)
    D = torch.randn(ED, generator=g)
    return dict(x=_cast(x, dtype), delta=_cast(delta, dtype), A=A.contiguous(),
                B=_cast(B, dtype), C=_cast(C, dtype), D=D.contiguous() if with_D else None)


def ssd_inputs(Bs: int, L: int, H: int, P: int, N: int, dtype: str = "bf16", seed: int = 0,
               with_D: bool = True, groups: int = 1):
    """Inputs of the chunked scalar-decay scan on the CPU: dict(x, dt, A_head, B, C, D).

    B and C have shape (Bs, L, groups, N); one group (the default) is shared
    by all heads.
    """
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = torch.randn(Bs, L, H, P, generator=g)
    dt = F.softplus(torch.randn(Bs, L, H, generator=g) - 2.0)
    A_head = -torch.exp(torch.rand(H, generator=g) * math.log(16.0))
    B = torch.randn(Bs, L, groups, N, generator=g) / math.sqrt(N)
    C = torch.randn(Bs, L, groups, N, generator=g) / math.sqrt(N)
    D = torch.randn(H, generator=g)
    return dict(x=_cast(x, dtype), dt=_cast(dt, dtype), A_head=A_head.contiguous(),
                B=_cast(B, dtype), C=_cast(C, dtype), D=D.contiguous() if with_D else None)


def option_inputs(x_shape, delta_shape, channels: int, state_shape, dtype: str = "bf16",
                  seed: int = 0):
    """Seeded inputs of the scan options on the CPU: dict(delta_raw, dt_bias, z, h0).

    delta_raw ~ N(0, 1) - 1 (delta / dt before the optional bias, softplus and
    clamp), shaped ``delta_shape``; dt_bias ~ 0.5 N(0, 1) per channel (ED or H);
    z ~ N(0, 1) shaped like x; h0 ~ 0.5 N(0, 1), fp32, shaped ``state_shape``.
    """
    g = torch.Generator(device="cpu").manual_seed(seed)
    delta_raw = torch.randn(*delta_shape, generator=g) - 1.0
    dt_bias = 0.5 * torch.randn(channels, generator=g)
    z = torch.randn(*x_shape, generator=g)
    h0 = 0.5 * torch.randn(*state_shape, generator=g)
    return dict(delta_raw=_cast(delta_raw, dtype), dt_bias=dt_bias.contiguous(),
                z=_cast(z, dtype), h0=h0.contiguous())


def grad_output(shape, seed: int = 0):
    """A seeded upstream gradient dy ~ N(0, 1), fp32, of the given shape (CPU)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    return torch.randn(*shape, generator=g)


def workload_inputs(w: Workload):
    s = w.shape
    if w.kind == "diag":
        return diag_inputs(s["Bs"], s["L"], s["ED"], s["N"], w.dtype, w.seed)
    return ssd_inputs(s["Bs"], s["L"], s["H"], s["P"], s["N"], w.dtype, w.seed,
                      groups=s.get("groups", 1))
