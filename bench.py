#!/usr/bin/env python3
"""Benchmark of the selective-scan hot path on GB300.

A step is one call of the scan on one batch of synthetic input resident in
HBM.  The default workload is the largest of the method's five benchmark
configurations by element-steps: the chunked scalar-decay (SSD) scan with
bf16 inputs, Bs=4 L=4096 H=32 P=64 N=128, chunk 256, on the tensor cores;
``--workload`` selects any workload in ``workloads.py``.  The default run also
measures every one of the five configurations (``configs`` in the JSON line):
time per call, throughput, roofline fraction, whole-output parity against
the fp64 oracle and the oracle's own CPU rate.

Prints ONE JSON line (rank 0).  ``value`` is element-steps/s (Bs*L*ED*N per
step, ED = H*P for the chunked scan, both directions counted when
bidirectional) over all ranks.  Inputs rotate over several resident sets so
no step finds its inputs in L2 (> 2x L2 bytes between reuses).

``e2e`` is the same metric through the public API with host buffers: each
step copies its inputs from pinned host memory, makes the call and copies y
back to pinned host memory, the three on three streams over a few device
buffer sets so that one step's copies overlap its neighbours' calls.

``--impl reference`` times the fp64 CPU oracle on a bounded sample of the
same workload on this host's cores (the reference arm).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

DEFAULT_WORKLOAD = "ssd_bf16_Bs4_L4096_H32_P64_N128_Q256"
# The method's five benchmark configurations, in their order.
METHOD_CONFIGS = [w.name for w in workloads.WORKLOADS[:5]]
L2_BYTES = 129 * 1024 * 1024
METRIC = "scan throughput (Bs·L·ED·N element-steps/s) and HBM GB/s vs roofline, 1 GB300"
UNIT = "element-steps/s"
FALLBACK_HBM_GBS = 6800.0
NUM_SMS = 152
ALU_ELEM_PER_CLK_SM = 32.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse_args():
    p = argparse.ArgumentParser(description=__doc__)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(workloads.BY_NAME))
    p.add_argument("--no-cpu-baseline", action="store_true",
                   help="skip the CPU oracle leg (used for profiler runs)")
    p.add_argument("--quick", action="store_true",
                   help="timed steps only: no clock sampling, pre/post roll or e2e leg "
                        "(used for profiler runs)")
    p.add_argument("--no-configs", action="store_true",
                   help="skip the leg that measures each of the five benchmark configurations")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="target wall time of the CPU oracle sample")
    p.add_argument("--mode", choices=["fwd", "options", "bwd"], default="fwd",
                   help="fwd: the plain forward scan (the headline); options: the forward scan "
                        "with every option on (delta bias + softplus + clamp, silu gate, initial "
                        "and final state); bwd: the gradients (diagonal scan, or the chunked "
                        "scan's CUDA-core correctness path)")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    sm_max_mhz=float(d.get("sm_max_mhz", 2070.0)), source="measured")
    except (OSError, KeyError, ValueError):
        return dict(hbm_gbs=FALLBACK_HBM_GBS, bf16_tflops=FALLBACK_BF16_TFLOPS,
                    bf16_tflops_sustained=1700.0, sm_max_mhz=2070.0, source="fallback")


# ---------------------------------------------------------------------------
# Traffic figures from the committed ncu summaries
# ---------------------------------------------------------------------------

def kernel_source_hash(kind: str) -> str:
    """Hash of the sources of the kernels a workload kind runs: "diag", "ssd"
    (the unidirectional tensor-core kernel) or "bissd" (the short-sequence
    bidirectional passes)."""
    csrc = os.path.join(ROOT, "linear_recurrence_ssm_gb300", "csrc")
    srcs = {"diag": ["diag_scan.cuh", "diag_scan.cu"],
            "ssd": ["ssd_chunk_scan.cu", "tc_ptx.cuh"],
            "bissd": ["ssd_bidir.cu", "tc_ptx.cuh"]}[kind]
    h = hashlib.sha256()
    for p in [os.path.join(csrc, f) for f in srcs] + [os.path.join(csrc, "ssm_common.cuh")]:
        with open(p, encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def _code_only(src: str) -> str:
    """C++ source without comments and blank lines (a comment edit leaves the
    compiled kernel, and so the recorded counters, valid)."""
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    lines = []
    for line in src.splitlines():
        # drop a // comment unless the // sits inside a string literal
        cut = line.find("//")
        if cut >= 0 and line[:cut].count('"') % 2 == 0:
            line = line[:cut]
        line = line.rstrip()
        if line.strip():
            lines.append(line)
    return "\n".join(lines)


def short_bidir(w) -> bool:
    """Whether the library runs this SSD workload on the short-sequence
    bidirectional passes: bf16, P = N = 64, at most four 128-row tiles."""
    s = w.shape
    return (w.kind != "diag" and s["bidirectional"] and w.dtype == "bf16" and s["N"] == 64
            and s["P"] == 64 and (s["L"] + 127) // 128 <= 4)


def source_kind(w) -> str:
    if w.kind == "diag":
        return "diag"
    return "bissd" if short_bidir(w) else "ssd"


def ncu_traffic(workload: str, kind: str):
    """dram read+write bytes per launch recorded in profiles/, if the kernel
    source still hashes to the value recorded with the counters."""
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    want = kernel_source_hash(kind)
    for name in sorted(os.listdir(pdir)):
        if not name.endswith(".md"):
            continue
        text = open(os.path.join(pdir, name)).read()
        for m in re.finditer(r"traffic_per_launch\[(?P<w>[^\]]+)\]\s*=\s*(?P<b>[0-9]+)\s*bytes"
                             r"\s*source_hash=(?P<h>[0-9a-f]+)", text):
            if m.group("w") == workload and m.group("h") == want:
                return int(m.group("b"))
    return None


# ---------------------------------------------------------------------------
# Clock sampling (nvidia-smi) around the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self._t is not None:
                self._t.join(timeout=2)

    def summary(self, t0: float, t1: float):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if not (t0 <= ts <= t1):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# The hot path
# ---------------------------------------------------------------------------

def kernels_per_call(w, lrs) -> int:
    """Kernels one library call launches: the unidirectional chunked scan is
    one kernel, the bidirectional one two (chunk states, then outputs) for
    sequences of at most four 128-row tiles with N = 64 and one otherwise; the
    diagonal scan is one, or two when the library splits the sequence into
    time segments (segment pass + carry pass)."""
    if w.kind != "diag":
        return 2 if short_bidir(w) else 1
    s = w.shape
    _, _, k = lrs.ssm_scan_fwd_plan(s["Bs"], s["L"], s["ED"], s["N"], w.dtype == "bf16")
    return 2 if k > 1 else 1


class nvtx_range:
    """An NVTX range (named in profiler timelines) around a block; a no-op
    where NVTX is unavailable."""

    def __init__(self, name: str):
        self.name = name

    def __enter__(self):
        try:
            torch.cuda.nvtx.range_push(self.name)
            self.pushed = True
        except Exception:
            self.pushed = False
        return self

    def __exit__(self, *exc):
        if self.pushed:
            try:
                torch.cuda.nvtx.range_pop()
            except Exception:
                pass
        return False


def max_over_ranks(values, world: int, device):
    """Element-wise maximum of per-rank timings over all ranks (the slowest
    rank defines the step time); identity on one rank."""
    if world <= 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(values), device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def shard_seed(base_seed: int, rank: int) -> int:
    """Each rank draws its own batch of the workload (weak scaling)."""
    return base_seed + 1000 * rank


OPTION_LIMIT = (1e-4, 100.0)


def option_host_inputs(w, seed):
    """Seeded option inputs for the workload (delta / dt before activation,
    bias, gate z, initial state)."""
    s = w.shape
    if w.kind == "diag":
        return workloads.option_inputs((s["Bs"], s["L"], s["ED"]), (s["Bs"], s["L"], s["ED"]),
                                       s["ED"], (s["Bs"], s["ED"], s["N"]), w.dtype, seed + 7)
    state = None if s["bidirectional"] else (s["Bs"], s["H"], s["P"], s["N"])
    o = workloads.option_inputs((s["Bs"], s["L"], s["H"], s["P"]), (s["Bs"], s["L"], s["H"]),
                                s["H"], state or (1,), w.dtype, seed + 7)
    if state is None:
        o["h0"] = None
    return o


def make_step(w, lrs, bufs, mode="fwd"):
    s = w.shape
    if mode == "bwd" and w.kind == "diag":
        def step(i):
            b = bufs[i % len(bufs)]
            lrs.ssm_scan_bwd(b["x"], b["delta"], b["A"], b["B"], b["C"], b["D"], b["dy"])
    elif mode == "bwd":
        def step(i):
            b = bufs[i % len(bufs)]
            lrs.ssd_chunk_scan_bwd(b["x"], b["dt"], b["A_head"], b["B"], b["C"], b["D"], b["dy"],
                                   bidirectional=s["bidirectional"])
    elif w.kind == "diag":
        def step(i):
            b = bufs[i % len(bufs)]
            if mode == "options":
                lrs.ssm_scan_fwd(b["x"], b["delta_raw"], b["A"], b["B"], b["C"], b["D"], y=b["y"],
                                 dt_bias=b["dt_bias"], dt_softplus=True, dt_limit=OPTION_LIMIT,
                                 z=b["z"], h0=b["h0"], return_final_state=True)
            else:
                lrs.ssm_scan_fwd(b["x"], b["delta"], b["A"], b["B"], b["C"], b["D"], y=b["y"])
    else:
        def step(i):
            b = bufs[i % len(bufs)]
            if mode == "options":
                st = {} if s["bidirectional"] else dict(h0=b["h0"], return_final_state=True)
                lrs.ssd_chunk_scan_fwd(b["x"], b["delta_raw"], b["A_head"], b["B"], b["C"], b["D"],
                                       chunk=s["chunk"], bidirectional=s["bidirectional"],
                                       y=b["y"], dt_bias=b["dt_bias"], dt_softplus=True,
                                       dt_limit=OPTION_LIMIT, z=b["z"], **st)
            else:
                lrs.ssd_chunk_scan_fwd(b["x"], b["dt"], b["A_head"], b["B"], b["C"], b["D"],
                                       chunk=s["chunk"], bidirectional=s["bidirectional"],
                                       y=b["y"])
    return step


def mode_bytes(w, mode) -> int:
    """Algorithmic bytes of one call in the given mode (inputs read once,
    outputs written once)."""
    s = w.shape
    esz = 2 if w.dtype == "bf16" else 4
    if mode == "fwd":
        return w.algorithmic_bytes
    if mode == "options":
        if w.kind == "diag":
            xs, state = s["Bs"] * s["L"] * s["ED"], s["Bs"] * s["ED"] * s["N"]
            return w.algorithmic_bytes + xs * esz + 2 * state * 4 + s["ED"] * 4
        xs = s["Bs"] * s["L"] * s["H"] * s["P"]
        state = 0 if s["bidirectional"] else s["Bs"] * s["H"] * s["P"] * s["N"]
        return w.algorithmic_bytes + xs * esz + 2 * state * 4 + s["H"] * 4
    if w.kind != "diag":
        # backward of the chunked scan: x, dt, B, C, A, D, dy in; dx, ddt, dA, dB, dC, dD out
        xs, dts = s["Bs"] * s["L"] * s["H"] * s["P"], s["Bs"] * s["L"] * s["H"]
        bc = s["Bs"] * s["L"] * s.get("groups", 1) * s["N"]
        return (xs * esz + dts * esz + 2 * bc * esz + xs * 4 + xs * 4 + dts * 4 + 2 * bc * 4
                + 4 * s["H"] * 4)
    # backward of the diagonal scan: x, delta, B, C, A, D, dy in; dx, ddelta, dA, dB, dC, dD out
    xs, bc = s["Bs"] * s["L"] * s["ED"], s["Bs"] * s["L"] * s["N"]
    return (2 * xs * esz + 2 * bc * esz + xs * 4 + 2 * xs * 4 + 2 * bc * 4
            + 2 * s["ED"] * s["N"] * 4 + 2 * s["ED"] * 4)


def out_shape(w):
    s = w.shape
    if w.kind == "diag":
        return (s["Bs"], s["L"], s["ED"])
    return (s["Bs"], s["L"], s["H"], s["P"])


E2E_SETS = 3          # device buffer sets the end-to-end leg cycles through
L2_POLICY = "inputs rotate over resident sets, > 2x L2 bytes between reuses"


def compute_dtype(w) -> str:
    """Arithmetic type of the path: the diagonal scan computes in fp32 (bf16
    or fp32 inputs); the chunked scan's products run on bf16 tensor-core
    operands with fp32 accumulation and state (fp32 inputs: fp32 CUDA cores)."""
    if w.kind == "diag" or w.dtype == "f32":
        return "f32"
    return "bf16"


def bench_config(w, mode: str) -> dict:
    """The ``config`` object of a bench line; both arms print the same one."""
    return {"workload": w.name, **{k: v for k, v in w.shape.items()}, "mode": mode,
            "input_dtype": w.dtype, "state_dtype": "f32", "output_dtype": "f32",
            "l2": L2_POLICY, "parallelism": "replica per GPU (batch shards, no collective)"}


def roofline_of(w, mode: str, per_launch_s: float, peaks: dict, with_traffic: bool) -> dict:
    """Roofline of one call: the diagonal scan against the ALU bound (MUFU
    ex2), the chunked scan against HBM bandwidth, both of the measured peaks."""
    call_bytes = mode_bytes(w, mode)
    hbm_achieved = call_bytes / per_launch_s / 1e9
    if w.kind == "diag":
        # One exp2 on the special-function unit and four fp32 operations per
        # element-step; both the MUFU (32 ex2 / clk / SM) and the FMA pipe
        # (128 lanes / clk / SM) allow 32 element-steps / clk / SM.
        alu_peak = ALU_ELEM_PER_CLK_SM * NUM_SMS * peaks["sm_max_mhz"] * 1e6 / 1e12
        achieved = w.element_steps / per_launch_s / 1e12
        return {
            "bound": "alu", "achieved": round(achieved, 4), "peak": round(alu_peak, 4),
            "unit": "T element-steps/s", "frac": round(achieved / alu_peak, 4),
            "traffic": ncu_traffic(w.name, source_kind(w)) if (with_traffic and mode == "fwd") else None,
            "peak_source": "derived: 152 SMs x 32 ex2/clk/SM (MUFU) x sm_max_mhz of "
                           "MEASURED_PEAKS.json; 1 ex2 + 4 fp32 ops per element-step"
                           + ("" if mode != "bwd" else
                              " of the forward scan (the gradients re-run the forward twice "
                              "and do about twice its work on the way back)"),
            "hbm": {"achieved_gbs": round(hbm_achieved, 1), "peak_gbs": peaks["hbm_gbs"],
                    "frac": round(hbm_achieved / peaks["hbm_gbs"], 4),
                    "algorithmic_bytes_per_launch": call_bytes},
            "launch_us": round(per_launch_s * 1e6, 3),
        }
    return {
        "bound": "hbm", "achieved": round(hbm_achieved, 1), "peak": peaks["hbm_gbs"],
        "unit": "GB/s", "frac": round(hbm_achieved / peaks["hbm_gbs"], 4),
        "traffic": ncu_traffic(w.name, source_kind(w)) if (with_traffic and mode == "fwd") else None,
        "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs, burst copy)",
        "algorithmic_bytes_per_launch": call_bytes,
        "launch_us": round(per_launch_s * 1e6, 3),
    }


def resident_sets(w, host, dev, per_set: int):
    """Enough copies of the inputs (and a y each) that > 2x L2 bytes pass
    between two uses of one set (at least three sets)."""
    import torch
    nsets = max(3, -(-3 * L2_BYTES // per_set))
    bufs = []
    for _ in range(nsets):
        b = {n: (t.to(dev) if t is not None else None) for n, t in host.items()}
        b["y"] = torch.empty(out_shape(w), dtype=torch.float32, device=dev)
        bufs.append(b)
    return bufs


def time_steps(step, stream, dev, steps: int, warmup: int) -> float:
    """Milliseconds for `steps` back-to-back steps, CUDA events on the
    launching stream, synchronised on both sides; raises if a kernel gave up
    a bounded wait meanwhile (its output would be wrong)."""
    import linear_recurrence_ssm_gb300 as lrs
    import torch
    for i in range(max(3, warmup)):
        step(i)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for k in range(steps):
        step(k)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    lrs.ssm_check_device_errors(dev)
    return e0.elapsed_time(e1)


def configs_leg(lrs, dev, peaks, seconds_per_config: float = 2.0) -> dict:
    """Every one of the method's five configurations: time per call (inputs
    rotating as in the headline), throughput, roofline, the GPU's whole y
    against the fp64 oracle, and the oracle's rate on this host's cores."""
    import oracle
    import torch
    stream = torch.cuda.current_stream(dev)
    out = {}
    for name in METHOD_CONFIGS:
        w = workloads.BY_NAME[name]
        host = workloads.workload_inputs(w)
        per_set = mode_bytes(w, "fwd")
        bufs = resident_sets(w, host, dev, per_set)
        nsets = len(bufs)
        step = make_step(w, lrs, bufs, "fwd")
        # about 0.2 s of timed GPU work, at least 20 and at most 5000 calls
        probe_ms = time_steps(step, stream, dev, 5, 3) / 5
        steps = int(min(5000, max(20, 200.0 / max(probe_ms, 1e-3))))
        ms = time_steps(step, stream, dev, steps, 3)
        per_launch_s = ms / 1e3 / steps
        # the last step used set (steps - 1) % nsets; rerun set 0 for parity
        step(0)
        torch.cuda.synchronize(dev)
        y = bufs[0]["y"].double().cpu().numpy()
        del step, bufs
        torch.cuda.empty_cache()
        # the oracle on the whole workload, repeated to fill the time budget
        args = {k: oracle._f64(v) for k, v in host.items()}
        t0 = time.perf_counter()
        if w.kind == "diag":
            ref = oracle.diag_scan(**args)
        else:
            ref = oracle.ssd_scan(**args, bidirectional=w.shape["bidirectional"])
        t_one = time.perf_counter() - t0
        reps = max(1, int(seconds_per_config / max(t_one, 1e-3)))
        t0 = time.perf_counter()
        for _ in range(reps - 1):
            if w.kind == "diag":
                oracle.diag_scan(**args)
            else:
                oracle.ssd_scan(**args, bidirectional=w.shape["bidirectional"])
        t_all = t_one + (time.perf_counter() - t0)
        err = float(np.max(np.abs(y - ref)))
        scale = float(np.max(np.abs(ref)))
        bound = 1e-4 * max(1.0, scale) if w.dtype == "f32" else 2e-2 * scale
        out[name] = {
            "us_per_call": round(per_launch_s * 1e6, 3),
            "value": w.element_steps / per_launch_s, "unit": UNIT, "steps": steps,
            "dtype": compute_dtype(w), "roofline": roofline_of(w, "fwd", per_launch_s, peaks, True),
            "parity": {"max_abs_err": err, "ref_max_abs": scale, "bound": bound,
                       "ok": bool(err <= bound), "sample": "whole output"},
            "cpu_baseline": {"value": w.element_steps * reps / t_all, "unit": UNIT,
                             "cores": oracle.max_threads(), "kind": "oracle",
                             "sample": "whole workload, %d pass(es) in %.2f s "
                                       "(fp64 sequential C, OpenMP)" % (reps, t_all)},
            "l2": "%s (%d sets of %.2f MB)" % (L2_POLICY, nsets, per_set / 1e6),
        }
    return out


def run_ours(args, rank, world, local):
    import torch
    import torch.distributed as dist
    import linear_recurrence_ssm_gb300 as lrs

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the library has no CPU path)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    w = workloads.BY_NAME[args.workload]
    lrs.library()

    # Resident input/output sets; each rank draws its own batch (weak scaling).
    host = workloads.workload_inputs(
        workloads.Workload(w.name, w.kind, w.dtype, w.shape, seed=shard_seed(w.seed, rank)))
    if args.mode == "options":
        host.update(option_host_inputs(w, shard_seed(w.seed, rank)))
    if args.mode == "bwd":
        host["dy"] = workloads.grad_output(out_shape(w), seed=shard_seed(w.seed, rank) + 11)
    per_set = mode_bytes(w, args.mode)
    bufs = resident_sets(w, host, dev, per_set)
    nsets = len(bufs)
    step = make_step(w, lrs, bufs, args.mode)
    stream = torch.cuda.current_stream(dev)

    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize(dev)

    # Busy pre-roll so that clocks are sampled under load around the timed region.
    sampler = ClockSampler(local)
    roll = 0.0 if args.quick else 0.6
    if not args.quick:
        sampler.start()
    t_roll = time.time()
    i = 0
    while time.time() - t_roll < roll:
        for _ in range(50):
            step(i)
            i += 1
        torch.cuda.synchronize(dev)

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with nvtx_range("%s %s: %d timed steps" % (w.name, args.mode, args.steps)):
        e0.record(stream)
        for k in range(args.steps):
            step(k)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    if world > 1:
        dist.barrier()
    ms = e0.elapsed_time(e1)
    # Busy post-roll, then stop sampling.
    t_roll = time.time()
    while time.time() - t_roll < (0.0 if args.quick else 0.4):
        for _ in range(50):
            step(i)
            i += 1
        torch.cuda.synchronize(dev)
    sampler.stop()
    clocks = sampler.summary(t_wall0 - 0.6, t_wall1 + 0.4)
    lrs.ssm_check_device_errors(dev)   # no kernel gave up a bounded wait

    # End to end through the public API with host buffers: every step copies
    # its inputs from pinned host memory, makes the call and copies y back to
    # pinned host memory.  The three run on three streams over NB device
    # buffer sets, so that the copies of one step overlap the calls of its
    # neighbours (a set is refilled only once its previous call has read it
    # and its previous y has been copied out).
    pinned = {n: (t.pin_memory() if t is not None else None) for n, t in host.items()}
    y_host = torch.empty(out_shape(w), dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in pinned.values() if t is not None)
    d2h = y_host.numel() * 4
    k_e2e = 0 if (args.quick or args.mode == "bwd") else max(1, min(args.steps, 200))
    nb = min(nsets, E2E_SETS)
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    in_done = [torch.cuda.Event() for _ in range(nb)]
    comp_done = [torch.cuda.Event() for _ in range(nb)]
    out_done = [torch.cuda.Event() for _ in range(nb)]

    def e2e_step(k):
        j = k % nb
        with torch.cuda.stream(s_in):
            if k >= nb:
                s_in.wait_event(comp_done[j])      # the call of step k - nb has read set j
            for n, t in pinned.items():
                if t is not None:
                    bufs[j][n].copy_(t, non_blocking=True)
            in_done[j].record(s_in)
        stream.wait_event(in_done[j])
        if k >= nb:
            stream.wait_event(out_done[j])         # y of step k - nb has left set j
        step(j)
        comp_done[j].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[j])
            y_host.copy_(bufs[j]["y"], non_blocking=True)
            out_done[j].record(s_out)

    for k in range(0 if args.quick else 2 * nb):
        e2e_step(k)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    with nvtx_range("%s %s: %d end-to-end steps" % (w.name, args.mode, k_e2e)):
        f0.record(stream)
        s_in.wait_event(f0)
        s_out.wait_event(f0)
        for k in range(k_e2e):
            e2e_step(k)
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)
        f1.record(stream)
    torch.cuda.synchronize(dev)
    lrs.ssm_check_device_errors(dev)
    ms_e2e = f0.elapsed_time(f1) if k_e2e else float("nan")

    ms, ms_e2e = max_over_ranks([ms, ms_e2e], world, dev)

    units = w.element_steps
    value = units * args.steps * world / (ms / 1e3)
    e2e_value = units * k_e2e * world / (ms_e2e / 1e3) if k_e2e else None
    peaks = load_peaks()
    if args.mode == "bwd":
        # diagonal: checkpointing forward + reverse pass; chunked (P = 64, N =
        # 64 or 128): chunk-local states, the pass over chunks, the per-chunk
        # gradients and the finishing sums, per direction
        launches_per_step = 2 if w.kind == "diag" else 4 * (2 if w.shape["bidirectional"] else 1)
    else:
        launches_per_step = kernels_per_call(w, lrs)
    per_launch_s = ms / 1e3 / args.steps
    roofline = roofline_of(w, args.mode, per_launch_s, peaks, True)
    achieved = mode_bytes(w, args.mode) / per_launch_s / 1e9
    config = bench_config(w, args.mode)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": compute_dtype(w),
        "data": "synthetic (seeded, distributions of the workload definition)",
        "config": config,
        "hbm_gbs": round(achieved, 1),
        "roofline": roofline,
        "clocks": clocks,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": k_e2e,
                "pipeline": "H2D, call and D2H of each step on three streams over %d device "
                            "buffer sets" % nb},
        "gpu_launches": args.steps * launches_per_step,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.mode == "fwd":
        # bufs[0] holds the workload's inputs and the y of its last step
        line["cpu_baseline"], parity = cpu_baseline(w, args.cpu_seconds, y_gpu=bufs[0]["y"])
        line["parity"] = parity
    if rank == 0 and world == 1 and args.mode == "fwd" and not (args.quick or args.no_configs):
        del step, bufs
        torch.cuda.empty_cache()
        line["configs"] = configs_leg(lrs, dev, peaks)
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# CPU oracle baseline (the reference arm)
# ---------------------------------------------------------------------------

def _oracle_sample(w, host, units_per_call_target):
    """Slice a contiguous block of channels (diag) or heads (SSD) of every batch
    row; returns (callable, element-steps it computes, description, view), the
    callable returning the sample's y and view(y) picking the same part of a
    whole-workload y."""
    import oracle
    s = w.shape
    if w.kind == "diag":
        Bs, L, ED, N = s["Bs"], s["L"], s["ED"], s["N"]
        per_chan = L * N
        ne = max(1, min(ED, int(units_per_call_target // (per_chan * Bs))))
        sl = dict(x=host["x"][:, :, :ne].contiguous(), delta=host["delta"][:, :, :ne].contiguous(),
                  A=host["A"][:ne].contiguous(), B=host["B"], C=host["C"],
                  D=host["D"][:ne].contiguous())
        sl = {k: oracle._f64(v) for k, v in sl.items()}
        fn = lambda: oracle.diag_scan(**sl)
        return fn, Bs * L * ne * N, "%d of %d channels (e < %d) of all %d batch rows" % (
            ne * Bs, Bs * ED, ne, Bs), (lambda y: y[:, :, :ne])
    Bs, L, H, P, N = s["Bs"], s["L"], s["H"], s["P"], s["N"]
    dirs = 2 if s["bidirectional"] else 1
    per_head = L * P * N * dirs
    nb = max(1, min(Bs, int(units_per_call_target // (per_head * H)) or 1))
    nh = H if nb > 1 else max(1, min(H, int(units_per_call_target // per_head)))
    G = host["B"].shape[2]
    ng = G
    if G > 1:   # whole groups only: head h reads group h // (H / G)
        hpg = H // G
        ng = max(1, nh // hpg)
        nh = ng * hpg
    sl = dict(x=host["x"][:nb, :, :nh].contiguous(), dt=host["dt"][:nb, :, :nh].contiguous(),
              A_head=host["A_head"][:nh].contiguous(), B=host["B"][:nb, :, :ng].contiguous(),
              C=host["C"][:nb, :, :ng].contiguous(), D=host["D"][:nh].contiguous())
    sl = {k: oracle._f64(v) for k, v in sl.items()}
    fn = lambda: oracle.ssd_scan(**sl, bidirectional=s["bidirectional"])
    return (fn, nb * L * nh * P * N * dirs, "%d of %d (batch, head) pairs" % (nb * nh, Bs * H),
            (lambda y: y[:nb, :, :nh]))


def parity_on_sample(w, y_full, ref, view, desc):
    """The GPU's y against the oracle's on the CPU baseline's sample, with the
    tolerance of the input type (fp32: 1e-4 * max(1, max|y_ref|); bf16:
    2e-2 * max|y_ref|)."""
    got = view(y_full).double().cpu().numpy()
    err = float(np.max(np.abs(got - ref)))
    scale = float(np.max(np.abs(ref)))
    bound = 1e-4 * max(1.0, scale) if w.dtype == "f32" else 2e-2 * scale
    return {"max_abs_err": err, "ref_max_abs": scale, "bound": bound, "ok": bool(err <= bound),
            "sample": desc}


def cpu_baseline(w, seconds: float, y_gpu=None):
    """The oracle timed on a sample of the workload; with y_gpu (the GPU's y
    for the same inputs) also the parity of that sample.  Returns
    (cpu_baseline, parity or None)."""
    import oracle
    host = workloads.workload_inputs(w)
    cores = oracle.max_threads()
    # Calibrate on a small sample, then size the sample to ~`seconds`.
    fn, units, _, _ = _oracle_sample(w, host, 2e6)
    t0 = time.perf_counter()
    fn()
    rate = units / max(1e-6, time.perf_counter() - t0)
    fn, units, desc, view = _oracle_sample(w, host, rate * seconds)
    # The sample is capped at the whole workload: time one pass, then repeat
    # it until the time budget is filled.
    t0 = time.perf_counter()
    fn()
    t_one = time.perf_counter() - t0
    reps = max(1, min(500, int(round(seconds / max(t_one, 1e-3)))))
    t0 = time.perf_counter()
    for _ in range(reps):
        ref = fn()
    dt = time.perf_counter() - t0
    cb = {"value": units * reps / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
          "sample": "%s, %d pass(es); %.3g element-steps in %.2f s (fp64 sequential C, OpenMP)"
                    % (desc, reps, units * reps, dt)}
    parity = parity_on_sample(w, y_gpu, ref, view, desc) if y_gpu is not None else None
    return cb, parity


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    w = workloads.BY_NAME[args.workload]
    host = workloads.workload_inputs(w)
    cores = oracle.max_threads()
    budget = 150.0  # seconds for the whole warm-up + timed run
    fn, units, _, _ = _oracle_sample(w, host, 2e6)
    t0 = time.perf_counter()
    fn()
    rate = units / max(1e-6, time.perf_counter() - t0)
    per_step = max(0.05, budget / max(1, args.steps + args.warmup))
    fn, units, desc, _ = _oracle_sample(w, host, rate * per_step)
    for _ in range(args.warmup):
        fn()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        fn()
    dt = time.perf_counter() - t0
    value = units * args.steps / dt
    s = w.shape
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded, distributions of the workload definition)",
        "config": bench_config(w, "fwd"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": "each step: " + desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
