"""Host checks of the workload definitions the benchmark and the tests share
(CPU only): the algorithmic byte count of each workload equals the bytes of
its inputs plus one fp32 y, the benchmark's oracle sample of a grouped
workload keeps whole groups, and its parity figure tells a right y from a
wrong one."""
import torch

import bench
import workloads


def test_algorithmic_bytes_are_inputs_plus_output():
    for w in workloads.WORKLOADS:
        inp = workloads.workload_inputs(w)
        in_bytes = sum(t.numel() * t.element_size() for t in inp.values() if t is not None)
        y_elems = inp["x"].numel()
        assert w.algorithmic_bytes == in_bytes + 4 * y_elems, w.name


def test_element_steps():
    for w in workloads.WORKLOADS:
        s = w.shape
        if w.kind == "diag":
            assert w.element_steps == s["Bs"] * s["L"] * s["ED"] * s["N"]
        else:
            dirs = 2 if s["bidirectional"] else 1
            assert w.element_steps == s["Bs"] * s["L"] * s["H"] * s["P"] * s["N"] * dirs


def test_grouped_oracle_sample_keeps_whole_groups():
    w = workloads.BY_NAME["ssd_bf16_Bs4_L4096_H32_G8_P64_N128_Q256"]
    host = workloads.workload_inputs(w)
    assert tuple(host["B"].shape) == (4, 4096, 8, 128)
    s = w.shape
    per_head = s["L"] * s["P"] * s["N"]
    # a target of 5 heads' work: one batch row, rounded down to one group of 4 heads
    fn, units, what, view = bench._oracle_sample(w, host, 5 * per_head)
    assert units == 4 * per_head
    y = fn()
    assert y.shape == (1, s["L"], 4, s["P"])
    assert tuple(view(torch.zeros(4, s["L"], s["H"], s["P"])).shape) == y.shape


def test_bench_parity_on_sample():
    """The benchmark's parity figure: the oracle's own y passes, a y off by
    more than the bf16 bound fails."""
    w = workloads.BY_NAME["diag_bf16_Bs8_L2048_ED1536_N16"]
    host = workloads.workload_inputs(w)
    fn, units, desc, view = bench._oracle_sample(w, host, 2e6)
    ref = fn()
    full = torch.zeros(8, 2048, 1536, dtype=torch.float32)
    view(full)[...] = torch.from_numpy(ref)
    p = bench.parity_on_sample(w, full, ref, view, desc)
    assert p["ok"] and p["max_abs_err"] < 1e-5 * p["ref_max_abs"]
    view(full)[0, 5, 0] += 0.05 * p["ref_max_abs"]
    assert not bench.parity_on_sample(w, full, ref, view, desc)["ok"]


def test_kernel_bookkeeping_of_the_benchmark():
    """Which kernels a workload runs, as the benchmark counts them: the
    short bidirectional SSD (bf16, P = N = 64, at most four 128-row tiles) is
    two passes and hashes the sources of ssd_bidir.cu; every other SSD
    workload is one kernel and hashes the tensor-core scan's sources."""
    by = workloads.BY_NAME
    short = by["bissd_bf16_Bs32_L400_H8_P64_N64_Q128"]
    uni = by["ssd_bf16_Bs4_L4096_H32_P64_N128_Q256"]
    assert bench.short_bidir(short) and not bench.short_bidir(uni)
    assert bench.kernels_per_call(short, None) == 2
    assert bench.kernels_per_call(uni, None) == 1
    assert bench.source_kind(short) == "bissd" and bench.source_kind(uni) == "ssd"
    assert bench.source_kind(by["diag_bf16_Bs8_L2048_ED1536_N16"]) == "diag"
    for w in workloads.WORKLOADS:
        if w.kind != "diag" and w.shape["bidirectional"]:
            s = w.shape
            fits = w.dtype == "bf16" and s["N"] == 64 and s["P"] == 64 and (s["L"] + 127) // 128 <= 4
            assert bench.short_bidir(w) == fits, w.name
    # the hashes of the three kernel families differ and ignore comments
    hashes = {k: bench.kernel_source_hash(k) for k in ("diag", "ssd", "bissd")}
    assert len(set(hashes.values())) == 3
    assert (bench._code_only("int a; // note\n\n/* block */ int b;")
            == bench._code_only("int a;\n/* another comment */ int b;  // x"))
