"""Host checks of the workload definitions the benchmark and the tests share
(CPU only): the algorithmic byte count of each workload equals the bytes of
its inputs plus one fp32 y, and the benchmark's oracle sample of a grouped
workload keeps whole groups."""
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
    fn, units, what = bench._oracle_sample(w, host, 5 * per_head)
    assert units == 4 * per_head
    y = fn()
    assert y.shape == (1, s["L"], 4, s["P"])
