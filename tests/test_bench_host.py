"""Host-side helpers of bench.py, on the CPU: the clock-sample summary that
decides whether a run saw throttling, and the link line-granularity rule the
dense-GNN line uses for its ceiling."""
import importlib.util
import os

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def test_clock_summary_reads_reasons_and_median():
    b = _bench()
    c = b.ClockSampler(0)
    c.lines = [
        # index, sm, max sm, power, active mask, hw_slowdown, hw_thermal, sw_thermal, sw_power_cap
        "0, 2070, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1390.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 950.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
        "0, [N/A], 2070, 1.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    s = c.summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 2070 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]
    c.lines.append("0, 1500, 2070, 1000.0, 0x8, Active, Not Active, Active, Not Active")
    assert c.summary()["reasons"] == ["hw_slowdown", "sw_power_cap", "sw_thermal_slowdown"]
    assert b.ClockSampler(0).summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                                           "samples": 0}


def test_line_bytes_follow_the_measured_size_classes():
    """The transfers workload measured rows per microsecond constant within
    X in {16, 32}, {48, 64}, {80..128}, {144, 160}, {176, 192}, {208..256}
    bytes read from a 128-byte boundary: one cost per class, rising between
    classes."""
    b = _bench()
    classes = [(16, 32), (48, 64), (80, 96, 112, 128), (144, 160), (176, 192),
               (208, 224, 240, 256)]
    costs = []
    for cl in classes:
        c = b.line_bytes(np.array(cl))
        assert len(set(c.tolist())) == 1, cl
        costs.append(int(c[0]))
    assert costs == [32, 64, 128, 160, 192, 256]
    assert b.line_bytes(np.array([0, 4, 452, 512, 513])).tolist() == [0, 32, 512, 512, 544]


def test_clock_sampler_without_nvidia_smi_records_nothing():
    """Where nvidia-smi is missing (this CPU-only check), entering and leaving
    the sampler, edge samples included, raises nothing and records no sample."""
    b = _bench()
    import shutil
    if shutil.which("nvidia-smi"):
        return
    with b.ClockSampler(0) as c:
        pass
    assert c.summary()["samples"] == 0
