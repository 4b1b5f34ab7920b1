"""The bench harness's replay schedule against the worked example printed on
the "advanced SGEMM on NVIDIA GPUs" page (benchmark section)."""
import os

import bench

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "replay_schedule.txt")


def _golden():
    for line in open(GOLDEN):
        if line.strip() and not line.startswith("#"):
            size, runs, averaged = (int(x) for x in line.split())
            yield size, runs, averaged


def test_worked_example():
    for size, runs, averaged in _golden():
        assert bench.replay_count(size) == runs
        times = [float(i) for i in range(runs)]
        # the mean of the last `averaged` replays
        assert bench.second_half_mean(times) == sum(times[runs - averaged:]) / averaged


def test_sweep_range():
    sizes = bench.sweep_sizes()
    assert sizes[0] == 1024 and sizes[-1] == 12800 and len(sizes) == 93
    assert all(b - a == 128 for a, b in zip(sizes, sizes[1:]))
    # exp(0) = 1 at the first size; the count only falls as the size grows
    assert bench.replay_count(1024) == 1000
    counts = [bench.replay_count(s) for s in sizes]
    assert all(a >= b for a, b in zip(counts, counts[1:])) and counts[-1] >= 1


def test_clock_summary_keeps_samples_inside_timed_windows():
    """Only samples taken inside the named timed windows count; idle samples
    (NVML reason bit 0x1, or a clock below half the maximum) are not 'under
    load'; reason bits map to their names."""
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.samples = [(0.5, 1000.0, 2070.0, 0x0, 90.0),      # outside every window
                 (1.1, 1900.0, 2070.0, 0x0, 900.0),
                 (1.2, 1800.0, 2070.0, 0x4, 950.0),     # sw_power_cap
                 (1.9, 300.0, 2070.0, 0x1, 80.0),       # idle
                 (3.0, 2000.0, 2070.0, 0x8, 1000.0)]    # hw_slowdown, second window
    s.windows = {"a": [1.0, 2.0], "b": [2.5, 3.5]}
    s.source = "test"
    r = s.summary(["a"])
    assert r["samples"] == 3 and r["samples_under_load"] == 2
    assert r["sm_mhz"] == 1850 and r["sm_max_mhz"] == 2070 and r["reasons"] == ["sw_power_cap"]
    assert r["power_w_max"] == 950.0
    r = s.summary(["a", "b"])
    assert r["sm_mhz"] == 1900 and r["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert s.summary(["missing"])["sm_mhz"] is None
