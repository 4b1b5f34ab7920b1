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


def test_clock_summary_parses_nvidia_smi_rows():
    rows = [["0", "t", "1900", "2070", "900.1", "0x0", "Not Active", "Not Active", "Not Active", "Active"],
            ["0", "t", "1800", "2070", "950.0", "0x4", "Not Active", "Not Active", "Not Active", "Not Active"],
            ["0", "t", "300", "2070", "90.0", "0x1", "Not Active", "Not Active", "Not Active", "Not Active"]]
    s = bench.ClockSampler._summary(rows)
    assert s["sm_mhz"] == 1850 and s["sm_max_mhz"] == 2070 and s["reasons"] == ["sw_power_cap"]
