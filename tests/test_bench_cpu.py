"""Host-side logic of the benchmark that needs no GPU: the clock summary
taken from nvidia-smi samples during the timed region."""
import bench


def _line(sm, mx=2070, reasons=("Not Active",) * 4):
    # index, clocks.sm, clocks.max.sm, power.draw, clocks_event_reasons.active, then the four reasons
    return ", ".join(["0", str(sm), str(mx), "1200.00", "0x0000000000000004", *reasons])


def test_median_clock_and_reasons():
    lines = [(0.0, _line(1500)), (0.1, _line(1800, reasons=("Not Active", "Not Active", "Not Active", "Active"))),
             (0.2, _line(1900))]
    out = bench.summarize_clocks(lines)
    assert out == {"sm_mhz": 1800.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}


def test_window_keeps_only_samples_of_the_timed_region():
    lines = [(0.0, _line(600))] + [(1.0 + 0.05 * k, _line(1900 + k)) for k in range(5)] + [(9.0, _line(700))]
    out = bench.summarize_clocks(lines, window=(1.0, 1.2))
    assert out["samples"] == 5 and out["sm_mhz"] == 1902.0
    # fewer than three samples inside: every sample counts
    out = bench.summarize_clocks(lines, window=(1.0, 1.01))
    assert out["samples"] == 7


def test_malformed_lines_are_skipped():
    assert bench.summarize_clocks([(0.0, "[N/A]"), (0.1, "garbage")]) is None
    lines = [(0.0, "0, [N/A], 2070, 1.0, 0x0, Not Active, Not Active, Not Active, Not Active"), (0.1, _line(1650))]
    assert bench.summarize_clocks(lines)["samples"] == 1
