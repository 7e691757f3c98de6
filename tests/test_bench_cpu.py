"""Host-side logic of the benchmark that needs no GPU: the clock summary
taken from nvidia-smi samples during the timed region, and the metric's
NS5 FLOP count."""
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


def test_ns5_algorithmic_flop_counts():
    """The metric's NS5 count, 5 (4 r^2 c + 2 r^3) per matrix, over the DiT
    sets: 5.884e13 per 1.3B refresh, 1.804e15 per 15B refresh, 2.774e13 per
    MuonBP block step (blocks of the 1.3B set along the long side)."""
    from matrix_aware_optimizer_gb300 import synth
    one = sum(bench._ns_flops(*s) for s in synth.MATRIX_SETS["dit_1p3b"].shapes)
    big = sum(bench._ns_flops(*s) for s in synth.MATRIX_SETS["dit_15b"].shapes)
    ms = synth.MATRIX_SETS["dit_1p3b_muonbp"]
    blk = sum(bench._ns_flops(*b) for s in ms.shapes for b in bench._block_shapes(s[0], s[1], ms.blocks))
    assert one == 58841051955200
    assert abs(big / 1.804e15 - 1) < 1e-3
    assert abs(blk / 2.774e13 - 1) < 1e-3
    # a square matrix: 5 (4 + 2) r^3
    assert bench._ns_flops(64, 64) == 30 * 64 ** 3
