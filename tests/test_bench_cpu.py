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


def test_leg_selection():
    a = bench.parse_args([])
    assert bench.leg_names(a) == ["dit_1p3b_muonbp", "dit_15b"]
    assert bench.leg_names(bench.parse_args(["--legs", "none"])) == []
    assert bench.leg_names(bench.parse_args(["--workload", "dit_15b"])) == []
    # the headline workload is never repeated as a leg
    assert bench.leg_names(bench.parse_args(["--workload", "dit_15b", "--legs", "dit_15b,dit_1p3b_muonbp"])) == \
        ["dit_1p3b_muonbp"]


def test_rate_summaries_are_fractions_of_the_peaks():
    """Executed NS5 rate and RowNorm bandwidth from per-family totals: the
    NS5 fraction divides executed FLOPs (what the launches compute) by the
    GEMM time; the metric count over the same time is reported beside it."""
    fam = {k: dict(ms=0.0, records=0, kernels=0, work=0.0) for k in
           ("rownorm_wide", "rownorm_tall", "ns_prep", "ns_gram", "ns_poly", "ns_combine", "ns_sym", "ns_small")}
    fam["ns_gram"].update(ms=2.0, records=1, work=3.0e12)
    fam["ns_combine"].update(ms=3.0, records=1, work=5.0e12)
    out = bench.ns5_summary(fam, alg_flops=1.2e13, cycles=2, tf_sus=1600.0, tf_burst=1900.0)
    assert out["gemm_ms_per_cycle"] == 2.5
    assert out["tflops_executed"] == 1600.0 and out["frac_executed"] == 1.0
    assert out["tflops_metric_count"] == 2400.0
    fam["rownorm_wide"].update(ms=1.0, records=2, work=6.0e9)
    fam["rownorm_tall"].update(ms=1.0, records=2, work=4.0e9)
    rn = bench.rownorm_summary(fam, hbm=6000.0)
    assert rn["wide"] == {"gbs": 6000.0, "frac": 1.0} and rn["tall"]["frac"] == round(4000 / 6000, 4)
    assert rn["gbs"] == 5000.0


def test_oracle_sample_is_bounded_and_labelled():
    """The one sampling both arms use: on the tiny set it times a 64 x 64 NS5
    and the RowNorm of every shape, well under a second, and says so."""
    from matrix_aware_optimizer_gb300 import synth
    v, sample, secs = bench.oracle_cycle_sample(synth.MATRIX_SETS["tiny"])
    assert v > 0 and secs < 5.0
    assert sample.startswith("timed:") and "64x64" in sample


def test_traffic_digest_follows_code_not_comments():
    """A stored DRAM figure stays valid across comment edits of its kernel's
    source and is dropped when the code changes."""
    from matrix_aware_optimizer_gb300 import build
    a = b"int f(int x) {  // doubles x\n  return 2 * x;  /* twice */\n}\n"
    b = b"// a new header line\nint f(int x) {  // twice x\n\n  return 2 * x;\n}\n"
    c = b"int f(int x) {  // doubles x\n  return 3 * x;\n}\n"
    assert build._code_only(a) == build._code_only(b)
    assert build._code_only(a) != build._code_only(c)
    digests = {f: build.source_digest(f) for f in build.FAMILY_SOURCES}
    assert len(set(digests.values())) == len(set(build.FAMILY_SOURCES.values()))  # one per kernel source
    traffic = bench.load_traffic()
    assert set(traffic) <= set(build.FAMILY_SOURCES)
