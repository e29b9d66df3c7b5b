"""Host-side helpers of bench.py (no GPU): clock-sample parsing and throttle
reasons, the peak fallback, and the kernel-source hash that gates the
recorded DRAM traffic."""
import json
import os

import bench


def test_clock_summary_median_and_reasons():
    cs = bench.ClockSampler(0)
    cs.lines = [(10.0, "1980, 2070, 900.1, Not Active, Not Active, Not Active, Not Active"),
                (10.1, "2070, 2070, 1200.5, Not Active, Not Active, Not Active, Active"),
                (10.2, "2070, 2070, 1250.0, Not Active, Not Active, Not Active, Active"),
                (20.0, "300, 2070, 100.0, Active, Not Active, Not Active, Not Active"),   # outside the window
                (10.3, "garbage line")]
    s = cs.summary(9.9, 10.5)
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_summary_without_samples():
    s = bench.ClockSampler(0).summary(0, 1)
    assert s["samples"] == 0 and s["sm_mhz"] is None


def test_measured_peak_or_fallback(tmp_path, monkeypatch):
    peak, kind = bench.measured_peaks()
    if os.path.exists(os.path.join(bench.ROOT, "MEASURED_PEAKS.json")):
        with open(os.path.join(bench.ROOT, "MEASURED_PEAKS.json")) as fh:
            assert peak == json.load(fh)["hbm_gbs"] and kind == "measured"
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peaks() == (bench.FALLBACK_HBM_GBS, "fallback")


def test_source_hash_is_stable_and_tracks_the_kernel_files():
    a, b = bench.sources_sha(), bench.sources_sha()
    assert a == b and len(a) == 16
    assert all(os.path.exists(os.path.join(bench.ROOT, f)) for f in bench.KERNEL_SOURCES)


def test_cpu_model_is_named():
    m = bench.cpu_model()
    assert isinstance(m, str) and m


def test_oracle_per_config_covers_every_measured_configuration():
    rows = bench.oracle_per_config(reps=1)
    names = [r["workload"] for r in rows]
    want = [bench.W.C1] + bench.W.C3 + [bench.W.C4, bench.W.C4_B15] + bench.W.C5
    assert names == [w.name for w in want]
    for r, w in zip(rows, want):
        assert r["elements_per_rank"] == min(w.count, bench.ORACLE_SAMPLE)
        assert r["whole"] == (w.count <= bench.ORACLE_SAMPLE)
        assert r["us_per_call"] > 0 and r["GBps"] > 0
