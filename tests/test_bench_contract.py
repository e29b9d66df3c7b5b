"""The JSON line bench.py prints: every key the measurement contract names,
for the reference arm (on the CPU) and for our arm (on the GPU)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _line(args, timeout):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT, capture_output=True,
                         text=True, timeout=timeout)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


def _common(d):
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "e2e", "cpu_baseline"):
        assert k in d, k
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["vs_baseline"] is None and d["value"] > 0 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "rsag_8x64MiB_fp16"
    for k in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"):
        assert k in d["e2e"], k


def test_reference_arm_line():
    d = _line(["--impl", "reference", "--steps", "3", "--warmup", "3"], timeout=600)
    _common(d)
    assert d["impl"] == "reference" and d["steps"] == 3 and d["warmup"] == 3
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0


def test_warmup_below_three_is_refused():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2"], cwd=ROOT,
                         capture_output=True, text=True, timeout=120)
    assert out.returncode != 0 and "--warmup" in out.stderr


@pytest.mark.gpu
def test_gpu_arm_line():
    d = _line(["--steps", "5", "--warmup", "3", "--settle-s", "0", "--no-rows", "--no-cpu-baseline"], timeout=900)
    _common(d)
    assert "impl" not in d or d["impl"] != "reference"
    r = d["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in r, k
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    assert 0.5 < r["frac"] < 1.2
    e = d["e2e"]
    assert e["h2d_bytes_per_step"] == e["d2h_bytes_per_step"] == 8 * 64 * 2 ** 20
    assert e["outputs_identical"] and e["variant"] in e["variants_ms_per_step"]
    assert d["gpu_launches"] == 5
    assert set(d["clocks"]) >= {"sm_mhz", "sm_max_mhz", "reasons"}
    assert d["cpu_baseline"] is None


@pytest.mark.gpu
def test_gpu_ll_rows_match_rsag():
    """Every LL row at 1 KiB per rank (two-launch, double-buffered on two
    streams, fused, and both packet write-backs; fp32 and bf16): the status
    word is clean and the outputs equal the rsag allreduce of the same inputs."""
    d = _line(["--steps", "3", "--warmup", "3", "--settle-s", "0", "--no-cpu-baseline", "--rows-only", "^ll_8x1KiB_"],
              timeout=900)
    rows = d["rows"]
    assert len(rows) == 10
    for r in rows:
        assert r["status_ok"] and r["outputs_ok"], r["workload"]
