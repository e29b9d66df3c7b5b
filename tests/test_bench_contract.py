"""The JSON line bench.py prints: every key the measurement contract names,
for the reference arm (on the CPU) and for our arm (on the GPU).  The line is
the last line of stdout, the only JSON line there, and short enough that a
log which keeps only the tail of the output still holds all of it."""
import json
import os
import subprocess
import sys
from types import SimpleNamespace

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, timeout):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT, capture_output=True,
                         text=True, timeout=timeout)
    assert out.returncode == 0, out.stderr[-2000:]
    return out


def _line(args, timeout):
    out = _run(args, timeout)
    lines = out.stdout.strip().splitlines()
    assert lines, out.stderr[-2000:]
    assert sum(ln.startswith("{") for ln in lines) == 1, out.stdout[-2000:]
    last = lines[-1]
    assert last.startswith("{") and len(last) <= bench.HEADLINE_MAX_CHARS, len(last)
    return json.loads(last)


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
    assert d["same_config"] is False and d["sample"] == d["config"]["sample"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0


def test_all_core_oracle_line_covers_disjoint_slices():
    """The all-core CPU line calls the unchanged oracle on one slice per
    thread; the slices it times cover the first elements of every rank once."""
    import numpy as np
    n = 3000
    ins = [np.arange(n, dtype=np.float32) + r for r in range(3)]
    wl = SimpleNamespace(name="t", nranks=3, dtype="fp32", count=n)
    r = bench.cpu_all_cores(ins, wl, budget_s=0.0, per_thread=500)
    cores = bench.host_threads()
    assert r["cores"] == min(cores, n) and r["value"] > 0
    assert r["sample"].startswith(f"first {min(n, 500 * cores)} elements of each rank in {r['cores']} slices")


def test_warmup_below_three_is_refused():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2"], cwd=ROOT,
                         capture_output=True, text=True, timeout=120)
    assert out.returncode != 0 and "--warmup" in out.stderr


def test_headline_is_short_with_every_field_filled():
    """The headline built from plausible measurements, with the longest
    strings the bench puts in it, stays under the size cap."""
    wl = bench.W.C2
    args = SimpleNamespace(steps=20, warmup=5)
    e2e = {"value": 329.73, "unit": "GB/s", "h2d_bytes_per_step": 536870912, "d2h_bytes_per_step": 536870912,
           "steps": 20, "ms_per_step": 3.256, "outputs_identical": True, "how": "x" * 130,
           "best_variant": "pipelined_cuda_graph", "best_value": 331.0, "vs_copies_alone": 0.99}
    clk = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap", "hw_slowdown"], "samples": 300}
    cpu = {"value": 0.3479, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": "y" * 90,
           "us_per_call_sample": 48215.3, "host_cpus": 16, "cpu_model": "Neoverse-V2"}
    line = bench.headline(wl, 1, args, 6802.2, 0.15785, 0.155, 6802.2, 6779.0, "measured", 1025101312,
                          "0123456789abcdef", 132 << 20, e2e, clk, cpu)
    text = json.dumps(line, separators=(",", ":"))
    assert len(text) < 1700, len(text)
    _common(json.loads(text))
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in line["roofline"], k
    assert "rows" not in line and "per_config" not in line["cpu_baseline"]


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
    assert e["outputs_identical"] and e["best_value"] >= e["value"] > 0
    assert d["gpu_launches"] == 5
    assert set(d["clocks"]) >= {"sm_mhz", "sm_max_mhz", "reasons"}
    assert d["cpu_baseline"] is None


@pytest.mark.gpu
def test_gpu_default_command_line(tmp_path):
    """The default measurement command (`bench.py --gpus 1 --steps 20
    --warmup 5`), rows and CPU baseline included: the last stdout line is the
    whole headline."""
    side = tmp_path / "side.json"
    d = _line(["--gpus", "1", "--steps", "20", "--warmup", "5", "--rows-out", str(side)], timeout=1500)
    _common(d)
    assert d["steps"] == 20 and d["warmup"] == 5 and d["gpu_launches"] == 20
    assert d["roofline"]["frac"] > 0.8
    assert d["e2e"]["h2d_bytes_per_step"] > 0 and d["e2e"]["d2h_bytes_per_step"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["cpu_baseline"]["all_cores"]["cores"] >= 1 and d["cpu_baseline"]["all_cores"]["value"] > 0
    s = json.loads(side.read_text())
    assert len(s["rows"]) > 50
    assert len(s["oracle_per_config"]) == len([bench.W.C1] + bench.W.C3 + [bench.W.C4, bench.W.C4_B15] + bench.W.C5)
    for r in s["rows"]:
        if "outputs_ok" in r:
            assert r["outputs_ok"] and r.get("status_ok", True), r["workload"]


@pytest.mark.gpu
def test_gpu_ll_rows_match_rsag(tmp_path):
    """Every LL row at 1 KiB per rank (two-launch, through sar_allreduce,
    double-buffered on two streams, fused, cluster, and both packet
    write-backs; fp32 and bf16): the status
    word is clean and the outputs equal the rsag allreduce of the same inputs."""
    side = tmp_path / "side.json"
    _line(["--steps", "3", "--warmup", "3", "--settle-s", "0", "--no-cpu-baseline", "--rows-only", "^ll_8x1KiB_",
           "--rows-out", str(side)], timeout=900)
    rows = json.loads(side.read_text())["rows"]
    assert len(rows) == 14
    for r in rows:
        assert r["outputs_ok"], r["workload"]
        assert r.get("status_ok", True), r["workload"]
