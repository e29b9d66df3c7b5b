"""Structure (no GPU): the oracle and the CUDA library share no code, the
oracle is used only by tests / smoke / the bench's CPU legs, and the product
path refuses to run without its compiled library (no fallback)."""
import os
import re
import shutil
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "allreduce_reduction_rank_gb300")
ORACLE = os.path.join(ROOT, "oracle")


def _sources(d, exts):
    for base, _, files in os.walk(d):
        if "_build" in base:
            continue
        for f in files:
            if f.endswith(exts):
                yield os.path.join(base, f)


def test_library_never_touches_the_oracle():
    for path in _sources(PKG, (".py", ".cu", ".cuh", ".h", ".c")):
        text = open(path).read()
        assert not re.search(r"^\s*(import oracle|from oracle)", text, re.M), path
        assert "sar_oracle" not in text and "orc_" not in text, path


def test_oracle_never_touches_the_library():
    for path in _sources(ORACLE, (".py", ".c", ".h")):
        text = open(path).read()
        assert "allreduce_reduction_rank_gb300" not in text, path
        assert "sar.h" not in text and "libsar" not in text, path
        assert "#include \"" not in text, path            # no local headers at all


def test_only_tests_smoke_and_bench_import_the_oracle():
    allowed = {os.path.join(ROOT, "__graft_entry__.py"), os.path.join(ROOT, "bench.py")}
    for path in _sources(ROOT, (".py",)):
        if path.startswith(os.path.join(ROOT, "tests")) or path.startswith(ORACLE) or \
                path.startswith(os.path.join(ROOT, "_work")):
            continue
        if re.search(r"^\s*(import oracle|from oracle)", open(path).read(), re.M):
            assert path in allowed, path


def test_package_import_fails_loudly_without_the_library(tmp_path):
    pkg = tmp_path / "allreduce_reduction_rank_gb300"
    pkg.mkdir()
    shutil.copy(os.path.join(PKG, "__init__.py"), pkg / "__init__.py")
    out = subprocess.run([sys.executable, "-c", "import allreduce_reduction_rank_gb300"], cwd=tmp_path,
                         capture_output=True, text=True)
    assert out.returncode != 0 and "ImportError" in out.stderr and "libsar is not built" in out.stderr
