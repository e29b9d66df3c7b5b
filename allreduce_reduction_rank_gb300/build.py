"""Build libsar.so in-tree with nvcc for sm_103a (GB300).

Usage: ``python allreduce_reduction_rank_gb300/build.py [--force] [--verbose-ptxas]``

Each CUDA translation unit is compiled in parallel into an object file under
``_build/`` and the objects are linked into ``_build/libsar.so`` (C ABI,
declared in ``include/sar.h``; the CUDA runtime is linked statically and its
symbols are kept private).  Floating point is compiled without fast-math,
flush-to-zero or contraction so that the binary32 adds are exactly IEEE adds
with gradual underflow.

This file imports nothing from the package, so it runs before the library
exists.
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_build")
LIB = os.path.join(OUT, "libsar.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

# Slowest first, so the parallel build finishes sooner.
SOURCES = ["ll_writeback.cu", "ll_fused.cu", "ll_cluster.cu", "ll_cta.cu", "rsag_e4m3b15.cu", "rsag_e4m3b15_acc.cu",
           "ll.cu", "rsag_e4m3fn_acc.cu", "rsag_e4m3fn.cu", "rsag_bf16_acc.cu", "rsag_fp16_acc.cu", "rsag_fp32_acc.cu", "rsag_fp16.cu",
           "rsag_bf16.cu", "rsag_fp32.cu", "convert.cu", "rsag.cu", "sar_api.cu", "noalloc.cu"]
HEADERS = ["sar_device.cuh", "sar_internal.h", "rsag_kernels.cuh", "ll_coop.cuh", "ll_packets.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + [
    "-O3", "-std=c++17", "-lineinfo",
    "-fmad=false", "-ftz=false", "-prec-div=true", "-prec-sqrt=true",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "-I", INCLUDE,
]


def nvcc_path() -> str:
    for cand in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        p = os.path.join(cand, "bin", "nvcc") if cand else ""
        if p and os.path.exists(p):
            return p
    p = shutil.which("nvcc")
    if not p:
        raise RuntimeError("nvcc not found: libsar needs the CUDA toolkit to build")
    return p


def _stale(target: str, deps: list) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    os.makedirs(OUT, exist_ok=True)
    nvcc = nvcc_path()
    headers = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "sar.h")]
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []

    def compile_one(src: str) -> str:
        path = os.path.join(CSRC, src)
        obj = os.path.join(OUT, src.replace(".cu", ".o"))
        if force or verbose_ptxas or _stale(obj, [path] + headers):
            cmd = [nvcc] + NVCC_FLAGS + extra + ["-c", path, "-o", obj + ".tmp"]
            res = subprocess.run(cmd, capture_output=True, text=True)
            if res.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
            if verbose_ptxas:
                sys.stderr.write(res.stderr)
            os.replace(obj + ".tmp", obj)
        return obj

    with ThreadPoolExecutor(min(len(SOURCES), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    if force or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs + [
            "-Xlinker", "--exclude-libs,ALL", "-Xlinker", "-z,defs"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
        os.replace(tmp, LIB)
    return LIB


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose-ptxas", action="store_true", help="print registers/spills per kernel")
    a = ap.parse_args()
    print(build(force=a.force, verbose_ptxas=a.verbose_ptxas))


if __name__ == "__main__":
    main()
