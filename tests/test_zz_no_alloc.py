"""sar_allreduce_ll_noalloc: the LL allreduce for callers that cannot
allocate device memory (a framework that owns the allocator, a plugin with a
fixed memory budget, a path where cudaMalloc is not allowed).  Its packet
scratch is a fixed array inside the library instead of a caller buffer.

It must give exactly the outputs of sar_allreduce_ll with caller-provided
scratch, on consecutive calls (the shared array keeps the previous call's
packets), and reject sizes beyond the array before launching anything.
This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from tests.gpu_util import ESIZE, Guarded

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sar():
    import allreduce_reduction_rank_gb300 as s
    return s


def _ptrs(bufs):
    return (ctypes.c_void_p * len(bufs))(*[b.ptr for b in bufs])


@pytest.mark.parametrize("dt,n,count", [("fp32", 8, 262144), ("bf16", 8, 524288), ("fp16", 2, 4097),
                                        ("e4m3fn", 32, 1001), ("bf16", 1, 33)])
def test_noalloc_matches_caller_scratch_on_two_calls(sar, dt, n, count):
    L = sar.lib
    stream = torch.cuda.current_stream().cuda_stream
    es = ESIZE[dt]
    pk = [Guarded(sar.sar_ll_packet_bytes(count, dt), 0, fill=0) for _ in range(n)]
    st_ref = torch.zeros(1, dtype=torch.int32, device="cuda")
    st_new = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call, seed in enumerate((21, 22)):
        ins = [Guarded.from_codes(x) for x in W.rank_inputs("uniform", seed, dt, count, n)]
        ref = [Guarded(count * es) for _ in range(n)]
        new = [Guarded(count * es, fill=0x5A) for _ in range(n)]
        rc = L.sar_allreduce_ll(_ptrs(ins), _ptrs(ref), _ptrs(pk), n, count, sar.DTYPE_CODES[dt], call + 1,
                                1 << 20, st_ref.data_ptr(), stream)
        assert rc == sar.SAR_OK
        status = st_new.data_ptr() if call == 0 else None          # second call: internal status word
        rc = L.sar_allreduce_ll_noalloc(_ptrs(ins), _ptrs(new), n, count, sar.DTYPE_CODES[dt], 1 << 20,
                                        status, stream)
        assert rc == sar.SAR_OK
        torch.cuda.synchronize()
        for j in range(n):
            assert np.array_equal(new[j].bytes(), ref[j].bytes()), f"call {call} out[{j}]"
            assert new[j].guards_intact()
    assert sar.sar_read_device_status(st_ref) == sar.SAR_OK
    assert sar.sar_read_device_status(st_new) == sar.SAR_OK


def test_noalloc_rejects_sizes_beyond_the_array(sar):
    L = sar.lib
    n, dt = 8, "fp32"
    bufs = [Guarded(64) for _ in range(n)]
    per_rank_max = sar.SAR_LL_NOALLOC_SCRATCH_BYTES // n          # packet bytes per rank that still fit
    fits = per_rank_max // 8 * 4 // ESIZE[dt]                     # elements whose packets fill that
    too_big = fits + 1
    rc = L.sar_allreduce_ll_noalloc(_ptrs(bufs), _ptrs(bufs), n, too_big, sar.DTYPE_CODES[dt], 1 << 20, None,
                                    torch.cuda.current_stream().cuda_stream)
    assert rc == sar.SAR_ERR_INVALID_ARG
    rc = L.sar_allreduce_ll_noalloc(_ptrs(bufs), _ptrs(bufs), 33, 16, sar.DTYPE_CODES[dt], 1 << 20, None, None)
    assert rc == sar.SAR_ERR_UNSUPPORTED_NRANKS
    rc = L.sar_allreduce_ll_noalloc(_ptrs(bufs), _ptrs(bufs), n, 16, sar.DTYPE_CODES[dt], 0, None, None)
    assert rc == sar.SAR_ERR_INVALID_ARG


def test_noalloc_largest_fitting_call(sar):
    """The largest per-rank size that fits with 8 ranks (1 MiB of fp32) runs
    and matches the caller-scratch path."""
    n, dt = 8, "fp32"
    count = (1 << 20) // 4
    ins = [Guarded.from_codes(x) for x in W.rank_inputs("uniform", 3, dt, count, n)]
    ref = [Guarded(count * 4) for _ in range(n)]
    new = [Guarded(count * 4) for _ in range(n)]
    pk = [Guarded(sar.sar_ll_packet_bytes(count, dt), 0, fill=0) for _ in range(n)]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sar.sar_allreduce_ll([b.ptr for b in ins], [b.ptr for b in ref], [b.ptr for b in pk], 5, st, count=count, dtype=dt)
    sar.sar_allreduce_ll_noalloc([b.ptr for b in ins], [b.ptr for b in new], st, count=count, dtype=dt)
    assert sar.sar_read_device_status(st) == sar.SAR_OK
    for j in range(n):
        assert np.array_equal(new[j].bytes(), ref[j].bytes())


def test_noalloc_epoch_wrap_clears_the_array(sar, tmp_path):
    """After 2^32 - 1 calls on a device the internal epoch wraps: the call
    that wraps zeroes the whole array, then uses epoch 1.  A test program
    linked against the library's object files sets the epoch counter through
    an internal hook and checks the outputs, the packets' flags and that the
    bytes past the wrapping call's packets are zero."""
    import glob
    import os
    import subprocess
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    objs = sorted(glob.glob(os.path.join(root, "allreduce_reduction_rank_gb300", "_build", "*.o")))
    assert objs, "library objects missing (build first)"
    exe = tmp_path / "noalloc_wrap_check"
    nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    build = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17", "-I",
                            os.path.join(root, "include"), os.path.join(root, "tests", "noalloc_wrap_check.cu")]
                           + objs + ["-o", str(exe)], capture_output=True, text=True, timeout=600)
    assert build.returncode == 0, build.stderr[-3000:]
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert run.returncode == 0 and run.stdout.strip().endswith("OK"), run.stdout + run.stderr
