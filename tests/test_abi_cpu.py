"""The C ABI without a GPU: the library builds and loads, exports every entry
point that include/sar.h declares, and its host-side argument checks return
the documented status codes before touching the device."""
import ctypes
import os
import re

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sar.h")


@pytest.fixture(scope="module")
def sar():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "_sar_build", os.path.join(ROOT, "allreduce_reduction_rank_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()
    import allreduce_reduction_rank_gb300 as s
    return s


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"SAR_API\s+[\w\s\*]+?\b(sar_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("sar_allreduce", "sar_ll_pack", "sar_ll_unpack_reduce", "sar_fp8_convert",
                 "sar_ll_packet_bytes", "sar_read_device_status", "sar_status_string"):
        assert must in names


def test_every_declared_symbol_is_exported(sar):
    lib = ctypes.CDLL(sar.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in sar.h but not exported"


def test_only_declared_symbols_are_exported(sar):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", sar.LIB_PATH], capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("nm unavailable")
    exported = sorted({ln.split()[-1] for ln in out.stdout.splitlines() if " T " in ln})
    assert exported == declared_functions()


def test_status_strings(sar):
    for st in range(7):
        assert sar.sar_status_string(st).startswith("SAR_")
    assert "unknown" in sar.sar_status_string(99)


@pytest.mark.parametrize("dt", ["bf16", "fp16", "fp32", "e4m3fn", "e4m3b15"])
def test_chunk_rule_matches_oracle(sar, dt):
    for count in (0, 1, 7, 9, 4097, 1 << 20, (1 << 25) + 3):
        for n in (1, 2, 4, 8, 16, 32):
            c = sar.sar_rsag_chunk(count, n, dt)
            b, e = oracle.rsag_chunk(count, n, dt, 1 if n > 1 else 0)
            if n > 1 and b < count:
                assert b == c
            assert all(oracle.rsag_chunk(count, n, dt, r)[0] == min(count, r * c) for r in range(n))
    assert sar.sar_rsag_chunk(10, 33, dt) == 0 and sar.sar_rsag_chunk(10, 0, dt) == 0
    for n in (3, 5, 6, 7, 12, 31):                      # any count up to 32 is valid
        c = sar.sar_rsag_chunk(100003, n, dt)
        assert c == oracle.rsag_chunk(100003, n, dt, 1)[0]


@pytest.mark.parametrize("dt", ["bf16", "fp16", "fp32", "e4m3fn", "e4m3b15"])
def test_packet_bytes_match_oracle(sar, dt):
    for count in (0, 1, 2, 3, 5, 1000, 262144):
        assert sar.sar_ll_packet_bytes(count, dt) == 8 * oracle.ll_packets(count, dt)
    assert sar.lib.sar_ll_packet_bytes(4, 7) == 0


def _arr(vals):
    return (ctypes.c_void_p * len(vals))(*vals)


def test_argument_errors_before_launch(sar):
    L = sar.lib
    ptrs2 = _arr([4096, 8192])
    # rank counts outside 1..32
    for n in (0, 33, 64, -1):
        assert L.sar_allreduce(ptrs2, ptrs2, n, 16, sar.SAR_BF16, 0, None) == sar.SAR_ERR_UNSUPPORTED_NRANKS
        assert L.sar_ll_pack(ptrs2, ptrs2, n, 16, sar.SAR_BF16, 1, None) == sar.SAR_ERR_UNSUPPORTED_NRANKS
    assert L.sar_allreduce(ptrs2, ptrs2, 2, 16, 5, 0, None) == sar.SAR_ERR_UNSUPPORTED_DTYPE
    assert L.sar_allreduce(ptrs2, ptrs2, 2, 16, sar.SAR_BF16, 7, None) == sar.SAR_ERR_INVALID_ARG
    assert L.sar_allreduce(None, ptrs2, 2, 16, sar.SAR_BF16, 0, None) == sar.SAR_ERR_INVALID_ARG
    assert L.sar_allreduce(_arr([4096, 0]), ptrs2, 2, 16, sar.SAR_BF16, 0, None) == sar.SAR_ERR_INVALID_ARG
    assert L.sar_allreduce(_arr([4096, 4097]), ptrs2, 2, 16, sar.SAR_BF16, 0, None) == sar.SAR_ERR_MISALIGNED
    assert L.sar_allreduce(_arr([4096, 4098]), ptrs2, 2, 16, sar.SAR_FP32, 0, None) == sar.SAR_ERR_MISALIGNED
    assert L.sar_allreduce(ptrs2, ptrs2, 2, 2 ** 62, sar.SAR_FP32, 0, None) == sar.SAR_ERR_INVALID_ARG
    # count == 0: nothing to do, nothing launched
    assert L.sar_allreduce(ptrs2, ptrs2, 2, 0, sar.SAR_BF16, 0, None) == sar.SAR_OK
    assert L.sar_reduce_scatter(ptrs2, ptrs2, 2, 0, sar.SAR_BF16, None) == sar.SAR_OK
    assert L.sar_all_gather(ptrs2, 2, 0, sar.SAR_BF16, None) == sar.SAR_OK
    # LL: epoch 0 is reserved, packets must be 16-byte aligned, status required
    assert L.sar_ll_pack(ptrs2, ptrs2, 2, 16, sar.SAR_BF16, 0, None) == sar.SAR_ERR_INVALID_ARG
    assert L.sar_ll_pack(ptrs2, _arr([4096, 8200]), 2, 16, sar.SAR_BF16, 1, None) == sar.SAR_ERR_MISALIGNED
    assert L.sar_ll_unpack_reduce(ptrs2, ptrs2, 2, 16, sar.SAR_BF16, 1, 100, None, None) == sar.SAR_ERR_INVALID_ARG
    assert L.sar_ll_unpack_reduce(ptrs2, ptrs2, 2, 16, sar.SAR_BF16, 1, 0, 4096, None) == sar.SAR_ERR_INVALID_ARG
    assert L.sar_ll_unpack_reduce(ptrs2, ptrs2, 2, 16, sar.SAR_BF16, 1, 9, 4098, None) == sar.SAR_ERR_MISALIGNED
    assert L.sar_allreduce_ll(ptrs2, ptrs2, ptrs2, 33, 16, sar.SAR_BF16, 1, 9, 4096, None) == \
        sar.SAR_ERR_UNSUPPORTED_NRANKS
    assert L.sar_allreduce_ll(ptrs2, None, ptrs2, 2, 16, sar.SAR_BF16, 1, 9, 4096, None) == sar.SAR_ERR_INVALID_ARG
    # double-buffered LL: the same checks as sar_allreduce_ll
    assert L.sar_allreduce_ll_double(ptrs2, ptrs2, ptrs2, 33, 16, sar.SAR_BF16, 1, 9, 4096, None) == \
        sar.SAR_ERR_UNSUPPORTED_NRANKS
    assert L.sar_allreduce_ll_double(ptrs2, None, ptrs2, 2, 16, sar.SAR_BF16, 1, 9, 4096, None) == \
        sar.SAR_ERR_INVALID_ARG
    assert L.sar_allreduce_ll_double(ptrs2, ptrs2, ptrs2, 2, 16, sar.SAR_BF16, 0, 9, 4096, None) == \
        sar.SAR_ERR_INVALID_ARG
    assert L.sar_allreduce_ll_double(ptrs2, ptrs2, _arr([4096, 8200]), 2, 16, sar.SAR_BF16, 2, 9, 4096, None) == \
        sar.SAR_ERR_MISALIGNED
    assert L.sar_allreduce_ll_double(ptrs2, ptrs2, ptrs2, 2, 16, sar.SAR_BF16, 2, 0, 4096, None) == \
        sar.SAR_ERR_INVALID_ARG
    assert L.sar_allreduce_ll_double(ptrs2, ptrs2, ptrs2, 2, 0, sar.SAR_BF16, 3, 9, 4096, None) == sar.SAR_OK
    # conversion pairs: one side FP8 (e4m3fn or e4m3b15), the other fp32/fp16/bf16
    assert L.sar_fp8_convert(4096, sar.SAR_FP8_E4M3FN, 8192, sar.SAR_FP8_E4M3B15, 16, None) == \
        sar.SAR_ERR_UNSUPPORTED_DTYPE
    assert L.sar_fp8_convert(4096, sar.SAR_FP32, 8192, sar.SAR_BF16, 16, None) == sar.SAR_ERR_UNSUPPORTED_DTYPE
    assert L.sar_fp8_convert(4096, sar.SAR_FP8_E4M3FN, 8192, sar.SAR_FP8_E4M3FN, 16, None) == \
        sar.SAR_ERR_UNSUPPORTED_DTYPE
    assert L.sar_fp8_convert(4097, sar.SAR_FP32, 8192, sar.SAR_FP8_E4M3FN, 16, None) == sar.SAR_ERR_MISALIGNED
    assert L.sar_fp8_convert(None, sar.SAR_FP32, 8192, sar.SAR_FP8_E4M3FN, 16, None) == sar.SAR_ERR_INVALID_ARG
    assert L.sar_fp8_convert(4096, sar.SAR_FP32, 8192, sar.SAR_FP8_E4M3FN, 0, None) == sar.SAR_OK
    assert L.sar_read_device_status(None, None) == sar.SAR_ERR_INVALID_ARG
    # accumulation types: fp32, fp16, bf16 or the input type itself
    assert L.sar_allreduce_accum(ptrs2, ptrs2, 0, 16, sar.SAR_BF16, sar.SAR_FP16, None) == \
        sar.SAR_ERR_UNSUPPORTED_NRANKS
    assert L.sar_allreduce_accum(ptrs2, ptrs2, 2, 16, sar.SAR_BF16, sar.SAR_FP8_E4M3FN, None) == \
        sar.SAR_ERR_UNSUPPORTED_DTYPE
    assert L.sar_allreduce_accum(ptrs2, ptrs2, 2, 16, sar.SAR_BF16, 9, None) == sar.SAR_ERR_UNSUPPORTED_DTYPE
    assert L.sar_allreduce_accum(ptrs2, ptrs2, 2, 0, sar.SAR_FP8_E4M3FN, sar.SAR_FP8_E4M3FN, None) == sar.SAR_OK
    # fused LL: host epoch 0 is reserved unless a device epoch counter supplies it
    assert L.sar_allreduce_ll_fused(ptrs2, ptrs2, ptrs2, 2, 16, sar.SAR_FP32, 0, None, 9, 4096, None) == \
        sar.SAR_ERR_INVALID_ARG
    assert L.sar_allreduce_ll_fused(ptrs2, ptrs2, ptrs2, 2, 16, sar.SAR_FP32, 0, 4100, 9, 4096, None) == \
        sar.SAR_ERR_MISALIGNED
    assert L.sar_allreduce_ll_fused(ptrs2, ptrs2, ptrs2, 2, 0, sar.SAR_FP32, 0, 4096, 9, 4096, None) == sar.SAR_OK
    assert L.sar_allreduce_ll_fused(ptrs2, ptrs2, ptrs2, 40, 16, sar.SAR_FP32, 1, None, 9, 4096, None) == \
        sar.SAR_ERR_UNSUPPORTED_NRANKS
    # packet write-back: result buffer required and 16-byte aligned
    assert L.sar_allreduce_ll_writeback(ptrs2, ptrs2, ptrs2, None, 2, 16, sar.SAR_FP32, 1, None, 1, 9, 4096,
                                        None) == sar.SAR_ERR_INVALID_ARG
    assert L.sar_allreduce_ll_writeback(ptrs2, ptrs2, ptrs2, 4104, 2, 16, sar.SAR_FP32, 1, None, 1, 9, 4096,
                                        None) == sar.SAR_ERR_MISALIGNED
    assert L.sar_allreduce_ll_writeback(ptrs2, ptrs2, ptrs2, 4096, 2, 16, sar.SAR_FP32, 0, None, 1, 9, 4096,
                                        None) == sar.SAR_ERR_INVALID_ARG


def test_binding_raises_on_error(sar):
    with pytest.raises(sar.SarError) as ei:
        sar.sar_allreduce([4096] * 33, [8192] * 33, count=16, dtype="bf16", stream=0)
    assert ei.value.status == sar.SAR_ERR_UNSUPPORTED_NRANKS


def test_binding_pointer_arrays_are_cached_and_bounded(sar):
    import torch
    a1, n1 = sar._ptrs([0x1000, 0x2000])
    a2, n2 = sar._ptrs((0x1000, 0x2000))
    assert a1 is a2 and n1 == n2 == 2 and [a1[0], a1[1]] == [0x1000, 0x2000]
    t = torch.empty(3)
    a3, n3 = sar._ptrs([t, 0x2000])              # tensors and raw addresses mix
    assert n3 == 2 and [a3[0], a3[1]] == [t.data_ptr(), 0x2000]
    for i in range(2 * sar._PTR_CACHE_MAX):
        sar._ptrs([0x10000 + 16 * i])
    assert len(sar._PTR_CACHE) <= sar._PTR_CACHE_MAX
    a4, n4 = sar._ptrs([])
    assert n4 == 0


@pytest.mark.parametrize("dt", ["bf16", "fp16", "fp32", "e4m3fn", "e4m3b15"])
def test_double_buffer_halves_stay_16_byte_aligned(sar, dt):
    for count in (0, 1, 2, 3, 5, 7, 8, 9, 1023, 1024, 4097):
        pb = sar.sar_ll_packet_bytes(count, dt)
        total = sar.ll_double_packet_bytes(count, dt)
        assert total % 32 == 0 and total >= 2 * pb and total - 2 * pb < 32


C_PROGRAM = r"""
#include "sar.h"
#include <stdio.h>
#include <string.h>

static int bad = 0;
#define EXPECT(call, want)                                                              \
    do {                                                                                \
        sar_status got_ = (call);                                                       \
        if (got_ != (want)) {                                                           \
            printf("%s -> %d, want %d\n", #call, (int)got_, (int)(want));               \
            bad = 1;                                                                    \
        }                                                                               \
    } while (0)

int main(void) {
    const void* in[2] = {(const void*)(uintptr_t)4096, (const void*)(uintptr_t)8192};
    void* out[2] = {(void*)(uintptr_t)4096, (void*)(uintptr_t)8192};
    EXPECT(sar_allreduce(in, out, 0, 16, SAR_BF16, SAR_ALGO_RSAG, NULL), SAR_ERR_UNSUPPORTED_NRANKS);
    EXPECT(sar_allreduce(in, out, 2, 16, (sar_dtype)5, SAR_ALGO_RSAG, NULL), SAR_ERR_UNSUPPORTED_DTYPE);
    EXPECT(sar_allreduce(in, out, 2, 0, SAR_BF16, SAR_ALGO_RSAG, NULL), SAR_OK);
    EXPECT(sar_allreduce(in, out, 33, 16, SAR_FP32, SAR_ALGO_LL_ALLPAIR, NULL), SAR_ERR_UNSUPPORTED_NRANKS);
    EXPECT(sar_allreduce(in, out, 2, 0, SAR_FP32, SAR_ALGO_LL_ALLPAIR, NULL), SAR_OK);
    {
        const void* odd[2] = {(const void*)(uintptr_t)4098, (const void*)(uintptr_t)8192};
        EXPECT(sar_allreduce(odd, out, 2, 16, SAR_FP32, SAR_ALGO_LL_ALLPAIR, NULL), SAR_ERR_MISALIGNED);
    }
    EXPECT(sar_allreduce(in, out, 2, 16, SAR_FP32, (sar_algo)3, NULL), SAR_ERR_INVALID_ARG);
    EXPECT(sar_ll_pack(in, out, 2, 16, SAR_BF16, 0, NULL), SAR_ERR_INVALID_ARG);
    EXPECT(sar_read_device_status(NULL, NULL), SAR_ERR_INVALID_ARG);
    if (sar_ll_packet_bytes(5, SAR_FP32) != 40) {
        printf("sar_ll_packet_bytes(5, fp32) = %zu\n", sar_ll_packet_bytes(5, SAR_FP32));
        bad = 1;
    }
    if (strncmp(sar_status_string(SAR_ERR_TIMEOUT), "SAR_ERR_TIMEOUT", 15) != 0) {
        printf("status string: %s\n", sar_status_string(SAR_ERR_TIMEOUT));
        bad = 1;
    }
    printf(bad ? "FAIL\n" : "OK\n");
    return bad;
}
"""


def test_plain_c_program_uses_the_boundary(sar, tmp_path):
    """A C11 program that includes only sar.h (no CUDA or C++ header) compiles
    with -Wall -Wextra -pedantic -Werror, links against libsar.so, and gets
    the argument errors back before any launch, so it needs no GPU."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src, exe = tmp_path / "use_sar.c", tmp_path / "use_sar"
    src.write_text(C_PROGRAM)
    libdir = os.path.dirname(sar.LIB_PATH)
    include = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    build = subprocess.run([cc, "-std=c11", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", include, str(src),
                            "-L", libdir, "-lsar", f"-Wl,-rpath,{libdir}", "-o", str(exe)],
                           capture_output=True, text=True)
    assert build.returncode == 0, build.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0 and run.stdout.strip() == "OK", run.stdout + run.stderr
