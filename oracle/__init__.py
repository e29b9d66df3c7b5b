"""CPU oracle for the simulated allreduce (ctypes wrapper over sar_oracle.c).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, the package smoke
check in ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this module.  The CUDA library never imports it, and it imports
nothing from the CUDA library.

Every function takes and returns numpy arrays holding the raw element codes
(uint16 for bf16/fp16, float32 for fp32, uint8 for e4m3fn) so that results can
be compared bit for bit.  The arithmetic itself lives in ``sar_oracle.c``;
see its header for the definitions followed and where the pages state them.

Parity of the LL packet image, the rsag chunk rule, every rounding function
and the sum semantics is pinned by tests that do not call this module's
arithmetic (format-definition brute force, library conversions, closed forms).
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sar_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

BF16, FP16, FP32, E4M3FN, E4M3B15 = 0, 1, 2, 3, 4
DTYPES = {"bf16": BF16, "fp16": FP16, "fp32": FP32, "e4m3fn": E4M3FN, "e4m3b15": E4M3B15}
ESIZE = {BF16: 2, FP16: 2, FP32: 4, E4M3FN: 1, E4M3B15: 1}
NP_STORAGE = {BF16: np.uint16, FP16: np.uint16, FP32: np.float32, E4M3FN: np.uint8, E4M3B15: np.uint8}

OK, BAD_ARG, NOT_ARRIVED = 0, 1, 2

_lock = threading.Lock()
_lib = None


def compile_library(src: str, out: str) -> str:
    """Compile an oracle C source into a shared library with the oracle's
    flags (also used by the tests to build deliberately broken copies)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-Wall", "-Wextra", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile sar_oracle.c into a shared library (plain gcc, no CUDA)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    return compile_library(_SRC, _LIB_PATH)


def _bind(lib):
    vp, sz, i32, u32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_uint32
    vpp = ctypes.POINTER(ctypes.c_void_p)
    lib.orc_esize.argtypes, lib.orc_esize.restype = [i32], i32
    lib.orc_bf16_to_f32.argtypes, lib.orc_bf16_to_f32.restype = [ctypes.c_uint16], ctypes.c_float
    lib.orc_fp16_to_f32.argtypes, lib.orc_fp16_to_f32.restype = [ctypes.c_uint16], ctypes.c_float
    lib.orc_e4m3fn_to_f32.argtypes, lib.orc_e4m3fn_to_f32.restype = [ctypes.c_uint8], ctypes.c_float
    lib.orc_f32_to_bf16.argtypes, lib.orc_f32_to_bf16.restype = [ctypes.c_float], ctypes.c_uint16
    lib.orc_f32_to_fp16.argtypes, lib.orc_f32_to_fp16.restype = [ctypes.c_float], ctypes.c_uint16
    lib.orc_f32_to_e4m3fn.argtypes, lib.orc_f32_to_e4m3fn.restype = [ctypes.c_float], ctypes.c_uint8
    lib.orc_e4m3b15_to_f32.argtypes, lib.orc_e4m3b15_to_f32.restype = [ctypes.c_uint8], ctypes.c_float
    lib.orc_f32_to_e4m3b15.argtypes, lib.orc_f32_to_e4m3b15.restype = [ctypes.c_float], ctypes.c_uint8
    lib.orc_round_array.argtypes, lib.orc_round_array.restype = [i32, vp, vp, sz], None
    lib.orc_decode_array.argtypes, lib.orc_decode_array.restype = [i32, vp, vp, sz], None
    lib.orc_add_f32.argtypes, lib.orc_add_f32.restype = [ctypes.c_float, ctypes.c_float], ctypes.c_float
    lib.orc_allreduce.argtypes, lib.orc_allreduce.restype = [vpp, vpp, i32, sz, i32], i32
    lib.orc_allreduce_accum.argtypes, lib.orc_allreduce_accum.restype = [vpp, vpp, i32, sz, i32, i32], i32
    lib.orc_reduce_scatter.argtypes, lib.orc_reduce_scatter.restype = [vpp, vpp, i32, sz, i32], i32
    lib.orc_all_gather.argtypes, lib.orc_all_gather.restype = [vpp, i32, sz, i32], i32
    lib.orc_rsag_chunk.argtypes = [sz, i32, i32, i32, ctypes.POINTER(sz), ctypes.POINTER(sz)]
    lib.orc_rsag_chunk.restype = None
    lib.orc_ll_packets.argtypes, lib.orc_ll_packets.restype = [sz, i32], sz
    lib.orc_ll_pack.argtypes, lib.orc_ll_pack.restype = [vpp, vpp, i32, sz, i32, u32], i32
    lib.orc_ll_unpack_reduce.argtypes = [vpp, vpp, i32, sz, i32, u32]
    lib.orc_ll_unpack_reduce.restype = i32
    lib.orc_convert.argtypes, lib.orc_convert.restype = [vp, i32, vp, i32, sz], i32
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


@contextlib.contextmanager
def using_library(path: str):
    """Temporarily route every oracle call to another build of the oracle
    source (the tests use it to check that planted mistakes are caught)."""
    global _lib
    with _lock:
        saved = _lib
        _lib = _bind(ctypes.CDLL(path))
    try:
        yield
    finally:
        with _lock:
            _lib = saved


def _dt(dtype) -> int:
    return DTYPES[dtype] if isinstance(dtype, str) else int(dtype)


def _ptrs(arrays):
    return (ctypes.c_void_p * len(arrays))(*[a.ctypes.data for a in arrays])


def _check_ranks(arrays, count, dt):
    for a in arrays:
        if not a.flags.c_contiguous or a.nbytes < count * ESIZE[dt]:
            raise ValueError("oracle buffers must be contiguous and hold count elements")


# --------------------------------------------------------------------------
# Number formats
# --------------------------------------------------------------------------

def round_f32(x: np.ndarray, dtype) -> np.ndarray:
    """Round binary32 values to the element type (RNE; e4m3fn saturates)."""
    dt = _dt(dtype)
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, dtype=NP_STORAGE[dt])
    _load().orc_round_array(dt, x.ctypes.data, y.ctypes.data, x.size)
    return y


def decode(codes: np.ndarray, dtype) -> np.ndarray:
    """Exact binary32 value of every element code."""
    dt = _dt(dtype)
    codes = np.ascontiguousarray(codes, dtype=NP_STORAGE[dt])
    y = np.empty(codes.shape, dtype=np.float32)
    _load().orc_decode_array(dt, codes.ctypes.data, y.ctypes.data, codes.size)
    return y


def add_f32(a: float, b: float) -> float:
    return float(_load().orc_add_f32(a, b))


# --------------------------------------------------------------------------
# Allreduce and its steps
# --------------------------------------------------------------------------

def allreduce(ins, dtype) -> list:
    """Every output = R_dt(in-order binary32 sum over ranks 0..N-1)."""
    dt = _dt(dtype)
    ins = [np.ascontiguousarray(a) for a in ins]
    count = ins[0].size
    _check_ranks(ins, count, dt)
    outs = [np.empty(count, dtype=NP_STORAGE[dt]) for _ in ins]
    rc = _load().orc_allreduce(_ptrs(ins), _ptrs(outs), len(ins), count, dt)
    if rc != OK:
        raise ValueError(f"oracle allreduce rejected arguments ({rc})")
    return outs


def allreduce_accum(ins, dtype, accum) -> list:
    """Every partial sum rounded into `accum` (native when accum == dtype)."""
    dt, at = _dt(dtype), _dt(accum)
    ins = [np.ascontiguousarray(a) for a in ins]
    count = ins[0].size
    _check_ranks(ins, count, dt)
    outs = [np.empty(count, dtype=NP_STORAGE[dt]) for _ in ins]
    rc = _load().orc_allreduce_accum(_ptrs(ins), _ptrs(outs), len(ins), count, dt, at)
    if rc != OK:
        raise ValueError(f"oracle allreduce_accum rejected arguments ({rc})")
    return outs


def rsag_chunk(count: int, nranks: int, dtype, r: int):
    b, e = ctypes.c_size_t(), ctypes.c_size_t()
    _load().orc_rsag_chunk(count, nranks, _dt(dtype), r, ctypes.byref(b), ctypes.byref(e))
    return b.value, e.value


def reduce_scatter(ins, outs, dtype) -> None:
    """In place on ``outs``: out[r][chunk r] = reduced chunk."""
    dt = _dt(dtype)
    count = ins[0].size
    _check_ranks(ins, count, dt)
    _check_ranks(outs, count, dt)
    rc = _load().orc_reduce_scatter(_ptrs(ins), _ptrs(outs), len(ins), count, dt)
    if rc != OK:
        raise ValueError(f"oracle reduce_scatter rejected arguments ({rc})")


def all_gather(outs, dtype) -> None:
    """In place on ``outs``: out[j][chunk r] = out[r][chunk r] for j != r."""
    dt = _dt(dtype)
    count = outs[0].size
    _check_ranks(outs, count, dt)
    rc = _load().orc_all_gather(_ptrs(outs), len(outs), count, dt)
    if rc != OK:
        raise ValueError(f"oracle all_gather rejected arguments ({rc})")


# --------------------------------------------------------------------------
# LL packets and conversion
# --------------------------------------------------------------------------

def ll_packets(count: int, dtype) -> int:
    return int(_load().orc_ll_packets(count, _dt(dtype)))


def ll_pack(ins, dtype, epoch: int) -> list:
    """Packet buffers as uint8 arrays of 8 bytes per packet."""
    dt = _dt(dtype)
    ins = [np.ascontiguousarray(a) for a in ins]
    count = ins[0].size
    _check_ranks(ins, count, dt)
    pk = [np.empty(8 * ll_packets(count, dt), dtype=np.uint8) for _ in ins]
    rc = _load().orc_ll_pack(_ptrs(ins), _ptrs(pk), len(ins), count, dt, epoch)
    if rc != OK:
        raise ValueError(f"oracle ll_pack rejected arguments ({rc})")
    return pk


def ll_unpack_reduce(pkts, count: int, dtype, epoch: int):
    """Returns (status, outputs); status NOT_ARRIVED if any flag != epoch."""
    dt = _dt(dtype)
    pkts = [np.ascontiguousarray(p, dtype=np.uint8) for p in pkts]
    outs = [np.zeros(count, dtype=NP_STORAGE[dt]) for _ in pkts]
    rc = _load().orc_ll_unpack_reduce(_ptrs(pkts), _ptrs(outs), len(pkts), count, dt, epoch)
    return rc, outs


def convert(src: np.ndarray, src_dtype, dst_dtype) -> np.ndarray:
    sdt, ddt = _dt(src_dtype), _dt(dst_dtype)
    src = np.ascontiguousarray(src, dtype=NP_STORAGE[sdt])
    dst = np.empty(src.shape, dtype=NP_STORAGE[ddt])
    rc = _load().orc_convert(src.ctypes.data, sdt, dst.ctypes.data, ddt, src.size)
    if rc != OK:
        raise ValueError("oracle convert rejected arguments")
    return dst
