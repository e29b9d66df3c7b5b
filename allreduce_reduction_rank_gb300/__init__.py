"""Python binding of libsar, the simulated allreduce on one GB300.

A thin ctypes layer over the C ABI declared in ``include/sar.h``: it turns
torch tensors (or raw device addresses) into pointer arrays and sizes, calls
the library, and raises :class:`SarError` on a non-OK status.  Every step of
the computation runs in the library's CUDA kernels; there is no fallback.
Importing this package fails if ``_build/libsar.so`` has not been built
(``python allreduce_reduction_rank_gb300/build.py``).

Function names follow the C ABI: :func:`sar_allreduce`,
:func:`sar_allreduce_accum`, :func:`sar_reduce_scatter`, :func:`sar_all_gather`,
:func:`sar_rsag_chunk`, :func:`sar_allreduce_ll_fused`, :func:`sar_allreduce_ll_writeback`,
:func:`sar_ll_packet_bytes`, :func:`sar_ll_pack`,
:func:`sar_ll_unpack_reduce`, :func:`sar_allreduce_ll`, :func:`sar_allreduce_ll_double`,
:func:`sar_allreduce_ll_noalloc`, :func:`sar_allreduce_ll_cluster`,
:func:`sar_fp8_convert`, :func:`sar_read_device_status`,
:func:`sar_status_string`.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libsar.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"libsar is not built ({LIB_PATH} missing); run "
        "`python allreduce_reduction_rank_gb300/build.py` (needs nvcc)")

lib = ctypes.CDLL(LIB_PATH)

# sar_dtype
SAR_BF16, SAR_FP16, SAR_FP32, SAR_FP8_E4M3FN, SAR_FP8_E4M3B15 = 0, 1, 2, 3, 4
# sar_algo
SAR_ALGO_RSAG, SAR_ALGO_RSAG_TWO_PHASE, SAR_ALGO_LL_ALLPAIR = 0, 1, 2
# sar_status
(SAR_OK, SAR_ERR_INVALID_ARG, SAR_ERR_UNSUPPORTED_NRANKS, SAR_ERR_UNSUPPORTED_DTYPE,
 SAR_ERR_MISALIGNED, SAR_ERR_CUDA, SAR_ERR_TIMEOUT) = range(7)
SAR_MAX_RANKS = 32
SAR_LL_NOALLOC_SCRATCH_BYTES = 16 << 20
SAR_LL_CLUSTER_MAX_RANKS = 16

DTYPE_CODES = {"bf16": SAR_BF16, "fp16": SAR_FP16, "fp32": SAR_FP32, "e4m3fn": SAR_FP8_E4M3FN,
               "e4m3b15": SAR_FP8_E4M3B15}
TORCH_DTYPES = {SAR_BF16: torch.bfloat16, SAR_FP16: torch.float16, SAR_FP32: torch.float32,
                SAR_FP8_E4M3FN: torch.float8_e4m3fn}
ESIZE = {SAR_BF16: 2, SAR_FP16: 2, SAR_FP32: 4, SAR_FP8_E4M3FN: 1, SAR_FP8_E4M3B15: 1}

_vp, _sz, _i32, _u32, _u64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_uint32, ctypes.c_uint64
_vpp = ctypes.POINTER(ctypes.c_void_p)

lib.sar_allreduce.argtypes = [_vpp, _vpp, _i32, _sz, _i32, _i32, _vp]
lib.sar_allreduce_accum.argtypes = [_vpp, _vpp, _i32, _sz, _i32, _i32, _vp]
lib.sar_reduce_scatter.argtypes = [_vpp, _vpp, _i32, _sz, _i32, _vp]
lib.sar_all_gather.argtypes = [_vpp, _i32, _sz, _i32, _vp]
lib.sar_rsag_chunk.argtypes = [_sz, _i32, _i32]
lib.sar_rsag_chunk.restype = _sz
lib.sar_ll_packet_bytes.argtypes = [_sz, _i32]
lib.sar_ll_packet_bytes.restype = _sz
lib.sar_ll_pack.argtypes = [_vpp, _vpp, _i32, _sz, _i32, _u32, _vp]
lib.sar_ll_unpack_reduce.argtypes = [_vpp, _vpp, _i32, _sz, _i32, _u32, _u64, _vp, _vp]
lib.sar_allreduce_ll.argtypes = [_vpp, _vpp, _vpp, _i32, _sz, _i32, _u32, _u64, _vp, _vp]
lib.sar_allreduce_ll_double.argtypes = [_vpp, _vpp, _vpp, _i32, _sz, _i32, _u32, _u64, _vp, _vp]
lib.sar_allreduce_ll_fused.argtypes = [_vpp, _vpp, _vpp, _i32, _sz, _i32, _u32, _vp, _u64, _vp, _vp]
lib.sar_allreduce_ll_writeback.argtypes = [_vpp, _vpp, _vpp, _vp, _i32, _sz, _i32, _u32, _vp, _i32, _u64, _vp, _vp]
lib.sar_allreduce_ll_noalloc.argtypes = [_vpp, _vpp, _i32, _sz, _i32, _u64, _vp, _vp]
lib.sar_allreduce_ll_cluster.argtypes = [_vpp, _vpp, _i32, _sz, _i32, _u64, _vp, _vp]
lib.sar_fp8_convert.argtypes = [_vp, _i32, _vp, _i32, _sz, _vp]
lib.sar_read_device_status.argtypes = [_vp, _vp]
lib.sar_status_string.argtypes = [_i32]
lib.sar_status_string.restype = ctypes.c_char_p
for _f in ("sar_allreduce", "sar_allreduce_accum", "sar_allreduce_ll_fused", "sar_allreduce_ll_writeback",
           "sar_reduce_scatter", "sar_all_gather", "sar_ll_pack", "sar_ll_unpack_reduce",
           "sar_allreduce_ll", "sar_allreduce_ll_double", "sar_allreduce_ll_noalloc", "sar_allreduce_ll_cluster",
           "sar_fp8_convert",
           "sar_read_device_status"):
    getattr(lib, _f).restype = _i32


class SarError(RuntimeError):
    def __init__(self, status: int):
        self.status = int(status)
        super().__init__(sar_status_string(self.status))


def sar_status_string(status: int) -> str:
    return lib.sar_status_string(int(status)).decode()


def _check(status: int) -> int:
    if status != SAR_OK:
        raise SarError(status)
    return status


def _addr(x) -> int:
    return x.data_ptr() if isinstance(x, torch.Tensor) else int(x)


# ctypes pointer arrays by address tuple: the library copies the pointers into
# kernel arguments and keeps nothing, so an array can serve every call with the
# same buffers.  Bounded; cleared when full.
_PTR_CACHE: dict = {}
_PTR_CACHE_MAX = 256


def _ptrs(xs):
    key = tuple(xs)
    if not key or set(map(type, key)) != {int}:
        key = tuple(x.data_ptr() if isinstance(x, torch.Tensor) else int(x) for x in key)
    arr = _PTR_CACHE.get(key)
    if arr is None:
        if len(_PTR_CACHE) >= _PTR_CACHE_MAX:
            _PTR_CACHE.clear()
        arr = (ctypes.c_void_p * max(1, len(key)))(*key)
        _PTR_CACHE[key] = arr
    return arr, len(key)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dtype_code(dtype, like=None) -> int:
    if dtype is None:
        if like is None:
            raise ValueError("dtype is required for raw pointers")
        for code, td in TORCH_DTYPES.items():
            if like.dtype == td:
                return code
        raise ValueError(f"unsupported tensor dtype {like.dtype}; pass dtype explicitly")
    if isinstance(dtype, str):
        return DTYPE_CODES[dtype]
    if isinstance(dtype, torch.dtype):
        return {v: k for k, v in TORCH_DTYPES.items()}[dtype]
    return int(dtype)


def _count(count, like) -> int:
    if count is not None:
        return int(count)
    if not isinstance(like, torch.Tensor):
        raise ValueError("count is required for raw pointers")
    return like.numel()


def sar_rsag_chunk(count: int, nranks: int, dtype) -> int:
    return int(lib.sar_rsag_chunk(count, nranks, _dtype_code(dtype)))


def sar_ll_packet_bytes(count: int, dtype) -> int:
    return int(lib.sar_ll_packet_bytes(count, _dtype_code(dtype)))


def sar_allreduce(ins, outs, count=None, dtype=None, algo=SAR_ALGO_RSAG, stream=None) -> None:
    """Allreduce: every outs[j] = R(sum over ranks 0..N-1 of ins[k]), by the
    rsag kernels or (SAR_ALGO_LL_ALLPAIR) LL packets in the shared memory of
    the CTAs that make and poll them."""
    pin, n = _ptrs(ins)
    pout, n_out = _ptrs(outs)
    if n != n_out:
        raise ValueError("ins and outs must have one buffer per rank")
    _check(lib.sar_allreduce(pin, pout, n, _count(count, ins[0]), _dtype_code(dtype, ins[0]), int(algo),
                             _stream(stream)))


def sar_allreduce_accum(ins, outs, accum, count=None, dtype=None, stream=None) -> None:
    """Fused rsag allreduce with every partial sum rounded into `accum`."""
    pin, n = _ptrs(ins)
    pout, _ = _ptrs(outs)
    _check(lib.sar_allreduce_accum(pin, pout, n, _count(count, ins[0]), _dtype_code(dtype, ins[0]),
                                   _dtype_code(accum), _stream(stream)))


def sar_reduce_scatter(ins, outs, count=None, dtype=None, stream=None) -> None:
    pin, n = _ptrs(ins)
    pout, _ = _ptrs(outs)
    _check(lib.sar_reduce_scatter(pin, pout, n, _count(count, ins[0]), _dtype_code(dtype, ins[0]),
                                  _stream(stream)))


def sar_all_gather(outs, count=None, dtype=None, stream=None) -> None:
    pout, n = _ptrs(outs)
    _check(lib.sar_all_gather(pout, n, _count(count, outs[0]), _dtype_code(dtype, outs[0]), _stream(stream)))


def sar_ll_pack(ins, pkts, epoch: int, count=None, dtype=None, stream=None) -> None:
    pin, n = _ptrs(ins)
    ppk, _ = _ptrs(pkts)
    _check(lib.sar_ll_pack(pin, ppk, n, _count(count, ins[0]), _dtype_code(dtype, ins[0]), epoch,
                           _stream(stream)))


def sar_ll_unpack_reduce(pkts, outs, epoch: int, status, max_spins: int = 1 << 20, count=None, dtype=None,
                         stream=None) -> None:
    ppk, n = _ptrs(pkts)
    pout, _ = _ptrs(outs)
    _check(lib.sar_ll_unpack_reduce(ppk, pout, n, _count(count, outs[0]), _dtype_code(dtype, outs[0]), epoch,
                                    max_spins, _addr(status), _stream(stream)))


def sar_allreduce_ll(ins, outs, pkts, epoch: int, status, max_spins: int = 1 << 20, count=None, dtype=None,
                     stream=None) -> None:
    pin, n = _ptrs(ins)
    pout, _ = _ptrs(outs)
    ppk, _ = _ptrs(pkts)
    _check(lib.sar_allreduce_ll(pin, pout, ppk, n, _count(count, ins[0]), _dtype_code(dtype, ins[0]), epoch,
                                max_spins, _addr(status), _stream(stream)))


def ll_double_packet_bytes(count: int, dtype) -> int:
    """Bytes of one rank's double-buffered packet scratch: two halves of
    sar_ll_packet_bytes rounded up to 16 bytes."""
    return 2 * ((sar_ll_packet_bytes(count, dtype) + 15) // 16 * 16)


def sar_allreduce_ll_double(ins, outs, pkts, epoch: int, status, max_spins: int = 1 << 20, count=None, dtype=None,
                            stream=None) -> None:
    """sar_allreduce_ll on a double-buffered scratch: half (epoch & 1) of each
    pkts[r] (see ll_double_packet_bytes)."""
    pin, n = _ptrs(ins)
    pout, _ = _ptrs(outs)
    ppk, _ = _ptrs(pkts)
    _check(lib.sar_allreduce_ll_double(pin, pout, ppk, n, _count(count, ins[0]), _dtype_code(dtype, ins[0]), epoch,
                                       max_spins, _addr(status), _stream(stream)))


def sar_allreduce_ll_fused(ins, outs, pkts, status, epoch: int = 0, epoch_ctrl=None, max_spins: int = 1 << 20,
                           count=None, dtype=None, stream=None) -> None:
    """LL allreduce in one launch (sliced up to 256 KiB per rank, cooperative
    above; see sar.h).  `epoch_ctrl`: optional device
    epoch counter (8 bytes, one uint64, zeroed once); when given, every launch
    takes the next epoch from it on the device (see ll_device_epoch)."""
    pin, n = _ptrs(ins)
    pout, _ = _ptrs(outs)
    ppk, _ = _ptrs(pkts)
    _check(lib.sar_allreduce_ll_fused(pin, pout, ppk, n, _count(count, ins[0]), _dtype_code(dtype, ins[0]), epoch,
                                      None if epoch_ctrl is None else _addr(epoch_ctrl), max_spins, _addr(status),
                                      _stream(stream)))


def sar_allreduce_ll_writeback(ins, outs, pkts, res, status, multi_dest: bool = True, epoch: int = 0,
                               epoch_ctrl=None, max_spins: int = 1 << 20, count=None, dtype=None, stream=None) -> None:
    """LL allreduce whose write-back is a second packet round through `res`."""
    pin, n = _ptrs(ins)
    pout, _ = _ptrs(outs)
    ppk, _ = _ptrs(pkts)
    _check(lib.sar_allreduce_ll_writeback(pin, pout, ppk, _addr(res), n, _count(count, ins[0]),
                                          _dtype_code(dtype, ins[0]), epoch,
                                          None if epoch_ctrl is None else _addr(epoch_ctrl), int(bool(multi_dest)),
                                          max_spins, _addr(status), _stream(stream)))


def sar_allreduce_ll_noalloc(ins, outs, status=None, max_spins: int = 1 << 20, count=None, dtype=None,
                             stream=None) -> None:
    """LL allreduce with the library's fixed packet scratch, for callers that
    cannot allocate device memory (see include/sar.h).  ``status`` is an
    optional device int32 that receives SAR_ERR_TIMEOUT."""
    pin, n = _ptrs(ins)
    pout, _ = _ptrs(outs)
    _check(lib.sar_allreduce_ll_noalloc(pin, pout, n, _count(count, ins[0]), _dtype_code(dtype, ins[0]), max_spins,
                                        None if status is None else _addr(status), _stream(stream)))


def sar_allreduce_ll_cluster(ins, outs, status, max_spins: int = 1 << 20, count=None, dtype=None,
                             stream=None) -> None:
    """LL allreduce with the packets exchanged through the shared memory of
    thread-block clusters (one CTA per simulated rank; at most 16 ranks)."""
    pin, n = _ptrs(ins)
    pout, _ = _ptrs(outs)
    _check(lib.sar_allreduce_ll_cluster(pin, pout, n, _count(count, ins[0]), _dtype_code(dtype, ins[0]), max_spins,
                                        _addr(status), _stream(stream)))


# The device epoch counter of sar_allreduce_ll_fused / _writeback: one uint64,
# launches so far in bits 20..63.
LL_EPOCH_SHIFT = 20
_EPOCH_PERIOD = 0xFFFFFFFF


def ll_device_epoch(ctrl) -> int:
    """The epoch the last launch on a device epoch counter used (0 before the
    first launch); ctrl is an 8-byte CUDA tensor.  Synchronises."""
    launches = int(ctrl.view(torch.int64)[0].item()) >> LL_EPOCH_SHIFT
    return 0 if launches == 0 else (launches - 1) % _EPOCH_PERIOD + 1


def ll_set_device_epoch(ctrl, last_epoch: int) -> None:
    """Make the next launch on the counter use last_epoch + 1 (1 after
    2^32 - 1), for example to continue after host epochs 1..last_epoch."""
    ctrl.view(torch.int64)[0] = int(last_epoch) << LL_EPOCH_SHIFT


def sar_fp8_convert(src, dst, src_dtype=None, dst_dtype=None, count=None, stream=None) -> None:
    _check(lib.sar_fp8_convert(_addr(src), _dtype_code(src_dtype, src), _addr(dst), _dtype_code(dst_dtype, dst),
                               _count(count, src), _stream(stream)))


def sar_read_device_status(status, stream=None) -> int:
    """Synchronises the stream and returns the status word as a sar_status."""
    return int(lib.sar_read_device_status(_addr(status), _stream(stream)))
