"""GPU parity of sar_allreduce with SAR_ALGO_LL_ALLPAIR: the LL all-pair
packet allreduce behind the one allreduce entry point, every packet in the
shared memory of the CTA that makes and polls it (one slice of the packets
per CTA, or one CTA for the whole call for small calls of rank counts without
an unrolled kernel).  Bar: bit-exact against the oracle (NaN by class),
canaries intact, inputs unchanged, at any size and with calls overlapping on
two streams."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.gpu_util import ESIZE, Guarded, assert_same, random_codes

pytestmark = pytest.mark.gpu

DTYPES = ["bf16", "fp16", "fp32", "e4m3fn", "e4m3b15"]
LL = 2


@pytest.fixture(scope="module")
def sar():
    import allreduce_reduction_rank_gb300 as s
    assert s.SAR_ALGO_LL_ALLPAIR == LL
    return s


def _run(sar, ins, dt, offsets=None, inplace=False):
    n, count = len(ins), ins[0].size
    offs = offsets or [0] * n
    gin = [Guarded.from_codes(c, o) for c, o in zip(ins, offs)]
    gout = gin if inplace else [Guarded(count * ESIZE[dt], o, fill=0x5A) for o in offs]
    sar.sar_allreduce([g.ptr for g in gin], [g.ptr for g in gout], count=count, dtype=dt, algo=LL)
    torch.cuda.synchronize()
    return gin, gout


def _check(gin, gout, ins, want, dt, inplace=False):
    for j, g in enumerate(gout):
        assert_same(g.codes(dt), want, dt, f"out[{j}]")
        assert g.guards_intact(), f"canary overwritten around out[{j}]"
    if not inplace:
        for r, g in enumerate(gin):
            assert_same(g.codes(dt), ins[r], dt, f"in[{r}] modified")


@pytest.mark.parametrize("count", [1, 3, 4097, 60001])
@pytest.mark.parametrize("n", [1, 2, 8, 32])
@pytest.mark.parametrize("dt", DTYPES)
def test_ll_allpair_matches_oracle(sar, dt, n, count):
    rng = np.random.default_rng([DTYPES.index(dt), n, count, 77])
    ins = [random_codes(rng, dt, count) for _ in range(n)]
    want = oracle.allreduce(ins, dt)[0]
    gin, gout = _run(sar, ins, dt)
    _check(gin, gout, ins, want, dt)


@pytest.mark.parametrize("n", [4, 5, 8, 16, 31])
@pytest.mark.parametrize("dt", DTYPES)
def test_ll_allpair_small_sizes(sar, dt, n):
    """Calls of at most 8 KiB over all ranks (one CTA for 5 and 31 ranks, one
    or a few slices otherwise): ragged counts up to that size, aligned and at
    odd element offsets."""
    limit = (8 << 10) // n // ESIZE[dt]
    rng = np.random.default_rng([DTYPES.index(dt), n, 31])
    for count in (1, 5, limit // 2 + 1, limit):
        ins = [random_codes(rng, dt, count) for _ in range(n)]
        want = oracle.allreduce(ins, dt)[0]
        gin, gout = _run(sar, ins, dt)
        _check(gin, gout, ins, want, dt)
    count = limit - 1
    ins = [random_codes(rng, dt, count) for _ in range(n)]
    want = oracle.allreduce(ins, dt)[0]
    gin, gout = _run(sar, ins, dt, offsets=[ESIZE[dt] * (r % 3) for r in range(n)])
    _check(gin, gout, ins, want, dt)


@pytest.mark.parametrize("n", [3, 5, 12])
def test_ll_allpair_any_rank_count_unaligned(sar, n):
    rng = np.random.default_rng(n + 100)
    ins = [random_codes(rng, "fp16", 2049) for _ in range(n)]
    want = oracle.allreduce(ins, "fp16")[0]
    gin, gout = _run(sar, ins, "fp16", offsets=[2 * (r % 5) for r in range(n)])
    _check(gin, gout, ins, want, "fp16")


def test_ll_allpair_in_place(sar):
    rng = np.random.default_rng(5)
    ins = [random_codes(rng, "bf16", 10007) for _ in range(8)]
    want = oracle.allreduce(ins, "bf16")[0]
    gin, gout = _run(sar, ins, "bf16", inplace=True)
    _check(gin, gout, ins, want, "bf16", inplace=True)


def test_ll_allpair_config5_sizes_back_to_back(sar):
    """8 ranks, fp32 and bf16, 1 KiB to 1 MiB per rank (the LL workloads),
    called back to back without synchronising: each call's outputs equal the
    oracle's."""
    outs = []
    for w in W.C5:
        ins = w.inputs()
        gin = [Guarded.from_codes(c) for c in ins]
        gout = [Guarded(w.count * ESIZE[w.dtype]) for _ in range(w.nranks)]
        sar.sar_allreduce([g.ptr for g in gin], [g.ptr for g in gout], count=w.count, dtype=w.dtype, algo=LL)
        outs.append((w, ins, gin, gout))
    torch.cuda.synchronize()
    for w, ins, gin, gout in outs:
        want = oracle.allreduce(ins, w.dtype)[0]
        _check(gin, gout, ins, want, w.dtype)


def test_ll_allpair_in_a_cuda_graph(sar):
    """Captured once and replayed on new inputs: each replay makes its packets
    afresh before it polls them, so each gives the sum of the inputs it saw."""
    n, count, dt = 8, 5000, "fp32"
    rng = np.random.default_rng(9)
    gin = [Guarded(count * 4) for _ in range(n)]
    gout = [Guarded(count * 4) for _ in range(n)]
    pin, pout = [g.ptr for g in gin], [g.ptr for g in gout]
    sar.sar_allreduce(pin, pout, count=count, dtype=dt, algo=LL)
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=s):
        sar.sar_allreduce(pin, pout, count=count, dtype=dt, algo=LL, stream=s)
    for _ in range(3):
        ins = [random_codes(rng, dt, count) for _ in range(n)]
        for g, c in zip(gin, ins):
            g.base[256: 256 + count * 4] = torch.from_numpy(c.view(np.uint8).copy()).cuda()
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            graph.replay()
        torch.cuda.synchronize()
        want = oracle.allreduce(ins, dt)[0]
        for g in gout:
            assert_same(g.codes(dt), want, dt)


@pytest.mark.parametrize("n,dt,count", [
    (5, "fp32", (8 << 10) // 5 // 4), (5, "fp32", (8 << 10) // 5 // 4 + 1),      # one CTA -> slices
    (31, "e4m3fn", (8 << 10) // 31), (31, "e4m3fn", (8 << 10) // 31 + 1),
    (8, "fp32", 151 * 512), (8, "fp32", 151 * 512 + 1),                           # 1 -> 4 packets per thread
    (2, "bf16", 2 * 151 * 512), (2, "bf16", 2 * 151 * 512 + 2),
    (16, "fp16", 2 * 151 * 512 + 2)])                                             # 16 ranks: 1 packet per thread
def test_ll_allpair_forms_at_their_boundaries(sar, n, dt, count):
    """Exact on either side of each switch between forms: one CTA for the
    whole call (rank counts without an unrolled kernel, at most 8 KiB over
    all ranks), slices of 1 packet per thread, slices of 4 packets per thread
    (at most 8 ranks, from 152 slices of 512 packets per rank)."""
    rng = np.random.default_rng([n, count])
    ins = [random_codes(rng, dt, count) for _ in range(n)]
    want = oracle.allreduce(ins, dt)[0]
    gin, gout = _run(sar, ins, dt)
    _check(gin, gout, ins, want, dt)


def test_ll_allpair_large_call(sar):
    """8 ranks x 8 MiB + 20 bytes of fp32 (64 MiB of packets, more than the
    fixed scratch of the no-alloc entry point holds): accepted and exact."""
    n, dt, count = 8, "fp32", (2 << 20) + 5
    rng = np.random.default_rng(4242)
    ins = [random_codes(rng, dt, count) for _ in range(n)]
    want = oracle.allreduce(ins, dt)[0]
    gin, gout = _run(sar, ins, dt)
    _check(gin, gout, ins, want, dt)


def test_ll_allpair_calls_on_two_streams_overlap_safely(sar):
    """No scratch and no state: calls on two streams without any ordering
    between them may run at the same time, and both give the oracle's
    outputs (sizes of one slice, several slices of 1 packet per thread and
    slices of 4 packets per thread)."""
    n, dt = 8, "fp32"
    rng = np.random.default_rng(23)
    for count in (256, 16384, 262144):
        cases = []
        for _ in range(2):
            ins = [random_codes(rng, dt, count) for _ in range(n)]
            gin = [Guarded.from_codes(c) for c in ins]
            gout = [Guarded(count * 4) for _ in range(n)]
            cases.append((ins, gin, gout, torch.cuda.Stream()))
        torch.cuda.synchronize()
        for _ in range(30):
            for ins, gin, gout, stream in cases:
                sar.sar_allreduce([g.ptr for g in gin], [g.ptr for g in gout], count=count, dtype=dt, algo=LL,
                                  stream=stream)
        torch.cuda.synchronize()
        for ins, gin, gout, stream in cases:
            _check(gin, gout, ins, oracle.allreduce(ins, dt)[0], dt)


def test_ll_allpair_argument_errors(sar):
    L = sar.lib
    n, dt = 8, "fp32"
    bufs = [Guarded(64) for _ in range(n)]
    import ctypes
    arr = (ctypes.c_void_p * n)(*[b.ptr for b in bufs])
    odd = (ctypes.c_void_p * n)(*([bufs[0].ptr + 2] + [b.ptr for b in bufs[1:]]))
    assert L.sar_allreduce(arr, arr, 33, 16, sar.DTYPE_CODES[dt], LL, None) == sar.SAR_ERR_UNSUPPORTED_NRANKS
    assert L.sar_allreduce(arr, arr, 0, 16, sar.DTYPE_CODES[dt], LL, None) == sar.SAR_ERR_UNSUPPORTED_NRANKS
    assert L.sar_allreduce(odd, arr, n, 16, sar.DTYPE_CODES[dt], LL, None) == sar.SAR_ERR_MISALIGNED
    assert L.sar_allreduce(arr, arr, n, 16, 7, LL, None) == sar.SAR_ERR_UNSUPPORTED_DTYPE
    assert L.sar_allreduce(arr, arr, n, 0, sar.DTYPE_CODES[dt], LL, None) == sar.SAR_OK
