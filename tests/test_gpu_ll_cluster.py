"""GPU parity of sar_allreduce_ll_cluster (LL packets exchanged through the
shared memory of thread-block clusters, one CTA per simulated rank) against
the CPU oracle, through the C ABI.  Bar: bit-exact (NaN by class), canaries
intact, inputs unchanged."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.gpu_util import ESIZE, Guarded, assert_same, random_codes

pytestmark = pytest.mark.gpu

DTYPES = ["bf16", "fp16", "fp32", "e4m3fn", "e4m3b15"]


@pytest.fixture(scope="module")
def sar():
    import allreduce_reduction_rank_gb300 as s
    return s


def _run(sar, ins, dt, offsets=None, inplace=False, max_spins=1 << 20):
    n, count = len(ins), ins[0].size
    offs = offsets or [0] * n
    gin = [Guarded.from_codes(c, o) for c, o in zip(ins, offs)]
    gout = gin if inplace else [Guarded(count * ESIZE[dt], o, fill=0x5A) for o in offs]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sar.sar_allreduce_ll_cluster([g.ptr for g in gin], [g.ptr for g in gout], st, max_spins=max_spins, count=count,
                                 dtype=dt)
    return gin, gout, sar.sar_read_device_status(st)


def _check(gin, gout, ins, want, dt, inplace=False):
    for j, g in enumerate(gout):
        assert_same(g.codes(dt), want, dt, f"out[{j}]")
        assert g.guards_intact(), f"canary overwritten around out[{j}]"
    if not inplace:
        for r, g in enumerate(gin):
            assert_same(g.codes(dt), ins[r], dt, f"in[{r}] modified")
            assert g.guards_intact()


@pytest.mark.parametrize("count", [1, 3, 5, 33, 1031, 20011, 65541, 262147])
@pytest.mark.parametrize("n", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("dt", DTYPES)
def test_cluster_matches_oracle(sar, dt, n, count):
    """The counts reach slices of 64, 128 and 256 packets per rank (the CTA
    size is chosen from the call's size)."""
    rng = np.random.default_rng([DTYPES.index(dt), n, count, 5])
    ins = [random_codes(rng, dt, count) for _ in range(n)]
    want = oracle.allreduce(ins, dt)[0]
    gin, gout, rc = _run(sar, ins, dt)
    assert rc == sar.SAR_OK
    _check(gin, gout, ins, want, dt)


@pytest.mark.parametrize("count", [7, 4099, 100003])
@pytest.mark.parametrize("n", [3, 5, 6, 7, 12, 15])
@pytest.mark.parametrize("dt", ["bf16", "fp32", "e4m3fn"])
def test_cluster_any_rank_count(sar, dt, n, count):
    rng = np.random.default_rng([DTYPES.index(dt), n, count, 6])
    ins = [random_codes(rng, dt, count) for _ in range(n)]
    want = oracle.allreduce(ins, dt)[0]
    gin, gout, rc = _run(sar, ins, dt)
    assert rc == sar.SAR_OK
    _check(gin, gout, ins, want, dt)


@pytest.mark.parametrize("dt", DTYPES)
def test_cluster_unaligned_and_in_place(sar, dt):
    """Buffers at odd element offsets take the byte-wise send and the
    element-wise write-back; in place the outputs are the inputs."""
    n, count = 8, 5003
    rng = np.random.default_rng([DTYPES.index(dt), 7])
    ins = [random_codes(rng, dt, count) for _ in range(n)]
    want = oracle.allreduce(ins, dt)[0]
    gin, gout, rc = _run(sar, ins, dt, offsets=[ESIZE[dt] * (r % 5) for r in range(n)])
    assert rc == sar.SAR_OK
    _check(gin, gout, ins, want, dt)
    gin, gout, rc = _run(sar, ins, dt, inplace=True)
    assert rc == sar.SAR_OK
    _check(gin, gout, ins, want, dt, inplace=True)


@pytest.mark.parametrize("wl", W.C5, ids=lambda w: w.name)
def test_cluster_on_the_ll_workloads(sar, wl):
    """8 ranks, fp32 and bf16, 1 KiB to 1 MiB per rank, 20 calls back to back
    on the same buffers: exact every time (no state is kept between calls)."""
    ins = wl.inputs()
    want = oracle.allreduce(ins, wl.dtype)[0]
    gin = [Guarded.from_codes(c) for c in ins]
    gout = [Guarded(wl.count * ESIZE[wl.dtype]) for _ in range(wl.nranks)]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(20):
        sar.sar_allreduce_ll_cluster([g.ptr for g in gin], [g.ptr for g in gout], st, count=wl.count, dtype=wl.dtype)
    assert sar.sar_read_device_status(st) == sar.SAR_OK
    _check(gin, gout, ins, want, wl.dtype)


def test_cluster_in_a_cuda_graph(sar):
    """Captured once and replayed on new inputs: every replay clears its
    slots and polls only its own packets, so each gives the sum of the inputs
    it saw."""
    n, count, dt = 8, 70001, "fp16"
    rng = np.random.default_rng(11)
    gin = [Guarded(count * 2) for _ in range(n)]
    gout = [Guarded(count * 2) for _ in range(n)]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=s):
        for _ in range(3):
            sar.sar_allreduce_ll_cluster([g.ptr for g in gin], [g.ptr for g in gout], st, count=count, dtype=dt,
                                         stream=s)
    for _ in range(3):
        ins = [random_codes(rng, dt, count) for _ in range(n)]
        for g, c in zip(gin, ins):
            g.base[256:256 + count * 2] = torch.from_numpy(c.view(np.uint8).copy()).cuda()
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            graph.replay()
        torch.cuda.synchronize()
        want = oracle.allreduce(ins, dt)[0]
        for g in gout:
            assert_same(g.codes(dt), want, dt)
    assert sar.sar_read_device_status(st) == sar.SAR_OK


def test_cluster_short_poll_bound_and_the_next_call(sar):
    """One re-read per poll at 16 x 1 MiB: the call may run out (status
    SAR_ERR_TIMEOUT) or finish; either way the launch ends, and the next call
    with the normal bound is exact."""
    n, count, dt = 16, 1 << 18, "fp32"
    rng = np.random.default_rng(13)
    ins = [random_codes(rng, dt, count) for _ in range(n)]
    want = oracle.allreduce(ins, dt)[0]
    gin, gout, rc = _run(sar, ins, dt, max_spins=1)
    assert rc in (sar.SAR_OK, sar.SAR_ERR_TIMEOUT)
    if rc == sar.SAR_OK:
        _check(gin, gout, ins, want, dt)
    gin, gout, rc = _run(sar, ins, dt)
    assert rc == sar.SAR_OK
    _check(gin, gout, ins, want, dt)


def test_cluster_argument_errors(sar):
    L = sar.lib
    bufs = [Guarded(64) for _ in range(17)]
    arr = (ctypes.c_void_p * 17)(*[b.ptr for b in bufs])
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    code = sar.DTYPE_CODES["fp32"]
    assert L.sar_allreduce_ll_cluster(arr, arr, 17, 16, code, 1 << 20, st.data_ptr(), None) == \
        sar.SAR_ERR_UNSUPPORTED_NRANKS
    assert L.sar_allreduce_ll_cluster(arr, arr, 8, 16, code, 0, st.data_ptr(), None) == sar.SAR_ERR_INVALID_ARG
    assert L.sar_allreduce_ll_cluster(arr, arr, 8, 16, code, 1 << 20, None, None) == sar.SAR_ERR_INVALID_ARG
    assert L.sar_allreduce_ll_cluster(arr, arr, 8, 0, code, 1 << 20, st.data_ptr(), None) == sar.SAR_OK


def test_cluster_calls_on_two_streams_overlap_safely(sar):
    """The cluster form keeps no state between calls, so calls on two streams
    without any ordering between them may run at the same time; both give
    the oracle's outputs (interleaved with SAR_ALGO_LL_ALLPAIR calls on the
    same streams, which keep no state either)."""
    n, count, dt = 8, 4096, "fp32"
    rng = np.random.default_rng(17)
    cases = []
    for s in range(2):
        ins = [random_codes(rng, dt, count) for _ in range(n)]
        gin = [Guarded.from_codes(c) for c in ins]
        gout = [Guarded(count * 4) for _ in range(n)]
        gall = [Guarded(count * 4) for _ in range(n)]
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        cases.append((ins, gin, gout, gall, st, torch.cuda.Stream()))
    torch.cuda.synchronize()
    for _ in range(50):
        for ins, gin, gout, gall, st, stream in cases:
            sar.sar_allreduce_ll_cluster([g.ptr for g in gin], [g.ptr for g in gout], st, count=count, dtype=dt,
                                         stream=stream)
            sar.sar_allreduce([g.ptr for g in gin], [g.ptr for g in gall], count=count, dtype=dt,
                              algo=sar.SAR_ALGO_LL_ALLPAIR, stream=stream)
    torch.cuda.synchronize()
    for ins, gin, gout, gall, st, stream in cases:
        want = oracle.allreduce(ins, dt)[0]
        assert sar.sar_read_device_status(st) == sar.SAR_OK
        for g in gout + gall:
            assert_same(g.codes(dt), want, dt)
