"""GPU parity of the LL-packet path (pack, poll/unpack/reduce, and the two
together) against the CPU oracle, through the C ABI, plus the bounded-wait
failure path: a flag that nothing ever sets makes the poll give up, record
SAR_ERR_TIMEOUT on the device and return, leaving the context usable."""
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


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _packets(sar, n, count, dt, fill=0):
    return [Guarded(sar.sar_ll_packet_bytes(count, dt), 0, fill=fill) for _ in range(n)]


@pytest.mark.parametrize("count", [1, 2, 3, 5, 8, 33, 1031, 65541])
@pytest.mark.parametrize("n", [1, 2, 3, 6, 8, 32])
@pytest.mark.parametrize("dt", DTYPES)
def test_pack_unpack_match_oracle(sar, dt, n, count):
    rng = np.random.default_rng([DTYPES.index(dt), n, count])
    ins = [random_codes(rng, dt, count) for _ in range(n)]
    epoch = 0x01020304 + count
    gin = [Guarded.from_codes(c) for c in ins]
    pk = _packets(sar, n, count, dt)
    sar.sar_ll_pack([g.ptr for g in gin], [g.ptr for g in pk], epoch, count=count, dtype=dt)
    torch.cuda.synchronize()
    want_pk = oracle.ll_pack(ins, dt, epoch)
    for r in range(n):
        assert np.array_equal(pk[r].bytes(), want_pk[r]), f"packet image of rank {r}"
        assert pk[r].guards_intact()
    # unpack the GPU's packets
    st = _status()
    gout = [Guarded(count * ESIZE[dt], 0, fill=0x5A) for _ in range(n)]
    sar.sar_ll_unpack_reduce([g.ptr for g in pk], [g.ptr for g in gout], epoch, st, count=count, dtype=dt)
    assert sar.sar_read_device_status(st) == sar.SAR_OK
    want = oracle.allreduce(ins, dt)[0]
    for j, g in enumerate(gout):
        assert_same(g.codes(dt), want, dt, f"out[{j}]")
        assert g.guards_intact()
    for r, g in enumerate(gin):
        assert_same(g.codes(dt), ins[r], dt, "input modified")


@pytest.mark.parametrize("which", ["rank0", "all"])
@pytest.mark.parametrize("count", [1, 7, 1031, 65541])
@pytest.mark.parametrize("dt", DTYPES)
def test_pack_into_16_but_not_32_byte_aligned_packets(sar, dt, count, which):
    """Packet buffers at 16 mod 32 (one rank, or all) take the two-16-byte-store
    pack instead of the 32-byte one; the packet image and the sums are the same."""
    n = 4
    rng = np.random.default_rng([DTYPES.index(dt), count, 16])
    ins = [random_codes(rng, dt, count) for _ in range(n)]
    epoch = 0x0A0B0C0D
    gin = [Guarded.from_codes(c) for c in ins]
    offs = [16 if (which == "all" or r == 0) else 0 for r in range(n)]
    pk = [Guarded(sar.sar_ll_packet_bytes(count, dt), o, fill=0) for o in offs]
    assert pk[0].ptr % 32 == 16
    sar.sar_ll_pack([g.ptr for g in gin], [g.ptr for g in pk], epoch, count=count, dtype=dt)
    torch.cuda.synchronize()
    want_pk = oracle.ll_pack(ins, dt, epoch)
    for r in range(n):
        assert np.array_equal(pk[r].bytes(), want_pk[r]), f"packet image of rank {r}"
        assert pk[r].guards_intact()
    st = _status()
    gout = [Guarded(count * ESIZE[dt]) for _ in range(n)]
    sar.sar_allreduce_ll([g.ptr for g in gin], [g.ptr for g in gout], [g.ptr for g in pk], epoch + 1, st,
                         count=count, dtype=dt)
    assert sar.sar_read_device_status(st) == sar.SAR_OK
    want = oracle.allreduce(ins, dt)[0]
    for g in gout:
        assert_same(g.codes(dt), want, dt)
        assert g.guards_intact()


@pytest.mark.parametrize("dt", DTYPES)
def test_unpack_reads_oracle_packets(sar, dt):
    """Packets written by the oracle (not by the GPU) unpack to the oracle's sums."""
    rng = np.random.default_rng(4)
    n, count = 8, 4099
    ins = [random_codes(rng, dt, count) for _ in range(n)]
    pk = [Guarded.from_codes(p) for p in oracle.ll_pack(ins, dt, 99)]
    gout = [Guarded(count * ESIZE[dt]) for _ in range(n)]
    st = _status()
    sar.sar_ll_unpack_reduce([g.ptr for g in pk], [g.ptr for g in gout], 99, st, count=count, dtype=dt)
    assert sar.sar_read_device_status(st) == sar.SAR_OK
    rc, want = oracle.ll_unpack_reduce(oracle.ll_pack(ins, dt, 99), count, dt, 99)
    assert rc == oracle.OK
    for g in gout:
        assert_same(g.codes(dt), want[0], dt)


@pytest.mark.parametrize("dt", DTYPES)
def test_allreduce_ll_unaligned_and_in_place(sar, dt):
    rng = np.random.default_rng(5)
    n, count = 4, 2053
    ins = [random_codes(rng, dt, count) for _ in range(n)]
    want = oracle.allreduce(ins, dt)[0]
    offs = [ESIZE[dt] * (r % 2) for r in range(n)]
    gin = [Guarded.from_codes(c, o) for c, o in zip(ins, offs)]
    gout = [Guarded(count * ESIZE[dt], o) for o in reversed(offs)]
    pk = _packets(sar, n, count, dt)
    st = _status()
    sar.sar_allreduce_ll([g.ptr for g in gin], [g.ptr for g in gout], [g.ptr for g in pk], 7, st,
                         count=count, dtype=dt)
    assert sar.sar_read_device_status(st) == sar.SAR_OK
    for g in gout:
        assert_same(g.codes(dt), want, dt)
        assert g.guards_intact()
    # in place: outputs are the inputs
    sar.sar_allreduce_ll([g.ptr for g in gin], [g.ptr for g in gin], [g.ptr for g in pk], 8, st,
                         count=count, dtype=dt)
    assert sar.sar_read_device_status(st) == sar.SAR_OK
    for g in gin:
        assert_same(g.codes(dt), want, dt)


def test_stale_epoch_times_out_and_context_survives(sar):
    """Packets that never carry the awaited epoch: zeroed scratch (epoch 0 =
    never written) and packets of an earlier epoch.  The bounded poll gives
    up, the device status reads SAR_ERR_TIMEOUT, and the GPU keeps working."""
    n, count, dt = 4, 1000, "fp32"
    rng = np.random.default_rng(6)
    ins = [random_codes(rng, dt, count) for _ in range(n)]
    gin = [Guarded.from_codes(c) for c in ins]
    gout = [Guarded(count * 4) for _ in range(n)]
    pk = _packets(sar, n, count, dt, fill=0)
    st = _status()
    sar.sar_ll_unpack_reduce([g.ptr for g in pk], [g.ptr for g in gout], 5, st, max_spins=64,
                             count=count, dtype=dt)
    assert sar.sar_read_device_status(st) == sar.SAR_ERR_TIMEOUT
    # packets of epoch 5, reader waits for 6
    st.zero_()
    sar.sar_ll_pack([g.ptr for g in gin], [g.ptr for g in pk], 5, count=count, dtype=dt)
    sar.sar_ll_unpack_reduce([g.ptr for g in pk], [g.ptr for g in gout], 6, st, max_spins=64,
                             count=count, dtype=dt)
    assert sar.sar_read_device_status(st) == sar.SAR_ERR_TIMEOUT
    # a single stale packet is enough
    st.zero_()
    sar.sar_ll_pack([g.ptr for g in gin], [g.ptr for g in pk], 6, count=count, dtype=dt)
    torch.cuda.synchronize()
    pk[2].base[256 + 8 * 517 + 4] ^= 1
    sar.sar_ll_unpack_reduce([g.ptr for g in pk], [g.ptr for g in gout], 6, st, max_spins=64,
                             count=count, dtype=dt)
    assert sar.sar_read_device_status(st) == sar.SAR_ERR_TIMEOUT
    # the context still works
    st.zero_()
    sar.sar_allreduce_ll([g.ptr for g in gin], [g.ptr for g in gout], [g.ptr for g in pk], 7, st,
                         count=count, dtype=dt)
    assert sar.sar_read_device_status(st) == sar.SAR_OK
    want = oracle.allreduce(ins, dt)[0]
    for g in gout:
        assert_same(g.codes(dt), want, dt)


def test_graph_capture_ll(sar):
    n, count, dt = 8, 4096, "bf16"
    rng = np.random.default_rng(8)
    gin = [Guarded(count * 2) for _ in range(n)]
    gout = [Guarded(count * 2) for _ in range(n)]
    pk = _packets(sar, n, count, dt)
    st = _status()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=s):
        sar.sar_allreduce_ll([g.ptr for g in gin], [g.ptr for g in gout], [g.ptr for g in pk], 11, st,
                             count=count, dtype=dt)
    for rep in range(3):
        ins = [random_codes(rng, dt, count) for _ in range(n)]
        for g, c in zip(gin, ins):
            g.base[256:256 + count * 2] = torch.from_numpy(c.view(np.uint8).copy()).cuda()
        graph.replay()
        torch.cuda.synchronize()
        want = oracle.allreduce(ins, dt)[0]
        for g in gout:
            assert_same(g.codes(dt), want, dt, f"replay {rep}")
    assert sar.sar_read_device_status(st) == sar.SAR_OK


@pytest.mark.parametrize("wl", W.C5, ids=[w.name for w in W.C5])
def test_thousand_epochs(sar, wl):
    """8 ranks, 1000 back-to-back calls with epoch 1..1000 on one packet
    scratch; every 100th call's outputs and packets are checked."""
    n, count, dt = wl.nranks, wl.count, wl.dtype
    ins = wl.inputs()
    gin = [Guarded.from_codes(c) for c in ins]
    gout = [Guarded(count * ESIZE[dt]) for _ in range(n)]
    pk = _packets(sar, n, count, dt, fill=0)
    st = _status()
    want = oracle.allreduce(ins, dt)[0]
    for epoch in range(1, W.LL_CALLS + 1):
        sar.sar_allreduce_ll([g.ptr for g in gin], [g.ptr for g in gout], [g.ptr for g in pk], epoch, st,
                             count=count, dtype=dt)
        if epoch % 100 == 0:
            torch.cuda.synchronize()
            for g in gout:
                assert_same(g.codes(dt), want, dt, f"epoch {epoch}")
            want_pk = oracle.ll_pack(ins, dt, epoch)
            for r in range(n):
                assert np.array_equal(pk[r].bytes(), want_pk[r])
    assert sar.sar_read_device_status(st) == sar.SAR_OK


def _double_scratch(sar, n, count, dt):
    return [Guarded(sar.ll_double_packet_bytes(count, dt), 0, fill=0) for _ in range(n)]


@pytest.mark.parametrize("count", [1, 5, 1031, 65541])
@pytest.mark.parametrize("n", [2, 3, 8])
@pytest.mark.parametrize("dt", DTYPES)
def test_double_buffer_halves_match_oracle(sar, dt, n, count):
    """Epoch 1 packs into and polls the second half, epoch 2 the first: after
    both calls each half holds exactly its own call's packet image, and each
    call's outputs are the oracle's sums."""
    rng = np.random.default_rng([DTYPES.index(dt), n, count, 7])
    half = sar.ll_double_packet_bytes(count, dt) // 2
    pk = _double_scratch(sar, n, count, dt)
    st = _status()
    seen = {}
    for epoch in (1, 2):
        ins = [random_codes(rng, dt, count) for _ in range(n)]
        gin = [Guarded.from_codes(c) for c in ins]
        gout = [Guarded(count * ESIZE[dt], 0, fill=0x5A) for _ in range(n)]
        sar.sar_allreduce_ll_double([g.ptr for g in gin], [g.ptr for g in gout], [g.ptr for g in pk], epoch, st,
                                    count=count, dtype=dt)
        assert sar.sar_read_device_status(st) == sar.SAR_OK
        want = oracle.allreduce(ins, dt)[0]
        for g in gout:
            assert_same(g.codes(dt), want, dt, f"epoch {epoch}")
            assert g.guards_intact()
        seen[epoch] = oracle.ll_pack(ins, dt, epoch)
    for r in range(n):
        b = pk[r].bytes()
        nb = seen[1][r].size
        assert np.array_equal(b[half: half + nb], seen[1][r]), "epoch 1 half overwritten"
        assert np.array_equal(b[:nb], seen[2][r]), "epoch 2 half"
        assert pk[r].guards_intact()


def test_double_buffer_two_streams_share_one_scratch(sar):
    """Two streams run LL allreduces on one double-buffered scratch at the same
    time, one with odd epochs and one with even: their packets never overlap,
    so both get their own sums.  (No kernel waits on the other stream's.)"""
    n, count, dt, iters = 8, 16384, "fp32", 50
    rng = np.random.default_rng(31)
    pk = _double_scratch(sar, n, count, dt)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    ins = [[random_codes(rng, dt, count) for _ in range(n)] for _ in range(2)]
    gin = [[Guarded.from_codes(c) for c in x] for x in ins]
    gout = [[Guarded(count * 4) for _ in range(n)] for _ in range(2)]
    st = [_status(), _status()]
    torch.cuda.synchronize()
    for i in range(iters):
        for s in range(2):
            sar.sar_allreduce_ll_double([g.ptr for g in gin[s]], [g.ptr for g in gout[s]], [g.ptr for g in pk],
                                        2 * i + 1 + s, st[s], max_spins=1 << 24, count=count, dtype=dt,
                                        stream=streams[s])
    torch.cuda.synchronize()
    for s in range(2):
        assert sar.sar_read_device_status(st[s]) == sar.SAR_OK
        want = oracle.allreduce(ins[s], dt)[0]
        for g in gout[s]:
            assert_same(g.codes(dt), want, dt, f"stream {s}")
