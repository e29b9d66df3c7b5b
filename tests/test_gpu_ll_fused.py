"""GPU parity of sar_allreduce_ll_fused (send, poll, reduce and write-back in
one launch: sliced up to 256 KiB per rank, where each block polls packets
its other warps have just written, cooperative above, where polls race
against packing blocks) against the CPU oracle, through the C ABI; and the
device-resident epoch counter that advances on every launch, including
CUDA-graph replays."""
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


def _packets(sar, n, count, dt):
    return [Guarded(sar.sar_ll_packet_bytes(count, dt), 0, fill=0) for _ in range(n)]


@pytest.mark.parametrize("count", [1, 3, 5, 33, 1031, 65541, 262147])
@pytest.mark.parametrize("n", [1, 2, 5, 8, 32])
@pytest.mark.parametrize("dt", DTYPES)
def test_fused_matches_oracle(sar, dt, n, count):
    rng = np.random.default_rng([DTYPES.index(dt), n, count])
    ins = [random_codes(rng, dt, count) for _ in range(n)]
    want = oracle.allreduce(ins, dt)[0]
    gin = [Guarded.from_codes(c) for c in ins]
    gout = [Guarded(count * ESIZE[dt], 0, fill=0x5A) for _ in range(n)]
    pk = _packets(sar, n, count, dt)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for epoch in (1, 2):
        sar.sar_allreduce_ll_fused([g.ptr for g in gin], [g.ptr for g in gout], [g.ptr for g in pk], st,
                                   epoch=epoch, count=count, dtype=dt)
    assert sar.sar_read_device_status(st) == sar.SAR_OK
    for j, g in enumerate(gout):
        assert_same(g.codes(dt), want, dt, f"out[{j}]")
        assert g.guards_intact()
    want_pk = oracle.ll_pack(ins, dt, 2)
    for r in range(n):
        assert np.array_equal(pk[r].bytes(), want_pk[r])
        assert pk[r].guards_intact()


@pytest.mark.parametrize("count", [7, 4099, 65541])
@pytest.mark.parametrize("dt", DTYPES)
def test_fused_packets_16_but_not_32_byte_aligned(sar, dt, count):
    """Packet buffers at 16 mod 32 take the two-16-byte-store send."""
    n = 4
    rng = np.random.default_rng([DTYPES.index(dt), count, 32])
    ins = [random_codes(rng, dt, count) for _ in range(n)]
    want = oracle.allreduce(ins, dt)[0]
    gin = [Guarded.from_codes(c) for c in ins]
    gout = [Guarded(count * ESIZE[dt]) for _ in range(n)]
    pk = [Guarded(sar.sar_ll_packet_bytes(count, dt), 16 if r % 2 else 0, fill=0) for r in range(n)]
    assert pk[1].ptr % 32 == 16
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sar.sar_allreduce_ll_fused([g.ptr for g in gin], [g.ptr for g in gout], [g.ptr for g in pk], st, epoch=5,
                               count=count, dtype=dt)
    assert sar.sar_read_device_status(st) == sar.SAR_OK
    for g in gout:
        assert_same(g.codes(dt), want, dt)
    want_pk = oracle.ll_pack(ins, dt, 5)
    for r in range(n):
        assert np.array_equal(pk[r].bytes(), want_pk[r])
        assert pk[r].guards_intact()


@pytest.mark.parametrize("dt", DTYPES)
def test_fused_unaligned(sar, dt):
    rng = np.random.default_rng(7)
    n, count = 4, 4099
    ins = [random_codes(rng, dt, count) for _ in range(n)]
    want = oracle.allreduce(ins, dt)[0]
    offs = [ESIZE[dt] * (r % 2) for r in range(n)]
    gin = [Guarded.from_codes(c, o) for c, o in zip(ins, offs)]
    gout = [Guarded(count * ESIZE[dt], o) for o in reversed(offs)]
    pk = _packets(sar, n, count, dt)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sar.sar_allreduce_ll_fused([g.ptr for g in gin], [g.ptr for g in gout], [g.ptr for g in pk], st, epoch=9,
                               count=count, dtype=dt)
    assert sar.sar_read_device_status(st) == sar.SAR_OK
    for g in gout:
        assert_same(g.codes(dt), want, dt)


def test_device_epoch_advances_per_launch_and_per_graph_replay(sar):
    n, count, dt = 8, 65536, "bf16"
    rng = np.random.default_rng(8)
    gin = [Guarded(count * 2) for _ in range(n)]
    gout = [Guarded(count * 2) for _ in range(n)]
    pk = _packets(sar, n, count, dt)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ctrl = torch.zeros(2, dtype=torch.int32, device="cuda")

    def fill():
        ins = [random_codes(rng, dt, count) for _ in range(n)]
        for g, c in zip(gin, ins):
            g.base[256:256 + count * 2] = torch.from_numpy(c.view(np.uint8).copy()).cuda()
        return ins

    def check(ins, epoch):
        torch.cuda.synchronize()
        want = oracle.allreduce(ins, dt)[0]
        for g in gout:
            assert_same(g.codes(dt), want, dt, f"epoch {epoch}")
        assert sar.ll_device_epoch(ctrl) == epoch
        assert np.array_equal(pk[3].bytes(), oracle.ll_pack(ins, dt, epoch)[3])

    for e in (1, 2, 3):
        ins = fill()
        sar.sar_allreduce_ll_fused([g.ptr for g in gin], [g.ptr for g in gout], [g.ptr for g in pk], st,
                                   epoch_ctrl=ctrl, count=count, dtype=dt)
        check(ins, e)
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=s):
        sar.sar_allreduce_ll_fused([g.ptr for g in gin], [g.ptr for g in gout], [g.ptr for g in pk], st,
                                   epoch_ctrl=ctrl, count=count, dtype=dt)
    for e in (4, 5, 6, 7):
        ins = fill()
        graph.replay()
        check(ins, e)
    assert sar.sar_read_device_status(st) == sar.SAR_OK


@pytest.mark.parametrize("wl", [w for w in W.C5 if w.bytes_per_rank in (1024, 1 << 20)], ids=lambda w: w.name)
def test_thousand_fused_calls(sar, wl):
    n, count, dt = wl.nranks, wl.count, wl.dtype
    ins = wl.inputs()
    gin = [Guarded.from_codes(c) for c in ins]
    gout = [Guarded(count * ESIZE[dt]) for _ in range(n)]
    pk = _packets(sar, n, count, dt)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    want = oracle.allreduce(ins, dt)[0]
    for epoch in range(1, W.LL_CALLS + 1):
        sar.sar_allreduce_ll_fused([g.ptr for g in gin], [g.ptr for g in gout], [g.ptr for g in pk], st,
                                   epoch=epoch, count=count, dtype=dt)
        if epoch % 250 == 0:
            torch.cuda.synchronize()
            for g in gout:
                assert_same(g.codes(dt), want, dt, f"epoch {epoch}")
    assert sar.sar_read_device_status(st) == sar.SAR_OK


@pytest.mark.parametrize("last,next_epoch", [(0xFFFFFFFE, 0xFFFFFFFF), (0xFFFFFFFF, 1)])
def test_device_epoch_wraps_past_zero(sar, last, next_epoch):
    """After epoch 2^32 - 1 the counter's next epoch is 1: the reserved 0 is
    skipped."""
    n, count, dt = 4, 3001, "fp32"
    rng = np.random.default_rng(12)
    ins = [random_codes(rng, dt, count) for _ in range(n)]
    want = oracle.allreduce(ins, dt)[0]
    gin = [Guarded.from_codes(c) for c in ins]
    gout = [Guarded(count * 4) for _ in range(n)]
    pk = _packets(sar, n, count, dt)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ctrl = torch.zeros(1, dtype=torch.int64, device="cuda")
    sar.ll_set_device_epoch(ctrl, last)
    sar.sar_allreduce_ll_fused([g.ptr for g in gin], [g.ptr for g in gout], [g.ptr for g in pk], st,
                               epoch_ctrl=ctrl, count=count, dtype=dt)
    assert sar.sar_read_device_status(st) == sar.SAR_OK
    assert sar.ll_device_epoch(ctrl) == next_epoch
    assert int(ctrl.item()) & ((1 << sar.LL_EPOCH_SHIFT) - 1) == 0      # no ticket left over
    for g in gout:
        assert_same(g.codes(dt), want, dt)
    assert np.array_equal(pk[0].bytes(), oracle.ll_pack(ins, dt, next_epoch)[0])


@pytest.mark.parametrize("n,dt,count", [(8, "fp32", 65536), (8, "fp32", 65537), (2, "bf16", 131072),
                                        (2, "bf16", 131073), (32, "e4m3fn", 262144), (32, "e4m3fn", 262145)])
def test_fused_on_both_sides_of_the_sliced_limit(sar, n, dt, count):
    """256 KiB per rank runs sliced, one element more runs cooperatively:
    both exact, and both leave the oracle's packet image."""
    rng = np.random.default_rng([n, count, 5])
    ins = [random_codes(rng, dt, count) for _ in range(n)]
    want = oracle.allreduce(ins, dt)[0]
    gin = [Guarded.from_codes(c) for c in ins]
    gout = [Guarded(count * ESIZE[dt], 0, fill=0x5A) for _ in range(n)]
    pk = _packets(sar, n, count, dt)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sar.sar_allreduce_ll_fused([g.ptr for g in gin], [g.ptr for g in gout], [g.ptr for g in pk], st, epoch=3,
                               count=count, dtype=dt)
    assert sar.sar_read_device_status(st) == sar.SAR_OK
    for g in gout:
        assert_same(g.codes(dt), want, dt)
        assert g.guards_intact()
    want_pk = oracle.ll_pack(ins, dt, 3)
    for r in range(n):
        assert np.array_equal(pk[r].bytes(), want_pk[r])
        assert pk[r].guards_intact()
