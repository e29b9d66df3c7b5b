"""GPU parity of sar_allreduce_ll_writeback: the LL allreduce whose
write-back is a second round of flagged packets (one launch: sliced up to 1
MiB per rank for the multi-destination fan-out and up to 256 KiB for the
per-output one, cooperative above), with each result packet either read once and
written to every output (multi-destination) or read by every rank for its
own output.  Outputs and the result-packet image are compared with the CPU
oracle bit for bit."""
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


def _run(sar, ins, dt, multi, epoch=None, ctrl=None, offsets=None, pk_offset=0):
    n, count = len(ins), ins[0].size
    offs = offsets or [0] * n
    gin = [Guarded.from_codes(c, o) for c, o in zip(ins, offs)]
    gout = [Guarded(count * ESIZE[dt], o, fill=0x5A) for o in offs]
    nbp = sar.sar_ll_packet_bytes(count, dt)
    pk = [Guarded(nbp, pk_offset, fill=0) for _ in range(n)]
    res = Guarded(nbp, 0, fill=0)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sar.sar_allreduce_ll_writeback([g.ptr for g in gin], [g.ptr for g in gout], [g.ptr for g in pk], res.ptr, st,
                                   multi_dest=multi, epoch=epoch or 0, epoch_ctrl=ctrl, count=count, dtype=dt)
    assert sar.sar_read_device_status(st) == sar.SAR_OK
    return gin, gout, pk, res


@pytest.mark.parametrize("multi", [True, False], ids=["multi_dest", "own_output"])
@pytest.mark.parametrize("count", [1, 3, 5, 33, 4099, 65541])
@pytest.mark.parametrize("n", [1, 2, 3, 8, 32])
@pytest.mark.parametrize("dt", DTYPES)
def test_writeback_matches_oracle(sar, dt, n, count, multi):
    rng = np.random.default_rng([DTYPES.index(dt), n, count, int(multi)])
    ins = [random_codes(rng, dt, count) for _ in range(n)]
    want = oracle.allreduce(ins, dt)[0]
    gin, gout, pk, res = _run(sar, ins, dt, multi, epoch=0x2468)
    for j, g in enumerate(gout):
        assert_same(g.codes(dt), want, dt, f"out[{j}]")
        assert g.guards_intact()
    # send packets: the closed-form image of each input; result packets: the
    # image of the reduced data (NaN payloads compared by class via the outputs)
    want_pk = oracle.ll_pack(ins, dt, 0x2468)
    for r in range(n):
        assert np.array_equal(pk[r].bytes(), want_pk[r])
    got_res = res.bytes().reshape(-1, 8)
    img = oracle.ll_pack([want], dt, 0x2468)[0].reshape(-1, 8)
    assert np.array_equal(got_res[:, 4:], img[:, 4:])                    # every flag is the epoch
    payload = np.ascontiguousarray(got_res[:, :4]).ravel()[: count * ESIZE[dt]]
    assert_same(payload.view(want.dtype), want, dt, "result packets")
    assert np.all(np.ascontiguousarray(got_res[:, :4]).ravel()[count * ESIZE[dt]:] == 0)   # zero padding
    assert res.guards_intact()


@pytest.mark.parametrize("multi", [True, False], ids=["multi_dest", "own_output"])
@pytest.mark.parametrize("dt", DTYPES)
def test_writeback_packets_16_but_not_32_byte_aligned(sar, dt, multi):
    """Send packet buffers at 16 mod 32 take the two-16-byte-store send."""
    rng = np.random.default_rng([DTYPES.index(dt), int(multi), 32])
    ins = [random_codes(rng, dt, 4099) for _ in range(5)]
    want = oracle.allreduce(ins, dt)[0]
    _, gout, pk, _ = _run(sar, ins, dt, multi, epoch=11, pk_offset=16)
    assert pk[0].ptr % 32 == 16
    for g in gout:
        assert_same(g.codes(dt), want, dt)
    want_pk = oracle.ll_pack(ins, dt, 11)
    for r in range(5):
        assert np.array_equal(pk[r].bytes(), want_pk[r])
        assert pk[r].guards_intact()


@pytest.mark.parametrize("multi", [True, False])
def test_writeback_unaligned_outputs(sar, multi):
    rng = np.random.default_rng(2)
    ins = [random_codes(rng, "fp16", 2051) for _ in range(4)]
    want = oracle.allreduce(ins, "fp16")[0]
    _, gout, _, _ = _run(sar, ins, "fp16", multi, epoch=3, offsets=[2 * (r % 2) for r in range(4)])
    for g in gout:
        assert_same(g.codes("fp16"), want, "fp16")


def test_writeback_device_epoch_and_graph(sar):
    n, count, dt = 8, 16384, "bf16"
    rng = np.random.default_rng(5)
    gin = [Guarded(count * 2) for _ in range(n)]
    gout = [Guarded(count * 2) for _ in range(n)]
    nbp = sar.sar_ll_packet_bytes(count, dt)
    pk = [Guarded(nbp, 0, fill=0) for _ in range(n)]
    res = Guarded(nbp, 0, fill=0)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ctrl = torch.zeros(2, dtype=torch.int32, device="cuda")

    def call():
        sar.sar_allreduce_ll_writeback([g.ptr for g in gin], [g.ptr for g in gout], [g.ptr for g in pk], res.ptr,
                                       st, multi_dest=True, epoch_ctrl=ctrl, count=count, dtype=dt)

    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=s):
        call()
    for e in (1, 2, 3):
        ins = [random_codes(rng, dt, count) for _ in range(n)]
        for g, c in zip(gin, ins):
            g.base[256:256 + count * 2] = torch.from_numpy(c.view(np.uint8).copy()).cuda()
        graph.replay()
        torch.cuda.synchronize()
        want = oracle.allreduce(ins, dt)[0]
        for g in gout:
            assert_same(g.codes(dt), want, dt, f"replay {e}")
        assert sar.ll_device_epoch(ctrl) == e
    assert sar.sar_read_device_status(st) == sar.SAR_OK


@pytest.mark.parametrize("wl", [w for w in W.C5 if w.bytes_per_rank in (1024, 1 << 20)], ids=lambda w: w.name)
def test_thousand_writeback_calls(sar, wl):
    n, count, dt = wl.nranks, wl.count, wl.dtype
    ins = wl.inputs()
    want = oracle.allreduce(ins, dt)[0]
    gin = [Guarded.from_codes(c) for c in ins]
    gout = [Guarded(count * ESIZE[dt]) for _ in range(n)]
    nbp = sar.sar_ll_packet_bytes(count, dt)
    pk = [Guarded(nbp, 0, fill=0) for _ in range(n)]
    res = Guarded(nbp, 0, fill=0)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for epoch in range(1, W.LL_CALLS + 1):
        sar.sar_allreduce_ll_writeback([g.ptr for g in gin], [g.ptr for g in gout], [g.ptr for g in pk], res.ptr,
                                       st, multi_dest=bool(epoch % 2), epoch=epoch, count=count, dtype=dt)
        if epoch % 250 == 0:
            torch.cuda.synchronize()
            for g in gout:
                assert_same(g.codes(dt), want, dt, f"epoch {epoch}")
    assert sar.sar_read_device_status(st) == sar.SAR_OK


@pytest.mark.parametrize("n,dt,count", [(8, "fp32", 262144), (8, "fp32", 262145), (2, "bf16", 524288),
                                        (2, "bf16", 524289)])
def test_multi_dest_on_both_sides_of_the_sliced_limit(sar, n, dt, count):
    """1 MiB per rank runs sliced, one element more cooperatively: both give
    the oracle's outputs and result-packet flags."""
    rng = np.random.default_rng([n, count, 6])
    ins = [random_codes(rng, dt, count) for _ in range(n)]
    want = oracle.allreduce(ins, dt)[0]
    gin, gout, pk, res = _run(sar, ins, dt, True, epoch=77)
    for j, g in enumerate(gout):
        assert_same(g.codes(dt), want, dt, f"out[{j}]")
        assert g.guards_intact()
    got_res = res.bytes().reshape(-1, 8)
    assert np.all(got_res[:, 4:].copy().view(np.uint32).ravel() == 77)
    assert res.guards_intact()


@pytest.mark.parametrize("n,dt,count", [(8, "fp32", 65536), (8, "fp32", 65537), (5, "bf16", 131072),
                                        (5, "bf16", 131073)])
def test_own_output_on_both_sides_of_the_sliced_limit(sar, n, dt, count):
    """256 KiB per rank runs sliced, one element more cooperatively: both give
    the oracle's outputs and result-packet flags."""
    rng = np.random.default_rng([n, count, 7])
    ins = [random_codes(rng, dt, count) for _ in range(n)]
    want = oracle.allreduce(ins, dt)[0]
    gin, gout, pk, res = _run(sar, ins, dt, False, epoch=78)
    for j, g in enumerate(gout):
        assert_same(g.codes(dt), want, dt, f"out[{j}]")
        assert g.guards_intact()
    got_res = res.bytes().reshape(-1, 8)
    assert np.all(got_res[:, 4:].copy().view(np.uint32).ravel() == 78)
    assert res.guards_intact()
