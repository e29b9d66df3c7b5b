"""The bounded polls of the one-launch LL kernels (sar_allreduce_ll_fused and
sar_allreduce_ll_writeback in both fan-outs) running out.

In the cooperative form the packets a block polls are written by other
blocks of the same launch, so with max_spins = 1 (one re-read) at 8 x 2 MiB
(cooperative for every kind) the polls give up: the status word reads
SAR_ERR_TIMEOUT, the launch ends, and the context stays usable.  The next
call on the same buffers with the normal bound gives the oracle's outputs.
With the device epoch counter the counter still advances by one per launch,
timed out or not, so the next launch gets a fresh epoch.  The sliced form
(direct and per-output write-backs up to 256 KiB per rank, multi-destination
up to 1 MiB) polls packets that warps of the same block have just written, so one
re-read may or may not run out; its test checks what must hold either way.
The failure is made by a short wait limit, the form of fault injection that
leaves the GPU healthy."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.gpu_util import ESIZE, Guarded, assert_same

pytestmark = pytest.mark.gpu

KINDS = ["fused", "writeback_multi_dest", "writeback_own_output"]


@pytest.fixture(scope="module")
def sar():
    import allreduce_reduction_rank_gb300 as s
    return s


def _call(sar, kind, gin, gout, pk, res, st, count, dt, max_spins, epoch=0, ctrl=None):
    args = ([g.ptr for g in gin], [g.ptr for g in gout], [g.ptr for g in pk])
    if kind == "fused":
        sar.sar_allreduce_ll_fused(*args, st, epoch=epoch, epoch_ctrl=ctrl, max_spins=max_spins, count=count,
                                   dtype=dt)
    else:
        sar.sar_allreduce_ll_writeback(*args, res.ptr, st, multi_dest=kind == "writeback_multi_dest", epoch=epoch,
                                       epoch_ctrl=ctrl, max_spins=max_spins, count=count, dtype=dt)


def _short_bound_then_exact(sar, kind, device_epoch, bytes_per_rank, must_time_out):
    n, dt = 8, "fp32"
    count = bytes_per_rank // 4
    rng = np.random.default_rng([bytes_per_rank, KINDS.index(kind), device_epoch])
    ins = [(rng.random(count, dtype=np.float32) * 2 - 1).astype(np.float32) for _ in range(n)]
    want = oracle.allreduce(ins, dt)[0]
    gin = [Guarded.from_codes(c) for c in ins]
    gout = [Guarded(count * ESIZE[dt]) for _ in range(n)]
    nbp = sar.sar_ll_packet_bytes(count, dt)
    pk = [Guarded(nbp, 0, fill=0) for _ in range(n)]
    res = Guarded(nbp, 0, fill=0)
    ctrl = torch.zeros(1, dtype=torch.int64, device="cuda") if device_epoch else None
    epoch, timeouts, launches = 0, 0, 0
    for _ in range(5):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        epoch += 1
        _call(sar, kind, gin, gout, pk, res, st, count, dt, max_spins=1, epoch=epoch, ctrl=ctrl)
        launches += 1
        rc = sar.sar_read_device_status(st)
        assert rc in (sar.SAR_OK, sar.SAR_ERR_TIMEOUT)
        if rc == sar.SAR_OK:                       # nothing ran out: the outputs are complete
            for g in gout:
                assert_same(g.codes(dt), want, dt)
        timeouts += rc == sar.SAR_ERR_TIMEOUT
        for g in gout:
            assert g.guards_intact()
        for g in pk:
            assert g.guards_intact()
        assert res.guards_intact()
    if must_time_out:
        assert timeouts > 0, "one re-read per poll never ran out in the cooperative form"
    # the same context, the normal bound: exact again
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for g in gout:
        g.base[256:256 + count * 4] = 0
    _call(sar, kind, gin, gout, pk, res, st, count, dt, max_spins=1 << 20, epoch=epoch + 1, ctrl=ctrl)
    launches += 1
    assert sar.sar_read_device_status(st) == sar.SAR_OK
    for g in gout:
        assert_same(g.codes(dt), want, dt)
    if device_epoch:
        assert sar.ll_device_epoch(ctrl) == launches


@pytest.mark.parametrize("device_epoch", [False, True], ids=["host_epoch", "device_epoch"])
@pytest.mark.parametrize("kind", KINDS)
def test_coop_polls_run_out_and_the_next_call_is_exact(sar, kind, device_epoch):
    _short_bound_then_exact(sar, kind, device_epoch, 2 << 20, must_time_out=True)


@pytest.mark.parametrize("device_epoch", [False, True], ids=["host_epoch", "device_epoch"])
@pytest.mark.parametrize("kind", KINDS)
def test_sliced_polls_with_one_reread_and_the_next_call_is_exact(sar, kind, device_epoch):
    _short_bound_then_exact(sar, kind, device_epoch, 256 << 10, must_time_out=False)
