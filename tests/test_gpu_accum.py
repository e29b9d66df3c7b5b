"""GPU parity of sar_allreduce_accum (partial sums rounded into fp16, bf16 or
the input type) against the CPU oracle, through the C ABI.  Bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.gpu_util import ESIZE, Guarded, assert_same, random_codes

pytestmark = pytest.mark.gpu

PAIRS = [("e4m3fn", "e4m3fn"), ("e4m3fn", "fp16"), ("e4m3fn", "bf16"), ("e4m3fn", "fp32"),
         ("bf16", "bf16"), ("bf16", "fp16"), ("fp16", "fp16"), ("fp16", "bf16"), ("fp32", "fp16"), ("fp32", "bf16"),
         ("e4m3b15", "e4m3b15"), ("e4m3b15", "fp16"), ("e4m3b15", "fp32")]


@pytest.fixture(scope="module")
def sar():
    import allreduce_reduction_rank_gb300 as s
    return s


def _run(sar, ins, dt, acc, offsets=None):
    n, count = len(ins), ins[0].size
    offs = offsets or [0] * n
    gin = [Guarded.from_codes(c, o) for c, o in zip(ins, offs)]
    gout = [Guarded(count * ESIZE[dt], o, fill=0x5A) for o in offs]
    sar.sar_allreduce_accum([g.ptr for g in gin], [g.ptr for g in gout], acc, count=count, dtype=dt)
    torch.cuda.synchronize()
    return gin, gout


@pytest.mark.parametrize("count", [1, 9, 4097, 100003])
@pytest.mark.parametrize("n", [1, 2, 6, 8, 32])
@pytest.mark.parametrize("dt,acc", PAIRS)
def test_accum_matches_oracle(sar, dt, acc, n, count):
    rng = np.random.default_rng([n, count, len(dt), len(acc)])
    ins = [random_codes(rng, dt, count) for _ in range(n)]
    want = oracle.allreduce_accum(ins, dt, acc)[0]
    gin, gout = _run(sar, ins, dt, acc)
    for j, g in enumerate(gout):
        assert_same(g.codes(dt), want, dt, f"out[{j}]")
        assert g.guards_intact()
    for r, g in enumerate(gin):
        assert_same(g.codes(dt), ins[r], dt, "input modified")


@pytest.mark.parametrize("dt,acc", [("e4m3fn", "e4m3fn"), ("e4m3fn", "fp16"), ("bf16", "bf16")])
def test_accum_unaligned(sar, dt, acc):
    rng = np.random.default_rng(3)
    ins = [random_codes(rng, dt, 3001) for _ in range(8)]
    want = oracle.allreduce_accum(ins, dt, acc)[0]
    _, gout = _run(sar, ins, dt, acc, offsets=[ESIZE[dt] * (r % 3) for r in range(8)])
    for g in gout:
        assert_same(g.codes(dt), want, dt)


def test_accum_fp32_is_sar_allreduce(sar):
    ins = W.rank_inputs("normal", 2, "e4m3fn", 65537, 8, 4.0)
    _, a = _run(sar, ins, "e4m3fn", "fp32")
    gin = [Guarded.from_codes(c) for c in ins]
    gout = [Guarded(65537) for _ in range(8)]
    sar.sar_allreduce([g.ptr for g in gin], [g.ptr for g in gout], count=65537, dtype="e4m3fn")
    torch.cuda.synchronize()
    assert np.array_equal(a[0].bytes(), gout[0].bytes())


def test_unsupported_accumulators_are_rejected(sar):
    bufs = [Guarded(64) for _ in range(2)]
    p = [b.ptr for b in bufs]
    with pytest.raises(sar.SarError) as ei:
        sar.sar_allreduce_accum(p, p, "e4m3fn", count=16, dtype="bf16")   # e4m3fn accumulator for bf16 data
    assert ei.value.status == sar.SAR_ERR_UNSUPPORTED_DTYPE


@pytest.mark.parametrize("acc", ["e4m3fn", "fp16", "fp32"])
def test_full_size_e4m3fn_workload_sampled(sar, acc):
    """The 8 x 16 MiB e4m3fn workload, sampled against the oracle."""
    wl = W.C4
    ins = wl.inputs()
    din = [torch.from_numpy(x).cuda() for x in ins]
    dout = [torch.empty_like(din[0]) for _ in range(wl.nranks)]
    sar.sar_allreduce_accum(din, dout, acc, count=wl.count, dtype="e4m3fn")
    torch.cuda.synchronize()
    idx = np.unique(np.concatenate([np.random.default_rng(1).integers(0, wl.count, 50000), [0, wl.count - 1]]))
    want = oracle.allreduce_accum([x[idx] for x in ins], "e4m3fn", acc)[0]
    tidx = torch.from_numpy(idx.astype(np.int64)).cuda()
    for j in range(wl.nranks):
        assert np.array_equal(dout[j][tidx].cpu().numpy(), want)
        assert torch.equal(dout[j], dout[0])


@pytest.mark.parametrize("n", [2, 3])
def test_native_e4m3fn_every_pair(sar, n):
    """Native e4m3fn accumulation over every ordered pair of codes (NaN
    included), then, with 3 ranks, a third code on top of every rounded pair
    sum: each step R(acc + x) on the vector path."""
    a = np.repeat(np.arange(256, dtype=np.uint8), 256)
    b = np.tile(np.arange(256, dtype=np.uint8), 256)
    ins = [a, b]
    if n == 3:
        ins.append(np.roll(b, 17) ^ 0x80)
    want = oracle.allreduce_accum(ins, "e4m3fn", "e4m3fn")[0]
    _, gout = _run(sar, ins, "e4m3fn", "e4m3fn")
    for g in gout:
        assert_same(g.codes("e4m3fn"), want, "e4m3fn")
        assert g.guards_intact()
