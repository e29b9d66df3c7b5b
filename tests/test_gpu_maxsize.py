"""Sizes past 32-bit indexing: more than 2^32 elements per rank for the rsag
kernels (fused and two-phase) and LL packet buffers past 4 GiB.

The inputs are seeded patterns generated on the host (length P, a prime, so
a truncated or wrapped index reads a different value) and tiled on the
device by plain copies; sampled outputs (around 2^31, 2^32, the rank-chunk
boundaries and the end, plus random indices) are checked against the oracle,
and every output must equal output 0."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

P = 1000003


@pytest.fixture(scope="module")
def sar():
    import allreduce_reduction_rank_gb300 as s
    return s


def _tiled(pattern: np.ndarray, count: int, torch_dtype) -> torch.Tensor:
    t = torch.empty(count, dtype=torch_dtype, device="cuda")
    pt = torch.from_numpy(pattern.view(np.int16) if pattern.dtype == np.uint16 else pattern).cuda()
    full, rem = divmod(count, P)
    t[: full * P].view(full, P).copy_(pt.expand(full, P))
    t[full * P:] = pt[:rem]
    return t


def _indices(count, n, dt, rng):
    idx = [0, 1, P - 1, P, (1 << 31) - 1, 1 << 31, (1 << 32) - 1, 1 << 32, (1 << 32) + 1, count - 2, count - 1]
    for r in range(1, n):
        b, _ = oracle.rsag_chunk(count, n, dt, r)
        idx += [b - 1, b, b + 1]
    idx += list(rng.integers(0, count, 20000))
    return np.unique(np.clip(np.array(idx, dtype=np.int64), 0, count - 1))


@pytest.mark.parametrize("algo", [0, 1], ids=["rsag", "two_phase"])
def test_rsag_past_2_32_elements(sar, algo):
    n, dt, count = 2, "e4m3fn", (1 << 32) + 4099
    pats = W.rank_inputs("normal", 7, dt, P, n, 4.0)
    din = [_tiled(p, count, torch.uint8) for p in pats]
    dout = [torch.empty_like(din[0]) for _ in range(n)]
    sar.sar_allreduce(din, dout, count=count, dtype=dt, algo=algo)
    torch.cuda.synchronize()
    idx = _indices(count, n, dt, np.random.default_rng(algo))
    want = oracle.allreduce([p[idx % P] for p in pats], dt)[0]
    tidx = torch.from_numpy(idx).cuda()
    for j in range(n):
        assert np.array_equal(dout[j][tidx].cpu().numpy(), want)
        assert torch.equal(dout[j], dout[0])
    del din, dout
    torch.cuda.empty_cache()


def test_ll_packets_past_4_gib(sar):
    n, dt, count = 2, "fp32", (1 << 29) + 5          # 2 GiB of input, 4 GiB of packets per rank
    pats = W.rank_inputs("uniform", 8, dt, P, n)
    din = [_tiled(p, count, torch.float32) for p in pats]
    dout = [torch.empty_like(din[0]) for _ in range(n)]
    nbp = sar.sar_ll_packet_bytes(count, dt)
    assert nbp > (1 << 32)
    pk = [torch.zeros(nbp, dtype=torch.uint8, device="cuda") for _ in range(n)]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sar.sar_allreduce_ll(din, dout, pk, 1, st, count=count, dtype=dt)
    assert sar.sar_read_device_status(st) == sar.SAR_OK
    idx = _indices(count, n, dt, np.random.default_rng(9))
    want = oracle.allreduce([p[idx % P] for p in pats], dt)[0]
    tidx = torch.from_numpy(idx).cuda()
    for j in range(n):
        assert np.array_equal(dout[j][tidx].cpu().numpy(), want)
    # the last packet of rank 1: payload = last element, flag = epoch 1
    last = pk[1][-8:].cpu().numpy()
    assert last[4:].tolist() == [1, 0, 0, 0]
    assert last[:4].view(np.float32)[0] == pats[1][(count - 1) % P]
    del din, dout, pk
    torch.cuda.empty_cache()


def test_cluster_ll_past_2_32_elements(sar):
    """sar_allreduce_ll_cluster with more than 2^32 elements per rank (2 ranks,
    e4m3fn): packet indices past 2^30, slices past 2^21 clusters."""
    n, dt, count = 2, "e4m3fn", (1 << 32) + 4099
    pats = W.rank_inputs("normal", 8, dt, P, n, 4.0)
    din = [_tiled(p, count, torch.uint8) for p in pats]
    dout = [torch.empty_like(din[0]) for _ in range(n)]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sar.sar_allreduce_ll_cluster(din, dout, st, count=count, dtype=dt)
    assert sar.sar_read_device_status(st) == sar.SAR_OK
    idx = _indices(count, n, dt, np.random.default_rng(5))
    want = oracle.allreduce([p[idx % P] for p in pats], dt)[0]
    tidx = torch.from_numpy(idx).cuda()
    for j in range(n):
        assert np.array_equal(dout[j][tidx].cpu().numpy(), want)
        assert torch.equal(dout[j], dout[0])
    del din, dout
    torch.cuda.empty_cache()


@pytest.mark.parametrize("n,count", [(2, (1 << 32) + 4099), (16, (1 << 31) + 4099)],
                         ids=["2_ranks_4_packets_per_thread", "16_ranks_1_packet_per_thread"])
def test_ll_allpair_past_2_31_bytes(sar, n, count):
    """sar_allreduce with SAR_ALGO_LL_ALLPAIR (e4m3fn) past 2^32 elements per
    rank with 2 ranks (slices of 4 packets per thread, slice offsets past
    2^30 packets) and past 2^31 bytes per rank with 16 ranks (slices of 1
    packet per thread)."""
    dt = "e4m3fn"
    pats = W.rank_inputs("normal", 10 + n, dt, P, n, 4.0)
    din = [_tiled(p, count, torch.uint8) for p in pats]
    dout = [torch.empty_like(din[0]) for _ in range(n)]
    sar.sar_allreduce(din, dout, count=count, dtype=dt, algo=sar.SAR_ALGO_LL_ALLPAIR)
    torch.cuda.synchronize()
    idx = _indices(count, n, dt, np.random.default_rng(n))
    want = oracle.allreduce([p[idx % P] for p in pats], dt)[0]
    tidx = torch.from_numpy(idx).cuda()
    for j in range(n):
        assert np.array_equal(dout[j][tidx].cpu().numpy(), want)
        assert torch.equal(dout[j], dout[0])
    del din, dout
    torch.cuda.empty_cache()
