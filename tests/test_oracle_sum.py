"""Pins for the oracle's allreduce, rsag steps, LL packets and conversion (no GPU).

Every expected value here comes from mathematics the oracle does not share:
exact sums (float64 or Fraction) rounded once by the brute-force nearest
search of tests/format_ref.py, closed forms (nranks == 1 identity, N*x,
the packet byte image), invariants (permutation invariance of exact sums,
chunks partition the index range) and a hand-built binary32 case whose value
depends on the summation order.
"""
import itertools
from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests import format_ref as ref

DTYPES = ["bf16", "fp16", "fp32", "e4m3fn"]
STORE = {"bf16": np.uint16, "fp16": np.uint16, "fp32": np.float32, "e4m3fn": np.uint8, "e4m3b15": np.uint8}


def _codes_from_values(vals: np.ndarray, dt: str) -> np.ndarray:
    """Codes of values that are exactly representable in dt."""
    if dt == "fp32":
        return vals.astype(np.float32)
    codes = ref.nearest_even(vals.astype(np.float64), dt).astype(STORE[dt])
    assert np.array_equal(oracle.decode(codes, dt).astype(np.float64), vals.astype(np.float64))
    return codes


def _expected(exact_sums: np.ndarray, dt: str) -> np.ndarray:
    if dt == "fp32":
        return exact_sums.astype(np.float32)      # caller ensures exactness
    return ref.nearest_even(exact_sums, dt).astype(STORE[dt])


def _same_bits(a, b):
    return np.array_equal(np.asarray(a).view(np.uint8), np.asarray(b).view(np.uint8))


def _random_codes(rng, dt, n):
    """Random non-NaN codes of dt (including zeros, subnormals, extremes)."""
    if dt == "fp32":
        bits = rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
        x = bits.view(np.float32)
        return np.where(np.isnan(x), np.float32(1.5), x).astype(np.float32)
    c = rng.integers(0, ref.n_codes(dt), n).astype(STORE[dt])
    vals = ref.all_values(dt)[c.astype(np.int64)]
    return np.where(np.isnan(vals), STORE[dt](0), c).astype(STORE[dt])


# ---------------------------------------------------------------- allreduce

@pytest.mark.parametrize("dt", DTYPES)
def test_one_rank_is_identity(dt):
    rng = np.random.default_rng(1)
    x = _random_codes(rng, dt, 20000)
    x[:4] = np.array([0, 0, 0, 0]).astype(STORE[dt])
    neg0 = {"bf16": 0x8000, "fp16": 0x8000, "e4m3fn": 0x80}
    if dt == "fp32":
        x[1] = np.float32(-0.0)
    else:
        x[1] = neg0[dt]
    (y,) = oracle.allreduce([x], dt)
    assert _same_bits(x, y)


@pytest.mark.parametrize("dt", DTYPES + ["e4m3b15"])
def test_reduce_scatter_of_negative_zeros_is_negative_zero(dt):
    """The in-order binary32 sum of -0 values is -0 (round to nearest: -0 + -0
    = -0), so every chunk the reduce-scatter writes holds -0 codes, as the
    allreduce's do (the seed is the first rank's value, not +0)."""
    n, count = 4, 37
    neg0 = {"bf16": 0x8000, "fp16": 0x8000, "fp32": np.float32(-0.0), "e4m3fn": 0x80, "e4m3b15": 0x80}[dt]
    ins = [np.full(count, neg0, dtype=STORE[dt]) for _ in range(n)]
    outs = [np.zeros(count, dtype=STORE[dt]) for _ in range(n)]
    oracle.reduce_scatter(ins, outs, dt)
    for r in range(n):
        b, e = oracle.rsag_chunk(count, n, dt, r)
        assert _same_bits(outs[r][b:e], ins[0][b:e]), r
    assert _same_bits(oracle.allreduce(ins, dt)[0], ins[0])


@pytest.mark.parametrize("dt", DTYPES + ["e4m3b15"])
@pytest.mark.parametrize("n", [2, 3, 4, 8, 16, 32])
def test_all_equal_inputs_give_n_times_x(dt, n):
    rng = np.random.default_rng(n)
    if dt == "fp32":
        # <= 19 significant bits keeps every partial sum k*x exact
        m = rng.integers(-(1 << 18), 1 << 18, 5000).astype(np.float64)
        x_vals = m * np.exp2(rng.integers(-140, 100, 5000).astype(np.float64))
        x_vals = x_vals.astype(np.float32).astype(np.float64)
        x = x_vals.astype(np.float32)
    else:
        x = _random_codes(rng, dt, 5000)
        x_vals = ref.all_values(dt)[x.astype(np.int64)]
        fin = np.isfinite(x_vals)
        x, x_vals = x[fin], x_vals[fin]
    outs = oracle.allreduce([x] * n, dt)
    want = _expected(n * x_vals, dt)
    for y in outs:
        assert _same_bits(y, want)


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("n", [2, 5, 8, 32])
def test_small_integers_sum_exactly_under_any_rank_order(dt, n):
    rng = np.random.default_rng(100 + n)
    vals = rng.integers(-8, 9, size=(n, 3000)).astype(np.float64)
    ins = [_codes_from_values(v, dt) for v in vals]
    want = _expected(vals.sum(axis=0), dt)
    outs = oracle.allreduce(ins, dt)
    for y in outs:
        assert _same_bits(y, want)
    perm = rng.permutation(n)
    outs_p = oracle.allreduce([ins[p] for p in perm], dt)
    assert _same_bits(outs_p[0], outs[0])


@pytest.mark.parametrize("n", [2, 5, 8, 32])
def test_e4m3b15_small_multiples_sum_exactly(n):
    """Multiples of 2^-9 up to 15 * 2^-9 are e4m3b15 values; their sums are
    exact in binary32, so the result is R_e4m3b15(exact sum), under any rank
    order."""
    rng = np.random.default_rng(40 + n)
    vals = rng.integers(-15, 16, size=(n, 3000)).astype(np.float64) * 2.0 ** -9
    ins = [_codes_from_values(v, "e4m3b15") for v in vals]
    want = _expected(vals.sum(axis=0), "e4m3b15")
    outs = oracle.allreduce(ins, "e4m3b15")
    assert _same_bits(outs[0], want) and _same_bits(outs[-1], want)
    perm = rng.permutation(n)
    assert _same_bits(oracle.allreduce([ins[p] for p in perm], "e4m3b15")[0], want)


def test_all_e4m3b15_pairs_bruteforce():
    vals = ref.all_values("e4m3b15")
    good = np.nonzero(np.isfinite(vals))[0]
    a, b = np.meshgrid(good, good, indexing="ij")
    a, b = a.ravel().astype(np.uint8), b.ravel().astype(np.uint8)
    exact = vals[a.astype(np.int64)] + vals[b.astype(np.int64)]
    want = ref.nearest_even(exact, "e4m3b15").astype(np.uint8)
    y0, _ = oracle.allreduce([a, b], "e4m3b15")
    assert np.array_equal(y0, want)


def test_all_e4m3fn_pairs_bruteforce():
    """All 256 x 256 code pairs, two ranks: two e4m3fn values always add
    exactly in binary32, so the result is the exact sum rounded once."""
    vals = ref.all_values("e4m3fn")
    good = np.nonzero(~np.isnan(vals))[0]
    a, b = np.meshgrid(good, good, indexing="ij")
    a, b = a.ravel().astype(np.uint8), b.ravel().astype(np.uint8)
    exact = vals[a.astype(np.int64)] + vals[b.astype(np.int64)]
    want = ref.nearest_even(exact, "e4m3fn").astype(np.uint8)
    y0, y1 = oracle.allreduce([a, b], "e4m3fn")
    assert np.array_equal(y0, want) and np.array_equal(y1, want)


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
@pytest.mark.parametrize("n", [2, 4, 8, 32])
def test_grid_values_round_once(dt, n):
    """Values on the 2^-14 grid with |x| < 2: every partial sum of up to 32 of
    them is exact in binary32, so the result is R_dt(exact sum), which
    exercises rounding of sums that are not representable in dt."""
    rng = np.random.default_rng(7 * n)
    raw = rng.integers(-(1 << 15) + 1, 1 << 15, size=(n, 4000)).astype(np.float64) * 2.0 ** -14
    ins = [ref.nearest_even(v, dt).astype(np.uint16) for v in raw]   # quantise inputs to dt
    vals = np.stack([ref.all_values(dt)[c.astype(np.int64)] for c in ins])
    assert np.all(np.abs(vals) <= 2) and np.all(vals * 2 ** 14 == np.round(vals * 2 ** 14))
    want = _expected(vals.sum(axis=0), dt)
    outs = oracle.allreduce(ins, dt)
    assert _same_bits(outs[0], want) and _same_bits(outs[-1], want)


def test_rank_order_is_0_to_n_minus_1():
    """In binary32, (((2^24 + 1) - 2^24) + 1) = 1 while the exact sum is 2 and
    the reversed order gives 2: the result fixes the order 0..N-1."""
    x = [np.array([v], np.float32) for v in (2.0 ** 24, 1.0, -(2.0 ** 24), 1.0)]
    assert oracle.allreduce(x, "fp32")[0][0] == 1.0
    assert oracle.allreduce(x[::-1], "fp32")[0][0] == 2.0
    xb = [oracle.round_f32(v, "bf16") for v in x]
    assert oracle.allreduce(xb, "bf16")[0][0] == 0x3F80       # bf16 1.0


def test_binary32_add_is_exact_rne_with_subnormals():
    tiny = float(np.float32(2.0 ** -149))
    assert oracle.add_f32(tiny, tiny) == 2.0 ** -148           # no flush to zero
    assert oracle.add_f32(2.0 ** -126, -(2.0 ** -126 - 2.0 ** -149)) == 2.0 ** -149
    # ties to even at the binary32 rounding point
    assert oracle.add_f32(1.0, 2.0 ** -24) == 1.0
    assert oracle.add_f32(1.0 + 2.0 ** -23, 2.0 ** -24) == 1.0 + 2.0 ** -22
    rng = np.random.default_rng(3)
    a = rng.standard_normal(2000).astype(np.float32)
    b = (rng.standard_normal(2000) * np.exp2(rng.integers(-30, 30, 2000))).astype(np.float32)
    for x, y in zip(a[:300], b[:300]):
        s = Fraction(float(x)) + Fraction(float(y))
        got = oracle.add_f32(float(x), float(y))
        # correctly rounded: no binary32 lies strictly closer to the exact sum
        lo = np.nextafter(np.float32(got), np.float32(-np.inf))
        hi = np.nextafter(np.float32(got), np.float32(np.inf))
        d = abs(Fraction(got) - s)
        assert d <= abs(Fraction(float(lo)) - s) and d <= abs(Fraction(float(hi)) - s)


def test_overflow_and_saturation_of_sums():
    bmax = np.array([0x7F7F], np.uint16)                    # bf16 max
    assert oracle.allreduce([bmax, bmax], "bf16")[0][0] == 0x7F80      # -> inf
    hmax = np.array([0x7BFF], np.uint16)                    # 65504
    assert oracle.allreduce([hmax, hmax], "fp16")[0][0] == 0x7C00
    emax = np.array([0x7E], np.uint8)                       # 448
    assert oracle.allreduce([emax] * 32, "e4m3fn")[0][0] == 0x7E       # saturates
    eneg = np.array([0xFE], np.uint8)
    assert oracle.allreduce([eneg, eneg], "e4m3fn")[0][0] == 0xFE


def test_nan_propagates_as_nan():
    for dt, nan_code in (("bf16", 0x7FC1), ("fp16", 0x7E01), ("e4m3fn", 0x7F)):
        x = np.array([nan_code], STORE[dt])
        one = _codes_from_values(np.array([1.0]), dt)
        y = oracle.allreduce([one, x], dt)[0]
        assert np.isnan(oracle.decode(y, dt)[0])
    y = oracle.allreduce([np.array([np.inf], np.float32), np.array([-np.inf], np.float32)], "fp32")
    assert np.isnan(y[0][0])


# ------------------------------------------------------------ rsag chunking

@pytest.mark.parametrize("dt", DTYPES)
def test_rsag_chunks_partition_the_range(dt):
    vec = 16 // oracle.ESIZE[oracle.DTYPES[dt]]
    for count, n in itertools.product([0, 1, 7, 8, 9, 15, 16, 17, 100, 4097, 65536, 1000003],
                                      [1, 2, 4, 8, 16, 32]):
        chunks = [oracle.rsag_chunk(count, n, dt, r) for r in range(n)]
        c = -(-count // n)
        c = -(-c // vec) * vec
        pos = 0
        for r, (b, e) in enumerate(chunks):
            assert b == min(count, r * c) and e == min(count, (r + 1) * c)
            assert b == pos and b <= e
            assert b % vec == 0 or b == count    # empty trailing chunks clamp to count
            pos = e
        assert pos == count


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("n,count", [(2, 33), (4, 1000), (8, 4097), (3, 50)])
def test_reduce_scatter_then_all_gather_is_allreduce(dt, n, count):
    rng = np.random.default_rng(count)
    vals = rng.integers(-8, 9, size=(n, count)).astype(np.float64)
    ins = [_codes_from_values(v, dt) for v in vals]
    want = _expected(vals.sum(axis=0), dt)
    canary = {"bf16": 0xABCD, "fp16": 0xABCD, "fp32": np.float32(-3.25), "e4m3fn": 0xAB}[dt]
    outs = [np.full(count, canary, dtype=STORE[dt]) for _ in range(n)]
    oracle.reduce_scatter(ins, outs, dt)
    for r in range(n):
        b, e = oracle.rsag_chunk(count, n, dt, r)
        assert _same_bits(outs[r][b:e], want[b:e])
        rest = np.concatenate([outs[r][:b], outs[r][e:]])
        assert _same_bits(rest, np.full(rest.size, canary, dtype=STORE[dt]))
    oracle.all_gather(outs, dt)
    for y in outs:
        assert _same_bits(y, want)


# ------------------------------------------------------------------ LL path

def _packet_image(x: np.ndarray, epoch: int) -> np.ndarray:
    """Closed form: payload words (input bytes, zero-padded to 4) interleaved
    with the little-endian epoch."""
    raw = np.frombuffer(x.tobytes(), dtype=np.uint8)
    pad = (-raw.size) % 4
    raw = np.concatenate([raw, np.zeros(pad, np.uint8)]).reshape(-1, 4)
    flag = np.frombuffer(np.array([epoch], "<u4").tobytes(), np.uint8)
    return np.concatenate([raw, np.broadcast_to(flag, raw.shape)], axis=1).ravel()


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("count", [1, 2, 3, 5, 64, 1001])
def test_ll_pack_byte_image(dt, count):
    rng = np.random.default_rng(count)
    ins = [_random_codes(rng, dt, count) for _ in range(4)]
    for epoch in (1, 0x12345678, 0xFFFFFFFF):
        pk = oracle.ll_pack(ins, dt, epoch)
        assert oracle.ll_packets(count, dt) == -(-count * oracle.ESIZE[oracle.DTYPES[dt]] // 4)
        for r in range(4):
            assert np.array_equal(pk[r], _packet_image(ins[r], epoch))


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("n,count", [(1, 9), (2, 7), (8, 257), (32, 33)])
def test_ll_unpack_reduce_gives_the_exact_sums(dt, n, count):
    rng = np.random.default_rng(n * count)
    vals = rng.integers(-8, 9, size=(n, count)).astype(np.float64)
    ins = [_codes_from_values(v, dt) for v in vals]
    want = _expected(vals.sum(axis=0), dt)
    pk = oracle.ll_pack(ins, dt, 77)
    rc, outs = oracle.ll_unpack_reduce(pk, count, dt, 77)
    assert rc == oracle.OK
    for y in outs:
        assert _same_bits(y, want)


def test_ll_stale_flag_is_not_arrived():
    x = [np.arange(10, dtype=np.float32) for _ in range(2)]
    pk = oracle.ll_pack(x, "fp32", 5)
    rc, _ = oracle.ll_unpack_reduce(pk, 10, "fp32", 6)        # wrong epoch
    assert rc == oracle.NOT_ARRIVED
    pk[1][8 * 7 + 4] ^= 1                                     # one stale packet
    rc, _ = oracle.ll_unpack_reduce(pk, 10, "fp32", 5)
    assert rc == oracle.NOT_ARRIVED
    with pytest.raises(ValueError):
        oracle.ll_pack(x, "fp32", 0)                          # epoch 0 is reserved


# --------------------------------------------------------------- conversion

def test_convert_e4m3fn_to_f32_every_code():
    c = np.arange(256, dtype=np.uint8)
    y = oracle.convert(c, "e4m3fn", "fp32").astype(np.float64)
    want = ref.all_values("e4m3fn")
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(y), nan) and np.array_equal(y[~nan], want[~nan])


@pytest.mark.parametrize("src", ["fp32", "bf16", "fp16"])
def test_convert_to_e4m3fn_rounds_once(src):
    rng = np.random.default_rng(11)
    x = _random_codes(rng, src, 50000)
    xv = oracle.decode(x, src).astype(np.float64) if src != "fp32" else x.astype(np.float64)
    ok = ~np.isnan(xv)
    y = oracle.convert(x[ok], src, "e4m3fn")
    assert np.array_equal(y.astype(np.int64), ref.nearest_even(xv[ok], "e4m3fn"))


@pytest.mark.parametrize("dst", ["bf16", "fp16", "fp32"])
def test_convert_from_e4m3fn_is_exact(dst):
    c = np.arange(256, dtype=np.uint8)
    vals = ref.all_values("e4m3fn")
    ok = ~np.isnan(vals)
    y = oracle.convert(c[ok], "e4m3fn", dst)
    back = y.astype(np.float64) if dst == "fp32" else ref.all_values(dst)[y.astype(np.int64)]
    assert np.array_equal(back, vals[ok])
