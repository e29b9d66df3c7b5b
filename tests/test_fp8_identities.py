"""Pins for the two identities the FP8 vector kernels rest on, checked on
the CPU with the oracle's conversions as the definition of each rounding.

1. e4m3fn accumulated in e4m3fn.  A step is R_fn(acc + x) with acc and x
   e4m3fn values (the binary32 add is exact: both are multiples of 2^-9
   below 2^9).  The kernel adds in binary16 first; for every pair of codes
   the e4m3fn rounding of the binary16 sum is the e4m3fn rounding of the
   exact sum.
2. e4m3b15 on the e4m3fn conversions.  A finite e4m3b15 code read as an
   e4m3fn code is 2^8 times its value, and rounding 2^8 s clamped to +-256
   (NaN kept) to e4m3fn gives the e4m3b15 code of s, with 0x78 (256 in
   e4m3fn) being e4m3b15 infinity."""
import numpy as np

import oracle

CODES = np.arange(256, dtype=np.uint8)


def _f32(codes, dt):
    return oracle.convert(np.asarray(codes, np.uint8), dt, "fp32")


def _same_codes(got, want, nan):
    got, want = np.asarray(got, np.uint8), np.asarray(want, np.uint8)
    return np.all((got == want) | (nan(got) & nan(want)))


def _fn_nan(c):
    return (c & 0x7F) == 0x7F


def _b15_nan(c):
    return ((c & 0x78) == 0x78) & ((c & 0x07) != 0)


def test_binary16_pair_sum_rounds_like_the_exact_sum_for_every_e4m3fn_pair():
    v = _f32(CODES, "e4m3fn")
    a, b = np.repeat(v, 256), np.tile(v, 256)
    exact = (a.astype(np.float64) + b.astype(np.float64)).astype(np.float32)
    assert np.array_equal(exact[~np.isnan(exact)].astype(np.float64),
                          (a.astype(np.float64) + b.astype(np.float64))[~np.isnan(exact)])
    h = (a.astype(np.float16) + b.astype(np.float16)).astype(np.float32)
    assert np.array_equal(a[~np.isnan(a)].astype(np.float16).astype(np.float32), a[~np.isnan(a)])
    want = oracle.convert(exact, "fp32", "e4m3fn")
    got = oracle.convert(h, "fp32", "e4m3fn")
    assert _same_codes(got, want, _fn_nan)
    # the binary16 sum really is inexact for some pairs: the identity is not vacuous
    fin = ~np.isnan(exact)
    assert np.count_nonzero(h[fin] != exact[fin]) > 1000


def test_finite_e4m3b15_code_read_as_e4m3fn_is_256_times_its_value():
    finite = CODES[(CODES & 0x78) != 0x78]
    assert finite.size == 240
    assert np.array_equal(_f32(finite, "e4m3fn"), np.float32(256) * _f32(finite, "e4m3b15"))
    # exponent field 15: e4m3fn reads 256 (e4m3b15 infinity) or more / NaN
    special = CODES[(CODES & 0x78) == 0x78]
    fn = np.abs(_f32(special, "e4m3fn"))
    assert np.all((fn >= 256) | np.isnan(fn))
    assert np.all((fn == 256) == ((special & 0x7F) == 0x78))


def _b15_via_fn(s):
    y = np.float32(256) * s.astype(np.float32)
    y = np.where(np.isnan(y), y, np.clip(y, -256, 256)).astype(np.float32)
    return oracle.convert(y, "fp32", "e4m3fn")


def test_scaled_e4m3fn_rounding_is_e4m3b15_rounding():
    grid = np.arange(-int(1.25 * 2 ** 17), int(1.25 * 2 ** 17) + 1, dtype=np.int64)
    s = (grid.astype(np.float64) * 2.0 ** -17).astype(np.float32)      # every kernel sum near the range
    halves = ((grid.astype(np.float64) + 0.5) * 2.0 ** -17).astype(np.float32)  # ties of the subnormal grid
    rng = np.random.default_rng(5)
    rand = (rng.standard_normal(200000) * np.exp2(rng.integers(-20, 8, 200000))).astype(np.float32)
    extra = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 0.9375, 0.96875, -0.96875, 0.968, 1.0, 30.0, -30.0,
                      2.0 ** -18, -(2.0 ** -18), 3 * 2.0 ** -18, 1e30, -1e30], np.float32)
    for x in (s, halves, rand, extra):
        want = oracle.convert(x, "fp32", "e4m3b15")
        got = _b15_via_fn(x)
        assert _same_codes(got, want, _b15_nan)
    assert _b15_via_fn(np.array([-0.0], np.float32))[0] == 0x80
