"""Pins for the oracle's number formats (no GPU).

The oracle's decode and round-to-nearest-even functions are checked against
(a) brute-force nearest search over each format's code table enumerated from
the field definitions (tests/format_ref.py), (b) library conversions (numpy
binary16, torch bfloat16 and float8_e4m3fn), and (c) named constants of the
format specifications (tests/golden/format_constants.txt).  None of these
shares code with the oracle.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from tests import format_ref as ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "format_constants.txt")


def _f32_points() -> np.ndarray:
    """Binary32 bit patterns aimed at every rounding decision of the three
    target formats: all upper halves with tie-class low halves, the exact
    midpoints of every target grid and their binary32 neighbours, per-exponent
    tie patterns at every drop position, and random patterns."""
    rng = np.random.default_rng(20261202)
    pts = []
    up = np.arange(1 << 16, dtype=np.uint32) << np.uint32(16)
    for low in (0x0000, 0x0001, 0x0FFF, 0x1000, 0x1001, 0x7FFF, 0x8000, 0x8001, 0xFFFF):
        pts.append(up | np.uint32(low))
    for fmt in ("bf16", "fp16", "e4m3fn", "e4m3b15"):
        vals, _ = ref.positive_table(fmt)
        mids = (vals[:-1] + vals[1:]) / 2
        over = vals[-1] + (vals[-1] - vals[-2]) / 2
        m32 = np.concatenate([mids, [over, vals[-1]]]).astype(np.float32)
        assert np.array_equal(m32.astype(np.float64), np.concatenate([mids, [over, vals[-1]]]))
        for v in (m32, np.nextafter(m32, np.float32(np.inf)), np.nextafter(m32, np.float32(0))):
            b = v.view(np.uint32)
            pts += [b, b | np.uint32(0x80000000)]
    exps = np.arange(255, dtype=np.uint32)
    for d in range(1, 24):
        tie = np.uint32(1 << (d - 1))
        for low in (tie, tie - np.uint32(1), tie + np.uint32(1), np.uint32((1 << d) - 1)):
            upper = rng.integers(0, 1 << (23 - d + 1), size=(255, 2), dtype=np.uint64).astype(np.uint32)
            m = ((upper << np.uint32(d)) | low) & np.uint32(0x7FFFFF)
            pts.append(((exps[:, None] << np.uint32(23)) | m).ravel())
    pts.append(rng.integers(0, 1 << 32, size=1 << 21, dtype=np.uint64).astype(np.uint32))
    bits = np.concatenate(pts).astype(np.uint32)
    e = (bits >> np.uint32(23)) & np.uint32(0xFF)
    frac = bits & np.uint32(0x7FFFFF)
    bits = bits[~((e == 0xFF) & (frac != 0))]        # NaN handled separately
    return np.unique(bits).view(np.float32)


@pytest.fixture(scope="module")
def points():
    return _f32_points()


@pytest.mark.parametrize("fmt", ["bf16", "fp16", "e4m3fn", "e4m3b15"])
def test_round_matches_bruteforce_nearest(points, fmt):
    got = oracle.round_f32(points, fmt).astype(np.int64)
    want = ref.nearest_even(points.astype(np.float64), fmt)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, (f"{bad.size} mismatches, e.g. x={points[bad[:5]]} "
                           f"got={got[bad[:5]]} want={want[bad[:5]]}")


def test_round_fp16_matches_numpy(points):
    got = oracle.round_f32(points, "fp16")
    with np.errstate(over="ignore"):      # the points include values that round to +-inf
        want = points.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)


def test_round_bf16_matches_torch(points):
    got = oracle.round_f32(points, "bf16")
    want = torch.from_numpy(points).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_round_e4m3fn_matches_torch_in_range(points):
    # torch's float8_e4m3fn conversion does not saturate; after clamping to
    # +-448 the saturating and non-saturating conversions coincide.
    got = oracle.round_f32(points, "e4m3fn")
    clamped = torch.from_numpy(points).clamp(-448.0, 448.0)
    want = clamped.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, want)


@pytest.mark.parametrize("fmt", ["bf16", "fp16", "e4m3fn", "e4m3b15"])
def test_decode_every_code(fmt):
    n = ref.n_codes(fmt)
    codes = np.arange(n).astype(oracle.NP_STORAGE[oracle.DTYPES[fmt]])
    got = oracle.decode(codes, fmt).astype(np.float64)
    want = ref.all_values(fmt)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    # the sign field decides the sign of every non-NaN value, zeros included
    sign_field = codes.astype(np.int64) >= n // 2
    assert np.array_equal(np.signbit(got[~nan]), sign_field[~nan])


def test_decode_matches_libraries():
    h = np.arange(1 << 16, dtype=np.uint16)
    lib16 = h.view(np.float16).astype(np.float32)
    o16 = oracle.decode(h, "fp16")
    ok = ~np.isnan(lib16)
    assert np.array_equal(np.isnan(o16), ~ok) and np.array_equal(o16[ok], lib16[ok])
    libb = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).float().numpy()
    ob = oracle.decode(h, "bf16")
    ok = ~np.isnan(libb)
    assert np.array_equal(np.isnan(ob), ~ok) and np.array_equal(ob[ok], libb[ok])
    c = np.arange(256, dtype=np.uint8)
    lib8 = torch.from_numpy(c).view(torch.float8_e4m3fn).float().numpy()
    o8 = oracle.decode(c, "e4m3fn")
    ok = ~np.isnan(lib8)
    assert np.array_equal(np.isnan(o8), ~ok) and np.array_equal(o8[ok], lib8[ok])


@pytest.mark.parametrize("fmt,canon", [("bf16", 0x7FC0), ("fp16", 0x7E00), ("e4m3fn", 0x7F), ("e4m3b15", 0x7F)])
def test_round_trip_every_code(fmt, canon):
    """decode then encode is the identity on every code except NaN, which
    becomes the canonical NaN."""
    n = ref.n_codes(fmt)
    codes = np.arange(n).astype(oracle.NP_STORAGE[oracle.DTYPES[fmt]])
    back = oracle.round_f32(oracle.decode(codes, fmt), fmt).astype(np.int64)
    vals = ref.all_values(fmt)
    nan = np.isnan(vals)
    assert np.array_equal(back[~nan], codes[~nan].astype(np.int64))
    assert np.all(back[nan] == canon)


def test_nan_and_infinity_rules():
    specials = np.array([np.nan, -np.nan, np.inf, -np.inf], dtype=np.float32)
    assert list(oracle.round_f32(specials, "bf16")) == [0x7FC0, 0x7FC0, 0x7F80, 0xFF80]
    assert list(oracle.round_f32(specials, "fp16")) == [0x7E00, 0x7E00, 0x7C00, 0xFC00]
    # e4m3fn has no infinity: satfinite sends +-inf to +-448.
    assert list(oracle.round_f32(specials, "e4m3fn")) == [0x7F, 0x7F, 0x7E, 0xFE]
    # e4m3b15 keeps infinities (S.1111.000); overflow past 0.96875 rounds to them
    assert list(oracle.round_f32(specials, "e4m3b15")) == [0x7F, 0x7F, 0x78, 0xF8]
    big = np.array([0.96875, 0.968, 1.0, -5.0], dtype=np.float32)
    assert list(oracle.round_f32(big, "e4m3b15")) == [0x78, 0x77, 0x78, 0xF8]


def test_subnormals_survive():
    # Smallest subnormals of each format map to code 1 (and their halves
    # round to zero by ties-to-even); binary32 subnormals reach bf16 subnormals.
    xs = np.array([2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -135], dtype=np.float32)
    assert list(oracle.round_f32(xs, "bf16")) == [1, 0, 1]
    xs = np.array([2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26], dtype=np.float32)
    assert list(oracle.round_f32(xs, "fp16")) == [1, 0, 1]
    xs = np.array([2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -11], dtype=np.float32)
    assert list(oracle.round_f32(xs, "e4m3fn")) == [1, 0, 1]
    xs = np.array([2.0 ** -17, 2.0 ** -18, 3 * 2.0 ** -19], dtype=np.float32)
    assert list(oracle.round_f32(xs, "e4m3b15")) == [1, 0, 1]


def test_e4m3b15_is_the_top_of_a_binary16():
    """The page converts e4m3b15 through fp16: with the same bias (15), every
    finite code is the binary16 whose bits are the code's sign, exponent and
    fraction shifted into place (checked against numpy's binary16)."""
    c = np.arange(256, dtype=np.uint16)
    finite = ((c >> 3) & 0xF) != 0xF
    half_bits = ((c & 0x80) << 8) | ((c & 0x7F) << 7)
    lib = half_bits.astype(np.uint16).view(np.float16).astype(np.float32)
    got = oracle.decode(c.astype(np.uint8), "e4m3b15")
    assert np.array_equal(got[finite], lib[finite])
    assert finite.sum() == 240 and float(np.max(got[finite])) == 0.9375


def _golden():
    rows = []
    with open(GOLDEN) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if line:
                fmt, code, value = line.split()
                rows.append((fmt, int(code, 16), float.fromhex(value)))
    return rows


def test_golden_format_constants():
    rows = _golden()
    assert len(rows) >= 12
    for fmt, code, value in rows:
        codes = np.array([code], dtype=oracle.NP_STORAGE[oracle.DTYPES[fmt]])
        assert float(oracle.decode(codes, fmt)[0]) == value, (fmt, hex(code))
        assert int(oracle.round_f32(np.array([value], np.float32), fmt)[0]) == code, (fmt, value)


@pytest.mark.parametrize("fmt", ["e4m3fn", "e4m3b15"])
def test_fp8_nan_is_the_positive_all_ones_code(fmt):
    """Reading of the pages' silence on NaN signs: narrowing any binary32 NaN
    (either sign, any payload) to an fp8 format gives the one code S=0,
    E=1111, M=111 (0x7F), which is NaN in both formats."""
    nans = np.array([0x7FC00000, 0xFFC00000, 0x7F800001, 0xFFFFFFFF], dtype=np.uint32).view(np.float32)
    got = oracle.round_f32(nans, fmt)
    assert np.all(got.astype(np.int64) == 0x7F), [hex(int(c)) for c in got]
    assert np.isnan(oracle.decode(np.array([0x7F], dtype=np.uint8), fmt)[0])
