"""Independent reference for the number formats, used only to pin the oracle.

Each format's code table is enumerated from its field definition with Python
integers and Fractions, and rounding is done by brute-force nearest search
over that table (ties to the even code), with no bit tricks and no shared
code with the oracle.  All values and all distances below are exact in
binary64: every table value and every binary32 input is a binary64 number,
and a binary32 input differs from its two neighbours in any of these formats
by at most 24 significant bits.

Formats:
  bfloat16 (1/8/7, bias 127), IEEE binary16 (1/5/10, bias 15): IEEE 754
  semantics, overflow rounds to infinity.
  e4m3fn (OCP 8-bit floating point, E4M3): 1/4/3, bias 7, no infinities,
  S.1111.111 is NaN, max finite 448; conversion saturates to +-448.
  e4m3b15: 1/4/3, bias 15, max finite 0.9375 (the page's definition), so the
  all-ones exponent is infinity / NaN and overflow rounds to infinity.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

FORMATS = {
    # name: (exponent bits, fraction bits, bias, has_inf)
    "bf16": (8, 7, 127, True),
    "fp16": (5, 10, 15, True),
    "e4m3fn": (4, 3, 7, False),
    # bias 15, max finite 0.9375: the all-ones exponent is infinity / NaN
    "e4m3b15": (4, 3, 15, True),
}


def code_value(fmt: str, code: int):
    """Exact value of a code as a Fraction, or 'inf'/'-inf'/'nan'."""
    eb, fb, bias, has_inf = FORMATS[fmt]
    sign = -1 if (code >> (eb + fb)) & 1 else 1
    e = (code >> fb) & ((1 << eb) - 1)
    f = code & ((1 << fb) - 1)
    all_ones = (1 << eb) - 1
    if has_inf and e == all_ones:
        if f == 0:
            return "inf" if sign > 0 else "-inf"
        return "nan"
    if not has_inf and e == all_ones and f == (1 << fb) - 1:
        return "nan"
    if e == 0:
        mag = Fraction(f, 1 << fb) * Fraction(2) ** (1 - bias)
    else:
        mag = (1 + Fraction(f, 1 << fb)) * Fraction(2) ** (e - bias)
    return sign * mag


def n_codes(fmt: str) -> int:
    eb, fb, _, _ = FORMATS[fmt]
    return 1 << (1 + eb + fb)


def positive_table(fmt: str):
    """(values as float64 ascending, codes) of every finite code with sign 0."""
    half = n_codes(fmt) // 2
    vals, codes = [], []
    for c in range(half):
        v = code_value(fmt, c)
        if isinstance(v, Fraction):
            vals.append(float(v))     # exact: a short binary fraction
            codes.append(c)
    order = np.argsort(vals, kind="stable")
    return np.asarray(vals, dtype=np.float64)[order], np.asarray(codes, dtype=np.int64)[order]


_TABLES = {}


def _table(fmt):
    if fmt not in _TABLES:
        _TABLES[fmt] = positive_table(fmt)
    return _TABLES[fmt]


def inf_code(fmt: str) -> int:
    eb, fb, _, _ = FORMATS[fmt]
    return ((1 << eb) - 1) << fb


def sign_bit(fmt: str) -> int:
    eb, fb, _, _ = FORMATS[fmt]
    return 1 << (eb + fb)


def nearest_even(x: np.ndarray, fmt: str) -> np.ndarray:
    """Round finite or infinite float64 values (each a binary32 number or an
    exact sum) to codes of ``fmt`` by brute-force nearest search, ties to the
    even code.  Overflow: infinity (bf16, fp16) or saturation to 448 (e4m3fn).
    NaN inputs are not allowed here."""
    x = np.asarray(x, dtype=np.float64)
    assert not np.isnan(x).any()
    vals, codes = _table(fmt)
    _, _, _, has_inf = FORMATS[fmt]
    ax = np.abs(x)
    vmax = vals[-1]
    i = np.searchsorted(vals, ax, side="left")
    i_hi = np.minimum(i, len(vals) - 1)
    i_lo = np.maximum(i - 1, 0)
    lo, hi = vals[i_lo], vals[i_hi]
    d_lo, d_hi = ax - lo, hi - ax
    c_lo, c_hi = codes[i_lo], codes[i_hi]
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (c_hi % 2 == 0))
    take_hi |= (i == 0)
    res = np.where(take_hi, c_hi, c_lo)
    above = ax > vmax
    if has_inf:
        # Past the largest finite value the next grid point is 2^(emax+1),
        # whose (virtual) code is even, so the midpoint already rounds up.
        ulp_max = vals[-1] - vals[-2]
        res = np.where(above & (ax >= vmax + ulp_max / 2), inf_code(fmt), np.where(above, codes[-1], res))
    else:
        res = np.where(above, codes[-1], res)
    res = np.where(np.signbit(x), res | sign_bit(fmt), res)
    return res.astype(np.int64)


def decode_ref(codes, fmt: str) -> np.ndarray:
    """float64 value of each code (NaN for NaN codes)."""
    out = np.empty(len(codes), dtype=np.float64)
    for j, c in enumerate(codes):
        v = code_value(fmt, int(c))
        if isinstance(v, str):
            out[j] = {"inf": np.inf, "-inf": -np.inf, "nan": np.nan}[v]
        else:
            # Fractions have no signed zero: take the sign from the sign field
            out[j] = np.copysign(float(abs(v)), -1.0 if int(c) & sign_bit(fmt) else 1.0)
    return out


_ALL = {}


def all_values(fmt: str) -> np.ndarray:
    """float64 value of every code, indexed by code (read-only, cached)."""
    if fmt not in _ALL:
        v = decode_ref(range(n_codes(fmt)), fmt)
        v.setflags(write=False)
        _ALL[fmt] = v
    return _ALL[fmt]
