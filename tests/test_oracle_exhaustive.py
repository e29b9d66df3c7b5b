"""Exhaustive pin of the oracle's binary32 -> element-type rounding: every one
of the 2^32 binary32 bit patterns, for bf16, fp16, e4m3fn and e4m3b15.

The reference here is integer arithmetic on the binary32 bit pattern, written
from the field definitions of each format (sign, exponent field with its
bias, fraction field; IEEE round to nearest, ties to even):

* A binary32 magnitude whose exponent is at least the target's smallest
  normal exponent is rounded on its bit pattern: adding (half a quantum - 1)
  plus the lowest kept bit and then dropping the low (24 - p) fraction bits is
  round-to-nearest-even, and a carry out of the fraction moves into the
  exponent field by itself.  Re-biasing the exponent field (127 -> the
  target's bias) gives the target code.
* A smaller magnitude is rounded the same way onto the target's subnormal
  grid (multiples of 2^(emin - p + 1)), from its significand and exponent.
* Results past the largest finite code are infinity (bf16, fp16, e4m3b15), or
  the largest finite value +-448 for e4m3fn, which saturates; binary32
  infinities map the same way.  NaN gives the canonical quiet NaN code.

This is a different algorithm from the oracle's (which builds the value as
significand x 2^exponent and rounds it to the target's grid with an explicit
remainder comparison), so a mistake in either shows up as a mismatch.

Marked slow: about 2^34 conversions on each side.  Run it with
``SAR_RUN_SLOW=1 python -m pytest tests/test_oracle_exhaustive.py``.
"""
from __future__ import annotations

import multiprocessing as mp
import os
import time

import numpy as np
import pytest

# name: (p = significand bits with the implicit one, exponent bias,
#        largest finite code magnitude, code for an overflow, NaN code)
FORMATS = {
    "bf16": (8, 127, 0x7F7F, 0x7F80, 0x7FC0),
    "fp16": (11, 15, 0x7BFF, 0x7C00, 0x7E00),
    "e4m3fn": (4, 7, 0x7E, 0x7E, 0x7F),
    "e4m3b15": (4, 15, 0x77, 0x78, 0x7F),
}
SIGN_BIT = {"bf16": 15, "fp16": 15, "e4m3fn": 7, "e4m3b15": 7}
CHUNK = 1 << 22


def _rne_shift(x: np.ndarray, s: np.ndarray) -> np.ndarray:
    """round(x / 2^s) to nearest, ties to even, for uint64 x and shifts s >= 1:
    add half - 1 and the lowest kept bit, then shift."""
    one = np.uint64(1)
    return (x + ((one << (s - one)) - one) + ((x >> s) & one)) >> s


def reference(u: np.ndarray, fmt: str) -> np.ndarray:
    """Target codes of the binary32 bit patterns u (uint64 array)."""
    p, bias, max_code, over_code, nan_code = FORMATS[fmt]
    u = u.astype(np.uint64)
    sign = (u >> np.uint64(31)) << np.uint64(SIGN_BIT[fmt])
    a = u & np.uint64(0x7FFFFFFF)
    E = a >> np.uint64(23)
    M = a & np.uint64(0x7FFFFF)
    emin = 1 - bias                                   # smallest normal exponent of the target
    shift = np.uint64(24 - p)                         # fraction bits dropped
    # normal target results: round on the bit pattern, then re-bias
    rebias = np.uint64((127 - bias) << (p - 1))
    normal_mag = _rne_shift(a, np.full(a.shape, shift, np.uint64))
    normal = E.astype(np.int64) - 127 >= emin
    normal_code = np.where(normal, normal_mag - np.where(normal, rebias, np.uint64(0)), np.uint64(0))
    # subnormal target results: significand * 2^exp2 onto the grid of 2^(emin - p + 1)
    sig = np.where(E == 0, M, M | np.uint64(1 << 23))
    exp2 = np.where(E == 0, -149, E.astype(np.int64) - 150)
    s = np.clip((emin - (p - 1)) - exp2, 1, 48).astype(np.uint64)
    sub_code = _rne_shift(sig, s)
    mag = np.where(normal, normal_code, sub_code)
    mag = np.where(mag > max_code, np.uint64(over_code), mag)
    mag = np.where(E == 255, np.uint64(over_code), mag)                # infinities
    code = sign | mag
    code = np.where((E == 255) & (M != 0), np.uint64(nan_code), code)  # NaN: canonical code
    return code


def _check_range(args):
    import oracle
    fmt, lo, hi = args
    bad = []
    for start in range(lo, hi, CHUNK):
        u = np.arange(start, min(hi, start + CHUNK), dtype=np.uint64)
        x = u.astype(np.uint32).view(np.float32)
        got = oracle.round_f32(x, fmt).astype(np.uint64)
        want = reference(u, fmt)
        diff = np.nonzero(got != want)[0]
        if diff.size:
            bad.extend((int(u[i]), int(got[i]), int(want[i])) for i in diff[:4])
            break
    return bad


def test_reference_on_known_values():
    """The reference itself on values fixed by the formats' definitions."""
    def f(x):
        return np.array([np.float32(x)]).view(np.uint32).astype(np.uint64)
    assert reference(f(1.0), "fp16")[0] == 0x3C00 and reference(f(65504.0), "fp16")[0] == 0x7BFF
    assert reference(f(65520.0), "fp16")[0] == 0x7C00                # the overflow midpoint rounds up
    assert reference(f(2.0 ** -24), "fp16")[0] == 0x0001 and reference(f(2.0 ** -25), "fp16")[0] == 0
    assert reference(f(3 * 2.0 ** -25), "fp16")[0] == 0x0002          # tie to even
    assert reference(f(1.0 + 2.0 ** -8), "bf16")[0] == 0x3F80         # tie to even (down)
    assert reference(f(1.0 + 3 * 2.0 ** -8), "bf16")[0] == 0x3F82     # tie to even (up)
    assert reference(f(-448.0), "e4m3fn")[0] == 0xFE and reference(f(1e30), "e4m3fn")[0] == 0x7E
    assert reference(f(2.0 ** -9), "e4m3fn")[0] == 0x01 and reference(f(1.0), "e4m3fn")[0] == 0x38
    assert reference(f(0.9375), "e4m3b15")[0] == 0x77 and reference(f(0.96875), "e4m3b15")[0] == 0x78
    assert reference(f(2.0 ** -17), "e4m3b15")[0] == 0x01 and reference(f(-0.0), "e4m3b15")[0] == 0x80
    assert reference(f(float("inf")), "bf16")[0] == 0x7F80 and reference(f(float("-inf")), "e4m3fn")[0] == 0xFE
    assert reference(np.array([0x7FC00001], np.uint64), "fp16")[0] == 0x7E00


def test_reference_matches_library_conversions_on_a_sample():
    """Where numpy and torch convert (binary16; bfloat16 and e4m3fn under
    torch's round-to-nearest-even), they agree with the reference on a
    random sample of bit patterns (non-NaN; torch's e4m3fn conversion does
    not saturate, so finite values beyond 464 are left out there)."""
    import torch
    rng = np.random.default_rng(31)
    u = rng.integers(0, 1 << 32, 1 << 20, dtype=np.uint64)
    x = u.astype(np.uint32).view(np.float32)
    keep = ~np.isnan(x)
    u, x = u[keep], x[keep]
    with np.errstate(over="ignore"):
        assert np.array_equal(x.astype(np.float16).view(np.uint16), reference(u, "fp16").astype(np.uint16))
    bf = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bf, reference(u, "bf16").astype(np.uint16))
    small = np.abs(x) < 464
    e4 = torch.from_numpy(x[small]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(e4, reference(u[small], "e4m3fn").astype(np.uint8))


@pytest.mark.slow
@pytest.mark.skipif(os.environ.get("SAR_RUN_SLOW") != "1", reason="set SAR_RUN_SLOW=1 (all 2^32 patterns)")
@pytest.mark.parametrize("fmt", list(FORMATS))
def test_oracle_rounding_on_every_binary32(fmt):
    workers = os.cpu_count() or 4
    parts = 4 * workers
    step = (1 << 32) // parts
    jobs = [(fmt, i * step, (i + 1) * step) for i in range(parts)]
    t = time.time()
    with mp.get_context("spawn").Pool(workers) as pool:
        bad = [b for r in pool.imap_unordered(_check_range, jobs) for b in r]
    assert not bad, f"{fmt}: oracle != reference at (bits, oracle, reference) {bad[:8]}"
    print(f"{fmt}: 2^32 patterns in {time.time() - t:.1f} s on {workers} processes")
