"""Pins for the oracle's accumulation-type variants (no GPU).

Semantics (mscclpp commit history, "Add mixed-precision accumulation for
allreduce": accumDtype, AUTO = the input type, FP8 reduced in float16 or
float32): every partial sum is rounded into the accumulator type,
    acc_0 = R_acc(x_0),  acc_k = R_acc(f32(acc_{k-1}) + f32(x_k)),  out = R_dt(acc).

Independent checks: a step-by-step reference built from exact float64 sums,
numpy's binary32 rounding and the brute-force nearest search of
tests/format_ref.py; the per-element optimality of binary32 accumulation for
e4m3fn inputs (their binary32 sums are exact, so no accumulator can land
closer to the exact sum); exact integer sums; and the page's invariant that
higher-precision accumulation is at least as accurate as native FP8.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from tests import format_ref as ref

STORE = {"bf16": np.uint16, "fp16": np.uint16, "fp32": np.float32, "e4m3fn": np.uint8}


def _vals(codes, dt):
    if dt == "fp32":
        return codes.astype(np.float64)
    return ref.all_values(dt)[codes.astype(np.int64)]


def _round_vals(x, dt):
    """Value of R_dt(x) for exact float64 x (independent rounding)."""
    if dt == "fp32":
        return x.astype(np.float32).astype(np.float64)
    return ref.all_values(dt)[ref.nearest_even(x, dt)]


def _stepwise(ins, dt, acc_dt):
    vals = [_vals(c, dt) for c in ins]
    acc = _round_vals(vals[0], acc_dt)
    for v in vals[1:]:
        s32 = (acc + v).astype(np.float32).astype(np.float64)    # binary32 add of exact operands
        acc = _round_vals(s32, acc_dt)
    if dt == "fp32":
        return acc.astype(np.float32)
    return ref.nearest_even(acc, dt).astype(STORE[dt])


CASES = [("e4m3fn", "e4m3fn"), ("e4m3fn", "fp16"), ("e4m3fn", "bf16"), ("bf16", "bf16"), ("bf16", "fp16"),
         ("fp16", "fp16"), ("fp32", "fp16"), ("fp16", "bf16")]


@pytest.mark.parametrize("dt,acc", CASES)
@pytest.mark.parametrize("n", [2, 3, 8, 32])
def test_stepwise_reference(dt, acc, n):
    rng = np.random.default_rng([n, len(dt), len(acc)])
    k = np.arange(4000, dtype=np.uint64) + np.uint64(rng.integers(0, 1 << 30))
    sigma = {"e4m3fn": 16.0, "bf16": 1.0, "fp16": 1.0, "fp32": 1.0}[dt]
    ins = [W.draw("normal", 9, k + np.uint64(r * 100000), dt, sigma) for r in range(n)]
    got = oracle.allreduce_accum(ins, dt, acc)
    want = _stepwise(ins, dt, acc)
    for y in got:
        assert np.array_equal(y.view(np.uint8), want.view(np.uint8))


@pytest.mark.parametrize("dt", ["bf16", "fp16", "fp32", "e4m3fn"])
def test_fp32_accumulation_is_the_plain_allreduce(dt):
    ins = W.rank_inputs("normal", 4, dt, 5000, 8, 4.0)
    a = oracle.allreduce_accum(ins, dt, "fp32")
    b = oracle.allreduce(ins, dt)
    assert np.array_equal(a[0].view(np.uint8), b[0].view(np.uint8))


def test_binary32_accumulation_is_optimal_for_e4m3fn():
    """Up to 32 e4m3fn values sum exactly in binary32, so fp32 accumulation
    returns the nearest e4m3fn value to the exact sum: every other
    accumulator is at best as close, element by element."""
    n = 8
    ins = W.rank_inputs("normal", 2, "e4m3fn", 20000, n, 4.0)
    exact = sum(_vals(c, "e4m3fn") for c in ins)
    err = {}
    for acc in ("fp32", "fp16", "bf16", "e4m3fn"):
        out = oracle.allreduce_accum(ins, "e4m3fn", acc)[0]
        err[acc] = np.abs(_vals(out, "e4m3fn") - exact)
    for acc in ("fp16", "bf16", "e4m3fn"):
        assert np.all(err["fp32"] <= err[acc])
    # the page's invariant: higher-precision accumulation at least as accurate as native FP8
    assert err["fp32"].mean() <= err["fp16"].mean() <= err["e4m3fn"].mean()
    assert err["e4m3fn"].mean() > err["fp32"].mean()       # native accumulation does lose accuracy


@pytest.mark.parametrize("dt,acc", [("e4m3fn", "fp16"), ("bf16", "fp16"), ("fp16", "fp16"), ("bf16", "bf16")])
def test_small_integer_sums_are_exact_in_any_wide_enough_accumulator(dt, acc):
    rng = np.random.default_rng(5)
    vals = rng.integers(-8, 9, size=(8, 3000)).astype(np.float64)
    ins = [ref.nearest_even(v, dt).astype(STORE[dt]) for v in vals]
    want = ref.nearest_even(vals.sum(axis=0), dt).astype(STORE[dt])
    got = oracle.allreduce_accum(ins, dt, acc)[0]
    assert np.array_equal(got, want)


def test_native_e4m3fn_rounds_every_partial_sum():
    """17 = 16 + 1 is not an e4m3fn value (the grid is 2 apart in [16, 32)):
    natively, 8 + 8 = 16, 16 + 1 -> 16 (tie to even), 16 + 1 -> 16, while
    fp32 accumulation gives R(18) = 18."""
    one, eight = np.array([0x38], np.uint8), np.array([0x50], np.uint8)
    ins = [eight, eight, one, one]
    assert ref.all_values("e4m3fn")[0x50] == 8.0
    native = oracle.allreduce_accum(ins, "e4m3fn", "e4m3fn")[0][0]
    wide = oracle.allreduce_accum(ins, "e4m3fn", "fp32")[0][0]
    assert ref.all_values("e4m3fn")[native] == 16.0
    assert ref.all_values("e4m3fn")[wide] == 18.0
