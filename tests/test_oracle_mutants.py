"""The oracle's pins have teeth: plausible mistakes planted in a copy of the
oracle source (a wrong tie rule, a dropped rank, a reversed rank order, a
lost sign, an off-by-one bias or scale, a missing saturation, a wrong packet
layout or count, an unrounded chunk size, a zero seed in the allreduce or the
reduce-scatter, infinity decoded as NaN, a NaN code that keeps its sign, a
conversion that rounds twice or decodes with the wrong type, an unpack that
ignores the epoch or reads the wrong half of a packet) must each fail at
least one pin.

Mistakes are planted only in a temporary copy of the C oracle, on the CPU.
"""
import os

import pytest

import oracle
from tests import test_oracle_accum as ta
from tests import test_oracle_formats as tf
from tests import test_oracle_sum as ts

SRC = os.path.join(os.path.dirname(oracle.__file__), "sar_oracle.c")

MUTANTS = {
    "ties away from zero":
        ("if (rest > half || (rest == half && (keep & 1))) keep += 1;",
         "if (rest >= half) keep += 1;"),
    "truncation instead of rounding":
        ("if (rest > half || (rest == half && (keep & 1))) keep += 1;", ";"),
    "last rank dropped":
        ("for (int k = 1; k < nranks; ++k) acc = acc + orc_load(dt, in[k], i);\n        for (int j",
         "for (int k = 1; k < nranks - 1; ++k) acc = acc + orc_load(dt, in[k], i);\n        for (int j"),
    "reversed rank order":
        ("float acc = orc_load(dt, in[0], i);\n        for (int k = 1; k < nranks; ++k) acc = acc + orc_load(dt, in[k], i);\n        for (int j",
         "float acc = orc_load(dt, in[nranks - 1], i);\n        for (int k = nranks - 2; k >= 0; --k) acc = acc + orc_load(dt, in[k], i);\n        for (int j"),
    "accumulator seeded with +0":
        ("float acc = orc_load(dt, in[0], i);\n        for (int k = 1; k < nranks; ++k) acc = acc + orc_load(dt, in[k], i);\n        for (int j",
         "float acc = 0.0f;\n        for (int k = 0; k < nranks; ++k) acc = acc + orc_load(dt, in[k], i);\n        for (int j"),
    "fp16 bias off by one":
        ("static const orc_fmt F = { 11, -14, 15 };", "static const orc_fmt F = { 11, -14, 16 };"),
    "bf16 sign dropped":
        ("    if (c < 0) return s | 0x7F80;                     /* overflow -> infinity */\n    return s | (uint16_t)c;",
         "    if (c < 0) return s | 0x7F80;                     /* overflow -> infinity */\n    return (uint16_t)c;"),
    "e4m3fn overflow to NaN":
        ("if (c < 0 || c > 0x7E) return s | 0x7E;", "if (c < 0 || c > 0x7E) return s | 0x7F;"),
    "fp16 subnormal scale":
        ("mag = ldexpf((float)f, -24);", "mag = ldexpf((float)f, -25);"),
    "e4m3fn normal scale":
        ("else mag = ldexpf((float)(8 + f), e - 10);", "else mag = ldexpf((float)(8 + f), e - 9);"),
    "packet flag big-endian":
        ("(uint8_t)(epoch >> (8 * k));", "(uint8_t)(epoch >> (8 * (3 - k)));"),
    "packet tail not zero-padded":
        ("at < bytes ? src[at] : 0;", "at < bytes ? src[at] : 0xFF;"),
    "chunk not rounded to a vector":
        ("    c = (c + vec - 1) / vec * vec;\n", ""),
    "partial sums not rounded into the accumulator":
        ("            acc = round_through(acc_dt, acc + orc_load(dt, in[k], i));",
         "            acc = acc + orc_load(dt, in[k], i);"),
    "accumulator seed not rounded":
        ("        float acc = round_through(acc_dt, orc_load(dt, in[0], i));",
         "        float acc = orc_load(dt, in[0], i);"),
    "e4m3b15 largest exponent field treated as finite":
        ("    int64_t c = encode_grid(n, q, &F, 14);", "    int64_t c = encode_grid(n, q, &F, 15);"),
    "e4m3b15 subnormal scale":
        ("        mag = ldexpf((float)f, -17);", "        mag = ldexpf((float)f, -16);"),
    "all-gather skips a peer":
        ("if (j == r || e == b) continue;", "if (j == r || j == 0 || e == b) continue;"),
    "unpack accepts any flag":
        ("if (flag != epoch) return ORC_NOT_ARRIVED;", "(void)flag;"),
    "unpack reads the payload from the flag half":
        ("rebuilt[r][at] = p[8 * (at / 4) + at % 4];", "rebuilt[r][at] = p[8 * (at / 4) + 4 + at % 4];"),
    "e4m3fn subnormal scale":
        ("    if (e == 0) mag = ldexpf((float)f, -9);", "    if (e == 0) mag = ldexpf((float)f, -8);"),
    "packet count rounds down":
        ("    return (bytes + 3) / 4;", "    return bytes / 4;"),
    "e4m3b15 infinity decoded as NaN":
        ("        if (f != 0) return bits_f32(0x7FC00000u);\n        mag = INFINITY;\n    } else if (e == 0) {\n"
         "        mag = ldexpf((float)f, -17);",
         "        return bits_f32(0x7FC00000u);\n    } else if (e == 0) {\n        mag = ldexpf((float)f, -17);"),
    "reduce-scatter seeded with +0":
        ("            float acc = orc_load(dt, in[0], i);\n            for (int k = 1; k < nranks; ++k) acc = acc + "
         "orc_load(dt, in[k], i);\n            orc_store(dt, out[r], i, acc);",
         "            float acc = 0.0f;\n            for (int k = 0; k < nranks; ++k) acc = acc + "
         "orc_load(dt, in[k], i);\n            orc_store(dt, out[r], i, acc);"),
    "e4m3fn NaN keeps its sign":
        ("    if (isnan(x)) return 0x7F;\n    if (isinf(x)) return s | 0x7E;",
         "    if (isnan(x)) return s | 0x7F;\n    if (isinf(x)) return s | 0x7E;"),
    "fp16 overflow saturates instead of going to infinity":
        ("    if (c < 0) return s | 0x7C00;", "    if (c < 0) return s | 0x7BFF;"),
    "conversion rounds twice, through bf16":
        ("orc_store(dst_dt, dst, i, orc_load(src_dt, src, i));",
         "orc_store(dst_dt, dst, i, orc_bf16_to_f32(orc_f32_to_bf16(orc_load(src_dt, src, i))));"),
    "conversion decodes with the destination type":
        ("orc_store(dst_dt, dst, i, orc_load(src_dt, src, i));", "orc_store(dst_dt, dst, i, orc_load(dst_dt, src, i));"),
}


def _battery(points):
    """Run a selection of pins; return how many failed."""
    checks = [
        lambda: [tf.test_round_matches_bruteforce_nearest(points, f) for f in ("bf16", "fp16", "e4m3fn", "e4m3b15")],
        lambda: [tf.test_decode_every_code(f) for f in ("bf16", "fp16", "e4m3fn", "e4m3b15")],
        lambda: tf.test_e4m3b15_is_the_top_of_a_binary16(),
        lambda: tf.test_golden_format_constants(),
        lambda: [ts.test_one_rank_is_identity(d) for d in ts.DTYPES],
        lambda: [ts.test_all_equal_inputs_give_n_times_x(d, 8) for d in ts.DTYPES],
        lambda: [ts.test_small_integers_sum_exactly_under_any_rank_order(d, 5) for d in ts.DTYPES],
        lambda: ts.test_all_e4m3fn_pairs_bruteforce(),
        lambda: ts.test_rank_order_is_0_to_n_minus_1(),
        lambda: [ts.test_rsag_chunks_partition_the_range(d) for d in ts.DTYPES],
        lambda: [ts.test_reduce_scatter_then_all_gather_is_allreduce(d, 8, 4097) for d in ts.DTYPES],
        lambda: [ts.test_reduce_scatter_of_negative_zeros_is_negative_zero(d) for d in ts.DTYPES + ["e4m3b15"]],
        lambda: [tf.test_fp8_nan_is_the_positive_all_ones_code(f) for f in ("e4m3fn", "e4m3b15")],
        lambda: [ts.test_ll_pack_byte_image(d, 5) for d in ts.DTYPES],
        lambda: [ts.test_ll_unpack_reduce_gives_the_exact_sums(d, 8, 257) for d in ts.DTYPES],
        lambda: ts.test_ll_stale_flag_is_not_arrived(),
        lambda: [ta.test_stepwise_reference(d, a, 8) for d, a in ta.CASES],
        lambda: ta.test_native_e4m3fn_rounds_every_partial_sum(),
        lambda: ts.test_convert_e4m3fn_to_f32_every_code(),
        lambda: [ts.test_convert_to_e4m3fn_rounds_once(d) for d in ("fp32", "bf16", "fp16")],
        lambda: [ts.test_convert_from_e4m3fn_is_exact(d) for d in ("bf16", "fp16", "fp32")],
    ]
    failed = 0
    for c in checks:
        try:
            c()
        except (AssertionError, ValueError):
            failed += 1
    return failed


@pytest.fixture(scope="module")
def points():
    return tf._f32_points()[::7]


def test_unmodified_oracle_passes_battery(points):
    assert _battery(points) == 0


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, points, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for '{name}' not found"
    mutated = src.replace(old, new, 1)
    path = tmp_path / "mutant.c"
    path.write_text(mutated)
    lib = oracle.compile_library(str(path), str(tmp_path / "libmutant.so"))
    with oracle.using_library(lib):
        failed = _battery(points)
    assert failed >= 1, f"no pin caught the planted mistake '{name}'"
