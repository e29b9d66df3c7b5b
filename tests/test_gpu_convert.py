"""GPU parity of sar_fp8_convert against the CPU oracle, through the C ABI:
every e4m3fn code widened, every bf16/fp16 code and a dense set of binary32
rounding cases narrowed, on the vector and the element paths."""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import ESIZE, Guarded, assert_same
from tests.test_oracle_formats import _f32_points

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sar():
    import allreduce_reduction_rank_gb300 as s
    return s


def _convert(sar, src_codes, src, dst, offset=0):
    count = src_codes.size
    g_src = Guarded.from_codes(src_codes, offset * ESIZE[src])
    g_dst = Guarded(count * ESIZE[dst], offset * ESIZE[dst], fill=0x5A)
    sar.sar_fp8_convert(g_src.ptr, g_dst.ptr, src_dtype=src, dst_dtype=dst, count=count)
    torch.cuda.synchronize()
    assert g_dst.guards_intact() and g_src.guards_intact()
    assert np.array_equal(g_src.bytes(), np.ascontiguousarray(src_codes).view(np.uint8))
    return g_dst.codes(dst)


@pytest.mark.parametrize("fp8", ["e4m3fn", "e4m3b15"])
@pytest.mark.parametrize("offset", [0, 1])
@pytest.mark.parametrize("dst", ["fp32", "fp16", "bf16"])
def test_every_fp8_code_widens_exactly(sar, dst, offset, fp8):
    codes = np.tile(np.arange(256, dtype=np.uint8), 9)[:2300]      # groups of 16 plus a tail
    got = _convert(sar, codes, fp8, dst, offset)
    assert_same(got, oracle.convert(codes, fp8, dst), dst)


@pytest.mark.parametrize("fp8", ["e4m3fn", "e4m3b15"])
@pytest.mark.parametrize("offset", [0, 3])
@pytest.mark.parametrize("src", ["fp16", "bf16"])
def test_every_16bit_code_narrows_once(sar, src, offset, fp8):
    codes = np.arange(1 << 16, dtype=np.uint16)
    codes = np.concatenate([codes, codes[:7]])
    got = _convert(sar, codes, src, fp8, offset)
    assert_same(got, oracle.convert(codes, src, fp8), fp8)


@pytest.mark.parametrize("offset", [0, 1])
def test_binary32_rounding_cases_narrow_once_e4m3b15(sar, offset):
    x = _f32_points()
    x = np.concatenate([x, np.array([np.inf, -np.inf, np.nan, 0.9375, 0.96875, 0.968, 1.0, -1e30], np.float32)])
    got = _convert(sar, x, "fp32", "e4m3b15", offset)
    assert_same(got, oracle.convert(x, "fp32", "e4m3b15"), "e4m3b15")
    assert got[-8:].tolist() == [0x78, 0xF8, got[-6], 0x77, 0x78, 0x77, 0x78, 0xF8]
    assert got[-6] & 0x78 == 0x78 and got[-6] & 0x07 != 0        # NaN stays NaN


@pytest.mark.parametrize("offset", [0, 1])
def test_binary32_rounding_cases_narrow_once(sar, offset):
    x = _f32_points()
    x = np.concatenate([x, np.array([np.inf, -np.inf, np.nan, 448.0, 464.0, 480.0, -1e30], np.float32)])
    got = _convert(sar, x, "fp32", "e4m3fn", offset)
    assert_same(got, oracle.convert(x, "fp32", "e4m3fn"), "e4m3fn")
    tail = got[-7:].tolist()
    assert tail[0] == 0x7E and tail[1] == 0xFE      # satfinite: +-inf -> +-448
    assert tail[3:6] == [0x7E, 0x7E, 0x7E] and tail[6] == 0xFE
    assert tail[2] & 0x7F == 0x7F                    # NaN stays NaN
