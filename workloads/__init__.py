"""Seeded synthetic workloads for the simulated allreduce.

This module only draws random numbers and quantises them to the element
types; it holds none of the reduction's arithmetic.  It is the one piece of
code shared by the CPU oracle's tests and the CUDA path's tests and benchmark:
both sides consume the same generated element codes, which are produced here
on the host and uploaded, never generated on the GPU.

Generator: splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", 2014) used as a counter-based stream, so any element can
be regenerated on its own: draw k of a stream with seed s is
``mix64(s + (k + 1) * 0x9E3779B97F4A7C15)`` (arithmetic mod 2^64), where
mix64 is the splitmix64 finaliser.  Rank r's element i is draw r*count + i of
the stream.

Distributions:
  * uniform[-1, 1): ``u24 * 2^-23 - 1`` with u24 the top 24 bits of a draw
    (exact in binary32);
  * normal N(0, sigma^2): Box-Muller in binary64 from draws 2j and 2j+1
    (u1 = (top53 + 0.5) * 2^-53, u2 = top53 * 2^-53; x = sqrt(-2 ln u1) *
    cos(2 pi u2) * sigma), then rounded to binary32.

Quantisation to the element type goes through library conversions, all
round-to-nearest-even from binary32: numpy for binary16, torch for bfloat16
and float8_e4m3fn (after clamping to +-448, which makes torch's
non-saturating conversion saturate).  e4m3b15 has no library conversion: its
values are rounded to binary16 by numpy and then to 3 fraction bits (a double
rounding, which only decides which input values are drawn).
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

ESIZE = {"bf16": 2, "fp16": 2, "fp32": 4, "e4m3fn": 1, "e4m3b15": 1}
STORAGE = {"bf16": np.uint16, "fp16": np.uint16, "fp32": np.float32, "e4m3fn": np.uint8, "e4m3b15": np.uint8}


def splitmix64(seed: int, k: np.ndarray) -> np.ndarray:
    """Draws k (uint64 array) of the splitmix64 stream with the given seed."""
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + (k.astype(np.uint64) + np.uint64(1)) * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def _uniform_f32(seed: int, k: np.ndarray) -> np.ndarray:
    u24 = (splitmix64(seed, k) >> np.uint64(40)).astype(np.int64).astype(np.float32)
    return u24 * np.float32(2.0 ** -23) - np.float32(1.0)


def _normal_f32(seed: int, k: np.ndarray, sigma: float) -> np.ndarray:
    k = k.astype(np.uint64)
    z1 = splitmix64(seed, np.uint64(2) * k)
    z2 = splitmix64(seed, np.uint64(2) * k + np.uint64(1))
    u1 = ((z1 >> np.uint64(11)).astype(np.float64) + 0.5) * 2.0 ** -53
    u2 = (z2 >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    x = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2) * sigma
    return x.astype(np.float32)


def quantise(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round binary32 values to element codes of ``dtype`` (library RNE)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "fp32":
        return x
    if dtype == "fp16":
        return x.astype(np.float16).view(np.uint16)
    import torch
    t = torch.from_numpy(x)
    if dtype == "bf16":
        return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    if dtype == "e4m3fn":
        t = t.clamp(-448.0, 448.0)
        return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    if dtype == "e4m3b15":
        # Same bias as binary16, so a finite e4m3b15 code is the top byte of a
        # binary16 with 3 fraction bits: round to binary16 (numpy RNE), then
        # round the 7 dropped fraction bits to nearest even (a double
        # rounding; it only picks the input values).  Values are clamped to
        # +-0.9375 first.
        h = np.clip(x, -0.9375, 0.9375).astype(np.float16).view(np.uint16).astype(np.uint32)
        mag = h & 0x7FFF
        keep, rest = mag >> 7, mag & 0x7F
        keep = keep + ((rest > 0x40) | ((rest == 0x40) & (keep & 1) == 1)).astype(np.uint32)
        return (((h >> 8) & 0x80) | keep).astype(np.uint8)
    raise ValueError(f"unknown dtype {dtype}")


def draw(dist: str, seed: int, k: np.ndarray, dtype: str, sigma: float = 1.0) -> np.ndarray:
    """Element codes for stream indices ``k``."""
    if dist == "uniform":
        x = _uniform_f32(seed, k)
    elif dist == "normal":
        x = _normal_f32(seed, k, sigma)
    else:
        raise ValueError(f"unknown distribution {dist}")
    return quantise(x, dtype)


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def rank_input(dist: str, seed: int, dtype: str, count: int, rank: int,
               sigma: float = 1.0, block: int = 1 << 22) -> np.ndarray:
    """All ``count`` element codes of one simulated rank (threaded in blocks)."""
    out = np.empty(count, dtype=STORAGE[dtype])
    base = rank * count

    def fill(lo: int) -> None:
        hi = min(count, lo + block)
        k = np.arange(base + lo, base + hi, dtype=np.uint64)
        out[lo:hi] = draw(dist, seed, k, dtype, sigma)

    starts = list(range(0, count, block))
    if len(starts) <= 1:
        for lo in starts:
            fill(lo)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, starts))
    return out


def rank_inputs(dist: str, seed: int, dtype: str, count: int, nranks: int,
                sigma: float = 1.0) -> list:
    return [rank_input(dist, seed, dtype, count, r, sigma) for r in range(nranks)]


def sample_inputs(dist: str, seed: int, dtype: str, count: int, nranks: int,
                  idx: np.ndarray, sigma: float = 1.0) -> list:
    """The codes of elements ``idx`` of every rank, regenerated on their own."""
    idx = np.asarray(idx, dtype=np.uint64)
    return [draw(dist, seed, np.uint64(r * count) + idx, dtype, sigma) for r in range(nranks)]


# --------------------------------------------------------------------------
# The workloads: the five configurations the measurements are quoted on.
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    nranks: int
    dtype: str
    count: int          # elements per rank
    dist: str
    seed: int
    sigma: float = 1.0
    algo: str = "rsag"

    @property
    def bytes_per_rank(self) -> int:
        return self.count * ESIZE[self.dtype]

    @property
    def algo_bytes(self) -> int:
        """Algorithmic HBM bytes of one allreduce: N*S read + N*S written."""
        return 2 * self.nranks * self.bytes_per_rank

    def inputs(self) -> list:
        return rank_inputs(self.dist, self.seed, self.dtype, self.count, self.nranks, self.sigma)


KiB, MiB = 1 << 10, 1 << 20

# 2 ranks, 1 MiB of bf16 each, uniform[-1,1], seed 0, rsag out of place.
C1 = Workload("rsag_2x1MiB_bf16", 2, "bf16", 524288, "uniform", 0)
# 8 ranks, 64 MiB of fp16 each (32M elements), N(0,1), rsag.
C2 = Workload("rsag_8x64MiB_fp16", 8, "fp16", 32 * MiB, "normal", 1, 1.0)
# 2 ranks, bf16, 16 KiB .. 256 MiB per rank in x4 steps, uniform, seed 0.
C3 = [Workload(f"rsag_2x{(8192 << (2 * k)) * 2 // KiB}KiB_bf16", 2, "bf16", 8192 << (2 * k),
               "uniform", 0) for k in range(8)]
# 8 ranks, e4m3fn, 16M elements (16 MiB) each, N(0,16) quantised with saturation.
C4 = Workload("rsag_8x16MiB_e4m3fn", 8, "e4m3fn", 16 * MiB, "normal", 2, 4.0)
# Added stress set for the saturation edge (sigma 256).
C4_STRESS = Workload("rsag_8x16MiB_e4m3fn_sigma256", 8, "e4m3fn", 16 * MiB, "normal", 2, 256.0)
# Added counterpart of the e4m3fn workload for the software e4m3b15 type
# (max finite 0.9375): 8 ranks, 16M elements, N(0, 0.05^2).
C4_B15 = Workload("rsag_8x16MiB_e4m3b15", 8, "e4m3b15", 16 * MiB, "normal", 2, 0.05)
# 8 ranks, LL all-pair, fp32 and bf16, 1 KiB .. 1 MiB per rank in x4 steps, uniform, seed 3.
C5 = [Workload(f"ll_8x{s // KiB}KiB_{dt}", 8, dt, s // ESIZE[dt], "uniform", 3, algo="ll")
      for dt in ("fp32", "bf16") for s in (1 * KiB, 4 * KiB, 16 * KiB, 64 * KiB, 256 * KiB, 1 * MiB)]
LL_CALLS = 1000
# Added: rank counts outside {1, 2, 4, 8, 16, 32}, which run the kernels with a
# rank count known only at run time, at the 64 MiB fp16 per rank of the 8-rank
# workload (same seed and stream, so rank r < 8 holds the same codes as there).
C6 = [Workload(f"rsag_{n}x64MiB_fp16", n, "fp16", 32 * MiB, "normal", 1, 1.0) for n in (3, 5, 6, 7, 12)]
