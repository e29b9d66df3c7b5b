"""Helpers for the GPU parity tests: guarded device buffers and bit-exact
comparison against the oracle's element codes."""
from __future__ import annotations

import numpy as np
import torch

GUARD = 256          # bytes of canary before and after every buffer
CANARY = 0xA5

STORE = {"bf16": np.uint16, "fp16": np.uint16, "fp32": np.float32, "e4m3fn": np.uint8, "e4m3b15": np.uint8}
ESIZE = {"bf16": 2, "fp16": 2, "fp32": 4, "e4m3fn": 1, "e4m3b15": 1}


class Guarded:
    """A device buffer of `nbytes` at byte offset `offset` inside a larger
    allocation whose other bytes hold a canary."""

    def __init__(self, nbytes: int, offset: int = 0, fill: int = CANARY):
        self.nbytes, self.offset = nbytes, offset
        self.base = torch.full((2 * GUARD + offset + nbytes,), CANARY, dtype=torch.uint8, device="cuda")
        if fill != CANARY:
            self.base[GUARD + offset: GUARD + offset + nbytes] = fill
        self.ptr = self.base.data_ptr() + GUARD + offset

    @classmethod
    def from_codes(cls, codes: np.ndarray, offset: int = 0) -> "Guarded":
        raw = np.ascontiguousarray(codes).view(np.uint8).ravel()
        g = cls(raw.size, offset)
        if raw.size:
            g.base[GUARD + offset: GUARD + offset + raw.size] = torch.from_numpy(raw.copy()).cuda()
        return g

    def bytes(self) -> np.ndarray:
        return self.base[GUARD + self.offset: GUARD + self.offset + self.nbytes].cpu().numpy()

    def codes(self, dt: str) -> np.ndarray:
        return self.bytes().view(STORE[dt])

    def guards_intact(self) -> bool:
        b = self.base.cpu().numpy()
        head = b[: GUARD + self.offset]
        tail = b[GUARD + self.offset + self.nbytes:]
        return bool(np.all(head == CANARY) and np.all(tail == CANARY))


def is_nan_code(codes: np.ndarray, dt: str) -> np.ndarray:
    c = np.asarray(codes)
    if dt == "fp32":
        return np.isnan(c.view(np.float32))
    if dt == "bf16":
        c = c.view(np.uint16)
        return ((c & 0x7F80) == 0x7F80) & ((c & 0x007F) != 0)
    if dt == "fp16":
        c = c.view(np.uint16)
        return ((c & 0x7C00) == 0x7C00) & ((c & 0x03FF) != 0)
    c = c.view(np.uint8)
    if dt == "e4m3b15":
        return ((c & 0x78) == 0x78) & ((c & 0x07) != 0)
    return (c & 0x7F) == 0x7F


def assert_same(got: np.ndarray, want: np.ndarray, dt: str, what: str = "") -> None:
    """Bit-exact equality; NaN is compared by class (both NaN)."""
    got = np.asarray(got).view(STORE[dt]).ravel()
    want = np.asarray(want).view(STORE[dt]).ravel()
    assert got.shape == want.shape, (what, got.shape, want.shape)
    gn, wn = is_nan_code(got, dt), is_nan_code(want, dt)
    gb = got.view(np.uint8).reshape(got.size, -1)
    wb = want.view(np.uint8).reshape(want.size, -1)
    diff = np.any(gb != wb, axis=1) & ~(gn & wn)
    bad = np.nonzero(diff)[0]
    assert bad.size == 0, (f"{what}: {bad.size} of {got.size} elements differ; first at {bad[:8]}: "
                           f"got {got[bad[:8]]} want {want[bad[:8]]}")


def random_codes(rng, dt: str, n: int, nan_ok: bool = False) -> np.ndarray:
    """Random bit patterns of dt (every class: zeros, subnormals, extremes)."""
    bits = rng.integers(0, 1 << (8 * ESIZE[dt]), n, dtype=np.uint64)
    if dt == "fp32":
        c = bits.astype(np.uint32).view(np.float32).copy()
    else:
        c = bits.astype(STORE[dt])
    if not nan_ok:
        nan = is_nan_code(c, dt)
        c[nan] = STORE[dt](0)
    return c
