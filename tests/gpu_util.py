"""Helpers for the GPU parity tests: byte-offset placement inside guarded
device buffers and host copies for the oracle.

Every output buffer sits inside a larger allocation filled with the guard
byte 0xA5, so a test can check that no byte before or after the output was
written (the page's size test fills its output storage with 0xA5 and checks
the bytes before and after ``out``).
"""
from __future__ import annotations

import numpy as np

GUARD = 0xA5
GUARD_BYTES = 64


def _torch():
    import torch

    return torch


class Placed:
    """A byte range at a chosen offset from a 256-byte boundary, with guard
    bytes on both sides."""

    def __init__(self, nbytes: int, offset: int, device="cuda", fill: int | None = GUARD):
        torch = _torch()
        total = GUARD_BYTES + 256 + offset + nbytes + GUARD_BYTES
        self.storage = torch.empty(total, dtype=torch.uint8, device=device)
        if fill is not None:
            self.storage.fill_(fill)
        base = self.storage.data_ptr()
        start = GUARD_BYTES + ((-(base + GUARD_BYTES)) % 256) + offset
        self.start, self.nbytes = start, nbytes
        self.view = self.storage[start:start + nbytes]

    def ptr(self) -> int:
        return self.storage.data_ptr() + self.start

    def write(self, data: np.ndarray) -> None:
        torch = _torch()
        assert data.size == self.nbytes
        if self.nbytes:
            self.view.copy_(torch.from_numpy(np.ascontiguousarray(data).view(np.uint8)))

    def read(self) -> np.ndarray:
        return self.view.cpu().numpy()

    def guards_intact(self) -> bool:
        s = self.storage.cpu().numpy()
        return bool((s[:self.start] == GUARD).all() and (s[self.start + self.nbytes:] == GUARD).all())


def bf16_tensor(bits: np.ndarray, device="cuda"):
    """A torch.bfloat16 device tensor holding the given 16-bit patterns."""
    torch = _torch()
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def bits_of(t) -> np.ndarray:
    """The 16-bit patterns of a bfloat16 tensor, on the host."""
    torch = _torch()
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_view_at(storage, byte_offset: int, count: int):
    """A bfloat16 view of `count` elements starting `byte_offset` bytes into
    a uint8 storage tensor (byte_offset must be even)."""
    torch = _torch()
    assert byte_offset % 2 == 0
    return storage[byte_offset:byte_offset + 2 * count].view(torch.bfloat16)


def is_nan_bits(h: np.ndarray) -> np.ndarray:
    return ((h & 0x7F80) == 0x7F80) & ((h & 0x007F) != 0)


def assert_bf16_equal(got: np.ndarray, want: np.ndarray, what: str = "") -> None:
    """Bit-exact equality, except that NaN is compared by class only."""
    gn, wn = is_nan_bits(got), is_nan_bits(want)
    if not np.array_equal(gn, wn):
        i = int(np.flatnonzero(gn != wn)[0])
        raise AssertionError(f"{what}: NaN class differs at {i}: got {got[i]:#06x} want {want[i]:#06x}")
    bad = np.flatnonzero((got != want) & ~wn)
    if bad.size:
        i = int(bad[0])
        raise AssertionError(f"{what}: {bad.size} elements differ, first at {i}: "
                             f"got {got[i]:#06x} want {want[i]:#06x}")


NP_OF = {"bf16": np.uint16, "f16": np.uint16, "f32": np.uint32}


def torch_dtype(dtype: str):
    torch = _torch()
    return {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[dtype]


def typed_tensor(bits: np.ndarray, dtype: str, device="cuda"):
    """A device tensor of element type `dtype` holding the given bit patterns."""
    torch = _torch()
    as_int = np.ascontiguousarray(bits).view(np.int16 if dtype != "f32" else np.int32)
    return torch.from_numpy(as_int).to(device).view(torch_dtype(dtype))


def typed_bits(t, dtype: str) -> np.ndarray:
    torch = _torch()
    iv = torch.int16 if dtype != "f32" else torch.int32
    return t.view(iv).cpu().numpy().view(NP_OF[dtype])


def is_nan_typed(h: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return is_nan_bits(h)
    if dtype == "f16":
        return ((h & 0x7C00) == 0x7C00) & ((h & 0x03FF) != 0)
    return ((h & 0x7F800000) == 0x7F800000) & ((h & 0x007FFFFF) != 0)


def assert_typed_equal(got: np.ndarray, want: np.ndarray, dtype: str, what: str = "") -> None:
    """Bit-exact equality except NaN, compared by class."""
    gn, wn = is_nan_typed(got, dtype), is_nan_typed(want, dtype)
    if not np.array_equal(gn, wn):
        i = int(np.flatnonzero(gn != wn)[0])
        raise AssertionError(f"{what}: NaN class differs at {i}: got {int(got[i]):#x} want {int(want[i]):#x}")
    bad = np.flatnonzero((got != want) & ~wn)
    if bad.size:
        i = int(bad[0])
        raise AssertionError(f"{what}: {bad.size} elements differ, first at {i}: "
                             f"got {int(got[i]):#x} want {int(want[i]):#x}")
