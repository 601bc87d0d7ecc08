"""Oracle for the deterministic collective's data-parallel core.

TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's
CPU-baseline leg may import this package; the CUDA library and its Python
binding never do.  It shares no code with the GPU path.

The oracle proper is the plain C code in ``dc_oracle.c``, loaded through
ctypes; this module only marshals numpy arrays into it.  Every parity test
compares the CUDA path against it.  The tests pin it to the page's
statements, to worked examples, to exact rational arithmetic and to library
routines before trusting it.

Page, by title:
  [PR491] "perf(cuda): vectorize the deterministic all-gather copy and
          right-size its single-block path" (RL-Kernel pull request 491).
"""
from __future__ import annotations

import ctypes
from typing import Sequence

import numpy as np

from . import build as _build

_default = None


def _configure(L: ctypes.CDLL) -> ctypes.CDLL:
    P = ctypes.c_void_p
    L.orc_all_gather.argtypes = [ctypes.POINTER(P), ctypes.c_int, ctypes.c_size_t, P]
    L.orc_all_gather_many.argtypes = [ctypes.POINTER(P), ctypes.POINTER(ctypes.c_size_t),
                                      ctypes.POINTER(P), ctypes.c_int, ctypes.c_int]
    L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
    L.orc_bf16_to_f32.restype = ctypes.c_float
    L.orc_f32_to_bf16_rne.argtypes = [ctypes.c_float]
    L.orc_f32_to_bf16_rne.restype = ctypes.c_uint16
    L.orc_f32_to_bf16_rne_array.argtypes = [P, P, ctypes.c_size_t]
    L.orc_all_reduce_bf16.argtypes = [ctypes.POINTER(P), ctypes.POINTER(P), ctypes.c_int,
                                      ctypes.c_size_t]
    L.orc_reduce_scatter_bf16.argtypes = [ctypes.POINTER(P), ctypes.POINTER(P),
                                          ctypes.c_int, ctypes.c_size_t]
    L.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
    L.orc_f16_to_f32.restype = ctypes.c_float
    L.orc_f32_to_f16_rne_array.argtypes = [P, P, ctypes.c_size_t]
    L.orc_all_reduce.argtypes = [ctypes.POINTER(P), ctypes.POINTER(P), ctypes.c_int,
                                 ctypes.c_size_t, ctypes.c_int, ctypes.c_int]
    L.orc_reduce_scatter.argtypes = [ctypes.POINTER(P), ctypes.POINTER(P), ctypes.c_int,
                                     ctypes.c_size_t, ctypes.c_int, ctypes.c_int]
    L.orc_subnormals_preserved.argtypes = []
    for f in ("orc_all_gather", "orc_all_gather_many", "orc_all_reduce_bf16",
              "orc_f32_to_bf16_rne_array", "orc_reduce_scatter_bf16", "orc_f32_to_f16_rne_array",
              "orc_all_reduce", "orc_reduce_scatter", "orc_subnormals_preserved"):
        getattr(L, f).restype = ctypes.c_int
    if L.orc_subnormals_preserved() != 1:
        raise RuntimeError("oracle host flushes binary32 subnormals; results would be wrong")
    return L


def _ptrs(arrs: Sequence[np.ndarray]):
    return (ctypes.c_void_p * max(1, len(arrs)))(*[a.ctypes.data for a in arrs])


def _u8(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    return a.view(np.uint8).reshape(-1)


DTYPES = {"bf16": (0, np.uint16), "f16": (1, np.uint16), "f32": (2, np.float32)}
ORDERS = {"linear": 0, "tree": 1}


def _as_elems(a, dtype: str) -> np.ndarray:
    """A contiguous 1-D view of the payload as the oracle's element type
    (16-bit patterns for bf16 / f16, binary32 for f32)."""
    want = DTYPES[dtype][1]
    a = np.ascontiguousarray(a)
    if a.dtype != want:
        if a.dtype.itemsize != np.dtype(want).itemsize:
            raise TypeError(f"{dtype} payloads need {np.dtype(want).itemsize}-byte elements")
        a = a.view(want)
    return a.reshape(-1)


def _as_bf16_bits(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        if a.dtype.itemsize != 2:
            raise TypeError("BF16 payloads are passed as 16-bit patterns")
        a = a.view(np.uint16)
    return a.reshape(-1)


class Oracle:
    """numpy front end over one loaded copy of the C oracle."""

    def __init__(self, L: ctypes.CDLL):
        self.L = L

    # ---------------------------------------------------------- gather ---
    def all_gather(self, peers: Sequence[np.ndarray]) -> np.ndarray:
        """Rank-ordered concatenation of the P payloads' bytes ([PR491]
        "What", copy_rank_ordered).  Every peer must have the same size."""
        bufs = [_u8(p) for p in peers]
        P = len(bufs)
        B = bufs[0].size if P else 0
        if any(b.size != B for b in bufs):
            raise ValueError("all peers must hold the same number of bytes")
        out = np.empty(P * B, dtype=np.uint8)
        rc = self.L.orc_all_gather(_ptrs(bufs), P, B, out.ctypes.data)
        if rc != 0:
            raise ValueError(f"orc_all_gather rejected its arguments ({rc})")
        return out

    def all_gather_many(self, peers_per_tensor) -> list[np.ndarray]:
        """T independent all-gathers, one output per tensor (no packing)."""
        T = len(peers_per_tensor)
        if T == 0:
            return []
        P = len(peers_per_tensor[0])
        flat, sizes = [], []
        for peers in peers_per_tensor:
            bufs = [_u8(p) for p in peers]
            if len(bufs) != P or any(b.size != bufs[0].size for b in bufs):
                raise ValueError("each tensor needs P peers of equal byte size")
            flat.extend(bufs)
            sizes.append(bufs[0].size)
        outs = [np.empty(P * s, dtype=np.uint8) for s in sizes]
        size_arr = (ctypes.c_size_t * T)(*sizes)
        rc = self.L.orc_all_gather_many(_ptrs(flat), size_arr, _ptrs(outs), T, P)
        if rc != 0:
            raise ValueError(f"orc_all_gather_many rejected its arguments ({rc})")
        return outs

    # -------------------------------------------------------- rounding ---
    def bf16_to_f32(self, h: int) -> float:
        return float(self.L.orc_bf16_to_f32(int(h) & 0xFFFF))

    def f32_to_bf16_rne_array(self, f32: np.ndarray) -> np.ndarray:
        """RNE of every binary32 value (uint32 bit patterns accepted)."""
        a = np.ascontiguousarray(f32)
        if a.dtype == np.uint32:
            a = a.view(np.float32)
        a = a.astype(np.float32, copy=False).reshape(-1)
        out = np.empty(a.size, dtype=np.uint16)
        if self.L.orc_f32_to_bf16_rne_array(a.ctypes.data, out.ctypes.data, a.size) != 0:
            raise ValueError("orc_f32_to_bf16_rne_array rejected its arguments")
        return out

    # ------------------------------------------------------ reductions ---
    def all_reduce_bf16_all_outputs(self, inputs) -> list[np.ndarray]:
        """Every rank's output buffer of the fixed-order BF16 all_reduce."""
        ins = [_as_bf16_bits(x) for x in inputs]
        P = len(ins)
        n = ins[0].size
        if any(x.size != n for x in ins):
            raise ValueError("all inputs must have the same element count")
        outs = [np.empty(n, dtype=np.uint16) for _ in range(P)]
        rc = self.L.orc_all_reduce_bf16(_ptrs(ins), _ptrs(outs), P, n)
        if rc != 0:
            raise ValueError(f"orc_all_reduce_bf16 rejected its arguments ({rc})")
        return outs

    def all_reduce_bf16(self, inputs) -> np.ndarray:
        """The fixed-order BF16 all_reduce of P equal-length 16-bit pattern
        arrays; returns the one result every rank receives."""
        outs = self.all_reduce_bf16_all_outputs(inputs)
        for r in range(1, len(outs)):
            if not np.array_equal(outs[0], outs[r]):
                raise AssertionError("oracle wrote different values to different ranks")
        return outs[0]

    def reduce_scatter_bf16(self, inputs) -> list[np.ndarray]:
        """Fixed-order BF16 reduce_scatter: each input holds P*C elements;
        rank r receives the reduced shard [r*C, (r+1)*C)."""
        ins = [_as_bf16_bits(x) for x in inputs]
        P = len(ins)
        n = ins[0].size
        if any(x.size != n for x in ins) or n % P != 0:
            raise ValueError("inputs must be equal length and divisible by P")
        C = n // P
        outs = [np.empty(C, dtype=np.uint16) for _ in range(P)]
        rc = self.L.orc_reduce_scatter_bf16(_ptrs(ins), _ptrs(outs), P, C)
        if rc != 0:
            raise ValueError(f"orc_reduce_scatter_bf16 rejected its arguments ({rc})")
        return outs

    # ------------------------------------------- other types and orders ---
    def f16_to_f32(self, h: int) -> float:
        return float(self.L.orc_f16_to_f32(int(h) & 0xFFFF))

    def f32_to_f16_rne_array(self, f32: np.ndarray) -> np.ndarray:
        a = np.ascontiguousarray(f32)
        if a.dtype == np.uint32:
            a = a.view(np.float32)
        a = a.astype(np.float32, copy=False).reshape(-1)
        out = np.empty(a.size, dtype=np.uint16)
        if self.L.orc_f32_to_f16_rne_array(a.ctypes.data, out.ctypes.data, a.size) != 0:
            raise ValueError("orc_f32_to_f16_rne_array rejected its arguments")
        return out

    def all_reduce_all_outputs(self, inputs, dtype="bf16", order="linear") -> list[np.ndarray]:
        """Every rank's output of the fixed-order all_reduce of element type
        `dtype` ("bf16", "f16", "f32") in summation order `order` ("linear",
        "tree")."""
        ins = [_as_elems(x, dtype) for x in inputs]
        P = len(ins)
        n = ins[0].size
        if any(x.size != n for x in ins):
            raise ValueError("all inputs must have the same element count")
        outs = [np.empty(n, dtype=DTYPES[dtype][1]) for _ in range(P)]
        rc = self.L.orc_all_reduce(_ptrs(ins), _ptrs(outs), P, n, DTYPES[dtype][0], ORDERS[order])
        if rc != 0:
            raise ValueError(f"orc_all_reduce rejected its arguments ({rc})")
        return outs

    def all_reduce(self, inputs, dtype="bf16", order="linear") -> np.ndarray:
        outs = self.all_reduce_all_outputs(inputs, dtype, order)
        for r in range(1, len(outs)):
            if not np.array_equal(outs[0].view(np.uint8), outs[r].view(np.uint8)):
                raise AssertionError("oracle wrote different values to different ranks")
        return outs[0]

    def reduce_scatter(self, inputs, dtype="bf16", order="linear") -> list[np.ndarray]:
        ins = [_as_elems(x, dtype) for x in inputs]
        P = len(ins)
        n = ins[0].size
        if any(x.size != n for x in ins) or n % P != 0:
            raise ValueError("inputs must be equal length and divisible by P")
        C = n // P
        outs = [np.empty(C, dtype=DTYPES[dtype][1]) for _ in range(P)]
        rc = self.L.orc_reduce_scatter(_ptrs(ins), _ptrs(outs), P, C, DTYPES[dtype][0],
                                       ORDERS[order])
        if rc != 0:
            raise ValueError(f"orc_reduce_scatter rejected its arguments ({rc})")
        return outs

    def reduce_bf16_at(self, inputs, index: np.ndarray) -> np.ndarray:
        """The fold evaluated only at the given element indices (for sampled
        checks of full-size outputs)."""
        cols = [np.ascontiguousarray(_as_bf16_bits(x)[index]) for x in inputs]
        return self.all_reduce_bf16(cols)


def load(path: str) -> Oracle:
    """Load a specific build of the C oracle (the tests use this to load
    deliberately broken copies and show that the pins reject them)."""
    return Oracle(_configure(ctypes.CDLL(path)))


def default() -> Oracle:
    global _default
    if _default is None:
        _default = load(_build.build())
    return _default


def all_gather(peers):
    return default().all_gather(peers)


def all_gather_many(peers_per_tensor):
    return default().all_gather_many(peers_per_tensor)


def f32_to_bf16_rne_array(f32):
    return default().f32_to_bf16_rne_array(f32)


def all_reduce_bf16(inputs):
    return default().all_reduce_bf16(inputs)


def all_reduce_bf16_all_outputs(inputs):
    return default().all_reduce_bf16_all_outputs(inputs)


def reduce_scatter_bf16(inputs):
    return default().reduce_scatter_bf16(inputs)


def reduce_bf16_at(inputs, index):
    return default().reduce_bf16_at(inputs, index)


def all_reduce(inputs, dtype="bf16", order="linear"):
    return default().all_reduce(inputs, dtype, order)


def reduce_scatter(inputs, dtype="bf16", order="linear"):
    return default().reduce_scatter(inputs, dtype, order)
