"""reduce_copy_rank_gb300 -- deterministic rank-ordered gather and fixed-order
BF16 reductions on one GPU, with the world's P ranks held as P buffers in the
GPU's own memory.

This module is a thin ctypes binding of ``libdc.so`` (C ABI in
``include/dc.h``): it only turns tensors into pointers, sizes and a stream
handle.  Every step of the work runs in the library's CUDA kernels; there is
no CPU or PyTorch fallback.  If the library has not been built the first call
raises :class:`LibraryMissing`.

Page, by title: "perf(cuda): vectorize the deterministic all-gather copy and
right-size its single-block path" (RL-Kernel PR 491).  Its Python API is
``DeterministicCollective.all_gather(input, out=)`` returning ``out``,
``all_gather_many(tensors)``, ``all_reduce`` and ``reduce_scatter``; the
functions here take the P ranks' buffers explicitly instead of one tensor
per process.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
from typing import Sequence

__all__ = [
    "DCError", "LibraryMissing", "all_gather", "all_gather_many", "all_reduce",
    "reduce_scatter", "set_option", "get_option", "launch_count", "last_error",
    "options", "lib", "LIB_PATH", "STATUS",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdc.so")

STATUS = {0: "DC_OK", 1: "DC_ERR_INVALID", 2: "DC_ERR_ALIGN", 3: "DC_ERR_OVERLAP",
          4: "DC_ERR_TOO_MANY", 5: "DC_ERR_CUDA", 6: "DC_ERR_TIMEOUT"}

MAX_RANKS = 64
MANY_MAX_TENSORS = 256
MANY_MAX_SEGMENTS = 1024


class LibraryMissing(RuntimeError):
    """libdc.so is not built (run ``python -m reduce_copy_rank_gb300._build``)."""


class DCError(RuntimeError):
    """A libdc call returned a non-zero status."""

    def __init__(self, status: int, message: str):
        self.status = status
        self.name = STATUS.get(status, f"status {status}")
        super().__init__(f"{self.name}: {message}")


_lib = None
_VP = ctypes.c_void_p


def lib() -> ctypes.CDLL:
    """The loaded C library (loaded on first use)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise LibraryMissing(
                f"{LIB_PATH} is missing: build it with `python -m reduce_copy_rank_gb300._build` "
                "(or __graft_entry__.build()); there is no fallback path")
        L = ctypes.CDLL(LIB_PATH)
        L.dc_all_gather.argtypes = [ctypes.POINTER(_VP), ctypes.c_int, ctypes.c_size_t, _VP, _VP]
        L.dc_all_gather_many.argtypes = [ctypes.POINTER(_VP), ctypes.POINTER(ctypes.c_size_t),
                                         ctypes.POINTER(_VP), ctypes.c_int, ctypes.c_int, _VP]
        L.dc_all_reduce_bf16.argtypes = [ctypes.POINTER(_VP), ctypes.POINTER(_VP), ctypes.c_int,
                                         ctypes.c_size_t, _VP]
        L.dc_reduce_scatter_bf16.argtypes = [ctypes.POINTER(_VP), ctypes.POINTER(_VP),
                                             ctypes.c_int, ctypes.c_size_t, _VP]
        for f in ("dc_all_gather", "dc_all_gather_many", "dc_all_reduce_bf16",
                  "dc_reduce_scatter_bf16"):
            getattr(L, f).restype = ctypes.c_int
        L.dc_last_error.argtypes = []
        L.dc_last_error.restype = ctypes.c_char_p
        L.dc_status_name.argtypes = [ctypes.c_int]
        L.dc_status_name.restype = ctypes.c_char_p
        L.dc_set_option.argtypes = [ctypes.c_char_p, ctypes.c_longlong]
        L.dc_set_option.restype = ctypes.c_int
        L.dc_get_option.argtypes = [ctypes.c_char_p]
        L.dc_get_option.restype = ctypes.c_longlong
        L.dc_launch_count.argtypes = []
        L.dc_launch_count.restype = ctypes.c_ulonglong
        L.dc_version.argtypes = []
        L.dc_version.restype = ctypes.c_int
        _lib = L
    return _lib


def _check(status: int) -> None:
    if status != 0:
        raise DCError(status, lib().dc_last_error().decode(errors="replace"))


def _ptr_array(ptrs: Sequence[int]):
    return (_VP * max(1, len(ptrs)))(*[int(p) for p in ptrs])


# ------------------------------------------------------------ raw (C ABI) ---
# Same names and arguments as include/dc.h; pointers are ints, the stream is a
# cudaStream_t handle as an int (0 = legacy default stream).  They return the
# status instead of raising, like the C functions.

def dc_all_gather(peer_ptrs: Sequence[int], P: int, bytes_per_rank: int, out: int,
                  stream: int = 0) -> int:
    return lib().dc_all_gather(_ptr_array(peer_ptrs), P, bytes_per_rank, out, stream)


def dc_all_gather_many(peer_ptrs: Sequence[int], bytes_per_rank: Sequence[int],
                       outs: Sequence[int], T: int, P: int, stream: int = 0) -> int:
    sizes = (ctypes.c_size_t * max(1, len(bytes_per_rank)))(*[int(b) for b in bytes_per_rank])
    return lib().dc_all_gather_many(_ptr_array(peer_ptrs), sizes, _ptr_array(outs), T, P, stream)


def dc_all_reduce_bf16(in_ptrs: Sequence[int], out_ptrs: Sequence[int], P: int, count: int,
                       stream: int = 0) -> int:
    return lib().dc_all_reduce_bf16(_ptr_array(in_ptrs), _ptr_array(out_ptrs), P, count, stream)


def dc_reduce_scatter_bf16(in_ptrs: Sequence[int], out_ptrs: Sequence[int], P: int,
                           count_per_shard: int, stream: int = 0) -> int:
    return lib().dc_reduce_scatter_bf16(_ptr_array(in_ptrs), _ptr_array(out_ptrs), P,
                                        count_per_shard, stream)


# ---------------------------------------------------------- tensor API ---

def _stream_handle(stream) -> int:
    import torch

    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def _device_tensor(t, what: str):
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor (got device {t.device})")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    return t


def all_gather(peers: Sequence, out, stream=None):
    """Rank-ordered all-gather: ``out`` receives the bytes of ``peers[0]``,
    ``peers[1]``, ... in order.  All peers must have the same byte size and
    ``out`` exactly P times that.  Returns ``out``."""
    P = len(peers)
    if P == 0:
        raise ValueError("need at least one peer")
    for r, p in enumerate(peers):
        _device_tensor(p, f"peers[{r}]")
    _device_tensor(out, "out")
    B = _nbytes(peers[0])
    if any(_nbytes(p) != B for p in peers):
        raise ValueError("all peers must have the same number of bytes")
    if _nbytes(out) != P * B:
        raise ValueError(f"out holds {_nbytes(out)} bytes, expected P * {B} = {P * B}")
    _check(dc_all_gather([p.data_ptr() for p in peers], P, B, out.data_ptr(),
                         _stream_handle(stream)))
    return out


def all_gather_many(peers_per_tensor: Sequence[Sequence], outs: Sequence, stream=None):
    """T independent all-gathers in one launch; ``outs[t]`` receives tensor
    t's P payloads in rank order (no packing across tensors).  Returns outs."""
    T = len(peers_per_tensor)
    if len(outs) != T:
        raise ValueError("need one output per tensor")
    if T == 0:
        return outs
    P = len(peers_per_tensor[0])
    ptrs, sizes = [], []
    for t, peers in enumerate(peers_per_tensor):
        if len(peers) != P:
            raise ValueError("every tensor needs the same number of peers")
        B = _nbytes(peers[0])
        for r, p in enumerate(peers):
            _device_tensor(p, f"peers_per_tensor[{t}][{r}]")
            if _nbytes(p) != B:
                raise ValueError(f"tensor {t}: all peers must have the same number of bytes")
        _device_tensor(outs[t], f"outs[{t}]")
        if _nbytes(outs[t]) != P * B:
            raise ValueError(f"outs[{t}] holds {_nbytes(outs[t])} bytes, expected {P * B}")
        ptrs.extend(p.data_ptr() for p in peers)
        sizes.append(B)
    _check(dc_all_gather_many(ptrs, sizes, [o.data_ptr() for o in outs], T, P,
                              _stream_handle(stream)))
    return outs


def _bf16_tensors(ts: Sequence, what: str, count: int | None):
    import torch

    for i, t in enumerate(ts):
        _device_tensor(t, f"{what}[{i}]")
        if t.dtype != torch.bfloat16:
            raise ValueError(f"{what}[{i}] must be torch.bfloat16 (got {t.dtype})")
        if count is not None and t.numel() != count:
            raise ValueError(f"{what}[{i}] has {t.numel()} elements, expected {count}")


def all_reduce(inputs: Sequence, outputs: Sequence, stream=None):
    """Deterministic BF16 all_reduce: every ``outputs[r]`` receives the sum of
    ``inputs[0..P-1]``, folded in rank order in binary32 and rounded once to
    BF16.  ``outputs[r]`` may be one of the inputs (in place).  Returns
    outputs."""
    P = len(inputs)
    if P == 0 or len(outputs) != P:
        raise ValueError("need P >= 1 inputs and P outputs")
    n = inputs[0].numel()
    _bf16_tensors(inputs, "inputs", n)
    _bf16_tensors(outputs, "outputs", n)
    _check(dc_all_reduce_bf16([t.data_ptr() for t in inputs], [t.data_ptr() for t in outputs],
                              P, n, _stream_handle(stream)))
    return outputs


def reduce_scatter(inputs: Sequence, outputs: Sequence, stream=None):
    """Deterministic BF16 reduce_scatter (input = world x output): each input
    holds P*C elements; ``outputs[r]`` (C elements) receives the rank-order
    fold of shard r of every input.  Returns outputs."""
    P = len(inputs)
    if P == 0 or len(outputs) != P:
        raise ValueError("need P >= 1 inputs and P outputs")
    n = inputs[0].numel()
    if n % P:
        raise ValueError(f"input length {n} is not divisible by P = {P}")
    C = n // P
    _bf16_tensors(inputs, "inputs", n)
    _bf16_tensors(outputs, "outputs", C)
    _check(dc_reduce_scatter_bf16([t.data_ptr() for t in inputs], [t.data_ptr() for t in outputs],
                                  P, C, _stream_handle(stream)))
    return outputs


# ------------------------------------------------------------- options ---

def set_option(key: str, value: int) -> None:
    if lib().dc_set_option(key.encode(), int(value)) != 0:
        raise KeyError(f"unknown option or bad value: {key}={value}")


def get_option(key: str) -> int:
    v = lib().dc_get_option(key.encode())
    if v < 0:
        raise KeyError(f"unknown option: {key}")
    return int(v)


@contextlib.contextmanager
def options(**kw):
    """Temporarily set library options, e.g. ``with options(force_path=1):``."""
    old = {k: get_option(k) for k in kw}
    try:
        for k, v in kw.items():
            set_option(k, v)
        yield
    finally:
        for k, v in old.items():
            set_option(k, v)


def launch_count() -> int:
    """Kernels this process has launched through the library."""
    return int(lib().dc_launch_count())


def last_error() -> str:
    return lib().dc_last_error().decode(errors="replace")
