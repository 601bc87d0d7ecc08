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

import array
import contextlib
import ctypes
import os
from typing import Sequence

__all__ = [
    "DCError", "LibraryMissing", "all_gather", "all_gather_many", "all_reduce",
    "reduce_scatter", "reduce", "all_reduce_many", "reduce_scatter_many", "inject_delay", "check_device",
    "fused_all_gather", "fused_workspace", "fused_reset",
    "set_option",
    "get_option",
    "launch_count", "last_grid", "last_error", "options", "lib", "LIB_PATH", "STATUS", "DTYPES", "ORDERS",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdc.so")
# The bounds-checked test build, loaded instead when DC_LIBRARY=bounds.
LIB_BOUNDS_PATH = os.path.join(_HERE, "libdc_bounds.so")

STATUS = {0: "DC_OK", 1: "DC_ERR_INVALID", 2: "DC_ERR_ALIGN", 3: "DC_ERR_OVERLAP",
          4: "DC_ERR_TOO_MANY", 5: "DC_ERR_CUDA", 6: "DC_ERR_TIMEOUT", 7: "DC_ERR_BOUNDS"}

MAX_RANKS = 64
MANY_MAX_TENSORS = 256
MANY_MAX_SEGMENTS = 1024
MANY_MAX_REDUCE_JOBS = 256
MANY_MAX_REDUCE_PTRS = 1024
MAX_DELAY_NS = 1_000_000_000

DTYPES = {"bf16": 0, "f16": 1, "f32": 2}      # dc_dtype_t
ORDERS = {"linear": 0, "tree": 1}             # dc_order_t


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
        path = LIB_BOUNDS_PATH if os.environ.get("DC_LIBRARY") == "bounds" else LIB_PATH
        if not os.path.exists(path):
            raise LibraryMissing(
                f"{path} is missing: build it with `python -m reduce_copy_rank_gb300._build` "
                "(--bounds for the checked build, or __graft_entry__.build()); there is no fallback path")
        L = ctypes.CDLL(path)
        A, I, Z = _VP, ctypes.c_int, ctypes.c_size_t  # A: address of a host array
        L.dc_all_gather.argtypes = [A, I, Z, _VP, _VP]
        L.dc_all_gather_many.argtypes = [A, A, A, I, I, _VP]
        L.dc_all_reduce_bf16.argtypes = [A, A, I, Z, _VP]
        L.dc_reduce_scatter_bf16.argtypes = [A, A, I, Z, _VP]
        L.dc_all_reduce.argtypes = [A, A, I, Z, I, I, _VP]
        L.dc_reduce_scatter.argtypes = L.dc_all_reduce.argtypes
        L.dc_reduce.argtypes = [A, I, Z, Z, _VP, I, I, _VP]
        L.dc_all_reduce_many.argtypes = [A, A, A, I, I, I, I, _VP]
        L.dc_reduce_scatter_many.argtypes = L.dc_all_reduce_many.argtypes
        L.dc_inject_delay_ns.argtypes = [ctypes.c_ulonglong, _VP]
        L.dc_check_device.argtypes = []
        L.dc_fused_workspace_bytes.argtypes = [I]
        L.dc_fused_workspace_bytes.restype = Z
        L.dc_fused_all_gather.argtypes = [A, A, A, I, Z, _VP, ctypes.c_uint, _VP]
        L.dc_fused_reset.argtypes = [_VP, I, _VP]
        L.dc_fused_all_gather_static.argtypes = [A, A, I, Z, _VP]
        for f in ("dc_all_gather", "dc_all_gather_many", "dc_all_reduce_bf16",
                  "dc_reduce_scatter_bf16", "dc_all_reduce", "dc_reduce_scatter", "dc_reduce",
                  "dc_all_reduce_many", "dc_reduce_scatter_many", "dc_inject_delay_ns",
                  "dc_check_device", "dc_fused_all_gather", "dc_fused_reset",
                  "dc_fused_all_gather_static"):
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
        L.dc_last_grid.argtypes = []
        L.dc_last_grid.restype = ctypes.c_int
        L.dc_version.argtypes = []
        L.dc_version.restype = ctypes.c_int
        L.dc_bounds_checked.argtypes = []
        L.dc_bounds_checked.restype = ctypes.c_int
        _lib = L
    return _lib


def _check(status: int) -> None:
    if status != 0:
        raise DCError(status, lib().dc_last_error().decode(errors="replace"))


# Host arrays of pointers and sizes are built as array("Q") (64-bit values;
# size_t and pointers are 64 bits on the supported platforms) and passed by
# address; the caller keeps the array object alive for the call.
assert ctypes.sizeof(ctypes.c_size_t) == 8 and ctypes.sizeof(ctypes.c_void_p) == 8
assert array.array("Q").itemsize == 8


def _u64(xs: Sequence[int]) -> array.array:
    return array.array("Q", xs) if len(xs) else array.array("Q", (0,))


def _addr(a: array.array) -> int:
    return a.buffer_info()[0]


# ------------------------------------------------------------ raw (C ABI) ---
# Same names and arguments as include/dc.h; pointers are ints, the stream is a
# cudaStream_t handle as an int (0 = legacy default stream).  They return the
# status instead of raising, like the C functions.

def dc_all_gather(peer_ptrs: Sequence[int], P: int, bytes_per_rank: int, out: int,
                  stream: int = 0) -> int:
    a = _u64(peer_ptrs)
    return lib().dc_all_gather(_addr(a), P, bytes_per_rank, out, stream)


def dc_all_gather_many(peer_ptrs: Sequence[int], bytes_per_rank: Sequence[int],
                       outs: Sequence[int], T: int, P: int, stream: int = 0) -> int:
    a, b, c = _u64(peer_ptrs), _u64(bytes_per_rank), _u64(outs)
    return lib().dc_all_gather_many(_addr(a), _addr(b), _addr(c), T, P, stream)


def dc_all_reduce_bf16(in_ptrs: Sequence[int], out_ptrs: Sequence[int], P: int, count: int,
                       stream: int = 0) -> int:
    a, b = _u64(in_ptrs), _u64(out_ptrs)
    return lib().dc_all_reduce_bf16(_addr(a), _addr(b), P, count, stream)


def dc_reduce_scatter_bf16(in_ptrs: Sequence[int], out_ptrs: Sequence[int], P: int,
                           count_per_shard: int, stream: int = 0) -> int:
    a, b = _u64(in_ptrs), _u64(out_ptrs)
    return lib().dc_reduce_scatter_bf16(_addr(a), _addr(b), P, count_per_shard, stream)


def dc_all_reduce(in_ptrs: Sequence[int], out_ptrs: Sequence[int], P: int, count: int,
                  dtype: int = 0, order: int = 0, stream: int = 0) -> int:
    a, b = _u64(in_ptrs), _u64(out_ptrs)
    return lib().dc_all_reduce(_addr(a), _addr(b), P, count, dtype, order, stream)


def dc_reduce_scatter(in_ptrs: Sequence[int], out_ptrs: Sequence[int], P: int,
                      count_per_shard: int, dtype: int = 0, order: int = 0, stream: int = 0) -> int:
    a, b = _u64(in_ptrs), _u64(out_ptrs)
    return lib().dc_reduce_scatter(_addr(a), _addr(b), P, count_per_shard, dtype, order, stream)


def dc_reduce(in_ptrs: Sequence[int], P: int, in_offset: int, count: int, out: int,
              dtype: int = 0, order: int = 0, stream: int = 0) -> int:
    a = _u64(in_ptrs)
    return lib().dc_reduce(_addr(a), P, in_offset, count, out, dtype, order, stream)


def dc_all_reduce_many(in_ptrs: Sequence[int], out_ptrs: Sequence[int], counts: Sequence[int],
                       T: int, P: int, dtype: int = 0, order: int = 0, stream: int = 0) -> int:
    a, b, c = _u64(in_ptrs), _u64(out_ptrs), _u64(counts)
    return lib().dc_all_reduce_many(_addr(a), _addr(b), _addr(c), T, P, dtype, order, stream)


def dc_reduce_scatter_many(in_ptrs: Sequence[int], out_ptrs: Sequence[int],
                           counts_per_shard: Sequence[int], T: int, P: int, dtype: int = 0,
                           order: int = 0, stream: int = 0) -> int:
    a, b, c = _u64(in_ptrs), _u64(out_ptrs), _u64(counts_per_shard)
    return lib().dc_reduce_scatter_many(_addr(a), _addr(b), _addr(c), T, P, dtype, order, stream)


def dc_inject_delay_ns(ns: int, stream: int = 0) -> int:
    return lib().dc_inject_delay_ns(int(ns), stream)


def dc_check_device() -> int:
    return lib().dc_check_device()


def dc_fused_workspace_bytes(P: int) -> int:
    return int(lib().dc_fused_workspace_bytes(P))


def dc_fused_all_gather(in_ptrs: Sequence[int], staging: Sequence[int], outs: Sequence[int], P: int,
                        bytes_per_rank: int, workspace: int, epoch: int, stream: int = 0) -> int:
    a, b, c = _u64(in_ptrs), _u64(staging), _u64(outs)
    return lib().dc_fused_all_gather(_addr(a), _addr(b), _addr(c), P, bytes_per_rank, workspace, epoch,
                                     stream)


def dc_fused_reset(workspace: int, P: int, stream: int = 0) -> int:
    return lib().dc_fused_reset(workspace, P, stream)


def dc_fused_all_gather_static(in_ptrs: Sequence[int], outs: Sequence[int], P: int, bytes_per_rank: int,
                               stream: int = 0) -> int:
    """dc_fused_all_gather for callers that cannot allocate device memory:
    its flags and staging buffers live in the library's static scratch
    (P * bytes_per_rank rounded up to 256 bytes per rank, 16 MiB at most);
    calls that overlap on the GPU race."""
    a, b = _u64(in_ptrs), _u64(outs)
    return lib().dc_fused_all_gather_static(_addr(a), _addr(b), P, bytes_per_rank, stream)


# ---------------------------------------------------------- tensor API ---

_raw_stream = None


def _stream_handle(stream) -> int:
    """cudaStream_t of `stream` (None: torch's current stream on the current
    device), read through torch's raw-stream accessor when it has one."""
    global _raw_stream
    if stream is None:
        import torch

        if _raw_stream is None:
            f = getattr(torch._C, "_cuda_getCurrentRawStream", None)
            _raw_stream = (lambda: f(torch.cuda.current_device())) if f is not None else \
                (lambda: torch.cuda.current_stream().cuda_stream)
        return _raw_stream()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def _cur_dev() -> int:
    """The current CUDA device: the library launches there, so every tensor
    must live there (a pointer of another device would fault the kernel)."""
    import torch

    return torch.cuda.current_device()


def _wrong_device(what: str, t, dev: int):
    raise ValueError(f"{what} is on {t.device}, but the current device is cuda:{dev}; "
                     "make it current (torch.cuda.set_device) or move the tensor")


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
    B = peers[0].nbytes
    if not peers[0].is_cuda:
        _explain_peers(peers)
    dev = _cur_dev()
    ptrs = []
    for r, p in enumerate(peers):
        if not p.is_cuda or p.nbytes != B or not p.is_contiguous():
            _explain_peers(peers)
        if p.get_device() != dev:
            _wrong_device(f"peers[{r}]", p, dev)
        ptrs.append(p.data_ptr())
    if not out.is_cuda or not out.is_contiguous():
        _device_tensor(out, "out")
    if out.get_device() != dev:
        _wrong_device("out", out, dev)
    if out.nbytes != P * B:
        raise ValueError(f"out holds {out.nbytes} bytes, expected P * {B} = {P * B}")
    a = array.array("Q", ptrs)
    _check(lib().dc_all_gather(_addr(a), P, B, out.data_ptr(), _stream_handle(stream)))
    return out


def fused_workspace(P: int, device=None):
    """A zeroed workspace tensor for dc_fused_all_gather with P ranks
    (allocated by torch; the library itself allocates nothing)."""
    import torch

    n = dc_fused_workspace_bytes(P)
    if n == 0:
        raise ValueError(f"P = {P} is outside 1..{MAX_RANKS}")
    return torch.zeros(n, dtype=torch.uint8, device=device if device is not None else "cuda")


def fused_all_gather(inputs: Sequence, staging: Sequence, outputs: Sequence, workspace, epoch: int,
                     stream=None):
    """The staged all-gather protocol (stage -> gather -> complete) over P
    ranks on one GPU: afterwards every ``outputs[r]`` holds ``inputs[0]``,
    ``inputs[1]``, ... in rank order and ``staging[r]`` a copy of
    ``inputs[r]``.  ``epoch`` is 1 for the first call on a cleared
    ``workspace`` (see :func:`fused_workspace`) and one more for each call.
    A rank that never arrives shows up as DC_ERR_TIMEOUT from
    :func:`check_device`.  Returns ``outputs``."""
    P = len(inputs)
    if P == 0 or len(staging) != P or len(outputs) != P:
        raise ValueError("need the same number (>= 1) of inputs, staging buffers and outputs")
    B = inputs[0].nbytes
    dev = _cur_dev()
    groups = (("inputs", inputs, B), ("staging", staging, B), ("outputs", outputs, P * B))
    ptrs = {}
    for name, ts, nbytes in groups:
        for r, t in enumerate(ts):
            if not t.is_cuda or not t.is_contiguous():
                _device_tensor(t, f"{name}[{r}]")
            if t.get_device() != dev:
                _wrong_device(f"{name}[{r}]", t, dev)
            if t.nbytes != nbytes:
                raise ValueError(f"{name}[{r}] holds {t.nbytes} bytes, expected {nbytes}")
        ptrs[name] = [t.data_ptr() for t in ts]
    _device_tensor(workspace, "workspace")
    _check(dc_fused_all_gather(ptrs["inputs"], ptrs["staging"], ptrs["outputs"], P, B,
                               workspace.data_ptr(), int(epoch), _stream_handle(stream)))
    return outputs


def fused_reset(workspace, P: int, stream=None) -> None:
    """Clear a fused workspace of P ranks (the next call uses epoch 1)."""
    _check(dc_fused_reset(workspace.data_ptr(), P, _stream_handle(stream)))


def _explain_peers(peers) -> None:
    for r, p in enumerate(peers):
        _device_tensor(p, f"peers[{r}]")
    raise ValueError("all peers must have the same number of bytes")


def all_gather_many(peers_per_tensor: Sequence[Sequence], outs: Sequence, stream=None):
    """T independent all-gathers in one launch; ``outs[t]`` receives tensor
    t's P payloads in rank order (no packing across tensors).  Returns outs."""
    T = len(peers_per_tensor)
    if len(outs) != T:
        raise ValueError("need one output per tensor")
    if T == 0:
        return outs
    P = len(peers_per_tensor[0])
    dev = _cur_dev()
    ptrs, sizes = [], []
    # one pass, few property reads per tensor (they dominate the host time of
    # large batches); on any mismatch the slow checks below name the culprit
    for t, peers in enumerate(peers_per_tensor):
        if len(peers) != P:
            raise ValueError("every tensor needs the same number of peers")
        B = peers[0].nbytes
        for r, p in enumerate(peers):
            if not (p.is_cuda and p.is_contiguous()) or p.nbytes != B or p.get_device() != dev:
                _device_tensor(p, f"peers_per_tensor[{t}][{r}]")
                if p.nbytes != B:
                    raise ValueError(f"tensor {t}: all peers must have the same number of bytes")
                _wrong_device(f"peers_per_tensor[{t}][{r}]", p, dev)
            ptrs.append(p.data_ptr())
        o = outs[t]
        if not (o.is_cuda and o.is_contiguous()) or o.get_device() != dev:
            _device_tensor(o, f"outs[{t}]")
            _wrong_device(f"outs[{t}]", o, dev)
        if o.nbytes != P * B:
            raise ValueError(f"outs[{t}] holds {o.nbytes} bytes, expected {P * B}")
        sizes.append(B)
    _check(dc_all_gather_many(ptrs, sizes, [o.data_ptr() for o in outs], T, P,
                              _stream_handle(stream)))
    return outs


_dtype_codes = None


def _dtype_code(t) -> int:
    global _dtype_codes
    if _dtype_codes is None:
        import torch

        _dtype_codes = {torch.bfloat16: 0, torch.float16: 1, torch.float32: 2}
    c = _dtype_codes.get(t.dtype)
    if c is None:
        raise ValueError(f"reductions take bfloat16, float16 or float32 tensors (got {t.dtype})")
    return c


def _reduce_ptrs(ts: Sequence, what: str, count: int, dtype) -> list:
    """Data pointers of `ts` after the checks of _reduce_tensors (which runs
    only to name the offending tensor)."""
    dev = None
    ptrs = []
    for i, t in enumerate(ts):
        if not t.is_cuda or t.dtype != dtype or t.numel() != count or not t.is_contiguous():
            _reduce_tensors(ts, what, count, dtype)
        if dev is None:
            dev = _cur_dev()
        if t.get_device() != dev:
            _wrong_device(f"{what}[{i}]", t, dev)
        ptrs.append(t.data_ptr())
    return ptrs


def _reduce_tensors(ts: Sequence, what: str, count: int | None, dtype):
    for i, t in enumerate(ts):
        _device_tensor(t, f"{what}[{i}]")
        if t.dtype != dtype:
            raise ValueError(f"{what}[{i}] has dtype {t.dtype}, expected {dtype}")
        if count is not None and t.numel() != count:
            raise ValueError(f"{what}[{i}] has {t.numel()} elements, expected {count}")


def _order_code(order: str) -> int:
    if order not in ORDERS:
        raise ValueError(f"order must be one of {sorted(ORDERS)} (got {order!r})")
    return ORDERS[order]


def all_reduce(inputs: Sequence, outputs: Sequence, order: str = "linear", stream=None):
    """Deterministic all_reduce: every ``outputs[r]`` receives the sum of
    ``inputs[0..P-1]`` (bfloat16, float16 or float32), each element widened to
    binary32, added in a fixed order (``"linear"``: rank 0, 1, 2, ...;
    ``"tree"``: pairs of neighbouring ranks, then pairs of pairs) and rounded
    once to the element type.  ``outputs[r]`` may be one of the inputs (in
    place).  Returns outputs."""
    P = len(inputs)
    if P == 0 or len(outputs) != P:
        raise ValueError("need P >= 1 inputs and P outputs")
    n = inputs[0].numel()
    dt = inputs[0].dtype
    a = array.array("Q", _reduce_ptrs(inputs, "inputs", n, dt))
    b = array.array("Q", _reduce_ptrs(outputs, "outputs", n, dt))
    _check(lib().dc_all_reduce(_addr(a), _addr(b), P, n, _dtype_code(inputs[0]), _order_code(order),
                               _stream_handle(stream)))
    return outputs


def reduce_scatter(inputs: Sequence, outputs: Sequence, order: str = "linear", stream=None):
    """Deterministic reduce_scatter (input = world x output): each input holds
    P*C elements; ``outputs[r]`` (C elements) receives the fixed-order fold of
    shard r of every input.  Returns outputs."""
    P = len(inputs)
    if P == 0 or len(outputs) != P:
        raise ValueError("need P >= 1 inputs and P outputs")
    n = inputs[0].numel()
    if n % P:
        raise ValueError(f"input length {n} is not divisible by P = {P}")
    C = n // P
    dt = inputs[0].dtype
    a = array.array("Q", _reduce_ptrs(inputs, "inputs", n, dt))
    b = array.array("Q", _reduce_ptrs(outputs, "outputs", C, dt))
    _check(lib().dc_reduce_scatter(_addr(a), _addr(b), P, C, _dtype_code(inputs[0]),
                                   _order_code(order), _stream_handle(stream)))
    return outputs


def reduce(inputs: Sequence, out, offset: int = 0, order: str = "linear", stream=None):
    """One rank's share of a reduction: ``out`` (n elements) receives the
    fixed-order fold of elements ``offset .. offset+n-1`` of every input, as
    all_reduce / reduce_scatter compute them (their rank-r output, for
    offset 0 or r*n).  For a rank that is its own process and reads its peers'
    buffers.  ``out`` may be exactly that range of one input.  Returns out."""
    P = len(inputs)
    if P == 0:
        raise ValueError("need at least one input")
    dt = out.dtype
    _device_tensor(out, "out")
    n = out.numel()
    if offset < 0:
        raise ValueError(f"offset must be >= 0 (got {offset})")
    dev = _cur_dev()
    if out.get_device() != dev:
        _wrong_device("out", out, dev)
    ptrs = []
    for i, t in enumerate(inputs):
        _device_tensor(t, f"inputs[{i}]")
        if t.dtype != dt:
            raise ValueError(f"inputs[{i}] has dtype {t.dtype}, expected {dt}")
        if n and t.numel() < offset + n:  # (nothing is read when n == 0)
            raise ValueError(f"inputs[{i}] has {t.numel()} elements, fewer than offset + n = {offset + n}")
        if t.get_device() != dev:
            _wrong_device(f"inputs[{i}]", t, dev)
        ptrs.append(t.data_ptr())
    a = array.array("Q", ptrs)
    _check(lib().dc_reduce(_addr(a), P, offset, n, out.data_ptr(), _dtype_code(out), _order_code(order),
                           _stream_handle(stream)))
    return out


def _many(inputs_per_tensor, outputs_per_tensor, scatter: bool):
    T = len(inputs_per_tensor)
    if len(outputs_per_tensor) != T:
        raise ValueError("need one output list per tensor")
    if T == 0:
        return [], [], [], 0, 0
    P = len(inputs_per_tensor[0])
    dt = inputs_per_tensor[0][0].dtype
    ins, outs, counts = [], [], []
    for t, (it, ot) in enumerate(zip(inputs_per_tensor, outputs_per_tensor)):
        if len(it) != P or len(ot) != P:
            raise ValueError("every tensor needs P inputs and P outputs")
        n = it[0].numel()
        if scatter and n % P:
            raise ValueError(f"tensor {t}: input length {n} is not divisible by P = {P}")
        c = n // P if scatter else n
        ins.extend(_reduce_ptrs(it, f"inputs[{t}]", n, dt))
        outs.extend(_reduce_ptrs(ot, f"outputs[{t}]", c, dt))
        counts.append(c)
    return ins, outs, counts, T, P


def all_reduce_many(inputs_per_tensor: Sequence[Sequence], outputs_per_tensor: Sequence[Sequence],
                    order: str = "linear", stream=None):
    """T independent all_reduces (same P, element type and order) in one
    launch.  Returns outputs_per_tensor."""
    ins, outs, counts, T, P = _many(inputs_per_tensor, outputs_per_tensor, False)
    if T:
        _check(dc_all_reduce_many(ins, outs, counts, T, P, _dtype_code(inputs_per_tensor[0][0]),
                                  _order_code(order), _stream_handle(stream)))
    return outputs_per_tensor


def reduce_scatter_many(inputs_per_tensor: Sequence[Sequence],
                        outputs_per_tensor: Sequence[Sequence], order: str = "linear", stream=None):
    """T independent reduce_scatters in one launch, into caller-given
    outputs.  Returns outputs_per_tensor."""
    ins, outs, counts, T, P = _many(inputs_per_tensor, outputs_per_tensor, True)
    if T:
        _check(dc_reduce_scatter_many(ins, outs, counts, T, P, _dtype_code(inputs_per_tensor[0][0]),
                                      _order_code(order), _stream_handle(stream)))
    return outputs_per_tensor


def inject_delay(ns: int, stream=None) -> None:
    """Delay `stream` (default: the current torch stream) by `ns` nanoseconds
    of the GPU's global timer (one-thread kernel; rank-skew calibration)."""
    _check(dc_inject_delay_ns(ns, _stream_handle(stream)))


def check_device() -> None:
    """Wait for the current device, then raise DCError(DC_ERR_TIMEOUT) if a
    bounded wait in one of the library's kernels ran out since the last check
    (the fault word is cleared)."""
    _check(dc_check_device())


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


def last_grid() -> int:
    """CTAs in the grid of this thread's last launch through the library."""
    return int(lib().dc_last_grid())


def last_error() -> str:
    return lib().dc_last_error().decode(errors="replace")
