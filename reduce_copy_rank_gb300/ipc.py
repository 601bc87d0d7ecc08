"""The staged collectives across processes: one process per rank, each with
its own buffers, the ranks' staging buffers shared between the processes.

Page, by title: "perf(cuda): vectorize the deterministic all-gather copy and
right-size its single-block path".  Its collective runs over CUDA IPC (the
backend id cuda_ipc_fixed_tree, in the author's replies): every rank stages
its payload in a buffer its peers have mapped, reads the peers' staged
payloads, and completes once every peer has read its buffer.  What happens
when a rank fails part-way is left open there: the review's reliability
finding notes that an interrupted staged gather leaves pending state with no
coordinated abort, and a review thread on the multi-process test notes that
peers of a failed rank block until the process-group timeout (minutes).

Here the handshakes run on the host, between the processes, and the work
runs in the library's kernels over the peers' mapped staging buffers; no
kernel ever waits for another process.  Each call (an epoch) is

  stage:    copy the local payload into the local staging buffer (the
            library's one-rank gather) and wait for the copy to finish;
  barrier:  every rank has staged this epoch (bounded by `timeout`);
  compute:  this rank's output from the P staging buffers, and wait for it:
            the rank-ordered gather (dc_all_gather; dc_all_gather_many for
            several tensors in one staging buffer), or the fixed-order fold
            of every buffer (dc_reduce) -- the whole buffer for all_reduce,
            shard r of it for rank r of reduce_scatter;
  barrier:  every rank has read every staging buffer (same bound), so the
            next epoch may overwrite them.

The barriers are either a monitored barrier of the process group
(handshake="gloo") or arrival counters in node-local shared memory
(handshake="shm": one 64-bit word per rank, polled; a few microseconds instead
of the process group's message round trips).  CUDA IPC only maps memory
between processes of one node, so the node-local handshake loses nothing
there, and it is the CUDA transport's default.  It is correct for payloads in
device memory on any host: a rank stores its counter only after its stream
synchronisation returned, so a peer that sees the counter launches its reads
after the copy finished.  (A transport whose payloads live in host memory
would need the payload's stores to become visible before the counter's,
which weakly ordered hosts do not promise: such a transport should keep the
gloo handshake.)

A barrier that runs out (a rank that never arrives, or died) raises
DCError(DC_ERR_TIMEOUT) naming the epoch and step; the collective is then
aborted: every later call raises at once, before it touches a peer's buffer.
close() drops the mappings of the peers' buffers, waits until every rank has
(within the bound), then releases the own buffer.  Signatures (operation,
world size, sizes, element type, order, transport, handshake and, for the
shared-memory handshake, the host) are compared once, when the collective is
built: a mismatch raises DCError(DC_ERR_INVALID) on every rank.

A transport provides: kind, default_handshake, alloc(nbytes) -> buffer,
export(buffer) -> descriptor (one per peer that opens it), open(descriptor)
-> the peer's buffer, opened_by_all(), stage(buffer, payload),
gather(buffers, out, nbytes), reduce(buffers, out, nbytes, offset, order),
stage_many(buffer, payloads, offsets), gather_many(buffers, outs, offsets,
sizes), close_peers(), release().  CudaIpcTransport is the product's: device buffers
shared through CUDA IPC handles, the work in dc_all_gather / dc_reduce.  The
process group must support monitored_barrier (gloo).
"""
from __future__ import annotations

import datetime
import os
import socket
import time

from . import DCError

_TIMEOUT = 6  # DC_ERR_TIMEOUT
_INVALID = 1  # DC_ERR_INVALID

# element types of the reductions and their sizes in bytes
ELEMENT_BYTES = {"bf16": 2, "f16": 2, "f32": 4}


class SharedBytes:
    """A file in node-local shared memory (/dev/shm, a tmpfs; the temporary
    directory where there is none) mapped into this process.  The creator
    names it and unlinks it; the others open it by path."""

    def __init__(self, size: int = 0, path: str | None = None):
        import mmap
        import tempfile
        import uuid

        self.owner = path is None
        if self.owner:
            d = "/dev/shm" if os.path.isdir("/dev/shm") else tempfile.gettempdir()
            path = os.path.join(d, f"dc_{uuid.uuid4().hex}")
            fd = os.open(path, os.O_CREAT | os.O_EXCL | os.O_RDWR, 0o600)
            os.ftruncate(fd, max(size, 8))
        else:
            fd = os.open(path, os.O_RDWR)
        try:
            self.size = os.fstat(fd).st_size
            self.mm = mmap.mmap(fd, self.size)
        finally:
            os.close(fd)
        self.path = path

    def array(self, dtype, count: int):
        import numpy as np

        return np.frombuffer(self.mm, dtype=dtype, count=count)

    def unlink(self) -> None:
        """Remove the name (creator only).  The mappings stay valid, so once
        every process has opened the file it is unlinked: nothing is left
        behind even if a process dies."""
        if self.owner:
            self.owner = False
            try:
                os.unlink(self.path)
            except FileNotFoundError:
                pass

    def close(self) -> None:
        try:
            self.mm.close()
        except BufferError:  # an array still views it: the mapping goes with the last one
            pass
        self.unlink()


class ShmHandshake:
    """Node-local barrier: one 64-bit arrival counter per rank in shared
    memory.  wait() stores the caller's next sequence number in its word,
    then polls until every word has reached it (spinning briefly, then
    sleeping 20 us between polls), for at most `timeout` seconds; it returns
    the ranks that had not arrived, or [] once all have.  A rank is at most
    one barrier ahead of any other, so `>=` is the arrival test."""

    kind = "shm"

    def __init__(self, group, rank: int, world: int, timeout: float):
        import numpy as np
        import torch.distributed as dist

        self.rank, self.world, self.timeout = rank, world, timeout
        self.seq = 0
        self.error = None  # set if this rank could not create or open the counters
        mem = None
        if rank == 0:
            try:
                mem = SharedBytes(8 * world)
            except OSError as e:
                self.error = e
        paths = [None] * world
        dist.all_gather_object(paths, mem.path if mem else None, group=group)
        self._mem, self.slots = mem, None
        if self._mem is None and paths[0] is not None:
            try:
                self._mem = SharedBytes(path=paths[0])
            except OSError as e:
                self.error = e
        elif paths[0] is None and self.error is None:
            self.error = RuntimeError("rank 0 could not create the arrival counters")
        if self._mem is not None:
            self.slots = self._mem.array(np.uint64, world)

    def wait(self) -> list:
        self.seq += 1
        seq = self.seq
        slots = self.slots
        slots[self.rank] = seq
        t0 = time.perf_counter()
        polls = 0
        while int(slots.min()) < seq:
            polls += 1
            if polls > 200:
                time.sleep(20e-6)
            if time.perf_counter() - t0 > self.timeout:
                return [q for q in range(self.world) if int(slots[q]) < seq]
        return []

    def opened_by_all(self) -> None:
        if self._mem is not None:
            self._mem.unlink()

    def close(self) -> None:
        if self._mem is None:
            return
        self.slots = None
        self._mem.close()
        self._mem = None


class CudaIpcTransport:
    """Device staging buffers shared between processes through CUDA IPC
    (torch's tensor sharing, torch.multiprocessing.reductions); the work is
    the library's dc_all_gather / dc_reduce over the mapped peer buffers on
    the current stream.  The processes' devices must be able to reach each
    other's memory (processes on one node)."""

    kind = "cuda-ipc"
    default_handshake = "shm"

    def __init__(self, device=None):
        import torch

        self.torch = torch
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
        self._opened = []

    def alloc(self, nbytes: int):
        return self.torch.empty(max(nbytes, 1), dtype=self.torch.uint8, device=self.device)

    def export(self, buf) -> object:
        from torch.multiprocessing.reductions import reduce_tensor

        return reduce_tensor(buf)

    def open(self, desc):
        fn, args = desc
        t = fn(*args)
        self._opened.append(t)
        return t

    def opened_by_all(self) -> None:
        pass

    def stage(self, buf, payload) -> None:
        from . import all_gather

        # a one-rank gather is a copy: the staging copy runs in the library too
        all_gather([payload.reshape(-1).view(self.torch.uint8)], buf[: payload.nbytes])
        self.torch.cuda.current_stream().synchronize()

    def gather(self, bufs, out, nbytes: int) -> None:
        from . import all_gather

        all_gather([b[:nbytes] for b in bufs], out.reshape(-1).view(self.torch.uint8))
        self.torch.cuda.current_stream().synchronize()

    def stage_many(self, buf, payloads, offsets) -> None:
        from . import all_gather_many

        # one launch: T one-rank gathers (copies) into the staging buffer
        live = [(p, o) for p, o in zip(payloads, offsets) if p.nbytes]
        if live:
            all_gather_many([[p.reshape(-1).view(self.torch.uint8)] for p, _o in live],
                            [buf[o:o + p.nbytes] for p, o in live])
        self.torch.cuda.current_stream().synchronize()

    def gather_many(self, bufs, outs, offsets, sizes) -> None:
        from . import all_gather_many

        live = [t for t, B in enumerate(sizes) if B]
        if live:
            all_gather_many([[b[offsets[t]:offsets[t] + sizes[t]] for b in bufs] for t in live],
                            [outs[t].reshape(-1).view(self.torch.uint8) for t in live])
        self.torch.cuda.current_stream().synchronize()

    def reduce(self, bufs, out, nbytes: int, offset: int, order: str) -> None:
        from . import reduce

        reduce([b[:nbytes].view(out.dtype) for b in bufs], out.reshape(-1), offset=offset, order=order)
        self.torch.cuda.current_stream().synchronize()

    def close_peers(self) -> None:
        self._opened = []
        self.torch.cuda.synchronize()

    def release(self) -> None:
        # frees this process's shared blocks once every peer has dropped them
        self.torch.cuda.ipc_collect()


class _Staged:
    """The protocol shared by the staged collectives: signature check,
    buffers and handshake at construction, stage / barrier / compute /
    barrier per call, abort and close."""

    op = ""

    def __init__(self, group, staging_bytes: int, transport, timeout: float, handshake: str | None,
                 extra: dict):
        import torch.distributed as dist

        self.dist, self.group, self.transport = dist, group, transport
        self.staging_bytes = int(staging_bytes)
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)
        self.timeout = datetime.timedelta(seconds=timeout)
        self.epoch = 0
        self.aborted = None
        self.closed = False
        # host seconds spent in each step, summed over the epochs
        self.seconds = dict.fromkeys(("stage", "stage_barrier", "compute", "complete_barrier"), 0.0)
        self.handshake = transport.default_handshake if handshake is None else handshake
        if self.handshake not in ("gloo", "shm"):
            raise ValueError(f"handshake must be 'gloo' or 'shm', not {self.handshake!r}")
        self._hs = None
        # every rank is here (bounded) before the exchanges below, which would
        # otherwise wait for a missing rank until the process group's timeout
        try:
            dist.monitored_barrier(group=group, timeout=self.timeout, wait_all_ranks=True)
        except RuntimeError as e:
            self.aborted = f"setup on rank {self.rank}: {e}"
            self.closed = True
            raise DCError(_TIMEOUT, self.aborted) from e
        sig = {"op": self.op, "world": self.world, "staging_bytes": self.staging_bytes,
               "transport": transport.kind, "handshake": self.handshake, **extra}
        if self.handshake == "shm":
            sig["host"] = socket.gethostname()
        sigs = [None] * self.world
        dist.all_gather_object(sigs, sig, group=group)
        if any(s != sig for s in sigs):
            raise DCError(_INVALID, f"ranks disagree on the collective: {sigs}")
        if self.handshake == "shm":
            self._hs = ShmHandshake(group, self.rank, self.world, timeout)
        # one descriptor per peer (CUDA IPC counts the references it hands
        # out: one export per process that opens it).  A rank that fails to
        # open the handshake's counters, allocate or export still takes part
        # in the exchange, with its error, so that every rank raises instead
        # of waiting for it.
        try:
            if self._hs is not None and self._hs.error is not None:
                raise self._hs.error
            self.local = transport.alloc(self.staging_bytes)
            mine = ("ok", [None if q == self.rank else transport.export(self.local) for q in range(self.world)])
        except Exception as e:  # reported to every rank below
            self.local = None
            mine = ("error", f"rank {self.rank}: {e!r}")
        descs = [None] * self.world
        dist.all_gather_object(descs, mine, group=group)
        failed = [d[1] for d in descs if d[0] != "ok"]
        if failed:
            self.aborted = "setup: " + "; ".join(failed)
            self._release_after_failed_setup()
            raise DCError(_INVALID, self.aborted)
        # a rank that fails to open a peer's buffer raises DC_ERR_INVALID and
        # never reaches the setup barrier: the others time out there (within
        # the bound), or fail to open its buffer once it released it; either
        # way every rank releases its buffers before it raises
        try:
            self.peers = [self.local if q == self.rank else self._open(q, descs[q][1][self.rank])
                          for q in range(self.world)]
            self._barrier("setup")
        except BaseException:
            self._release_after_failed_setup()
            raise
        # every rank has opened every shared buffer: their names can go
        self.transport.opened_by_all()
        if self._hs is not None:
            self._hs.opened_by_all()

    def _open(self, q: int, desc):
        try:
            return self.transport.open(desc)
        except Exception as e:
            self.aborted = f"setup: rank {self.rank} could not open the buffer of rank {q}: {e!r}"
            raise DCError(_INVALID, self.aborted) from e

    def _release_after_failed_setup(self) -> None:
        self.closed = True
        self.peers = []
        self.transport.close_peers()
        self.local = None
        self.transport.release()
        if self._hs is not None:
            self._hs.close()

    def _wait_all(self) -> str | None:
        """One barrier; None once every rank arrived, else what went wrong."""
        if self._hs is not None:
            missing = self._hs.wait()
            return f"ranks {missing} did not arrive within {self.timeout.total_seconds()} s" if missing else None
        try:
            self.dist.monitored_barrier(group=self.group, timeout=self.timeout, wait_all_ranks=True)
        except RuntimeError as e:
            return str(e)
        return None

    def _barrier(self, step: str) -> None:
        err = self._wait_all()
        if err is not None:
            self.aborted = f"{step} of epoch {self.epoch} on rank {self.rank}: {err}"
            raise DCError(_TIMEOUT, self.aborted)

    def _run(self, payload, out, payload_bytes: int, out_bytes: int, compute):
        """Stage, barrier, compute, barrier (the module docstring)."""
        self._check_open()
        if payload.nbytes != payload_bytes or out.nbytes != out_bytes:
            raise ValueError(f"{self.op} needs a payload of {payload_bytes} bytes and an output of "
                             f"{out_bytes} (got {payload.nbytes} and {out.nbytes})")
        self._steps(lambda: self.transport.stage(self.local, payload), compute)
        return out

    def _check_open(self) -> None:
        if self.aborted:
            raise DCError(_TIMEOUT, "the collective was aborted: " + self.aborted)
        if self.closed:
            raise ValueError("the collective is closed")

    def _steps(self, stage, compute) -> None:
        self.epoch += 1
        t0 = time.perf_counter()
        stage()
        t1 = time.perf_counter()
        self._barrier("stage")
        t2 = time.perf_counter()
        compute()
        t3 = time.perf_counter()
        self._barrier("complete")
        t4 = time.perf_counter()
        sec = self.seconds
        sec["stage"] += t1 - t0
        sec["stage_barrier"] += t2 - t1
        sec["compute"] += t3 - t2
        sec["complete_barrier"] += t4 - t3

    def close(self) -> None:
        """Drop the peers' mappings, wait (if the collective is healthy, within
        the bound) until every rank has dropped them, then release the own
        staging buffer.  Idempotent; later calls raise."""
        if self.closed:
            return
        self.closed = True
        self.peers = []
        self.transport.close_peers()
        if not self.aborted:
            err = self._wait_all()
            if err is not None:
                self.aborted = f"close on rank {self.rank}: {err}"
        self.local = None
        self.transport.release()
        if self._hs is not None:
            self._hs.close()


class StagedAllGather(_Staged):
    """Rank r's all_gather(payload, out) leaves in `out` the P ranks'
    payloads in rank order (P * nbytes bytes).  Payloads and outputs are
    contiguous buffers of the transport's kind."""

    op = "all_gather"

    def __init__(self, group, nbytes: int, transport, timeout: float = 5.0, handshake: str | None = None):
        self.nbytes = int(nbytes)
        super().__init__(group, self.nbytes, transport, timeout, handshake, {})

    def all_gather(self, payload, out):
        return self._run(payload, out, self.nbytes, self.world * self.nbytes,
                         lambda: self.transport.gather(self.peers, out, self.nbytes))


class StagedAllGatherMany(_Staged):
    """Several gathers in one epoch: rank r's all_gather_many(payloads, outs)
    leaves in outs[t] the P ranks' payloads of tensor t in rank order
    (P * sizes[t] bytes).  The T payloads share one staging buffer per rank
    (tensor t at a 256-byte aligned offset), staged by one launch, and the
    gather is one dc_all_gather_many over the mapped buffers."""

    op = "all_gather_many"

    def __init__(self, group, sizes, transport, timeout: float = 5.0, handshake: str | None = None):
        self.sizes = [int(b) for b in sizes]
        if any(b < 0 for b in self.sizes):
            raise ValueError("sizes must be >= 0")
        self.offsets, off = [], 0
        for b in self.sizes:
            self.offsets.append(off)
            off += (b + 255) // 256 * 256
        super().__init__(group, off, transport, timeout, handshake, {"sizes": self.sizes})

    def all_gather_many(self, payloads, outs):
        self._check_open()
        T = len(self.sizes)
        if len(payloads) != T or len(outs) != T:
            raise ValueError(f"{self.op} needs {T} payloads and {T} outputs")
        for t, B in enumerate(self.sizes):
            if payloads[t].nbytes != B or outs[t].nbytes != self.world * B:
                raise ValueError(f"tensor {t}: need a payload of {B} bytes and an output of {self.world * B} "
                                 f"(got {payloads[t].nbytes} and {outs[t].nbytes})")
        self._steps(lambda: self.transport.stage_many(self.local, payloads, self.offsets),
                    lambda: self.transport.gather_many(self.peers, outs, self.offsets, self.sizes))
        return outs


class StagedAllReduce(_Staged):
    """Rank r's all_reduce(payload, out): `out` (count elements of `dtype`,
    "bf16" / "f16" / "f32") receives the fixed-order fold of the P ranks'
    payloads -- bit-identical to rank r's output of dc_all_reduce over the
    same P buffers."""

    op = "all_reduce"

    def __init__(self, group, count: int, dtype: str, transport, order: str = "linear",
                 timeout: float = 5.0, handshake: str | None = None):
        if dtype not in ELEMENT_BYTES:
            raise ValueError(f"dtype must be one of {sorted(ELEMENT_BYTES)} (got {dtype!r})")
        self.count, self.dtype, self.order = int(count), dtype, order
        self.nbytes = self.count * ELEMENT_BYTES[dtype]
        super().__init__(group, self.nbytes, transport, timeout, handshake,
                         {"count": self.count, "dtype": dtype, "order": order})

    def all_reduce(self, payload, out):
        return self._run(payload, out, self.nbytes, self.nbytes,
                         lambda: self.transport.reduce(self.peers, out, self.nbytes, 0, self.order))


class StagedReduceScatter(_Staged):
    """Rank r's reduce_scatter(payload, out): the payload holds P shards of
    count_per_shard elements; `out` receives the fixed-order fold of shard r
    of every rank's payload -- bit-identical to rank r's output of
    dc_reduce_scatter."""

    op = "reduce_scatter"

    def __init__(self, group, count_per_shard: int, dtype: str, transport, order: str = "linear",
                 timeout: float = 5.0, handshake: str | None = None):
        import torch.distributed as dist

        if dtype not in ELEMENT_BYTES:
            raise ValueError(f"dtype must be one of {sorted(ELEMENT_BYTES)} (got {dtype!r})")
        self.count, self.dtype, self.order = int(count_per_shard), dtype, order
        self.shard_bytes = self.count * ELEMENT_BYTES[dtype]
        P = dist.get_world_size(group)
        super().__init__(group, P * self.shard_bytes, transport, timeout, handshake,
                         {"count_per_shard": self.count, "dtype": dtype, "order": order})

    def reduce_scatter(self, payload, out):
        return self._run(payload, out, self.world * self.shard_bytes, self.shard_bytes,
                         lambda: self.transport.reduce(self.peers, out, self.world * self.shard_bytes,
                                                       self.rank * self.count, self.order))


__all__ = ["StagedAllGather", "StagedAllGatherMany", "StagedAllReduce", "StagedReduceScatter", "CudaIpcTransport",
           "ShmHandshake", "SharedBytes", "ELEMENT_BYTES"]
