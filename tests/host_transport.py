"""A transport for the staged collectives' host protocol on machines without
a GPU (tests only): staging buffers are host memory in node-local shared
memory files, the gather is a byte copy and the reduction is the oracle's
fold.  It exercises everything of reduce_copy_rank_gb300.ipc but the device
work: signatures, descriptor exchange, handshakes, timeouts, abort, close.

Payloads are numpy arrays (bytes for the gather; 16- or 32-bit patterns for
the reductions, as the oracle takes them)."""
from __future__ import annotations

import numpy as np

import oracle
from reduce_copy_rank_gb300.ipc import SharedBytes


class HostTransport:
    kind = "host-shared-memory"
    # the shared-memory handshake needs the payload's stores visible before
    # the counter's: x86 (where these tests run) promises it, weakly ordered
    # hosts do not, so the default is the process group's barrier
    default_handshake = "gloo"

    def __init__(self, dtype: str = "u8", fail_alloc: bool = False, fail_open: bool = False):
        self.dtype = dtype
        self.fail_alloc, self.fail_open = fail_alloc, fail_open
        self._owned = []
        self._opened = []

    def alloc(self, nbytes: int):
        if self.fail_alloc:  # (tests: an allocation that fails on this rank)
            raise MemoryError("injected allocation failure")
        mem = SharedBytes(nbytes)
        self._owned.append(mem)
        return mem.array(np.uint8, nbytes), mem.path

    def export(self, buf) -> object:
        return buf[1]

    def open(self, desc):
        if self.fail_open:  # (tests: a peer buffer that cannot be mapped here)
            raise OSError("injected failure to open a peer's buffer")
        mem = SharedBytes(path=desc)
        self._opened.append(mem)
        return mem.array(np.uint8, mem.size), desc

    def opened_by_all(self) -> None:
        for mem in self._owned:
            mem.unlink()

    def stage(self, buf, payload) -> None:
        buf[0][: payload.nbytes] = np.ascontiguousarray(payload).view(np.uint8).reshape(-1)

    def gather(self, bufs, out, nbytes: int) -> None:
        for q, b in enumerate(bufs):
            out[q * nbytes:(q + 1) * nbytes] = b[0][:nbytes]

    def stage_many(self, buf, payloads, offsets) -> None:
        for p, o in zip(payloads, offsets):
            buf[0][o:o + p.nbytes] = np.ascontiguousarray(p).view(np.uint8).reshape(-1)

    def gather_many(self, bufs, outs, offsets, sizes) -> None:
        for t, (o, B) in enumerate(zip(offsets, sizes)):
            for q, b in enumerate(bufs):
                outs[t][q * B:(q + 1) * B] = b[0][o:o + B]

    def reduce(self, bufs, out, nbytes: int, offset: int, order: str) -> None:
        n = out.size
        cols = [b[0][:nbytes].view(out.dtype)[offset:offset + n] for b in bufs]
        out[:] = oracle.all_reduce(cols, self.dtype, order).view(out.dtype)

    def close_peers(self) -> None:
        for mem in self._opened:
            mem.close()
        self._opened = []

    def release(self) -> None:
        for mem in self._owned:
            mem.close()
        self._owned = []
