"""Seeded random reductions on the GPU against the oracle: all_reduce,
reduce_scatter, their batched forms and one rank's share (dc_reduce), over
random rank counts (1..8 and 13), element types, orders, element counts (0 to
200 000), element offsets of every input and output from a 16-byte boundary,
ranks in place, and grid / path options.  Bit exact, NaN by class; guard
bytes around every output that is not an input.

Page, by title: "perf(cuda): vectorize the deterministic all-gather copy and
right-size its single-block path" (author's replies: the reductions of the
collective; the fixed-order fold is the reading the oracle states).
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import GUARD, NP_OF, assert_typed_equal, torch_dtype, typed_bits, typed_tensor

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import reduce_copy_rank_gb300 as dc  # noqa: E402

ES = {"bf16": 2, "f16": 2, "f32": 4}
GUARD_BYTES = 64


class Slot:
    """`n` elements of `dtype` starting `off` elements past a 16-byte boundary
    inside a guarded allocation."""

    def __init__(self, n, dtype, off, fill=GUARD):
        es = ES[dtype]
        self.store = torch.full((GUARD_BYTES * 2 + 16 + (n + 8) * es,), fill, dtype=torch.uint8, device="cuda")
        self.start = GUARD_BYTES + ((-(self.store.data_ptr() + GUARD_BYTES)) % 16) + off * es
        self.nbytes = n * es
        self.view = self.store[self.start:self.start + self.nbytes].view(torch_dtype(dtype))

    def guards_intact(self):
        s = self.store.cpu().numpy()
        return bool((s[:self.start] == GUARD).all() and (s[self.start + self.nbytes:] == GUARD).all())


def random_bits(rng, n, dtype):
    if dtype == "f32":
        x = rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
        x[(x & 0x7F800000) == 0x7F800000] &= 0xBFFFFFFF  # finite, but for the injected NaN below
    else:
        x = rng.integers(0, 1 << 16, n, dtype=np.uint32).astype(np.uint16)
        e = 0x7F80 if dtype == "bf16" else 0x7C00
        x[(x & e) == e] &= 0xBFFF
    if n and rng.random() < 0.3:  # a NaN and an infinity somewhere
        nan = {"bf16": 0x7FC1, "f16": 0x7E01, "f32": 0x7FC00001}[dtype]
        inf = {"bf16": 0x7F80, "f16": 0x7C00, "f32": 0x7F800000}[dtype]
        x[int(rng.integers(0, n))] = nan
        x[int(rng.integers(0, n))] = inf
    return x


@pytest.mark.parametrize("case", range(80))
def test_random_reductions(case):
    rng = np.random.default_rng(W.seed_for(4, 9200 + case))
    op = ["all_reduce", "reduce_scatter", "all_reduce_many", "reduce_scatter_many", "reduce"][case % 5]
    dtype = str(rng.choice(["bf16", "f16", "f32"]))
    order = str(rng.choice(["linear", "tree"]))
    P = int(rng.choice([1, 2, 3, 4, 5, 6, 8, 13]))
    opts = [{}, {"grid_ctas": int(rng.integers(1, 9))}, {"reduce_staged": 0}, {"force_path": 1},
            {"prefetch": 0}][int(rng.integers(0, 5))]
    T = int(rng.integers(1, 6)) if op.endswith("_many") else 1
    scatter = op.startswith("reduce_scatter")
    counts = []
    for _ in range(T):
        c = int(rng.choice([0, 1, 7, 64, 1000, 4099, 33333, 200000]))
        counts.append(c if not scatter else max(c // P, 0))
    cols = [[random_bits(rng, counts[t] * (P if scatter else 1), dtype) for _ in range(P)] for t in range(T)]
    in_offs = [[int(x) for x in rng.integers(0, 16 // ES[dtype], P)] for _ in range(T)]
    ins = []
    for t in range(T):
        row = []
        for r in range(P):
            s = Slot(cols[t][r].size, dtype, in_offs[t][r], fill=0)
            if cols[t][r].size:
                s.view.copy_(typed_tensor(cols[t][r], dtype))
            row.append(s)
        ins.append(row)
    out_off = int(rng.integers(0, 16 // ES[dtype]))
    with dc.options(**opts):
        if op == "reduce":  # elements [offset, offset + n) of every input
            offset = int(rng.integers(0, 8))
            n = max(counts[0] - offset, 0)
            out = Slot(n, dtype, out_off)
            dc.reduce([x.view for x in ins[0]], out.view, offset=offset, order=order)
            torch.cuda.synchronize()
            if n == 0:
                assert out.guards_intact()
                return
            want = oracle.all_reduce([c[offset:offset + n] for c in cols[0]], dtype, order).view(NP_OF[dtype])
            assert_typed_equal(typed_bits(out.view, dtype), want, dtype, f"case {case} reduce")
            assert out.guards_intact()
            return
        in_place = [bool(rng.random() < 0.3) for _ in range(P)]
        outs = []
        for t in range(T):
            row = []
            for r in range(P):
                n = counts[t]
                if in_place[r] and not scatter and n:
                    row.append(None)  # in place: the output is the input
                else:
                    row.append(Slot(n, dtype, out_off))
            outs.append(row)
        out_views = [[ins[t][r].view if o is None else o.view for r, o in enumerate(outs[t])] for t in range(T)]
        in_views = [[x.view for x in ins[t]] for t in range(T)]
        if op == "all_reduce":
            dc.all_reduce(in_views[0], out_views[0], order=order)
        elif op == "reduce_scatter":
            dc.reduce_scatter(in_views[0], out_views[0], order=order)
        elif op == "all_reduce_many":
            dc.all_reduce_many(in_views, out_views, order=order)
        else:
            dc.reduce_scatter_many(in_views, out_views, order=order)
    torch.cuda.synchronize()
    for t in range(T):
        if scatter:
            want = oracle.reduce_scatter(cols[t], dtype, order) if counts[t] else [np.zeros(0)] * P
        else:
            w = oracle.all_reduce(cols[t], dtype, order) if counts[t] else np.zeros(0)
            want = [w] * P
        for r in range(P):
            got = typed_bits(out_views[t][r], dtype)
            assert_typed_equal(got, np.asarray(want[r]).view(NP_OF[dtype]) if counts[t] else got, dtype,
                               f"case {case} {op} {dtype} {order} P={P} t={t} r={r} {opts}")
            if outs[t][r] is not None:
                assert outs[t][r].guards_intact(), (case, t, r)
