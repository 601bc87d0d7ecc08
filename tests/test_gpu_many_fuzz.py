"""Seeded random batches for all_gather_many on the GPU, against the oracle:
the planner's every branch (one CTA, the general path, the split launch with
its aligned part in runs or round robin, the unaligned part on the ring or
across warps with its boundary CTAs, the small-job part) over random table
sizes, payload sizes from 0 B to 300 KiB, offsets 0..15 bytes, rank counts and
grid limits.  Every output byte and the guard bytes around every output are
checked.

Page, by title: "perf(cuda): vectorize the deterministic all-gather copy and
right-size its single-block path" (the author's reply on all_gather_many:
several gathers, one handshake, no packing).
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import Placed

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import reduce_copy_rank_gb300 as dc  # noqa: E402

SIZE_CLASSES = [(0, 1), (1, 16), (16, 128), (128, 4096), (4096, 70000), (70000, 300000)]


def random_batch(rng):
    P = int(rng.choice([1, 2, 3, 4, 5, 8]))
    T = int(rng.integers(1, min(200, 1024 // P) + 1))
    weights = rng.dirichlet(np.ones(len(SIZE_CLASSES)))
    sizes, in_offs, out_offs = [], [], []
    aligned_share = float(rng.random())
    for _ in range(T):
        lo, hi = SIZE_CLASSES[int(rng.choice(len(SIZE_CLASSES), p=weights))]
        B = int(rng.integers(lo, hi))
        if rng.random() < aligned_share:
            B = (B + 15) // 16 * 16
            in_offs.append([0] * P)
            out_offs.append(0)
        else:
            in_offs.append([int(x) for x in rng.integers(0, 16, P)])
            out_offs.append(int(rng.integers(0, 16)))
        sizes.append(B)
    return P, sizes, in_offs, out_offs


@pytest.mark.parametrize("case", range(120))
def test_random_batches(case):
    rng = np.random.default_rng(W.seed_for(5, 9100 + case))
    P, sizes, in_offs, out_offs = random_batch(rng)
    opts = [{}, {"grid_ctas": int(rng.integers(1, 12))}, {"gather_realign_warp": 0},
            {"gather_many_single_max_bytes": 0}, {"grid_ctas": 5000}][case % 5]
    tensors = [[rng.integers(0, 256, B, dtype=np.uint8) for _ in range(P)] for B in sizes]
    srcs, outs, ptrs = [], [], []
    for t, B in enumerate(sizes):
        for r in range(P):
            s = Placed(B, in_offs[t][r])
            s.write(tensors[t][r])
            srcs.append(s)
            ptrs.append(s.ptr())
        outs.append(Placed(P * B, out_offs[t]))
    with dc.options(**opts):
        st = dc.dc_all_gather_many(ptrs, sizes, [o.ptr() for o in outs], len(sizes), P,
                                   torch.cuda.current_stream().cuda_stream)
    assert st == 0, dc.last_error()
    torch.cuda.synchronize()
    want = oracle.all_gather_many(tensors)
    for t in range(len(sizes)):
        assert np.array_equal(outs[t].read(), want[t]), (case, t, sizes[t], P, opts)
        assert outs[t].guards_intact(), (case, t)
