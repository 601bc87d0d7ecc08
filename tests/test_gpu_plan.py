"""The planner's grid choices on the GPU (dc_last_grid), next to the bits.

Tiles are sized so that every SM gets the same share of a launch: an output
too small for a full tile per resident CTA is cut into tiles of at least 512
vectors (aligned gathers) or 64 units (an all_reduce of one tensor); a
realigning gather adds one CTA for its rank-boundary vectors; a launch with no
16-byte body at all runs one CTA.  Bits are checked against torch.cat / the
oracle on every call.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import reduce_copy_rank_gb300 as dc  # noqa: E402


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _gather(P, B, io=0, oo=0):
    peers = [torch.randint(0, 256, (B + io,), dtype=torch.uint8, device="cuda")[io:] for _ in range(P)]
    out = torch.empty(P * B + oo, dtype=torch.uint8, device="cuda")[oo:]
    dc.all_gather(peers, out)
    g = dc.last_grid()
    torch.cuda.synchronize()
    assert torch.equal(out, torch.cat(peers))
    return g


def test_aligned_gather_grids():
    sms = _sms()
    assert _gather(8, 8192) == 8          # 4096 vectors in tiles of 512
    assert _gather(8, 131072) == 128      # 65536 vectors in tiles of 512
    g = _gather(8, 1 << 20)               # one round over every SM
    assert sms <= g <= 4 * sms
    assert _gather(2, 1024) == 1          # one tile of the grid kernel


def test_unaligned_gather_grids():
    sms = _sms()
    assert _gather(8, 100, io=1) == 1     # under 128 B per rank: one CTA, bytes
    g = _gather(8, (1 << 20) + 1, io=1, oo=3)
    assert 2 <= g <= 3 * sms              # tiles plus the boundary CTA, a slot kept free


@pytest.mark.parametrize("n", [2, 4, 7])
def test_realigned_all_reduce_without_body_runs_one_cta(n):
    """An all_reduce of one tensor with inputs at other offsets than the
    outputs but too short for one 16-byte unit: the staged kernel's tile
    count is zero and the launch is one CTA (scalar head and tail only)."""
    P = 2
    cols = [W.normal_bf16(W.seed_for(4, 9998), r, n) for r in range(P)]
    store = [torch.empty(n + 16, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    ins = []
    for r, c in enumerate(cols):
        off = ((-store[r].data_ptr()) % 16) // 2 + r  # rank 1 one element off
        v = store[r][off:off + n]
        v.copy_(torch.from_numpy(c.view(np.int16)).cuda().view(torch.bfloat16))
        ins.append(v)
    outs = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    dc.all_reduce(ins, outs)
    assert dc.last_grid() == 1
    torch.cuda.synchronize()
    want = np.asarray(oracle.all_reduce(cols, "bf16", "linear")).view(np.uint16)
    for r in range(P):
        assert np.array_equal(outs[r].view(torch.int16).cpu().numpy().view(np.uint16), want)


def test_small_all_reduce_reaches_every_sm():
    sms = _sms()
    P, n = 8, 131072  # 16384 units: tiles of >= 64 units over the SMs
    ins = [torch.randn(n, device="cuda").bfloat16() for _ in range(P)]
    outs = [torch.empty_like(x) for x in ins]
    dc.all_reduce(ins, outs)
    g = dc.last_grid()
    assert sms // 2 <= g <= 2 * sms
    torch.cuda.synchronize()
    acc = ins[0].float()
    for x in ins[1:]:
        acc = acc + x.float()
    assert torch.equal(outs[3].view(torch.int16), acc.bfloat16().view(torch.int16))
