"""The allocation-free fused all-gather (dc_fused_all_gather_static), for
callers that are handed only their input and output buffers and may not call
cudaMalloc themselves (a plug-in inside a framework that owns all device
memory, code whose memory was planned up front, code that must not let an
allocation synchronise the device).  It keeps its flags and staging buffers in
the library's static device scratch.

Checked through the C ABI against the allocating entry point
(dc_fused_all_gather with a caller-allocated workspace and staging buffers),
byte for byte, on two calls in a row; the size limit of the static scratch is
checked as well.  This file is named so that pytest collects it last.
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

OK, INVALID = 0, 1
STATIC_STAGING_BYTES = 16 << 20


def test_static_scratch_matches_the_allocating_entry_point_two_calls_in_a_row():
    assert dc.dc_check_device() == OK, dc.last_error()
    P, B = 8, (256 << 10) + 16
    stream = torch.cuda.current_stream().cuda_stream
    ins = [torch.empty(B, dtype=torch.uint8, device="cuda") for _ in range(P)]
    outs_static = [torch.full((P * B,), 0xA5, dtype=torch.uint8, device="cuda") for _ in range(P)]
    outs_ref = [torch.full((P * B,), 0x5A, dtype=torch.uint8, device="cuda") for _ in range(P)]
    staging = [torch.empty(B, dtype=torch.uint8, device="cuda") for _ in range(P)]
    ws = torch.zeros(dc.dc_fused_workspace_bytes(P), dtype=torch.uint8, device="cuda")
    for call in (1, 2):
        host = [W.random_bytes(W.seed_for(2, 990 + call), r, B) for r in range(P)]
        for t, h in zip(ins, host):
            t.copy_(torch.from_numpy(h))
        st = dc.dc_fused_all_gather_static([t.data_ptr() for t in ins], [o.data_ptr() for o in outs_static],
                                           P, B, stream)
        assert st == OK, dc.last_error()
        st = dc.dc_fused_all_gather([t.data_ptr() for t in ins], [s.data_ptr() for s in staging],
                                    [o.data_ptr() for o in outs_ref], P, B, ws.data_ptr(), call, stream)
        assert st == OK, dc.last_error()
        torch.cuda.synchronize()
        assert dc.dc_check_device() == OK, dc.last_error()
        want = oracle.all_gather(host)
        for r in range(P):
            got = outs_static[r].cpu().numpy()
            assert np.array_equal(got, outs_ref[r].cpu().numpy()), (call, r)
            assert np.array_equal(got, want), (call, r)


def test_static_scratch_rejects_calls_beyond_its_size():
    stream = torch.cuda.current_stream().cuda_stream
    P = 8
    B = STATIC_STAGING_BYTES // P + 16  # one rank's buffer too many bytes
    x = torch.empty(16, dtype=torch.uint8, device="cuda")
    before = dc.launch_count()
    st = dc.dc_fused_all_gather_static([x.data_ptr()] * P, [x.data_ptr() + 4096 * (r + 1) for r in range(P)],
                                       P, B, stream)
    assert st == INVALID
    assert "static scratch" in dc.last_error()
    assert dc.launch_count() == before
