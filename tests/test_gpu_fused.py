"""GPU tests of the staged all-gather protocol (stage -> gather -> complete)
with the P ranks as CTA groups of one cooperative launch: every rank's
output against the oracle, bit exact, over consecutive epochs; and a rank
that never arrives, whose peers must give up within the wait bound, report
DC_ERR_TIMEOUT through dc_check_device, and leave a context that a cleared
workspace makes usable again.

Page, by title: "perf(cuda): vectorize the deterministic all-gather copy and
right-size its single-block path" (author's replies: the fused protocol of
the cuda_ipc_fixed_tree backend; section "Not in this PR" and the review
threads: no abort path for a pending protocol, peers of a dead rank wait
until the process-group timeout).
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

TIMEOUT = 6


@pytest.fixture(autouse=True)
def clean_fault_word():
    assert dc.dc_check_device() == 0, dc.last_error()
    yield
    assert dc.dc_check_device() == 0, dc.last_error()


def buffers(P, B):
    ins = [torch.empty(B, dtype=torch.uint8, device="cuda") for _ in range(P)]
    stg = [torch.full((B,), 0xA5, dtype=torch.uint8, device="cuda") for _ in range(P)]
    outs = [torch.full((P * B,), 0xA5, dtype=torch.uint8, device="cuda") for _ in range(P)]
    return ins, stg, outs


def fill(ins, seed):
    host = [W.random_bytes(seed, r, ins[r].numel()) for r in range(len(ins))]
    for t, h in zip(ins, host):
        t.copy_(torch.from_numpy(h))
    return host


def check(host, stg, outs):
    want = oracle.all_gather(host)
    for r, (s, o) in enumerate(zip(stg, outs)):
        assert np.array_equal(o.cpu().numpy(), want), f"output of rank {r}"
        assert np.array_equal(s.cpu().numpy(), host[r]), f"staging buffer of rank {r}"


@pytest.mark.parametrize("P,B,opts", [
    (1, 16, {}), (2, 1024, {}), (3, 4096 + 48, {"fused_chunk_min": 256}), (8, 1 << 20, {}),
    (8, 4 << 20, {}), (8, 65536 + 16, {"fused_chunk_min": 16}), (64, 4096, {"fused_chunk_min": 64}),
    (5, 3 * 65536, {"fused_chunk_min": 1 << 30})],
    ids=lambda v: str(v) if not isinstance(v, dict) else (",".join(f"{k}={x}" for k, x in v.items()) or "default"))
def test_fused_parity_over_epochs(P, B, opts):
    ins, stg, outs = buffers(P, B)
    ws = dc.fused_workspace(P)
    with dc.options(**opts):
        for epoch in (1, 2, 3):
            host = fill(ins, W.seed_for(2, 950 + epoch))
            dc.fused_all_gather(ins, stg, outs, ws, epoch)
            torch.cuda.synchronize()
            check(host, stg, outs)


def test_fused_rank_that_never_arrives():
    """Rank 3 of 8 never arrives: the others give up after wait_limit_ns (2
    ms here, not minutes), dc_check_device names a waiting rank and rank 3;
    after dc_fused_reset the same buffers work again from epoch 1."""
    P, B = 8, 1 << 18
    ins, stg, outs = buffers(P, B)
    ws = dc.fused_workspace(P)
    host = fill(ins, W.seed_for(2, 960))
    dc.fused_all_gather(ins, stg, outs, ws, 1)
    torch.cuda.synchronize()
    check(host, stg, outs)
    with dc.options(test_fused_absent_ranks=1 << 3, wait_limit_ns=2_000_000):
        fill(ins, W.seed_for(2, 961))
        dc.fused_all_gather(ins, stg, outs, ws, 2)
        assert dc.dc_check_device() == TIMEOUT
        msg = dc.last_error()
        assert "waiting for rank 3's staged flag" in msg and "epoch 2" in msg, msg
    assert dc.dc_check_device() == 0  # reported once
    dc.fused_reset(ws, P)
    for epoch in (1, 2):
        host = fill(ins, W.seed_for(2, 962 + epoch))
        dc.fused_all_gather(ins, stg, outs, ws, epoch)
        torch.cuda.synchronize()
        check(host, stg, outs)


def test_fused_every_rank_absent_but_one():
    P, B = 4, 4096
    ins, stg, outs = buffers(P, B)
    ws = dc.fused_workspace(P)
    fill(ins, W.seed_for(2, 970))
    with dc.options(test_fused_absent_ranks=0b1110, wait_limit_ns=1_000_000):
        dc.fused_all_gather(ins, stg, outs, ws, 1)
        with pytest.raises(dc.DCError) as e:
            dc.check_device()
        assert e.value.status == TIMEOUT
    dc.fused_reset(ws, P)
    host = fill(ins, W.seed_for(2, 971))
    dc.fused_all_gather(ins, stg, outs, ws, 1)
    torch.cuda.synchronize()
    check(host, stg, outs)


def test_fused_is_one_launch():
    P, B = 8, 65536
    ins, stg, outs = buffers(P, B)
    ws = dc.fused_workspace(P)
    fill(ins, W.seed_for(2, 980))
    before = dc.launch_count()
    dc.fused_all_gather(ins, stg, outs, ws, 1)
    assert dc.launch_count() - before == 1
    torch.cuda.synchronize()
