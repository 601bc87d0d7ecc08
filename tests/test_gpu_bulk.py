"""GPU parity of the TMA-engine all-gather (1-D bulk copies through a ring of
shared-memory stages) against the oracle, bit exact, and its bounded waits.

The bulk path takes the 16-byte aligned dc_all_gather calls when the
gather_bulk option is on (it is off by default: measured, it only wins back
to back at outputs of 32 MiB and more).  Covered here: the
aligned sweep at full size (P=8 and P=2, 1 KiB .. 4 MiB per rank); chunk,
stage and grid settings that put many chunks on each CTA (one stage, two
stages, deep rings, one CTA for the whole output), chunks that cross rank
boundaries or hold many ranks, P = 1 and P = 64, guard bytes around every
output; and a wait that is made to run out (the test option announces 16
bytes more than the loads bring), which must come back as DC_ERR_TIMEOUT from
dc_check_device and leave the context usable.

Page, by title: "perf(cuda): vectorize the deterministic all-gather copy and
right-size its single-block path" (section "What": a pure rank-ordered copy,
byte-identical; one flat copy across all ranks when everything is aligned).
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

TIMEOUT = 6


def gather_placed(peers_np, **opts):
    P, B = len(peers_np), peers_np[0].size
    srcs = []
    for r in range(P):
        s = Placed(B, 0)
        s.write(peers_np[r])
        srcs.append(s)
    out = Placed(P * B, 0)
    with dc.options(**opts):
        st = dc.dc_all_gather([s.ptr() for s in srcs], P, B, out.ptr(),
                              torch.cuda.current_stream().cuda_stream)
        grid = dc.last_grid()
    assert st == 0, dc.last_error()
    torch.cuda.synchronize()
    return out.read(), out.guards_intact(), grid


@pytest.fixture(autouse=True)
def bulk_path_and_clean_fault_word():
    """Every test here runs with the bulk path switched on (it is opt-in) and
    starts and ends with a clean device fault word."""
    assert dc.dc_check_device() == 0, dc.last_error()
    with dc.options(gather_bulk=1):
        yield
    assert dc.dc_check_device() == 0, dc.last_error()


@pytest.mark.parametrize("case", W.config2_cases(), ids=lambda c: f"P{c.P}-{c.bytes_per_rank}")
def test_bulk_config2_sweep(case):
    peers = [W.random_bf16_patterns(case.seed, r, case.bytes_per_rank // 2).view(np.uint8)
             for r in range(case.P)]
    want = oracle.all_gather(peers)
    got, guards, grid = gather_placed(peers, gather_bulk=1)
    assert np.array_equal(got, want)
    assert guards
    assert grid >= 1


RINGS = [
    {},
    {"bulk_chunk_bytes": 256, "bulk_stages": 1},
    {"bulk_chunk_bytes": 256, "bulk_stages": 2},
    {"bulk_chunk_bytes": 1024, "bulk_stages": 3, "bulk_ctas_per_sm": 1},
    {"bulk_chunk_bytes": 4096, "bulk_stages": 32},
    {"bulk_chunk_bytes": 65536, "bulk_stages": 3},
    {"bulk_chunk_bytes": 16, "bulk_chunk_min": 16, "bulk_stages": 5},
    {"grid_ctas": 1, "bulk_chunk_bytes": 2048, "bulk_stages": 4},
    {"grid_ctas": 7, "bulk_chunk_bytes": 48, "bulk_stages": 2},
    {"pdl": 0, "prefetch": 0},
]

SIZES = [(1, 16), (2, 16), (3, 48), (8, 1024), (5, 1040), (8, 65552), (2, 3 * 65536 + 48), (64, 4096),
         (8, 1 << 20)]


@pytest.mark.parametrize("ring", RINGS, ids=lambda o: ",".join(f"{k}={v}" for k, v in o.items()) or "default")
def test_bulk_rings_and_rank_crossings(ring):
    seed = W.seed_for(2, 900)
    for P, B in SIZES:
        peers = [W.random_bytes(seed, r, B, tensor=B) for r in range(P)]
        got, guards, _ = gather_placed(peers, gather_bulk=1, **ring)
        assert np.array_equal(got, oracle.all_gather(peers)), (P, B, ring)
        assert guards, (P, B, ring)


def test_bulk_large_output_many_rounds():
    """8 x (32 MiB + 16 B): several rounds of full chunks on every CTA; the
    chunks do not divide the rank size, so many cross a rank boundary."""
    P, B = 8, (32 << 20) + 16
    gen = torch.Generator(device="cuda").manual_seed(W.seed_for(2, 901))
    peers = [torch.randint(0, 256, (B,), dtype=torch.uint8, device="cuda", generator=gen) for _ in range(P)]
    out = torch.empty(P * B + 32, dtype=torch.uint8, device="cuda").fill_(0xA5)
    with dc.options(gather_bulk=1):
        dc.all_gather(peers, out[16:16 + P * B])
    torch.cuda.synchronize()
    assert torch.equal(out[16:16 + P * B], torch.cat(peers))
    assert bool((out[:16] == 0xA5).all()) and bool((out[16 + P * B:] == 0xA5).all())


def test_bulk_repeatable_across_plans():
    seed = W.seed_for(2, 902)
    P, B = 8, 3 * 65536 + 16
    peers = [W.random_bytes(seed, r, B) for r in range(P)]
    want = oracle.all_gather(peers)
    for opts in ({}, {"bulk_ctas_per_sm": 1}, {"bulk_ctas_per_sm": 4, "bulk_stages": 2},
                 {"bulk_chunk_bytes": 32768}, {"bulk_prefetch": 0}, {"bulk_prefetch": 64},
                 {"gather_bulk": 0}):
        got, guards, _ = gather_placed(peers, **opts)
        assert np.array_equal(got, want), opts
        assert guards


def test_bounded_wait_runs_out_and_the_context_survives():
    """Every CTA's first wait is made to run out (16 bytes announced that no
    copy brings): the kernel gives up after wait_limit_ns, records the fault
    and returns; dc_check_device reports DC_ERR_TIMEOUT once and clears it;
    the next call on the same context is correct."""
    seed = W.seed_for(2, 903)
    P, B = 8, 1 << 16
    peers = [W.random_bytes(seed, r, B) for r in range(P)]
    with dc.options(test_bulk_short_tx=1, wait_limit_ns=2_000_000):
        gather_placed(peers, gather_bulk=1)
        assert dc.dc_check_device() == TIMEOUT
        assert "gave up" in dc.last_error()
    assert dc.dc_check_device() == 0
    got, guards, _ = gather_placed(peers, gather_bulk=1)
    assert np.array_equal(got, oracle.all_gather(peers))
    assert guards
    with pytest.raises(dc.DCError):
        with dc.options(test_bulk_short_tx=1, wait_limit_ns=1_000_000):
            gather_placed(peers, gather_bulk=1, bulk_chunk_bytes=4096, bulk_stages=3)
            dc.check_device()
