"""GPU parity of the rank-ordered all-gather against the oracle (bit exact).

Covers the single-CTA workload (P=2, 1 KiB per rank), the aligned sweep
(P=8 and P=2, 1 KiB .. 4 MiB per rank, full size), all 336 misaligned / odd
cases (P in {2,3,8}, odd sizes up to 1 MiB+1, input and output offsets in
{0,1,8,15}), exhaustive small cases, independent per-rank offsets, guard
bytes around every output, path and grid independence and repeatability.

Page, by title: "perf(cuda): vectorize the deterministic all-gather copy and
right-size its single-block path" (section "What": a pure rank-ordered copy,
byte-identical; section "Tests": sizes across the threshold, odd tails,
misaligned input and output).
"""
from __future__ import annotations

import hashlib

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


def run_gather(peers_np, in_offsets, out_offset, **opts):
    """Place the payloads and the output at the given byte offsets, run the
    library's all-gather, return (output bytes, guards intact)."""
    P = len(peers_np)
    B = peers_np[0].size
    srcs = []
    for r in range(P):
        s = Placed(B, in_offsets[r])
        s.write(peers_np[r])
        srcs.append(s)
    out = Placed(P * B, out_offset)
    with dc.options(**opts):
        st = dc.dc_all_gather([s.ptr() for s in srcs], P, B, out.ptr(),
                              torch.cuda.current_stream().cuda_stream)
    assert st == 0, dc.last_error()
    torch.cuda.synchronize()
    return out.read(), out.guards_intact()


def test_config1_single_cta_workload():
    c = W.CONFIG1
    seed = W.seed_for(1, 0)
    peers = [W.random_bf16_patterns(seed, r, c["bytes_per_rank"] // 2).view(np.uint8)
             for r in range(c["P"])]
    want = oracle.all_gather(peers)
    for opts in ({}, {"force_path": 1}, {"force_path": 2}):
        got, guards = run_gather(peers, [0] * c["P"], 0, **opts)
        assert np.array_equal(got, want), opts
        assert guards


@pytest.mark.parametrize("case", W.config2_cases(), ids=lambda c: f"P{c.P}-{c.bytes_per_rank}")
def test_config2_aligned_sweep(case):
    peers = [W.random_bf16_patterns(case.seed, r, case.bytes_per_rank // 2).view(np.uint8)
             for r in range(case.P)]
    want = oracle.all_gather(peers)
    for opts in ({}, {"gather_staged": 0}, {"gather_bulk": 1}):
        got, guards = run_gather(peers, [0] * case.P, 0, **opts)
        assert np.array_equal(got, want), opts
        assert guards


def _config3_by_size():
    groups = {}
    for c in W.config3_cases():
        groups.setdefault((c.P, c.bytes_per_rank), []).append(c)
    return sorted(groups.items())


@pytest.mark.parametrize("key_cases", _config3_by_size(), ids=lambda kc: f"P{kc[0][0]}-B{kc[0][1]}")
def test_config3_misaligned_odd(key_cases):
    (P, B), cases = key_cases
    for c in cases:  # the 16 offset pairs of this (P, B)
        peers = [W.random_bytes(c.seed, r, B) for r in range(P)]
        want = oracle.all_gather(peers)
        got, guards = run_gather(peers, [c.in_offset] * P, c.out_offset)
        assert np.array_equal(got, want), (P, B, c.in_offset, c.out_offset)
        assert guards, (P, B, c.in_offset, c.out_offset)


def _batched_cases(cases, make_peers):
    """Run many small gathers back to back on the stream, then check all of
    them after one synchronisation."""
    pending = []
    stream = torch.cuda.current_stream().cuda_stream
    for (P, B, in_offs, out_off) in cases:
        peers = make_peers(P, B)
        srcs = []
        for r in range(P):
            s = Placed(B, in_offs[r])
            s.write(peers[r])
            srcs.append(s)
        out = Placed(P * B, out_off)
        st = dc.dc_all_gather([s.ptr() for s in srcs], P, B, out.ptr(), stream)
        assert st == 0, dc.last_error()
        pending.append((P, B, in_offs, out_off, peers, srcs, out))
    torch.cuda.synchronize()
    for (P, B, in_offs, out_off, peers, _srcs, out) in pending:
        want = oracle.all_gather(peers)
        got = out.read()
        assert np.array_equal(got, want), (P, B, in_offs, out_off)
        assert out.guards_intact(), (P, B, in_offs, out_off)


def test_tiny_exhaustive_byte_path():
    """P in {1,2,3}, every B in 0..48, every output offset 0..15, input
    offsets {0,1,7,8,15}: the byte path and its edges."""
    rng = np.random.default_rng(W.seed_for(3, 9000))
    cases = [(P, B, [io] * P, oo) for P in (1, 2, 3) for B in range(0, 49)
             for io in (0, 1, 7, 8, 15) for oo in range(16)]
    _batched_cases(cases, lambda P, B: [rng.integers(0, 256, B, dtype=np.uint8) for _ in range(P)])


def test_exhaustive_offsets_around_vector_threshold():
    """B from 120 to 160 (across the byte-path threshold, every residue mod
    16), P in {1,2,3,5}, all 16 x 16 input/output offsets."""
    rng = np.random.default_rng(W.seed_for(3, 9001))
    cases = [(P, B, [io] * P, oo) for P in (1, 2, 3, 5) for B in range(120, 161)
             for io in range(16) for oo in range(16)]
    _batched_cases(cases, lambda P, B: [rng.integers(0, 256, B, dtype=np.uint8) for _ in range(P)])


def test_independent_per_rank_offsets():
    """Each rank's payload at its own offset (the realignment shift differs
    per rank), P up to 64, sizes spanning vector runs and CTA chunks."""
    rng = np.random.default_rng(W.seed_for(3, 9002))
    cases = []
    for P in (2, 3, 7, 16, 64):
        for B in (129, 1000, 4097, 65537, 100003):
            if P * B > 8 << 20:
                continue
            cases.append((P, B, [int(x) for x in rng.integers(0, 16, P)], int(rng.integers(0, 16))))
    _batched_cases(cases, lambda P, B: [rng.integers(0, 256, B, dtype=np.uint8) for _ in range(P)])


def test_page_size_list_all_offsets():
    """The sizes the page's distributed test uses to straddle the single-block
    threshold (4095 B, 32 KiB+3 B, 96 KiB, 1 MiB, and 1 MiB+5 B, its largest
    per-rank case), for P = 2 and 8, every payload and the output at each of
    the offsets {0, 1, 8, 15} (16 pairs), against the oracle."""
    rng = np.random.default_rng(W.seed_for(3, 9300))
    cases = []
    for P in (2, 8):
        for B in (4095, 32 * 1024 + 3, 96 * 1024, 1024 * 1024, 1024 * 1024 + 5):
            for io in (0, 1, 8, 15):
                for oo in (0, 1, 8, 15):
                    cases.append((P, B, [io] * P, oo))
    _batched_cases(cases, lambda P, B: [rng.integers(0, 256, B, dtype=np.uint8) for _ in range(P)])


@pytest.mark.parametrize("opts", [
    {"force_path": 1}, {"force_path": 2}, {"force_generic": 1},
    {"force_path": 2, "grid_ctas": 1}, {"force_path": 2, "grid_ctas": 3},
    {"force_path": 2, "grid_ctas": 151}, {"force_path": 2, "grid_ctas": 5000},
    {"force_generic": 1, "force_path": 1},
    {"gather_staged": 1}, {"gather_staged": 1, "force_path": 2, "grid_ctas": 3},
    {"gather_staged": 1, "force_path": 2, "grid_ctas": 7000}, {"gather_staged": 1, "force_path": 1},
    {"pdl": 0}, {"gather_staged": 0}, {"gather_staged": 0, "force_path": 2, "grid_ctas": 3},
    {"prefetch": 0}, {"prefetch": 4, "force_path": 2, "grid_ctas": 2},
    {"gather_tile_min": 32}, {"gather_tile_min": 33}, {"gather_tile_min": 1 << 20},
    {"gather_tile_min": 33, "force_path": 2, "grid_ctas": 5}, {"gather_tile_min": 33, "prefetch": 3},
    {"gather_realign_warp": 0}, {"gather_realign_warp": 0, "force_path": 2, "grid_ctas": 2},
    {"gather_realign_warp": 1, "force_path": 2, "grid_ctas": 2},
    {"gather_realign_warp": 1, "gather_tile_min": 33}, {"gather_realign_warp": 1, "grid_ctas": 7},
], ids=lambda o: ",".join(f"{k}={v}" for k, v in o.items()))
def test_path_and_grid_independence(opts):
    """The bytes never depend on the path, the grid or the flat/generic
    choice (aligned and unaligned layouts)."""
    rng = np.random.default_rng(W.seed_for(2, 9003))
    for (P, B, io, oo) in [(8, 64 * 1024, 0, 0), (2, 200000, 0, 0), (3, 65537, 1, 8),
                           (8, 4096 + 5, 15, 0), (5, 1 << 20, 8, 8), (4, 300000 + 3, 7, 9),
                           (2, 128, 3, 5), (64, 129, 1, 0)]:
        peers = [rng.integers(0, 256, B, dtype=np.uint8) for _ in range(P)]
        want = oracle.all_gather(peers)
        got, guards = run_gather(peers, [io] * P, oo, **opts)
        assert np.array_equal(got, want), (P, B, io, oo, opts)
        assert guards


@pytest.mark.parametrize("B", [4 * 1024 * 1024 + 1, 32 * 1024 * 1024 + 1])
def test_large_unaligned_full_size(B):
    """The bench's unaligned rows at full size (8 ranks, payloads at +1 B,
    output at +3 B; the warp realigning path, and the shared-memory ring once),
    byte for byte against the oracle, with per-rank offsets varied as well."""
    rng = np.random.default_rng(W.seed_for(3, 9100))
    P = 8
    peers = [rng.integers(0, 256, B, dtype=np.uint8) for _ in range(P)]
    want = oracle.all_gather(peers)
    for in_offs, out_off, opts in (([1] * P, 3, {}), ([int(x) for x in rng.integers(0, 16, P)], 9, {}),
                                   ([1] * P, 3, {"gather_realign_warp": 0})):
        got, guards = run_gather(peers, in_offs, out_off, **opts)
        assert np.array_equal(got, want), (B, in_offs, out_off)
        assert guards


def test_p1_identity_and_repeatability():
    rng = np.random.default_rng(W.seed_for(2, 9004))
    x = rng.integers(0, 256, 3 * 1024 * 1024 + 7, dtype=np.uint8)
    got, _ = run_gather([x], [5], 11)
    assert np.array_equal(got, x)
    peers = [rng.integers(0, 256, 4 << 20, dtype=np.uint8) for _ in range(8)]
    digests = {hashlib.sha256(run_gather(peers, [0] * 8, 0)[0].tobytes()).hexdigest()
               for _ in range(5)}
    assert len(digests) == 1


def test_tensor_api_returns_out():
    P, n = 4, 1000
    peers = [torch.randint(0, 256, (n,), dtype=torch.uint8, device="cuda") for _ in range(P)]
    out = torch.empty(P * n, dtype=torch.uint8, device="cuda")
    ret = dc.all_gather(peers, out)
    assert ret is out
    assert torch.equal(out, torch.cat(peers))


def test_every_call_is_one_launch():
    P, n = 8, 4096
    peers = [torch.randint(0, 256, (n,), dtype=torch.uint8, device="cuda") for _ in range(P)]
    out = torch.empty(P * n, dtype=torch.uint8, device="cuda")
    before = dc.launch_count()
    for _ in range(10):
        dc.all_gather(peers, out)
    assert dc.launch_count() - before == 10


def _free_bytes():
    torch.cuda.empty_cache()  # memory cached for earlier tests counts as used
    free, _total = torch.cuda.mem_get_info()
    return free


@pytest.mark.parametrize("P,B,in_off,out_off,path", [
    (2, (9 << 28) + 1, 1, 3, "unaligned, 4.5 GiB output: 64-bit staged realign indices"),
    (2, (16 << 30) + 16, 0, 0, "aligned, 32 GiB output: more than 2^31 vectors, 64-bit flat path"),
])
def test_huge_outputs_take_64_bit_paths(P, B, in_off, out_off, path):
    """Outputs past 4 GiB (unaligned) and past 2^31 16-byte vectors (aligned)
    switch the kernels to 64-bit indices.  At these sizes the oracle is the
    definition itself, checked on the device: slice r of the output equals
    payload r byte for byte (and the guard bytes around it are untouched)."""
    need = 2 * P * B + (1 << 30)
    if _free_bytes() < need:
        pytest.skip(f"needs {need >> 30} GiB of free device memory")
    g = torch.Generator(device="cuda")
    g.manual_seed(W.device_seed(W.seed_for(3, 9200), 0))
    store = [torch.empty(B + 16, dtype=torch.uint8, device="cuda") for _ in range(P)]
    peers = []
    for s in store:
        v = s[in_off:in_off + B]
        v.random_(0, 256, generator=g)
        peers.append(v)
    out_store = torch.full((P * B + 64,), 0xA5, dtype=torch.uint8, device="cuda")
    out = out_store[out_off:out_off + P * B]
    dc.all_gather(peers, out)
    torch.cuda.synchronize()
    for r in range(P):
        assert torch.equal(out[r * B:(r + 1) * B], peers[r]), (path, r)
    assert bool((out_store[:out_off] == 0xA5).all()) and bool((out_store[out_off + P * B:] == 0xA5).all())
