"""GPU parity of all_gather_many (several gathers in one launch, one output
per tensor) against the oracle, bit exact, plus CUDA-graph capture and
replay of every entry point.

Workload: 6 tensors per rank of {3 B, 4 KiB, 100000 B, 1 MiB, 7 MiB+5 B,
32 MiB}, P=8, random bytes.  Page, by title: "perf(cuda): vectorize the
deterministic all-gather copy and right-size its single-block path"
(results paragraph and the author's reply on all_gather_many: several
gathers, one handshake, no packing).
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import Placed, assert_bf16_equal, bf16_tensor, bits_of

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import reduce_copy_rank_gb300 as dc  # noqa: E402


def run_many(tensors_np, in_offs, out_offs, **opts):
    T = len(tensors_np)
    P = len(tensors_np[0])
    srcs, outs, ptrs, sizes = [], [], [], []
    for t in range(T):
        B = tensors_np[t][0].size
        sizes.append(B)
        for r in range(P):
            s = Placed(B, in_offs[t][r])
            s.write(tensors_np[t][r])
            srcs.append(s)
            ptrs.append(s.ptr())
        outs.append(Placed(P * B, out_offs[t]))
    with dc.options(**opts):
        st = dc.dc_all_gather_many(ptrs, sizes, [o.ptr() for o in outs], T, P,
                                   torch.cuda.current_stream().cuda_stream)
    assert st == 0, dc.last_error()
    torch.cuda.synchronize()
    return [o.read() for o in outs], all(o.guards_intact() for o in outs)


def test_config5_gather_many_full_size():
    P = W.CONFIG5_MANY_P
    seed = W.seed_for(5, 1)
    tensors = [[W.random_bytes(seed, r, B, tensor=t) for r in range(P)]
               for t, B in enumerate(W.CONFIG5_MANY_SIZES)]
    want = oracle.all_gather_many(tensors)
    T = len(tensors)
    for opts in ({}, {"force_generic": 1}):
        got, guards = run_many(tensors, [[0] * P] * T, [0] * T, **opts)
        for t in range(T):
            assert np.array_equal(got[t], want[t]), (t, opts)
        assert guards


def test_many_random_layouts():
    rng = np.random.default_rng(W.seed_for(5, 9000))
    for trial in range(12):
        P = int(rng.choice([1, 2, 3, 8]))
        T = int(rng.integers(1, 20))
        tensors = [[rng.integers(0, 256, int(B), dtype=np.uint8) for _ in range(P)]
                   for B in rng.choice([0, 1, 15, 16, 17, 127, 128, 129, 4096, 65537, 300000], T)]
        in_offs = [[int(x) for x in rng.integers(0, 16, P)] for _ in range(T)]
        out_offs = [int(x) for x in rng.integers(0, 16, T)]
        want = oracle.all_gather_many(tensors)
        got, guards = run_many(tensors, in_offs, out_offs)
        for t in range(T):
            assert np.array_equal(got[t], want[t]), (trial, t)
        assert guards


@pytest.mark.parametrize("opts", [{}, {"grid_ctas": 1}, {"grid_ctas": 2}, {"grid_ctas": 3},
                                  {"grid_ctas": 7}, {"grid_ctas": 5000}, {"gather_staged": 0},
                                  {"force_path": 2, "grid_ctas": 2}],
                         ids=lambda o: ",".join(f"{k}={v}" for k, v in o.items()) or "default")
def test_many_split_aligned_and_unaligned(opts):
    """Aligned and unaligned tensors interleaved: the aligned ones are staged
    by the first part of the grid, the others realigned by the rest; every
    grid size (one CTA falls back to one path) gives the same bytes."""
    rng = np.random.default_rng(W.seed_for(5, 9002))
    P = 8
    sizes = [4096, 100003, 65536, 7, 1 << 20, 33, 300000 + 16, 129]
    tensors = [[rng.integers(0, 256, B, dtype=np.uint8) for _ in range(P)] for B in sizes]
    in_offs = [[0] * P if B % 16 == 0 else [int(x) for x in rng.integers(0, 16, P)] for B in sizes]
    out_offs = [0 if B % 16 == 0 else int(rng.integers(1, 16)) for B in sizes]
    want = oracle.all_gather_many(tensors)
    got, guards = run_many(tensors, in_offs, out_offs, **opts)
    for t in range(len(sizes)):
        assert np.array_equal(got[t], want[t]), (t, opts)
    assert guards


@pytest.mark.parametrize("grid", [0, 1, 2, 5, 5000])
def test_many_all_aligned(grid):
    rng = np.random.default_rng(W.seed_for(5, 9003))
    P = 4
    sizes = [16, 4096, 1 << 20, 48, 262144 + 32]
    tensors = [[rng.integers(0, 256, B, dtype=np.uint8) for _ in range(P)] for B in sizes]
    want = oracle.all_gather_many(tensors)
    got, guards = run_many(tensors, [[0] * P] * len(sizes), [0] * len(sizes), grid_ctas=grid)
    for t in range(len(sizes)):
        assert np.array_equal(got[t], want[t]), (t, grid)
    assert guards


@pytest.mark.parametrize("grid", [0, 1, 2, 7, 5000])
def test_many_all_unaligned(grid):
    """No aligned tensor: every CTA stages and realigns; small jobs (under
    128 B per rank) and rank boundaries go byte by byte."""
    rng = np.random.default_rng(W.seed_for(5, 9004))
    P = 5
    sizes = [3, 127, 128, 129, 4097, 100001, 300007]
    tensors = [[rng.integers(0, 256, B, dtype=np.uint8) for _ in range(P)] for B in sizes]
    in_offs = [[int(x) for x in rng.integers(1, 16, P)] for _ in sizes]
    out_offs = [int(x) for x in rng.integers(1, 16, len(sizes))]
    want = oracle.all_gather_many(tensors)
    got, guards = run_many(tensors, in_offs, out_offs, grid_ctas=grid)
    for t in range(len(sizes)):
        assert np.array_equal(got[t], want[t]), (t, grid)
    assert guards


@pytest.mark.parametrize("opts", [{}, {"grid_ctas": 1}, {"grid_ctas": 2}, {"grid_ctas": 3},
                                  {"grid_ctas": 5000}, {"gather_many_single_max_bytes": 0},
                                  {"gather_many_single_max_bytes": 1 << 20}],
                         ids=lambda o: ",".join(f"{k}={v}" for k, v in o.items()) or "default")
def test_many_tiny_tensors(opts):
    """120 tensors x 8 ranks of 3..100 B at random offsets: every job is
    assembled from bytes by the split launch's small-job CTAs (tables in
    shared memory), or by one CTA, or on the general path when the grid is
    too small to split."""
    rng = np.random.default_rng(W.seed_for(5, 9005))
    P, T = 8, 120
    tensors = [[rng.integers(0, 256, int(B), dtype=np.uint8) for _ in range(P)]
               for B in rng.integers(3, 101, T)]
    in_offs = [[int(x) for x in rng.integers(0, 16, P)] for _ in range(T)]
    out_offs = [int(x) for x in rng.integers(0, 16, T)]
    want = oracle.all_gather_many(tensors)
    got, guards = run_many(tensors, in_offs, out_offs, **opts)
    for t in range(T):
        assert np.array_equal(got[t], want[t]), (t, opts)
    assert guards


@pytest.mark.parametrize("grid", [0, 2, 3, 4, 9, 5000])
def test_many_three_parts(grid):
    """Aligned, unaligned and small tensors in one launch: three parts of the
    grid (or fewer CTAs than parts: the general path)."""
    rng = np.random.default_rng(W.seed_for(5, 9006))
    P = 8
    sizes = [5, 4096, 127, 100003, 1, 65536, 77, 300000 + 16, 2000, 3]
    tensors = [[rng.integers(0, 256, B, dtype=np.uint8) for _ in range(P)] for B in sizes]
    in_offs = [[0] * P if B % 16 == 0 else [int(x) for x in rng.integers(0, 16, P)] for B in sizes]
    out_offs = [0 if B % 16 == 0 else int(rng.integers(1, 16)) for B in sizes]
    want = oracle.all_gather_many(tensors)
    got, guards = run_many(tensors, in_offs, out_offs, grid_ctas=grid)
    for t in range(len(sizes)):
        assert np.array_equal(got[t], want[t]), (t, grid)
    assert guards


def test_many_small_jobs_at_the_table_limit():
    """P = 64 ranks x 16 tensors of 1..127 B (1024 sources): the shared
    pointer table of the small-job CTAs at its largest."""
    rng = np.random.default_rng(W.seed_for(5, 9007))
    P, T = 64, 16
    tensors = [[rng.integers(0, 256, int(B), dtype=np.uint8) for _ in range(P)]
               for B in rng.integers(1, 128, T)]
    in_offs = [[int(x) for x in rng.integers(0, 16, P)] for _ in range(T)]
    want = oracle.all_gather_many(tensors)
    got, guards = run_many(tensors, in_offs, [int(x) for x in rng.integers(0, 16, T)])
    for t in range(T):
        assert np.array_equal(got[t], want[t]), t
    assert guards


def test_many_large_table():
    """More tensors than the small parameter block holds (T=100, P=8)."""
    rng = np.random.default_rng(W.seed_for(5, 9001))
    P, T = 8, 100
    tensors = [[rng.integers(0, 256, int(B), dtype=np.uint8) for _ in range(P)]
               for B in rng.integers(1, 3000, T)]
    want = oracle.all_gather_many(tensors)
    got, guards = run_many(tensors, [[0] * P] * T, [int(x) for x in rng.integers(0, 16, T)])
    for t in range(T):
        assert np.array_equal(got[t], want[t]), t
    assert guards


@pytest.mark.parametrize("opts", [{}, {"gather_realign_warp": 0}, {"grid_ctas": 3}, {"grid_ctas": 4},
                                  {"grid_ctas": 6}, {"grid_ctas": 40}, {"grid_ctas": 5000},
                                  {"gather_split_cost_warp_pct": 400}],
                         ids=lambda o: ",".join(f"{k}={v}" for k, v in o.items()) or "default")
def test_many_jobs_runs_and_warp_realign(opts):
    """More than 16 jobs in each part: contiguous runs of tiles per CTA from
    the host's start-job tables; the unaligned part realigned across the
    lanes of a warp, its rank-boundary vectors copied by their own CTAs (or
    through the ring with gather_realign_warp=0); small grids fall back to
    fewer parts."""
    rng = np.random.default_rng(W.seed_for(5, 9010))
    P, T = 4, 90
    sizes = [int(B) for B in rng.integers(128, 70000, T)]
    sizes = [((B + 15) // 16) * 16 if t % 3 == 0 else B for t, B in enumerate(sizes)]
    tensors = [[rng.integers(0, 256, B, dtype=np.uint8) for _ in range(P)] for B in sizes]
    in_offs = [[0] * P if t % 3 == 0 else [int(x) for x in rng.integers(0, 16, P)] for t in range(T)]
    out_offs = [0 if t % 3 == 0 else int(rng.integers(0, 16)) for t in range(T)]
    want = oracle.all_gather_many(tensors)
    got, guards = run_many(tensors, in_offs, out_offs, **opts)
    for t in range(T):
        assert np.array_equal(got[t], want[t]), (t, opts)
    assert guards


def test_many_tensor_api():
    P = 4
    tensors = [[torch.randint(0, 256, (n,), dtype=torch.uint8, device="cuda") for _ in range(P)]
               for n in (5, 4096, 777)]
    outs = [torch.empty(P * p[0].numel(), dtype=torch.uint8, device="cuda") for p in tensors]
    ret = dc.all_gather_many(tensors, outs)
    assert ret is outs
    for p, o in zip(tensors, outs):
        assert torch.equal(o, torch.cat(p))


def test_cuda_graph_capture_and_replay():
    """Every entry point captured into one CUDA graph and replayed with new
    input values: the launches read no host memory after capture."""
    P, n, B = 8, 65536 + 8, 4096 * 3 + 4
    ar_in = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    ar_out = [torch.empty_like(x) for x in ar_in]
    rs_in = [torch.empty(P * 1024, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    rs_out = [torch.empty(1024, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    g_in = [torch.empty(B, dtype=torch.uint8, device="cuda") for _ in range(P)]
    g_out = torch.empty(P * B, dtype=torch.uint8, device="cuda")
    m_in = [[torch.empty(s, dtype=torch.uint8, device="cuda") for _ in range(P)] for s in (3, 5000)]
    m_out = [torch.empty(P * s, dtype=torch.uint8, device="cuda") for s in (3, 5000)]

    def fill(seed):
        for r in range(P):
            ar_in[r].copy_(bf16_tensor(W.normal_bf16(seed, r, n)))
            rs_in[r].copy_(bf16_tensor(W.normal_bf16(seed + 1, r, P * 1024)))
            g_in[r].copy_(torch.from_numpy(W.random_bytes(seed, r, B)))
            for t in range(2):
                m_in[t][r].copy_(torch.from_numpy(W.random_bytes(seed, r, m_in[t][r].numel(), t + 1)))

    def body():
        dc.all_reduce(ar_in, ar_out)
        dc.reduce_scatter(rs_in, rs_out)
        dc.all_gather(g_in, g_out)
        dc.all_gather_many(m_in, m_out)

    fill(W.seed_for(5, 9100))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        body()  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    before = dc.launch_count()
    with torch.cuda.graph(g):
        body()
    assert dc.launch_count() - before == 4
    for seed in (W.seed_for(5, 9101), W.seed_for(5, 9102)):
        fill(seed)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        host_ar = [bits_of(x) for x in ar_in]
        want = oracle.all_reduce_bf16(host_ar)
        for r in range(P):
            assert_bf16_equal(bits_of(ar_out[r]), want, "graph all_reduce")
        want_rs = oracle.reduce_scatter_bf16([bits_of(x) for x in rs_in])
        for r in range(P):
            assert_bf16_equal(bits_of(rs_out[r]), want_rs[r], "graph reduce_scatter")
        assert np.array_equal(g_out.cpu().numpy(), oracle.all_gather([x.cpu().numpy() for x in g_in]))
        for t in range(2):
            assert np.array_equal(m_out[t].cpu().numpy(),
                                  oracle.all_gather([x.cpu().numpy() for x in m_in[t]]))
