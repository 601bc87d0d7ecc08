"""GPU parity of dc_reduce, one rank's share of a reduction (the P inputs
folded into one output), against the oracle's fold of the same slices and
against the rank's output of the all-rank entry points: bit exact (0 ULP),
NaN compared by class.

Page, by title: "perf(cuda): vectorize the deterministic all-gather copy and
right-size its single-block path" -- author's replies: the collective's
ranks exchange payloads through buffers their peers map, so each rank
computes its own output; the arithmetic is the fold the oracle states.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import NP_OF, Placed, assert_typed_equal, typed_bits, typed_tensor, torch_dtype

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import reduce_copy_rank_gb300 as dc  # noqa: E402

DTYPES = ["bf16", "f16", "f32"]
ORDERS = ["linear", "tree"]
ES = {"bf16": 2, "f16": 2, "f32": 4}


def random_bits(seed, rank, n, dtype, finite=True):
    rng = np.random.default_rng(np.random.SeedSequence([seed, rank, 11]))
    if dtype == "f32":
        x = rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
        if finite:
            x[(x & 0x7F800000) == 0x7F800000] &= 0xBFFFFFFF
        return x
    x = rng.integers(0, 1 << 16, n, dtype=np.uint32).astype(np.uint16)
    if finite:
        x[(x & (0x7F80 if dtype == "bf16" else 0x7C00)) == (0x7F80 if dtype == "bf16" else 0x7C00)] &= 0xBFFF
    return x


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("order", ORDERS)
def test_reduce_slices_every_p(dtype, order):
    for P in (1, 2, 3, 5, 8):
        for n in (1, 9, 4099, 100003):
            length = 3 * n + 5
            cols = [random_bits(W.seed_for(4, 9900 + P), r, length, dtype, finite=(n % 2 == 0))
                    for r in range(P)]
            ins = [typed_tensor(c, dtype) for c in cols]
            for off in (0, n, 2 * n + 5, 1):
                want = oracle.all_reduce([c[off:off + n] for c in cols], dtype, order).view(NP_OF[dtype])
                out = torch.empty(n, dtype=torch_dtype(dtype), device="cuda")
                dc.reduce(ins, out, offset=off, order=order)
                torch.cuda.synchronize()
                assert_typed_equal(typed_bits(out, dtype), want, dtype, f"P={P} n={n} off={off} {order}")


@pytest.mark.parametrize("dtype", DTYPES)
def test_reduce_matches_the_all_rank_entry_points(dtype):
    P, C = 8, 12345
    cols = [random_bits(W.seed_for(4, 9950), r, P * C, dtype) for r in range(P)]
    ins = [typed_tensor(c, dtype) for c in cols]
    for order in ORDERS:
        ar = [torch.empty_like(x) for x in ins]
        dc.all_reduce(ins, ar, order=order)
        shards = [torch.empty(C, dtype=torch_dtype(dtype), device="cuda") for _ in range(P)]
        dc.reduce_scatter(ins, shards, order=order)
        for r in range(P):
            mine = torch.empty(P * C, dtype=torch_dtype(dtype), device="cuda")
            dc.reduce(ins, mine, order=order)
            shard = torch.empty(C, dtype=torch_dtype(dtype), device="cuda")
            dc.reduce(ins, shard, offset=r * C, order=order)
            torch.cuda.synchronize()
            assert np.array_equal(typed_bits(mine, dtype), typed_bits(ar[r], dtype)), (order, r)
            assert np.array_equal(typed_bits(shard, dtype), typed_bits(shards[r], dtype)), (order, r)


@pytest.mark.parametrize("dtype", DTYPES)
def test_reduce_at_any_alignment_with_guards(dtype):
    """Inputs and output at every element offset from 16 bytes (vector,
    realigning and element paths), no byte outside the output written."""
    es = ES[dtype]
    P, n = 4, 5003
    cols = [random_bits(W.seed_for(4, 9960), r, n + 64, dtype) for r in range(P)]
    for in_shift in range(0, 16, es):
        for out_shift in range(0, 16, es):
            srcs = []
            for r in range(P):
                s = Placed((n + 64) * es, in_shift + (r % 2) * es * (in_shift // es % 2), fill=0)
                s.write(cols[r].view(np.uint8))
                srcs.append(s)
            ins = [s.view.view(torch_dtype(dtype)) for s in srcs]
            out = Placed(n * es, out_shift)
            off = 3
            dc.reduce(ins, out.view.view(torch_dtype(dtype)), offset=off)
            torch.cuda.synchronize()
            want = oracle.all_reduce([c[off:off + n] for c in cols], dtype, "linear").view(NP_OF[dtype])
            got = out.read().view(NP_OF[dtype])
            assert_typed_equal(got, want, dtype, f"in+{in_shift} out+{out_shift}")
            assert out.guards_intact(), (in_shift, out_shift)


@pytest.mark.parametrize("dtype", DTYPES)
def test_reduce_in_place(dtype):
    """The output may be exactly the range of one input that is read."""
    P, C = 4, 3001
    cols = [random_bits(W.seed_for(4, 9970), r, P * C, dtype) for r in range(P)]
    for r in range(P):
        ins = [typed_tensor(c, dtype) for c in cols]
        want = oracle.all_reduce([c[r * C:(r + 1) * C] for c in cols], dtype, "tree").view(NP_OF[dtype])
        out = ins[r][r * C:(r + 1) * C]
        dc.reduce(ins, out, offset=r * C, order="tree")
        torch.cuda.synchronize()
        assert_typed_equal(typed_bits(out, dtype), want, dtype, f"in place, rank {r}")
        # the rest of input r is untouched
        rest = typed_bits(ins[r], dtype)
        assert np.array_equal(rest[:r * C], cols[r][:r * C])
        assert np.array_equal(rest[(r + 1) * C:], cols[r][(r + 1) * C:])


def test_reduce_rejects_a_partial_overlap_on_the_gpu_buffers():
    ins = [torch.zeros(1024, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    with pytest.raises(dc.DCError) as e:
        dc.reduce(ins, ins[1][101:357], offset=100)
    assert e.value.status == 3  # DC_ERR_OVERLAP


def test_reduce_full_size_one_launch_and_graph():
    """P = 8 ranks x 8627x8192 BF16 (the all_reduce workload's large shape):
    every rank's output through dc_reduce equals its all_reduce output, one
    kernel per call, and a captured graph replays it."""
    P, N = 8, 8627 * 8192
    ins = [W.normal_bf16_device(W.seed_for(4, 4), r, N, "cuda") for r in range(P)]
    ref = torch.empty(N, dtype=torch.bfloat16, device="cuda")
    dc.all_reduce(ins, [ref] + [torch.empty_like(ref) for _ in range(P - 1)])
    out = torch.empty_like(ref)
    n0 = dc.launch_count()
    dc.reduce(ins, out)
    assert dc.launch_count() - n0 == 1
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    # sampled against the oracle
    idx = np.random.default_rng(5).integers(0, N, 4096)
    host = [x.view(torch.int16).cpu().numpy().view(np.uint16) for x in ins]
    want = oracle.reduce_bf16_at(host, idx)
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)[idx]
    assert np.array_equal(got, want)
    out.fill_(0)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            dc.reduce(ins, out)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
