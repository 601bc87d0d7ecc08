"""GPU parity of the typed reductions (BF16, FP16, FP32), the tree summation
order, and the batched forms all_reduce_many / reduce_scatter_many, against
the oracle: bit exact (0 ULP), NaN compared by class.

Page, by title: "perf(cuda): vectorize the deterministic all-gather copy and
right-size its single-block path" -- author's replies: the backend is a fixed
tree ("cuda_ipc_fixed_tree"); section "Tests": reduce_scatter_many with
caller-given outputs (outs=).  The tree shape and the arithmetic are the
readings the oracle states.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import oracle_pins
import workloads as W
from gpu_util import assert_typed_equal, typed_bits, typed_tensor, torch_dtype, NP_OF

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import reduce_copy_rank_gb300 as dc  # noqa: E402

DTYPES = ["bf16", "f16", "f32"]
ORDERS = ["linear", "tree"]


def random_bits(seed, rank, n, dtype, finite=True):
    rng = np.random.default_rng(np.random.SeedSequence([seed, rank, 7]))
    if dtype == "f32":
        x = rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
        if finite:
            x[(x & 0x7F800000) == 0x7F800000] &= 0xBFFFFFFF
        return x
    x = rng.integers(0, 1 << 16, n, dtype=np.uint32).astype(np.uint16)
    if finite:
        if dtype == "bf16":
            x[(x & 0x7F80) == 0x7F80] &= 0xBFFF
        else:
            x[(x & 0x7C00) == 0x7C00] &= 0xBFFF
    return x


def normal_bits(seed, rank, n, dtype):
    """N(0,1) draws in the element type (cast by torch)."""
    g = torch.Generator(device="cuda")
    g.manual_seed(W.device_seed(seed, rank))
    return torch.randn(n, generator=g, device="cuda", dtype=torch.float32).to(torch_dtype(dtype))


def test_typed_worked_examples_on_gpu():
    for name, dtype, order, inputs, expected in oracle_pins.load_typed_examples():
        cols = [np.full(19, h, dtype=NP_OF[dtype]) for h in inputs]
        ins = [typed_tensor(c, dtype) for c in cols]
        outs = [torch.empty_like(x) for x in ins]
        dc.all_reduce(ins, outs, order=order)
        torch.cuda.synchronize()
        for o in outs:
            assert (typed_bits(o, dtype) == expected).all(), name


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("order", ORDERS)
def test_all_reduce_every_p(dtype, order):
    for P in (1, 2, 3, 4, 5, 6, 8, 13, 64):
        for n in (1, 7, 9, 1000, 4099, 100003):
            if P * n > 2_000_000:
                continue
            cols = [random_bits(W.seed_for(4, 9800 + P), r, n, dtype, finite=(n % 2 == 1))
                    for r in range(P)]
            want = oracle.all_reduce(cols, dtype, order)
            ins = [typed_tensor(c, dtype) for c in cols]
            outs = [torch.empty_like(x) for x in ins]
            dc.all_reduce(ins, outs, order=order)
            torch.cuda.synchronize()
            for r in range(P):
                assert_typed_equal(typed_bits(outs[r], dtype), np.asarray(want).view(NP_OF[dtype]),
                                   dtype, f"{dtype} {order} P={P} n={n} rank {r}")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("order", ORDERS)
def test_reduce_scatter_in_place_and_offsets(dtype, order):
    es = 4 if dtype == "f32" else 2
    for P, C in ((8, 1001), (3, 7), (5, 4096 + 3)):
        cols = [random_bits(W.seed_for(5, 9800 + P), r, P * C, dtype) for r in range(P)]
        want = oracle.reduce_scatter(cols, dtype, order)
        # inputs at an element offset from 16 bytes (scalar head), in place
        stores = [torch.empty(P * C * es + 64, dtype=torch.uint8, device="cuda") for _ in range(P)]
        ins = []
        for r in range(P):
            off = ((-stores[r].data_ptr()) % 16) + es
            v = stores[r][off:off + P * C * es].view(torch_dtype(dtype))
            v.copy_(typed_tensor(cols[r], dtype))
            ins.append(v)
        outs = [ins[r][r * C:(r + 1) * C] for r in range(P)]
        dc.reduce_scatter(ins, outs, order=order)
        torch.cuda.synchronize()
        for r in range(P):
            assert_typed_equal(typed_bits(outs[r], dtype), want[r].view(NP_OF[dtype]), dtype,
                               f"{dtype} {order} P={P} C={C} shard {r}")


@pytest.mark.parametrize("dtype,order,shape", [
    ("f16", "tree", "8627x8192"), ("f32", "linear", "8627x8192"), ("bf16", "tree", "16384x8192"),
])
def test_full_size_typed_all_reduce(dtype, order, shape):
    P, n = 8, W.CONFIG4_COUNTS[shape]
    ins = [normal_bits(W.seed_for(4, 9900), r, n, dtype) for r in range(P)]
    outs = [torch.empty_like(x) for x in ins]
    dc.all_reduce(ins, outs, order=order)
    torch.cuda.synchronize()
    want = oracle.all_reduce([typed_bits(x, dtype) for x in ins], dtype, order)
    want = np.asarray(want).view(NP_OF[dtype])
    for r in range(P):
        assert_typed_equal(typed_bits(outs[r], dtype), want, dtype, f"{shape} rank {r}")


def test_full_size_reduce_scatter_tree():
    c = W.CONFIG5_RS
    P, n = c["P"], c["rows"] * c["cols"]
    ins = [W.normal_bf16_device(W.seed_for(5, 0), r, n, "cuda") for r in range(P)]
    outs = [torch.empty(n // P, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    dc.reduce_scatter(ins, outs, order="tree")
    torch.cuda.synchronize()
    want = oracle.reduce_scatter([typed_bits(x, "bf16") for x in ins], "bf16", "tree")
    for r in range(P):
        assert_typed_equal(typed_bits(outs[r], "bf16"), want[r], "bf16", f"shard {r}")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("order", ORDERS)
def test_all_reduce_many(dtype, order):
    rng = np.random.default_rng(W.seed_for(4, 9950))
    for P, T in ((8, 6), (3, 40), (2, 200)):  # small and large parameter blocks
        counts = [int(x) for x in rng.choice([0, 1, 7, 8, 100, 4099, 65536 + 5], T)]
        cols = [[random_bits(W.seed_for(4, 9951 + t), r, max(n, 1), dtype)[:n] for r in range(P)]
                for t, n in enumerate(counts)]
        ins = [[typed_tensor(c, dtype) for c in tc] for tc in cols]
        outs = [[torch.empty_like(x) for x in t] for t in ins]
        dc.all_reduce_many(ins, outs, order=order)
        torch.cuda.synchronize()
        for t in range(T):
            if counts[t] == 0:
                continue
            want = np.asarray(oracle.all_reduce(cols[t], dtype, order)).view(NP_OF[dtype])
            for r in range(P):
                assert_typed_equal(typed_bits(outs[t][r], dtype), want, dtype,
                                   f"{dtype} {order} P={P} tensor {t} rank {r}")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("order", ORDERS)
def test_reduce_scatter_many_with_outs(dtype, order):
    rng = np.random.default_rng(W.seed_for(5, 9960))
    for P, T in ((8, 5), (4, 50)):  # reduce_scatter jobs: T*P
        counts = [int(x) for x in rng.choice([0, 1, 3, 8, 1001, 8192], T)]
        cols = [[random_bits(W.seed_for(5, 9961 + t), r, max(P * n, 1), dtype)[:P * n]
                 for r in range(P)] for t, n in enumerate(counts)]
        ins = [[typed_tensor(c, dtype) for c in tc] for tc in cols]
        outs = [[torch.empty(n, dtype=torch_dtype(dtype), device="cuda") for _ in range(P)]
                for n in counts]
        ret = dc.reduce_scatter_many(ins, outs, order=order)
        assert ret is outs
        torch.cuda.synchronize()
        for t in range(T):
            if counts[t] == 0:
                continue
            want = oracle.reduce_scatter(cols[t], dtype, order)
            for r in range(P):
                assert_typed_equal(typed_bits(outs[t][r], dtype), want[r].view(NP_OF[dtype]), dtype,
                                   f"{dtype} {order} P={P} tensor {t} shard {r}")


@pytest.mark.parametrize("opts", [{"force_path": 1}, {"force_path": 2, "grid_ctas": 3},
                                  {"force_path": 2, "grid_ctas": 999}, {"pdl": 0}],
                         ids=lambda o: ",".join(f"{k}={v}" for k, v in o.items()))
def test_typed_path_and_grid_independence(opts):
    for dtype in DTYPES:
        for order in ORDERS:
            P, n = 8, 65536 + 7
            cols = [random_bits(W.seed_for(4, 9970), r, n, dtype) for r in range(P)]
            want = np.asarray(oracle.all_reduce(cols, dtype, order)).view(NP_OF[dtype])
            ins = [typed_tensor(c, dtype) for c in cols]
            outs = [torch.empty_like(x) for x in ins]
            with dc.options(**opts):
                dc.all_reduce(ins, outs, order=order)
            torch.cuda.synchronize()
            assert_typed_equal(typed_bits(outs[3], dtype), want, dtype, f"{dtype} {order} {opts}")


def test_tree_and_linear_differ_on_gpu():
    """The two orders really are different folds.  Eight N(0,1) BF16 values
    sum exactly in FP32 whatever the order, and a reordered sum that is off
    by one FP32 ulp changes the BF16 result only next to a rounding
    midpoint, so each column here holds +L and -L (L = 2^24..2^30) at two
    random ranks among small values: which small values the big partial sum
    absorbs depends on the order."""
    P, n = 8, 1 << 16
    rng = np.random.default_rng(W.seed_for(4, 9980))
    vals = rng.standard_normal((P, n)).astype(np.float32) * 16
    big = np.exp2(rng.integers(24, 31, n)).astype(np.float32)
    pos = np.argsort(rng.random((P, n)), axis=0)[:2]
    vals[pos[0], np.arange(n)] = big
    vals[pos[1], np.arange(n)] = -big
    cols = [(vals[r].view(np.uint32) >> 16).astype(np.uint16) for r in range(P)]
    lin = np.asarray(oracle.all_reduce(cols, "bf16", "linear"))
    tree = np.asarray(oracle.all_reduce(cols, "bf16", "tree"))
    differ = lin != tree
    assert differ.sum() > n // 100
    ins = [typed_tensor(c, "bf16") for c in cols]
    a = [torch.empty_like(x) for x in ins]
    b = [torch.empty_like(x) for x in ins]
    dc.all_reduce(ins, a, order="linear")
    dc.all_reduce(ins, b, order="tree")
    torch.cuda.synchronize()
    ga, gb = typed_bits(a[0], "bf16"), typed_bits(b[0], "bf16")
    assert_typed_equal(ga, lin, "bf16", "linear")
    assert_typed_equal(gb, tree, "bf16", "tree")
    assert (ga[differ] != gb[differ]).all()


def _at_offsets(cols, dtype, offs):
    """Device copies of `cols`, rank r's starting `offs[r]` elements past a
    16-byte boundary."""
    es = 4 if dtype == "f32" else 2
    out = []
    for c, o in zip(cols, offs):
        n = c.size
        store = torch.empty(n * es + 64, dtype=torch.uint8, device="cuda")
        start = ((-store.data_ptr()) % 16) + o * es
        v = store[start:start + n * es].view(torch_dtype(dtype))
        v.copy_(typed_tensor(c, dtype))
        out.append(v)
    return out


@pytest.mark.parametrize("staged", [1, 0])
@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("order", ORDERS)
def test_realigned_inputs(dtype, order, staged):
    """Inputs at different offsets from 16 bytes, outputs aligned: 16-byte
    units anchored at the outputs, every input realigned (all_reduce and
    reduce_scatter, compile-time and runtime P), with the all_reduce of one
    tensor on the shared-memory staged kernel (P = 2, 4, 8) or on the
    register path."""
    epv = 4 if dtype == "f32" else 8
    rng = np.random.default_rng(W.seed_for(4, 9990))
    for P in (2, 3, 4, 8, 13):
        for C in (1, 9, 1000, 65536 + 3):
            offs = [int(x) for x in rng.integers(0, epv, P)]
            offs[0] = (offs[0] + 1) % epv if len(set(offs)) == 1 else offs[0]  # not all equal
            cols = [random_bits(W.seed_for(4, 9991 + P), r, P * C, dtype) for r in range(P)]
            ins = _at_offsets(cols, dtype, offs)
            outs = [torch.empty(P * C, dtype=torch_dtype(dtype), device="cuda") for _ in range(P)]
            shards = [torch.empty(C, dtype=torch_dtype(dtype), device="cuda") for _ in range(P)]
            with dc.options(reduce_staged=staged):
                dc.all_reduce(ins, outs, order=order)
                dc.reduce_scatter(ins, shards, order=order)
            torch.cuda.synchronize()
            want = np.asarray(oracle.all_reduce(cols, dtype, order)).view(NP_OF[dtype])
            for r in range(P):
                assert_typed_equal(typed_bits(outs[r], dtype), want, dtype,
                                   f"all_reduce {dtype} {order} P={P} C={C} offs={offs} rank {r}")
            want_rs = oracle.reduce_scatter(cols, dtype, order)
            for r in range(P):
                assert_typed_equal(typed_bits(shards[r], dtype), want_rs[r].view(NP_OF[dtype]), dtype,
                                   f"reduce_scatter {dtype} {order} P={P} C={C} offs={offs} shard {r}")


def test_in_place_at_disagreeing_offsets():
    """In-place all_reduce with each rank's buffer at its own offset: the
    outputs disagree mod 16, so the job runs element by element."""
    P, n = 4, 10007
    cols = [random_bits(W.seed_for(4, 9995), r, n, "bf16") for r in range(P)]
    want = np.asarray(oracle.all_reduce(cols, "bf16", "linear")).view(np.uint16)
    bufs = _at_offsets(cols, "bf16", [0, 1, 2, 5])
    dc.all_reduce(bufs, bufs)
    torch.cuda.synchronize()
    for r in range(P):
        assert_typed_equal(typed_bits(bufs[r], "bf16"), want, "bf16", f"rank {r}")


@pytest.mark.parametrize("opts", [{}, {"grid_ctas": 1}, {"grid_ctas": 3}, {"grid_ctas": 5000},
                                  {"prefetch": 0}, {"prefetch": 5}, {"pdl": 0}, {"force_path": 1}],
                         ids=lambda o: ",".join(f"{k}={v}" for k, v in o.items()) or "default")
def test_realigned_in_place_and_grids(opts):
    """The staged realigning all_reduce with two ranks in place (their
    outputs are exactly their inputs, at the outputs' offset) and two ranks'
    inputs off by 1 and 3 elements; sizes around the tile and the ring (256
    units per tile), odd grids and prefetch depths."""
    P = 4
    for n in (8 * 256 * 3 + 5, 8 * 256 * 7 + 8 * 3 + 1, 100003):
        cols = [random_bits(W.seed_for(4, 9997), r, n, "bf16") for r in range(P)]
        want = np.asarray(oracle.all_reduce(cols, "bf16", "tree")).view(np.uint16)
        ins = _at_offsets(cols, "bf16", [0, 1, 0, 3])
        outs = [ins[0], torch.empty(n, dtype=torch.bfloat16, device="cuda"), ins[2],
                torch.empty(n, dtype=torch.bfloat16, device="cuda")]
        with dc.options(**opts):
            dc.all_reduce(ins, outs, order="tree")
        torch.cuda.synchronize()
        for r in range(P):
            assert_typed_equal(typed_bits(outs[r], "bf16"), want, "bf16", f"n={n} {opts} rank {r}")


def test_full_size_realigned_all_reduce():
    """8627x8192 per rank, P = 8, rank 1's input one element off: bit exact
    at full size on the realigning path."""
    P, n = 8, W.CONFIG4_COUNTS["8627x8192"]
    store = [normal_bits(W.seed_for(4, 9996), r, n + 8, "bf16") for r in range(P)]
    ins = [store[r][(1 if r == 1 else 0):(1 if r == 1 else 0) + n] for r in range(P)]
    outs = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    dc.all_reduce(ins, outs)
    torch.cuda.synchronize()
    want = oracle.all_reduce([typed_bits(x, "bf16") for x in ins], "bf16", "linear")
    assert_typed_equal(typed_bits(outs[5], "bf16"), np.asarray(want), "bf16", "rank 5")
