"""GPU parity of the fixed-order BF16 all_reduce and reduce_scatter against
the oracle: bit exact (0 ULP); NaN compared by class.

Covers the worked examples, brute force over rank orders, the all_reduce
workload (P=8; 256 KiB, 512 KiB, 8x8192, 8627x8192 and 16384x8192 elements
per rank, N(0,1)) and the reduce_scatter workload (P=8, 16384x8192 per rank)
at full size, ragged counts, 2-byte-aligned pointers (same and mixed
offsets), every P from 1 to 9 plus 13, 16 and 64, in-place calls, special
values, path and grid independence and repeatability.

Page, by title: "perf(cuda): vectorize the deterministic all-gather copy and
right-size its single-block path" (sections "What" and "Not in this PR" name
the deterministic all_reduce / reduce_scatter; the author's reply gives the
reduce_scatter shape, input = world x output).  The arithmetic is the
reading the oracle states: rank order 0..P-1, binary32 accumulation, one
round to nearest even.
"""
from __future__ import annotations

import hashlib
import itertools

import numpy as np
import pytest

import oracle
import oracle_pins
import workloads as W
from gpu_util import assert_bf16_equal, bf16_tensor, bf16_view_at, bits_of

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import reduce_copy_rank_gb300 as dc  # noqa: E402


def gpu_all_reduce(cols, **opts):
    """all_reduce of host bit-pattern arrays; returns every rank's output."""
    ins = [bf16_tensor(c) for c in cols]
    outs = [torch.empty_like(x) for x in ins]
    with dc.options(**opts):
        dc.all_reduce(ins, outs)
    torch.cuda.synchronize()
    return [bits_of(o) for o in outs]


def check_all_reduce(cols, what="", **opts):
    want = oracle.all_reduce_bf16(cols)
    for r, got in enumerate(gpu_all_reduce(cols, **opts)):
        assert_bf16_equal(got, want, f"{what} rank {r} {opts}")


def test_worked_examples_on_gpu():
    for name, P, inputs, expected in oracle_pins.load_worked_examples():
        outs = gpu_all_reduce([np.array([h], dtype=np.uint16) for h in inputs])
        for got in outs:
            if expected is None:
                assert oracle_pins.is_bf16_nan(int(got[0])), name
            else:
                assert int(got[0]) == expected, (name, hex(int(got[0])), hex(expected))


def test_worked_examples_in_vector_groups():
    """The worked examples placed inside 16-byte groups (vector path) and
    repeated, so every lane position of the 8-element group is exercised."""
    for name, P, inputs, expected in oracle_pins.load_worked_examples():
        cols = [np.full(64 + 3, h, dtype=np.uint16) for h in inputs]
        outs = gpu_all_reduce(cols)
        for got in outs:
            if expected is None:
                assert oracle_pins.is_bf16_nan(int(got[0])), name
            else:
                assert (got == expected).all(), name


def test_rank_order_bruteforce_on_gpu():
    """Every permutation of order-sensitive columns: the GPU must follow the
    oracle's rank order exactly, for each permutation."""
    small = [0x3F80, 0xBF80, 0x3B80, 0xBB80, 0x3C00, 0xBC00, 0x4000, 0x4B80]
    rng = np.random.default_rng(W.seed_for(4, 9000))
    for P in (2, 3, 4, 5, 6):
        for _ in range(8):
            big = int(rng.choice([0x4B80, 0xCB80]))
            col = [big, big ^ 0x8000] + [int(rng.choice(small)) for _ in range(P - 2)]
            perms = sorted(set(itertools.permutations(col)))
            cols = [np.array([p[r] for p in perms], dtype=np.uint16) for r in range(P)]
            check_all_reduce(cols, f"perm P={P}")


@pytest.mark.parametrize("name", list(W.CONFIG4_COUNTS))
def test_config4_all_reduce_full_size(name):
    n = W.CONFIG4_COUNTS[name]
    P = W.CONFIG4_P
    seed = W.seed_for(4, list(W.CONFIG4_COUNTS).index(name))
    ins = [W.normal_bf16_device(seed, r, n, "cuda") for r in range(P)]
    outs = [torch.empty_like(x) for x in ins]
    dc.all_reduce(ins, outs)
    torch.cuda.synchronize()
    host_in = [bits_of(x) for x in ins]
    want = oracle.all_reduce_bf16(host_in)
    for r in range(P):
        assert_bf16_equal(bits_of(outs[r]), want, f"{name} rank {r}")


def test_config5_reduce_scatter_full_size():
    c = W.CONFIG5_RS
    P, n = c["P"], c["rows"] * c["cols"]
    seed = W.seed_for(5, 0)
    ins = [W.normal_bf16_device(seed, r, n, "cuda") for r in range(P)]
    C = n // P
    outs = [torch.empty(C, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    dc.reduce_scatter(ins, outs)
    torch.cuda.synchronize()
    want = oracle.reduce_scatter_bf16([bits_of(x) for x in ins])
    for r in range(P):
        assert_bf16_equal(bits_of(outs[r]), want[r], f"shard {r}")


@pytest.mark.parametrize("P", [1, 2, 3, 4, 5, 6, 7, 8, 9, 13, 16, 64])
def test_every_rank_count_ragged(P):
    rng = np.random.default_rng(W.seed_for(4, 9100 + P))
    for n in (1, 7, 8, 9, 1000, 4096 + 5, 300007):
        cols = [W.random_bf16_patterns(W.seed_for(4, 9200 + P), r, n) for r in range(P)]
        if rng.integers(0, 2):
            for c in cols:  # mostly finite values, sometimes raw patterns (NaN, inf)
                c[(c & 0x7F80) == 0x7F80] &= 0xBFFF
        check_all_reduce(cols, f"P={P} n={n}")


@pytest.mark.parametrize("offset_elems", [0, 1, 3, 7])
def test_two_byte_aligned_same_offset(offset_elems):
    """Every pointer at the same 2-byte offset from 16: head + vector body."""
    P, n = 8, 100003
    cols = [W.random_bf16_patterns(W.seed_for(4, 9300), r, n) for r in range(P)]
    for c in cols:
        c[(c & 0x7F80) == 0x7F80] &= 0xBFFF
    want = oracle.all_reduce_bf16(cols)
    stores = [torch.empty(2 * n + 64, dtype=torch.uint8, device="cuda") for _ in range(2 * P)]
    ins, outs = [], []
    for r in range(P):
        v = bf16_view_at(stores[r], 2 * offset_elems + ((-stores[r].data_ptr()) % 16), n)
        v.copy_(bf16_tensor(cols[r]))
        ins.append(v)
        outs.append(bf16_view_at(stores[P + r], 2 * offset_elems + ((-stores[P + r].data_ptr()) % 16), n))
    dc.all_reduce(ins, outs)
    torch.cuda.synchronize()
    for r in range(P):
        assert_bf16_equal(bits_of(outs[r]), want, f"offset {offset_elems} rank {r}")


def test_two_byte_aligned_mixed_offsets():
    """Pointers at different 2-byte offsets: the element-wise path."""
    P, n = 5, 20011
    cols = [W.random_bf16_patterns(W.seed_for(4, 9301), r, n) for r in range(P)]
    want = oracle.all_reduce_bf16(cols)
    rng = np.random.default_rng(3)
    stores = [torch.empty(2 * n + 64, dtype=torch.uint8, device="cuda") for _ in range(2 * P)]
    ins, outs = [], []
    for r in range(P):
        a = 2 * int(rng.integers(0, 8)) + ((-stores[r].data_ptr()) % 16)
        b = 2 * int(rng.integers(0, 8)) + ((-stores[P + r].data_ptr()) % 16)
        v = bf16_view_at(stores[r], a, n)
        v.copy_(bf16_tensor(cols[r]))
        ins.append(v)
        outs.append(bf16_view_at(stores[P + r], b, n))
    dc.all_reduce(ins, outs)
    torch.cuda.synchronize()
    for r in range(P):
        assert_bf16_equal(bits_of(outs[r]), want, f"mixed rank {r}")


def test_all_reduce_in_place():
    P, n = 8, 123457
    cols = [W.random_bf16_patterns(W.seed_for(4, 9302), r, n) for r in range(P)]
    want = oracle.all_reduce_bf16(cols)
    ins = [bf16_tensor(c) for c in cols]
    dc.all_reduce(ins, ins)
    torch.cuda.synchronize()
    for r in range(P):
        assert_bf16_equal(bits_of(ins[r]), want, f"in place rank {r}")


def test_reduce_scatter_in_place_and_ragged():
    for P, C in ((8, 1001), (3, 7), (4, 65536 + 3), (1, 100)):
        cols = [W.random_bf16_patterns(W.seed_for(5, 9400 + P), r, P * C) for r in range(P)]
        want = oracle.reduce_scatter_bf16(cols)
        ins = [bf16_tensor(c) for c in cols]
        outs = [ins[r][r * C:(r + 1) * C] for r in range(P)]  # each rank's own shard
        dc.reduce_scatter(ins, outs)
        torch.cuda.synchronize()
        for r in range(P):
            assert_bf16_equal(bits_of(outs[r]), want[r], f"P={P} C={C} shard {r}")


@pytest.mark.parametrize("opts", [
    {"force_path": 1}, {"force_path": 2}, {"force_path": 2, "grid_ctas": 1},
    {"force_path": 2, "grid_ctas": 7}, {"force_path": 2, "grid_ctas": 4000},
    {"reduce_tile_min": 32}, {"reduce_tile_min": 33}, {"reduce_tile_min": 1 << 20},
    {"reduce_tile_min": 33, "force_path": 2, "grid_ctas": 9}, {"reduce_tile_min": 33, "prefetch": 3},
], ids=lambda o: ",".join(f"{k}={v}" for k, v in o.items()))
def test_path_and_grid_independence(opts):
    P = 8
    for n in (8 * 8192, 262144 + 5):
        cols = [W.normal_bf16(W.seed_for(4, 9500), r, n) for r in range(P)]
        check_all_reduce(cols, f"n={n}", **opts)
    cols = [W.normal_bf16(W.seed_for(5, 9501), r, 8 * 4099) for r in range(P)]
    want = oracle.reduce_scatter_bf16(cols)
    ins = [bf16_tensor(c) for c in cols]
    outs = [torch.empty(4099, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    with dc.options(**opts):
        dc.reduce_scatter(ins, outs)
    torch.cuda.synchronize()
    for r in range(P):
        assert_bf16_equal(bits_of(outs[r]), want[r], f"rs {opts}")


def test_special_values():
    """Subnormals, signed zeros, infinities, NaN, overflow, in every lane."""
    specials = np.array([0x0000, 0x8000, 0x0001, 0x8001, 0x007F, 0x0080, 0x7F7F, 0xFF7F,
                         0x7F80, 0xFF80, 0x7FC0, 0xFFC1, 0x3F80, 0xBF80, 0x4B80, 0xCB80],
                        dtype=np.uint16)
    rng = np.random.default_rng(W.seed_for(4, 9600))
    for P in (2, 3, 8):
        cols = [rng.choice(specials, 4099).astype(np.uint16) for _ in range(P)]
        check_all_reduce(cols, f"specials P={P}")


def test_repeatable_bits():
    P, n = 8, 1 << 22
    ins = [W.normal_bf16_device(W.seed_for(4, 9700), r, n, "cuda") for r in range(P)]
    outs = [torch.empty_like(x) for x in ins]
    digests = set()
    for grid, tmin in ((0, 64), (0, 64), (0, 64), (17, 64), (1000, 64), (0, 33), (0, 1 << 20)):
        with dc.options(grid_ctas=grid, reduce_tile_min=tmin):
            dc.all_reduce(ins, outs)
        torch.cuda.synchronize()
        digests.add(hashlib.sha256(bits_of(outs[0]).tobytes()).hexdigest())
    assert len(digests) == 1
