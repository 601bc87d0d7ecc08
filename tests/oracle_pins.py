"""Pins for the oracle: checks against what the page and the mathematics fix.

Each check takes an :class:`oracle.Oracle` and raises AssertionError when the
oracle disagrees with something other than itself:

* worked examples derived by hand (``tests/golden/*_worked_examples.txt``),
* exact rational arithmetic with IEEE round-to-nearest-even from its
  definition (``exact_ieee``),
* library routines for the special cases that reduce to them (numpy
  concatenation for the gather; torch's float->bfloat16 cast for the final
  rounding; torch CPU binary32 adds for the fold),
* brute force over tiny inputs and over all rank orders,
* invariants the page states (slice r of the gather is peer r's payload,
  byte for byte; P=1 is the identity).

The same checks run against deliberately broken builds of the oracle in
``test_oracle_mutants.py`` to show that each plausible mistake is caught.

Page, by title: "perf(cuda): vectorize the deterministic all-gather copy and
right-size its single-block path" (section "What": the copy is a pure
rank-ordered copy, so results are byte-identical).
"""
from __future__ import annotations

import itertools
import os
import random

import numpy as np

import exact_ieee as ex

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ------------------------------------------------------------ fixtures ---

def load_worked_examples():
    """Parse the reduction fixture: (name, P, inputs, expected or None)."""
    rows = []
    with open(os.path.join(GOLDEN, "reduction_worked_examples.txt")) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, P, ins, exp, _why = [c.strip() for c in line.split("|", 4)]
            inputs = [int(h, 16) for h in ins.split()]
            assert len(inputs) == int(P), name
            expected = None if exp == "NAN" else int(exp, 16)
            rows.append((name, int(P), inputs, expected))
    return rows


def load_gather_examples():
    """Parse the gather fixture: (name, [peer bytes], expected bytes)."""
    rows = []
    with open(os.path.join(GOLDEN, "gather_worked_examples.txt")) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, peers, expected, _why = [c.strip() for c in line.split("|", 3)]
            peer_bytes = [bytes.fromhex(p) if p != "-" else b"" for p in peers.split()]
            rows.append((name, peer_bytes, bytes.fromhex(expected) if expected != "-" else b""))
    return rows


def is_bf16_nan(h: int) -> bool:
    return (h & 0x7F80) == 0x7F80 and (h & 0x007F) != 0


# ------------------------------------------------------- gather checks ---

def check_gather_worked_examples(orc):
    for name, peers, expected in load_gather_examples():
        got = orc.all_gather([np.frombuffer(p, dtype=np.uint8) for p in peers]).tobytes()
        assert got == expected, (name, got.hex(), expected.hex())


def check_gather_matches_concatenate(orc, seed=1):
    """Library special case: the gather equals numpy's concatenation, and
    slice r equals peer r byte for byte, for random P and odd sizes."""
    rng = np.random.default_rng(seed)
    for _ in range(40):
        P = int(rng.integers(1, 9))
        B = int(rng.integers(0, 3000))
        peers = [rng.integers(0, 256, B, dtype=np.uint8) for _ in range(P)]
        out = orc.all_gather(peers)
        assert np.array_equal(out, np.concatenate(peers))
        for r in range(P):
            assert np.array_equal(out[r * B:(r + 1) * B], peers[r]), (P, B, r)


def check_gather_tiny_bruteforce(orc):
    """Every P in {1,2,3} and B in 0..48: each output byte is the byte of
    the peer whose rank-ordered block contains it (checked one by one)."""
    for P in (1, 2, 3):
        for B in range(0, 49):
            peers = [np.array([(31 * r + 7 * j + 1) & 0xFF for j in range(B)], dtype=np.uint8)
                     for r in range(P)]
            out = orc.all_gather(peers)
            assert out.size == P * B
            for k in range(P * B):
                r, j = divmod(k, B)
                assert out[k] == peers[r][j], (P, B, k)


def check_gather_identity_p1(orc, seed=2):
    rng = np.random.default_rng(seed)
    for B in (0, 1, 15, 16, 17, 4097):
        x = rng.integers(0, 256, B, dtype=np.uint8)
        assert np.array_equal(orc.all_gather([x]), x)


def check_gather_many_independent(orc, seed=3):
    """all_gather_many equals one gather per tensor, each its own output."""
    rng = np.random.default_rng(seed)
    P = 4
    sizes = [3, 0, 17, 4096, 1001]
    tensors = [[rng.integers(0, 256, s, dtype=np.uint8) for _ in range(P)] for s in sizes]
    outs = orc.all_gather_many(tensors)
    assert len(outs) == len(sizes)
    for peers, out in zip(tensors, outs):
        assert np.array_equal(out, np.concatenate(peers))


# ---------------------------------------------------- rounding checks ---

def _rounding_probe_values(seed=4, n_random=200_000):
    rng = np.random.default_rng(seed)
    special = [0x00000000, 0x80000000, 0x00000001, 0x80000001, 0x007FFFFF, 0x00800000,
               0x7F7FFFFF, 0xFF7FFFFF, 0x7F800000, 0xFF800000, 0x7FC00000, 0xFFC00001,
               0x7F800001, 0x7FBFFFFF, 0x3F808000, 0x3F818000, 0x3F807FFF, 0x3F808001,
               0x7F7F8000, 0x7F7F7FFF, 0x00008000, 0x00018000, 0x0000FFFF, 0x80008000]
    # ties (low half exactly 0x8000) and their neighbours, over many exponents
    hi = rng.integers(0, 1 << 16, 4000, dtype=np.uint64)
    ties = (hi << np.uint64(16)) | np.uint64(0x8000)
    near = np.concatenate([ties - np.uint64(1), ties + np.uint64(1)])
    rand = rng.integers(0, 1 << 32, n_random, dtype=np.uint64)
    allv = np.concatenate([np.array(special, dtype=np.uint64), ties, near, rand])
    return (allv & np.uint64(0xFFFFFFFF)).astype(np.uint32)


def check_rounding_matches_torch_cast(orc):
    """Library routine: torch's float32 -> bfloat16 cast rounds to nearest
    even; the oracle's final rounding must agree on every non-NaN input and
    give a NaN for every NaN input."""
    import torch

    u = _rounding_probe_values()
    got = orc.f32_to_bf16_rne_array(u)
    ref = torch.from_numpy(u.view(np.float32).copy()).to(torch.bfloat16).view(torch.int16)
    ref = ref.numpy().view(np.uint16)
    nan = np.isnan(u.view(np.float32))
    assert np.array_equal(got[~nan], ref[~nan]), "rounding differs from torch's cast"
    assert all(is_bf16_nan(int(h)) for h in got[nan]), "NaN inputs must stay NaN"


def check_rounding_matches_exact(orc, seed=5):
    """Exact definition: the nearest BF16 value, ties to the even
    significand, computed on rationals."""
    rng = np.random.default_rng(seed)
    u = np.concatenate([
        rng.integers(0, 1 << 32, 3000, dtype=np.uint64).astype(np.uint32),
        ((rng.integers(0, 1 << 16, 1000, dtype=np.uint64) << np.uint64(16))
         | np.uint64(0x8000)).astype(np.uint32),
        np.array([0x00000001, 0x00008000, 0x00018000, 0x007FFFFF, 0x7F7F8000, 0x7F7F7FFF,
                  0x80000000, 0x3F808000, 0x3F818000], dtype=np.uint32),
    ])
    got = orc.f32_to_bf16_rne_array(u)
    for ui, gi in zip(u.tolist(), got.tolist()):
        if (ui & 0x7F800000) == 0x7F800000:
            continue  # inf / NaN: covered by the library check
        assert gi == ex.f32_to_bf16_exact(ui), (hex(ui), hex(gi))


# ---------------------------------------------------- reduction checks ---

def check_reduction_worked_examples(orc):
    rows = load_worked_examples()
    for name, P, inputs, expected in rows:
        got = int(orc.all_reduce_bf16([np.array([h], dtype=np.uint16) for h in inputs])[0])
        if expected is None:
            assert is_bf16_nan(got), (name, hex(got))
        else:
            assert got == expected, (name, hex(got), hex(expected))
    # the same examples as one multi-element reduction per P, every rank's
    # output checked: elements must not interact
    by_p = {}
    for name, P, inputs, expected in rows:
        by_p.setdefault(P, []).append((name, inputs, expected))
    for P, items in by_p.items():
        cols = [np.array([it[1][r] for it in items], dtype=np.uint16) for r in range(P)]
        outs = orc.all_reduce_bf16_all_outputs(cols)
        for r in range(P):
            for k, (name, _i, expected) in enumerate(items):
                got = int(outs[r][k])
                if expected is None:
                    assert is_bf16_nan(got), (name, r)
                else:
                    assert got == expected, (name, r, hex(got), hex(expected))


def _bf16_column(rng, P, wide):
    """Random finite BF16 patterns: N(0,1)-like or with a wide exponent spread."""
    out = []
    for _ in range(P):
        sign = int(rng.integers(0, 2))
        exp = int(rng.integers(1, 255)) if wide else int(rng.integers(120, 131))
        frac = int(rng.integers(0, 128))
        out.append((sign << 15) | (exp << 7) | frac)
    return out


def check_fold_matches_exact(orc, seed=6, n_cols=400):
    """Exact definition of each binary32 add (nearest, ties to even) and of
    the final BF16 rounding, on rationals, for random columns of P values."""
    rng = np.random.default_rng(seed)
    for P in (1, 2, 3, 5, 8):
        cols = []
        for k in range(n_cols):
            while True:
                c = _bf16_column(rng, P, wide=(k % 4 == 0))
                try:
                    e = ex.fold_bf16_exact(c)
                except ValueError:  # a partial sum overflowed to inf: redraw
                    continue
                cols.append((c, e))
                break
        inputs = [np.array([c[r] for c, _ in cols], dtype=np.uint16) for r in range(P)]
        got = orc.all_reduce_bf16(inputs)
        for k, (c, e) in enumerate(cols):
            assert int(got[k]) == e, (P, [hex(h) for h in c], hex(int(got[k])), hex(e))


def check_fold_matches_torch_cpu(orc, seed=7):
    """Library routine: torch CPU binary32 tensor adds in rank order, then
    torch's cast to bfloat16."""
    import torch

    rng = np.random.default_rng(seed)
    for P in (2, 3, 8):
        n = 5000
        xs = [rng.integers(0, 65536, n, dtype=np.uint16) for _ in range(P)]
        for x in xs:  # finite values only (NaN is compared by class elsewhere)
            x[(x & 0x7F80) == 0x7F80] &= 0xBFFF
        t = [torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16) for x in xs]
        acc = t[0].float()
        for q in range(1, P):
            acc = acc + t[q].float()
        ref = acc.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        got = orc.all_reduce_bf16(xs)
        nan = np.array([is_bf16_nan(int(h)) for h in ref], dtype=bool)
        assert np.array_equal(got[~nan], ref[~nan]), P
        assert all(is_bf16_nan(int(h)) for h in got[nan]), P


def check_order_bruteforce(orc):
    """Brute force over every rank permutation of small columns that hold
    +-2^24, its negation and small values from {+-1, +-2^-8, +-2^-7, 2, 2^24}:
    the oracle's result for each permutation must equal the exact fold in
    that rank order, and most columns must give different results for
    different orders (so the check can tell orders apart)."""
    small = [0x3F80, 0xBF80, 0x3B80, 0xBB80, 0x3C00, 0xBC00, 0x4000, 0x4B80]
    rng = random.Random(8)
    sensitive = total = 0
    for P in (2, 3, 4, 5):
        for _ in range(20):
            big = rng.choice([0x4B80, 0xCB80])
            col = [big, big ^ 0x8000] + [rng.choice(small) for _ in range(P - 2)]
            rng.shuffle(col)
            perms = sorted(set(itertools.permutations(col)))
            inputs = [np.array([p[r] for p in perms], dtype=np.uint16) for r in range(P)]
            got = orc.all_reduce_bf16(inputs)
            exact = [ex.fold_bf16_exact(list(p)) for p in perms]
            assert [int(g) for g in got] == exact, (P, [hex(h) for h in col])
            total += 1
            sensitive += len(set(exact)) > 1
    assert sensitive >= total // 2, (sensitive, total)


def check_reduce_scatter_shards(orc, seed=9):
    """reduce_scatter's shard r is the all_reduce restricted to elements
    [r*C, (r+1)*C) of the inputs (input = world x output)."""
    rng = np.random.default_rng(seed)
    for P in (1, 2, 3, 8):
        C = int(rng.integers(1, 300))
        xs = [rng.integers(0, 65536, P * C, dtype=np.uint16) for _ in range(P)]
        for x in xs:
            x[(x & 0x7F80) == 0x7F80] &= 0xBFFF
        full = orc.all_reduce_bf16(xs)
        shards = orc.reduce_scatter_bf16(xs)
        assert len(shards) == P
        for r in range(P):
            assert np.array_equal(shards[r], full[r * C:(r + 1) * C]), (P, C, r)


def check_reduce_scatter_worked_example(orc):
    """P=2, C=2: in_0 = [1, 2, 3, 4], in_1 = [10, 20, 30, 40] (all exact in
    BF16): rank 0 gets [11, 22], rank 1 gets [33, 44]."""
    in0 = np.array([0x3F80, 0x4000, 0x4040, 0x4080], dtype=np.uint16)
    in1 = np.array([0x4120, 0x41A0, 0x41F0, 0x4220], dtype=np.uint16)
    out = orc.reduce_scatter_bf16([in0, in1])
    assert [int(v) for v in out[0]] == [0x4130, 0x41B0], [hex(int(v)) for v in out[0]]
    assert [int(v) for v in out[1]] == [0x4204, 0x4230], [hex(int(v)) for v in out[1]]


ALL_CHECKS = [
    check_gather_worked_examples,
    check_gather_matches_concatenate,
    check_gather_tiny_bruteforce,
    check_gather_identity_p1,
    check_gather_many_independent,
    check_rounding_matches_torch_cast,
    check_rounding_matches_exact,
    check_reduction_worked_examples,
    check_fold_matches_exact,
    check_fold_matches_torch_cpu,
    check_order_bruteforce,
    check_reduce_scatter_shards,
    check_reduce_scatter_worked_example,
]


# ------------------------------------------- other element types and orders ---

def load_typed_examples():
    rows = []
    with open(os.path.join(GOLDEN, "typed_reduction_worked_examples.txt")) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, dtype, order, ins, exp, _why = [c.strip() for c in line.split("|", 5)]
            rows.append((name, dtype, order, [int(h, 16) for h in ins.split()], int(exp, 16)))
    return rows


_NP = {"bf16": np.uint16, "f16": np.uint16, "f32": np.uint32}


def _bits(arr, dtype):
    return np.ascontiguousarray(arr).view(_NP[dtype])


def check_typed_worked_examples(orc):
    for name, dtype, order, inputs, expected in load_typed_examples():
        cols = [np.array([h], dtype=_NP[dtype]) for h in inputs]
        got = int(_bits(orc.all_reduce(cols, dtype, order), dtype)[0])
        assert got == expected, (name, hex(got), hex(expected))
        # every rank's output, and several copies of the column (no interaction)
        cols = [np.full(9, h, dtype=_NP[dtype]) for h in inputs]
        for out in orc.all_reduce_all_outputs(cols, dtype, order):
            assert (_bits(out, dtype) == expected).all(), (name, "all outputs")


def check_f16_rounding_matches_torch_cast(orc):
    """Library routine: torch's float32 -> float16 cast (round to nearest
    even)."""
    import torch

    u = _rounding_probe_values()
    # also the binary16 neighbourhoods: ties on the 13 dropped bits
    rng = np.random.default_rng(11)
    hi = rng.integers(0, 1 << 19, 4000, dtype=np.uint64)
    ties = ((hi << np.uint64(13)) | np.uint64(0x1000)).astype(np.uint32)
    u = np.concatenate([u, ties, ties - 1, ties + 1,
                        np.array([0x477FF000, 0x477FEFFF, 0x38800000, 0x387FFFFF, 0x33800000,
                                  0x33000000, 0x33000001, 0x337FFFFF, 0x00000001], dtype=np.uint32)])
    got = orc.f32_to_f16_rne_array(u)
    ref = torch.from_numpy(u.view(np.float32).copy()).to(torch.float16).view(torch.int16)
    ref = ref.numpy().view(np.uint16)
    nan = np.isnan(u.view(np.float32))
    assert np.array_equal(got[~nan], ref[~nan]), "binary16 rounding differs from torch's cast"
    assert all(((h & 0x7C00) == 0x7C00 and (h & 0x3FF)) for h in got[nan].tolist())


def check_f16_rounding_matches_exact(orc, seed=12):
    rng = np.random.default_rng(seed)
    u = np.concatenate([
        rng.integers(0, 1 << 32, 2000, dtype=np.uint64).astype(np.uint32),
        # values inside the binary16 range, where the rounding does work
        (rng.integers(0x33000000, 0x477FFFFF, 3000, dtype=np.uint64)).astype(np.uint32),
        np.array([0x477FF000, 0x477FEFFF, 0x38800000, 0x387FFFFF, 0x33000000, 0x33000001],
                 dtype=np.uint32),
    ])
    got = orc.f32_to_f16_rne_array(u)
    for ui, gi in zip(u.tolist(), got.tolist()):
        if (ui & 0x7F800000) == 0x7F800000:
            continue
        assert gi == ex.f32_to_f16_exact(ui), (hex(ui), hex(gi))


def check_f16_widening_exhaustive(orc):
    """Every binary16 pattern widens to the value torch's float16 -> float32
    cast gives (NaN by class)."""
    import torch

    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(h.view(np.int16).copy()).view(torch.float16).float().numpy()
    got = np.array([orc.f16_to_f32(int(x)) for x in range(0, 65536, 1)], dtype=np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def _typed_column(rng, P, dtype, wide):
    out = []
    for _ in range(P):
        s = int(rng.integers(0, 2))
        if dtype == "bf16":
            e = int(rng.integers(1, 255)) if wide else int(rng.integers(120, 131))
            out.append((s << 15) | (e << 7) | int(rng.integers(0, 128)))
        elif dtype == "f16":
            e = int(rng.integers(0, 31)) if wide else int(rng.integers(12, 18))
            out.append((s << 15) | (e << 10) | int(rng.integers(0, 1024)))
        else:
            e = int(rng.integers(1, 255)) if wide else int(rng.integers(120, 131))
            out.append((s << 31) | (e << 23) | int(rng.integers(0, 1 << 23)))
    return out


def check_typed_folds_match_exact(orc, seed=13, n_cols=120):
    """Exact rational fold (every binary32 add and the final rounding from
    their definitions) for every element type, both orders, several P."""
    rng = np.random.default_rng(seed)
    for dtype in ("bf16", "f16", "f32"):
        for order in ("linear", "tree"):
            for P in (1, 2, 3, 4, 5, 6, 7, 8, 13):
                cols = []
                for k in range(n_cols):
                    while True:
                        c = _typed_column(rng, P, dtype, wide=(k % 3 == 0))
                        try:
                            cols.append((c, ex.fold_exact(c, dtype, order)))
                            break
                        except ValueError:
                            continue
                inputs = [np.array([c[r] for c, _ in cols], dtype=_NP[dtype]) for r in range(P)]
                got = _bits(orc.all_reduce(inputs, dtype, order), dtype)
                for k, (c, e) in enumerate(cols):
                    assert int(got[k]) == e, (dtype, order, P, [hex(h) for h in c], hex(int(got[k])), hex(e))


def check_typed_linear_matches_torch_cpu(orc, seed=14):
    """Library routine: torch CPU binary32 adds in rank order, then torch's
    cast back, for float16 and float32 (and the bfloat16 path again)."""
    import torch

    rng = np.random.default_rng(seed)
    for dtype, tdt in (("f16", torch.float16), ("f32", torch.float32), ("bf16", torch.bfloat16)):
        for P in (2, 3, 8):
            xs = [_bits(np.array(_typed_column(rng, 4000, dtype, wide=False)), dtype) for _ in range(1)]
            cols = [np.array(_typed_column(rng, 4000, dtype, wide=False), dtype=_NP[dtype]) for _ in range(P)]
            t = [torch.from_numpy(c.view(np.int16 if dtype != "f32" else np.int32).copy()).view(tdt) for c in cols]
            acc = t[0].float()
            for q in range(1, P):
                acc = acc + t[q].float()
            ref = acc.to(tdt).view(torch.int16 if dtype != "f32" else torch.int32).numpy().view(_NP[dtype])
            got = _bits(orc.all_reduce(cols, dtype, "linear"), dtype)
            assert np.array_equal(got, ref), (dtype, P)
            del xs


def check_tree_order_bruteforce(orc):
    """Every rank permutation of order-sensitive columns in the tree order:
    the oracle equals the exact tree fold in that rank order, and the tree
    and linear orders disagree on some of them."""
    small = [0x3F80, 0xBF80, 0x3B80, 0xBB80, 0x3C00, 0xBC00, 0x4000, 0x4B80]
    rng = random.Random(15)
    differs = total = 0
    for P in (4, 5, 6):
        for _ in range(6):
            big = rng.choice([0x4B80, 0xCB80])
            col = [big, big ^ 0x8000] + [rng.choice(small) for _ in range(P - 2)]
            perms = sorted(set(itertools.permutations(col)))[:400]
            inputs = [np.array([p[r] for p in perms], dtype=np.uint16) for r in range(P)]
            got = orc.all_reduce(inputs, "bf16", "tree")
            lin = orc.all_reduce(inputs, "bf16", "linear")
            exact = [ex.fold_exact(list(p), "bf16", "tree") for p in perms]
            assert [int(g) for g in got] == exact, (P, col)
            total += 1
            differs += int(not np.array_equal(got, lin))
    assert differs >= total // 2, (differs, total)


def check_typed_reduce_scatter_shards(orc, seed=16):
    rng = np.random.default_rng(seed)
    for dtype in ("bf16", "f16", "f32"):
        for order in ("linear", "tree"):
            P, C = int(rng.integers(1, 9)), int(rng.integers(1, 200))
            xs = [np.array(_typed_column(rng, P * C, dtype, wide=False), dtype=_NP[dtype]) for _ in range(P)]
            full = _bits(orc.all_reduce(xs, dtype, order), dtype)
            shards = orc.reduce_scatter(xs, dtype, order)
            for r in range(P):
                assert np.array_equal(_bits(shards[r], dtype), full[r * C:(r + 1) * C]), (dtype, order, r)


def check_bf16_entry_points_agree(orc, seed=17):
    """The BF16 functions and the typed functions with bf16 / linear are the
    same fold."""
    rng = np.random.default_rng(seed)
    xs = [rng.integers(0, 65536, 3000, dtype=np.uint16) for _ in range(5)]
    assert np.array_equal(orc.all_reduce_bf16(xs).view(np.uint8),
                          orc.all_reduce(xs, "bf16", "linear").view(np.uint8))


ALL_CHECKS += [
    check_typed_worked_examples,
    check_f16_rounding_matches_torch_cast,
    check_f16_rounding_matches_exact,
    check_f16_widening_exhaustive,
    check_typed_folds_match_exact,
    check_typed_linear_matches_torch_cpu,
    check_tree_order_bruteforce,
    check_typed_reduce_scatter_shards,
    check_bf16_entry_points_agree,
]
