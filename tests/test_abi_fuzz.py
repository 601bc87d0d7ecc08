"""Randomised checks of the C ABI's argument validation against a model of
the rules include/dc.h states (no GPU: calls that pass validation report
DC_ERR_CUDA through the test_fail_launch option instead of launching).

Rules modelled (the header fixes no priority between two faults of one
call, so the model takes the library's order): rank count and type checks,
table limits; for the reductions, for every live tensor and rank a NULL
pointer (DC_ERR_INVALID) or a pointer not aligned to the element size
(DC_ERR_ALIGN), then overlaps: two outputs (DC_ERR_OVERLAP), or an output
and an input unless the output is exactly that input (all_reduce) or
exactly its own shard of it (reduce_scatter); for the gather, rank by rank
a NULL payload or one overlapping the output.
"""
from __future__ import annotations

import pytest

import reduce_copy_rank_gb300 as dc

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")
from hypothesis import given, settings  # noqa: E402

OK, INVALID, ALIGN, OVERLAP, TOO_MANY, CUDA = 0, 1, 2, 3, 4, 5
ESIZE = {0: 2, 1: 2, 2: 4}


@pytest.fixture(autouse=True)
def no_launch():
    with dc.options(test_fail_launch=1):
        yield


def model_reduce(ins, outs, counts, T, P, dtype, scatter):
    if not 1 <= P <= 64:
        return INVALID
    jobs = T * (P if scatter else 1)
    if jobs > 256 or 2 * T * P > 1024:
        return TOO_MANY
    live = [t for t in range(T) if counts[t]]
    if not live:
        return OK
    es = ESIZE[dtype]
    ranges = []
    for t in live:
        n = counts[t]
        out_b = n * es
        in_b = out_b * (P if scatter else 1)
        for q in range(P):
            i, o = ins[t * P + q], outs[t * P + q]
            if i == 0 or o == 0:
                return INVALID
            if (i | o) % es:
                return ALIGN
            ranges.append((i, i + in_b, t, q, False))
            ranges.append((o, o + out_b, t, q, True))
    for x in range(len(ranges)):
        for y in range(x + 1, len(ranges)):
            a, b = ranges[x], ranges[y]
            if not (a[0] < b[1] and b[0] < a[1]):
                continue
            if not a[4] and not b[4]:
                continue
            if a[4] and b[4]:
                return OVERLAP
            o, i = (a, b) if a[4] else (b, a)
            alias = i[0] + (o[3] * counts[o[2]] * es if scatter else 0)
            if not (o[2] == i[2] and o[0] == alias):
                return OVERLAP
    return CUDA


def model_gather(peers, P, B, out):
    if not 1 <= P <= 64:
        return INVALID
    if B == 0:
        return OK
    if out == 0:
        return INVALID
    for r in range(P):  # rank by rank: a NULL payload, then its overlap with the output
        if peers[r] == 0:
            return INVALID
        if out < peers[r] + B and peers[r] < out + P * B:
            return OVERLAP
    return CUDA


# Buffers are drawn from a few 64 KiB slots so that overlaps, exact aliases
# and shard aliases all occur; offsets include odd and 2-mod-4 addresses.
SLOT = 1 << 16
offsets = st.sampled_from([0, 0, 0, 2, 16, 18, 1, 3, 4096])


@st.composite
def reduce_case(draw):
    P = draw(st.integers(1, 6))
    T = draw(st.integers(1, 3))
    dtype = draw(st.sampled_from([0, 1, 2]))
    scatter = draw(st.booleans())
    counts = [draw(st.sampled_from([0, 1, 5, 64])) for _ in range(T)]
    ins, outs = [], []
    for t in range(T):
        for q in range(P):
            ins.append(draw(st.integers(1, 6)) * SLOT + draw(offsets))
        for q in range(P):
            how = draw(st.sampled_from(["fresh", "fresh", "alias", "shard", "null"]))
            if how == "alias":
                outs.append(ins[t * P + draw(st.integers(0, P - 1))])
            elif how == "shard":
                outs.append(ins[t * P + draw(st.integers(0, P - 1))] + q * counts[t] * ESIZE[dtype])
            elif how == "null":
                outs.append(0)
            else:
                outs.append(draw(st.integers(7, 12)) * SLOT + draw(offsets))
    return ins, outs, counts, T, P, dtype, scatter


@settings(max_examples=400, deadline=None)
@given(reduce_case())
def test_reduce_validation_matches_model(case):
    ins, outs, counts, T, P, dtype, scatter = case
    want = model_reduce(ins, outs, counts, T, P, dtype, scatter)
    fn = dc.dc_reduce_scatter_many if scatter else dc.dc_all_reduce_many
    got = fn(ins, outs, counts, T, P, dtype, 0, 0)
    assert got == want, (case, dc.last_error())


@st.composite
def gather_case(draw):
    P = draw(st.integers(1, 6))
    B = draw(st.sampled_from([0, 1, 15, 16, 4096, 70000]))
    peers = [0 if draw(st.integers(0, 20)) == 0 else draw(st.integers(1, 6)) * SLOT + draw(offsets)
             for _ in range(P)]
    out = draw(st.sampled_from([0, 1])) * draw(st.integers(1, 8)) * SLOT + draw(offsets)
    return peers, P, B, out


@settings(max_examples=400, deadline=None)
@given(gather_case())
def test_gather_validation_matches_model(case):
    peers, P, B, out = case
    got = dc.dc_all_gather(peers, P, B, out, 0)
    assert got == model_gather(peers, P, B, out), (case, dc.last_error())
