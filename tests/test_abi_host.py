"""C-ABI checks that need no GPU: the library loads, exports every function
declared in include/dc.h, and rejects bad arguments before any CUDA call.

Pointers here are fake device addresses: every rejected call returns before
touching them.  Calls that pass validation use the ``test_fail_launch``
option, which makes the library report a launch failure instead of
launching, so nothing here ever reaches a GPU.
"""
from __future__ import annotations

import os
import re
import threading

import pytest

import reduce_copy_rank_gb300 as dc
from reduce_copy_rank_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dc.h")

OK, INVALID, ALIGN, OVERLAP, TOO_MANY, CUDA = 0, 1, 2, 3, 4, 5
BASE = 0x7F00_0000_0000  # a fake, 256-byte aligned device address


@pytest.fixture(scope="module", autouse=True)
def built_library():
    _build.build()
    dc.lib()
    yield


@pytest.fixture
def no_launch():
    with dc.options(test_fail_launch=1):
        yield


def declared_functions() -> list[str]:
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dc_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for needed in ("dc_all_gather", "dc_all_gather_many", "dc_all_reduce_bf16",
                   "dc_reduce_scatter_bf16", "dc_last_error", "dc_set_option"):
        assert needed in names


def test_library_exports_every_declared_function():
    L = dc.lib()
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_which_build_is_loaded():
    """libdc.so unless DC_LIBRARY=bounds selects the bounds-checked build."""
    want = 1 if os.environ.get("DC_LIBRARY") == "bounds" else 0
    assert dc.lib().dc_bounds_checked() == want


def test_version_and_status_names():
    assert dc.lib().dc_version() == 1
    for code, name in dc.STATUS.items():
        assert dc.lib().dc_status_name(code).decode() == name


# ------------------------------------------------------------- all_gather ---

def test_gather_rejects_bad_rank_counts():
    assert dc.dc_all_gather([], 0, 16, BASE) == INVALID
    assert "P = 0" in dc.last_error()
    assert dc.dc_all_gather([BASE] * 65, 65, 16, BASE + (1 << 30)) == INVALID


def test_gather_zero_bytes_is_a_noop_without_launch():
    before = dc.launch_count()
    assert dc.dc_all_gather([0, 0], 2, 0, 0) == OK
    assert dc.launch_count() == before


def test_gather_rejects_null_pointers():
    assert dc.dc_all_gather([BASE, 0], 2, 16, BASE + 4096) == INVALID
    assert dc.dc_all_gather([BASE, BASE + 64], 2, 16, 0) == INVALID


@pytest.mark.parametrize("out_off", [-31, -1, 0, 1, 15])
def test_gather_rejects_overlap(out_off):
    peers = [BASE + 1024, BASE + 2048]
    out = peers[1] + out_off  # a 32-byte output starting here touches rank 1's 16 bytes
    assert dc.dc_all_gather(peers, 2, 16, out) == OVERLAP
    assert "overlaps" in dc.last_error()


@pytest.mark.parametrize("out_off", [-32, 16])
def test_gather_adjacent_is_not_overlap(no_launch, out_off):
    peers = [BASE + 1024, BASE + 2048]
    assert dc.dc_all_gather(peers, 2, 16, peers[1] + out_off) == CUDA  # passed validation
    assert "injected" in dc.last_error()


def test_gather_peers_may_repeat(no_launch):
    assert dc.dc_all_gather([BASE, BASE, BASE], 3, 100, BASE + 4096) == CUDA


def test_gather_rejects_size_overflow():
    assert dc.dc_all_gather([BASE, BASE], 2, (1 << 63) + 1, BASE + 4096) == INVALID


# -------------------------------------------------------- all_gather_many ---

def test_many_limits():
    P = 8
    T = 129  # 1032 segments
    assert dc.dc_all_gather_many([BASE] * (T * P), [16] * T, [BASE + 4096] * T, T, P) == TOO_MANY
    assert dc.dc_all_gather_many([BASE] * 257, [16] * 257, [BASE] * 257, 257, 1) == TOO_MANY
    assert dc.dc_all_gather_many([], [], [], 0, 4) == OK


def test_many_rejects_overlapping_outputs():
    P = 2
    peers = [BASE, BASE + 64, BASE + 128, BASE + 192]
    outs = [BASE + 4096, BASE + 4096 + 16]  # first output is 32 bytes long
    assert dc.dc_all_gather_many(peers, [16, 16], outs, 2, P) == OVERLAP


def test_many_rejects_output_over_another_tensors_payload():
    P = 2
    peers = [BASE, BASE + 64, BASE + 4096, BASE + 128]  # tensor 1 rank 0 sits in output 0
    outs = [BASE + 4096, BASE + 8192]
    assert dc.dc_all_gather_many(peers, [16, 16], outs, 2, P) == OVERLAP


def test_many_zero_sized_tensors_are_skipped(no_launch):
    before = dc.launch_count()
    assert dc.dc_all_gather_many([0, 0, 0, 0], [0, 0], [0, 0], 2, 2) == OK
    assert dc.launch_count() == before
    peers = [0, 0, BASE, BASE + 64]
    assert dc.dc_all_gather_many(peers, [0, 32], [0, BASE + 4096], 2, 2) == CUDA


def _many_overlap_model(peers, sizes, outs, T, P):
    """The rule of dc_all_gather_many, pair by pair: an output may overlap no
    other output and no payload; payloads may overlap each other."""
    if not any(sizes[:T]):
        return OK  # nothing to gather: a no-op
    rng = []
    for t in range(T):
        if sizes[t] == 0:
            continue
        rng.append((outs[t], outs[t] + P * sizes[t], True))
        rng.extend((peers[t * P + r], peers[t * P + r] + sizes[t], False) for r in range(P))
    for i in range(len(rng)):
        for k in range(i + 1, len(rng)):
            a, b = rng[i], rng[k]
            if (a[2] or b[2]) and a[0] < b[1] and b[0] < a[1]:
                return OVERLAP
    return CUDA


def test_many_overlap_check_matches_pairwise_model(no_launch):
    import random

    rnd = random.Random(0xDC17)
    for _ in range(400):
        P, T = rnd.randint(1, 5), rnd.randint(1, 6)
        sizes = [rnd.choice([0, 1, 16, 100, 4096]) for _ in range(T)]
        slots = [BASE + k * 8192 for k in range(10)]
        peers = [rnd.choice(slots) + rnd.choice([0, 1, 16, 4000]) for _ in range(T * P)]
        outs = [rnd.choice(slots) + rnd.choice([0, 3, 2048, 8000]) for _ in range(T)]
        want = _many_overlap_model(peers, sizes, outs, T, P)
        got = dc.dc_all_gather_many(peers, sizes, outs, T, P)
        assert got == want, (peers, sizes, outs, T, P, dc.last_error())


def test_many_overlap_check_at_the_table_limits(no_launch):
    """T = 256 tensors x P = 4 ranks (1024 payloads): a clean layout passes,
    one planted payload inside an output, or two touching outputs that
    overlap by one byte, are found; the check is a sort and one sweep, so a
    call costs microseconds of host time, not the ~0.3 M range tests of an
    all-pairs check."""
    import time

    T, P, B = 256, 4, 4096
    peers = [BASE + (t * P + r) * 2 * B for t in range(T) for r in range(P)]
    out0 = BASE + (T * P + 16) * 2 * B
    outs = [out0 + t * P * B for t in range(T)]  # back to back, not overlapping
    assert dc.dc_all_gather_many(peers, [B] * T, outs, T, P) == CUDA
    t0 = time.perf_counter()
    for _ in range(20):
        dc.dc_all_gather_many(peers, [B] * T, outs, T, P)
    per_call_us = (time.perf_counter() - t0) / 20 * 1e6
    print(f"all_gather_many validation at T={T}, P={P}: {per_call_us:.1f} us of host time per call")
    assert per_call_us < 20000
    planted = list(peers)
    planted[T * P - 1] = outs[100] + 17  # tensor 255 rank 3's payload inside output 100
    assert dc.dc_all_gather_many(planted, [B] * T, outs, T, P) == OVERLAP
    assert "output of tensor 100 overlaps the payload of tensor 255 rank 3" in dc.last_error()
    bumped = list(outs)
    bumped[201] -= 1  # output 201 starts one byte inside output 200
    assert dc.dc_all_gather_many(peers, [B] * T, bumped, T, P) == OVERLAP
    assert "outputs of tensors 200 and 201 overlap" in dc.last_error()


# ------------------------------------------------------------- reductions ---

def test_reduce_rejects_misaligned_bf16():
    ins = [BASE, BASE + 1024 + 1]
    outs = [BASE + 4096, BASE + 8192]
    assert dc.dc_all_reduce_bf16(ins, outs, 2, 8) == ALIGN
    assert dc.dc_reduce_scatter_bf16(ins, outs, 2, 8) == ALIGN


def test_reduce_zero_count_is_a_noop():
    before = dc.launch_count()
    assert dc.dc_all_reduce_bf16([0] * 4, [0] * 4, 4, 0) == OK
    assert dc.dc_reduce_scatter_bf16([0] * 4, [0] * 4, 4, 0) == OK
    assert dc.launch_count() == before


def test_all_reduce_in_place_allowed(no_launch):
    ins = [BASE + i * 4096 for i in range(4)]
    assert dc.dc_all_reduce_bf16(ins, ins, 4, 100) == CUDA  # validation passed
    # outputs that are other ranks' inputs are also exact aliases
    assert dc.dc_all_reduce_bf16(ins, ins[::-1], 4, 100) == CUDA


def test_all_reduce_rejects_partial_overlap():
    ins = [BASE + i * 4096 for i in range(4)]
    outs = [BASE + 64 * 1024 + i * 4096 for i in range(4)]
    outs[2] = ins[1] + 2  # shifted by one element
    assert dc.dc_all_reduce_bf16(ins, outs, 4, 100) == OVERLAP
    outs[2] = outs[1] + 100  # two outputs overlap
    assert dc.dc_all_reduce_bf16(ins, outs, 4, 100) == OVERLAP


def test_reduce_scatter_in_place_shard_allowed(no_launch):
    P, C = 4, 64
    ins = [BASE + i * 4096 for i in range(P)]
    outs = [ins[r] + 2 * r * C for r in range(P)]  # each rank's own shard
    assert dc.dc_reduce_scatter_bf16(ins, outs, P, C) == CUDA


def test_reduce_scatter_rejects_other_shard():
    P, C = 4, 64
    ins = [BASE + i * 4096 for i in range(P)]
    outs = [BASE + 64 * 1024 + r * 1024 for r in range(P)]
    outs[1] = ins[0]  # shard 0 of input 0 is not rank 1's shard
    assert dc.dc_reduce_scatter_bf16(ins, outs, P, C) == OVERLAP


def test_reduce_rejects_null():
    assert dc.dc_all_reduce_bf16([BASE, 0], [BASE + 4096, BASE + 8192], 2, 8) == INVALID


# ---------------------------------------------------------------- options ---

def test_options_roundtrip():
    assert dc.get_option("force_path") in (0, 1, 2)
    with dc.options(force_path=2, grid_ctas=7):
        assert dc.get_option("force_path") == 2
        assert dc.get_option("grid_ctas") == 7
    assert dc.lib().dc_set_option(b"no_such_option", 1) == -1
    assert dc.lib().dc_get_option(b"no_such_option") == -1
    assert dc.lib().dc_set_option(b"grid_ctas", -5) == -1


def test_rejected_calls_launch_nothing():
    before = dc.launch_count()
    dc.dc_all_gather([BASE], 1, 16, BASE + 8)
    dc.dc_all_reduce_bf16([BASE + 1], [BASE + 4096], 1, 4)
    assert dc.launch_count() == before


def test_last_error_is_per_thread():
    msgs = {}

    def worker(name, P):
        dc.dc_all_gather([BASE] * max(P, 1), P, 16, BASE + 4096)
        msgs[name] = dc.last_error()

    t1 = threading.Thread(target=worker, args=("a", 0))
    t1.start()
    t1.join()
    dc.dc_all_gather([BASE, BASE], 2, 16, BASE + 8)  # overlap on this thread
    assert "P = 0" in msgs["a"]
    assert "overlaps" in dc.last_error()


def test_tensor_api_requires_cuda_tensors():
    import torch

    x = torch.zeros(16, dtype=torch.uint8)
    with pytest.raises(ValueError):
        dc.all_gather([x], torch.zeros(16, dtype=torch.uint8))


# ------------------------------------------------- typed and batched reductions ---

def test_typed_reduce_rejects_bad_type_and_order():
    ins = [BASE, BASE + 4096]
    outs = [BASE + 8192, BASE + 12288]
    assert dc.dc_all_reduce(ins, outs, 2, 8, 3, 0) == INVALID
    assert dc.dc_all_reduce(ins, outs, 2, 8, 0, 2) == INVALID
    assert dc.dc_reduce_scatter(ins, outs, 2, 8, -1, 0) == INVALID


def test_f32_needs_4_byte_alignment(no_launch):
    ins = [BASE, BASE + 4096 + 2]
    outs = [BASE + 8192, BASE + 12288]
    assert dc.dc_all_reduce(ins, outs, 2, 8, 2, 0) == ALIGN
    assert dc.dc_all_reduce(ins, outs, 2, 8, 1, 0) == CUDA  # 2-byte aligned is enough for FP16


def test_batched_reduce_limits():
    P = 8
    assert dc.dc_all_reduce_many([BASE] * (257 * 1), [BASE] * 257, [4] * 257, 257, 1) == TOO_MANY
    T = 65  # 2 * 65 * 8 = 1040 pointers
    assert dc.dc_all_reduce_many([BASE] * (T * P), [BASE] * (T * P), [4] * T, T, P) == TOO_MANY
    T = 33  # 264 reduce_scatter jobs
    assert dc.dc_reduce_scatter_many([BASE] * (T * P), [BASE] * (T * P), [4] * T, T, P) == TOO_MANY
    assert dc.dc_all_reduce_many([], [], [], 0, P) == OK


def test_batched_reduce_aliasing(no_launch):
    P, n = 2, 64
    ins = [BASE + i * 4096 for i in range(2 * P)]        # tensor 0: 0,1  tensor 1: 2,3
    outs = [BASE + 65536 + i * 4096 for i in range(2 * P)]
    assert dc.dc_all_reduce_many(ins, outs, [n, n], 2, P) == CUDA
    outs_inplace = [ins[0], ins[1], ins[2], ins[3]]     # each tensor in place
    assert dc.dc_all_reduce_many(ins, outs_inplace, [n, n], 2, P) == CUDA
    outs_cross = [outs[0], outs[1], ins[0], outs[3]]    # tensor 1 writes over tensor 0's input
    assert dc.dc_all_reduce_many(ins, outs_cross, [n, n], 2, P) == OVERLAP
    assert "tensor 1" in dc.last_error()


def test_batched_reduce_scatter_inplace_shards(no_launch):
    P, C = 4, 32
    ins = [BASE + i * 8192 for i in range(2 * P)]
    outs = [ins[t * P + r] + 2 * r * C for t in range(2) for r in range(P)]
    assert dc.dc_reduce_scatter_many(ins, outs, [C, C], 2, P) == CUDA
    outs[5] = ins[0] + 2 * 1 * C  # tensor 1 rank 1 writes into tensor 0's input
    assert dc.dc_reduce_scatter_many(ins, outs, [C, C], 2, P) == OVERLAP


def test_batched_zero_counts_launch_nothing():
    before = dc.launch_count()
    assert dc.dc_all_reduce_many([0] * 6, [0] * 6, [0, 0, 0], 3, 2) == OK
    assert dc.dc_reduce_scatter_many([0] * 6, [0] * 6, [0, 0, 0], 3, 2) == OK
    assert dc.launch_count() == before


def test_delay_limit_checked_before_cuda(no_launch):
    assert dc.dc_inject_delay_ns(dc.MAX_DELAY_NS + 1, 0) == 1  # DC_ERR_INVALID
    assert "limit" in dc.last_error()
    # a valid request reaches the (refused) launch
    assert dc.dc_inject_delay_ns(0, 0) == 5
    assert dc.dc_inject_delay_ns(dc.MAX_DELAY_NS, 0) == 5


def test_every_documented_option_exists_and_round_trips():
    keys = re.findall(r'\*   "([a-z_]+)"', open(HEADER).read())
    assert {"gather_single_max_bytes", "reduce_single_max_bytes", "prefetch",
            "gather_split_cost_pct", "gather_staged", "pdl", "gather_tile_min",
            "reduce_tile_min", "reduce_staged"} <= set(keys)
    for k in keys:
        v = dc.get_option(k)
        assert v >= 0, k
        with dc.options(**{k: v}):
            assert dc.get_option(k) == v


class _FakeCudaTensor:
    """Just enough of a CUDA tensor for the binding's checks (never launched)."""

    def __init__(self, nbytes, device_index, dtype=None):
        import torch

        self.is_cuda = True
        self.nbytes = nbytes
        self.dtype = dtype if dtype is not None else torch.uint8
        self._dev = device_index
        self.device = f"cuda:{device_index}"

    def is_contiguous(self):
        return True

    def get_device(self):
        return self._dev

    def numel(self):
        return self.nbytes

    def element_size(self):
        return 1

    def data_ptr(self):
        return 0x10000 * (self._dev + 1)


def test_tensors_on_another_device_are_rejected(monkeypatch):
    """The library launches on the current device; a tensor elsewhere must be
    refused before the call, not fault the kernel."""
    monkeypatch.setattr(dc, "_cur_dev", lambda: 0)
    peers = [_FakeCudaTensor(64, 0), _FakeCudaTensor(64, 1)]
    with pytest.raises(ValueError, match="current device"):
        dc.all_gather(peers, _FakeCudaTensor(128, 0))
    with pytest.raises(ValueError, match="current device"):
        dc.all_gather([_FakeCudaTensor(64, 0)], _FakeCudaTensor(64, 1))
    with pytest.raises(ValueError, match="current device"):
        dc.all_gather_many([[_FakeCudaTensor(64, 0)]], [_FakeCudaTensor(64, 2)])
    with pytest.raises(ValueError, match="current device"):
        dc.all_reduce([_FakeCudaTensor(64, 0), _FakeCudaTensor(64, 0)],
                      [_FakeCudaTensor(64, 0), _FakeCudaTensor(64, 3)])


# ------------------------------------------------- one rank's reduction ---

def test_reduce_rejects_bad_arguments():
    ins = [BASE, BASE + 4096]
    out = BASE + 8192
    assert dc.dc_reduce(ins, 0, 0, 8, out) == INVALID
    assert dc.dc_reduce([BASE] * 65, 65, 0, 8, out) == INVALID
    assert dc.dc_reduce(ins, 2, 0, 8, out, dtype=3) == INVALID
    assert dc.dc_reduce(ins, 2, 0, 8, out, order=2) == INVALID
    assert dc.dc_reduce([BASE, 0], 2, 0, 8, out) == INVALID
    assert dc.dc_reduce(ins, 2, 0, 8, 0) == INVALID
    assert dc.dc_reduce(ins, 2, 1 << 63, 1 << 63, out) == INVALID  # offset + count overflows
    assert "overflows" in dc.last_error()


def test_reduce_alignment_follows_the_element_type(no_launch):
    ins = [BASE, BASE + 4096]
    assert dc.dc_reduce(ins, 2, 0, 8, BASE + 8193) == ALIGN           # BF16 output at an odd byte
    assert dc.dc_reduce([BASE + 1, BASE + 4096], 2, 0, 8, BASE + 8192) == ALIGN
    assert dc.dc_reduce(ins, 2, 0, 8, BASE + 8194, dtype=2) == ALIGN  # FP32 at 2 mod 4
    assert dc.dc_reduce(ins, 2, 0, 8, BASE + 8194) == CUDA            # BF16 at 2 mod 16: fine


def test_reduce_zero_count_is_a_noop_without_launch():
    before = dc.launch_count()
    assert dc.dc_reduce([0, 0], 2, 0, 0, 0) == OK
    assert dc.launch_count() == before


@pytest.mark.parametrize("shift", [-2, 2, 14])
def test_reduce_rejects_partial_overlap_with_the_elements_read(shift):
    ins = [BASE, BASE + 4096]
    # reads elements [16, 24) of every input (BF16): bytes [32, 48) of each
    assert dc.dc_reduce(ins, 2, 16, 8, BASE + 4096 + 32 + shift) == OVERLAP
    assert "overlaps" in dc.last_error()


def test_reduce_in_place_and_unread_overlaps_are_allowed(no_launch):
    ins = [BASE, BASE + 4096]
    assert dc.dc_reduce(ins, 2, 16, 8, BASE + 4096 + 32) == CUDA  # exactly the range read: in place
    assert dc.dc_reduce(ins, 2, 16, 8, BASE + 4096) == CUDA       # input 1's unread elements [0, 8)
    assert dc.dc_reduce(ins, 2, 16, 8, BASE + 4096 + 48) == CUDA  # just past the range read
    assert dc.dc_reduce([BASE, BASE], 2, 0, 8, BASE + 4096) == CUDA  # inputs may repeat


# ------------------------------------------------------- fused all-gather ---

def _fused_layout(P, B, base=BASE):
    """Disjoint, 256-byte spaced inputs, staging buffers, outputs and workspace."""
    step = ((P * B + 255) // 256) * 256 + 256
    ins = [base + r * step for r in range(P)]
    stg = [base + (P + r) * step for r in range(P)]
    outs = [base + (2 * P + r) * step for r in range(P)]
    ws = base + 3 * P * step
    return ins, stg, outs, ws


def test_fused_workspace_size():
    assert dc.dc_fused_workspace_bytes(0) == 0 and dc.dc_fused_workspace_bytes(65) == 0
    assert dc.dc_fused_workspace_bytes(8) == 8 * 128 * 2 * 4


def test_fused_argument_checks(no_launch):
    P, B = 4, 4096
    ins, stg, outs, ws = _fused_layout(P, B)
    assert dc.dc_fused_all_gather(ins, stg, outs, P, B, ws, 1) == CUDA  # valid: reaches the launch
    assert dc.dc_fused_all_gather(ins, stg, outs, P, 0, ws, 1) == OK  # zero bytes: a no-op
    assert dc.dc_fused_all_gather(ins, stg, outs, 0, B, ws, 1) == INVALID
    assert dc.dc_fused_all_gather(ins, stg, outs, P, B, ws, 0) == INVALID  # epoch 0 is reserved
    assert dc.dc_fused_all_gather(ins, stg, outs, P, B, 0, 1) == INVALID
    assert dc.dc_fused_all_gather(ins, stg, outs, P, B + 8, ws, 1) == ALIGN
    assert dc.dc_fused_all_gather(ins, stg, [outs[0] + 8] + outs[1:], P, B, ws, 1) == ALIGN
    assert dc.dc_fused_all_gather(ins, [0] + stg[1:], outs, P, B, ws, 1) == INVALID
    # inputs may overlap inputs (the same payload on every rank)
    assert dc.dc_fused_all_gather([ins[0]] * P, stg, outs, P, B, ws, 1) == CUDA
    # a staging buffer inside another rank's input, an output over the workspace,
    # two staging buffers on one another
    assert dc.dc_fused_all_gather(ins, [ins[1]] + stg[1:], outs, P, B, ws, 1) == OVERLAP
    assert "staging buffer of rank 0" in dc.last_error() or "input of rank 1" in dc.last_error()
    assert dc.dc_fused_all_gather(ins, stg, outs[:-1] + [ws - 16], P, B, ws, 1) == OVERLAP
    assert dc.dc_fused_all_gather(ins, [stg[0], stg[0] + 16] + stg[2:], outs, P, B, ws, 1) == OVERLAP


def test_fused_reset_checks():
    assert dc.dc_fused_reset(0, 4) == INVALID
    assert dc.dc_fused_reset(BASE, 0) == INVALID
