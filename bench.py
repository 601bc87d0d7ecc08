#!/usr/bin/env python3
"""Benchmark of the deterministic rank-ordered all-gather (and, beside it,
the fixed-order BF16 reductions) on one GB300.

Metric: all-gather / all-reduce GB/s and us per call vs size, and the
fraction of the HBM roofline (bytes read + bytes written per call).

Workload of the headline line: the all-gather sweep with P=8 and P=2
simulated ranks, per-rank sizes 1, 8, 32, 64, 128 KiB, 1 MiB and 4 MiB of
BF16 bit patterns, 16-byte aligned (the sizes of the results tables of
"perf(cuda): vectorize the deterministic all-gather copy and right-size its
single-block path").  One step = the 14 gathers of the sweep, captured once
into a CUDA graph and replayed: an L2 flush (write, then read, of a buffer
four times the L2 size), a timing event, the 14 calls back to back, a timing
event.  Inputs are resident in HBM; every call reads inputs that no kernel
has touched since the flush, so they come from HBM.  `value` = algorithmic
bytes of a step / the time between the two events.  In the same timed
region every call is also timed on its own (flush, event, the one launch,
event): that gives `per_call` (us per call vs size, as the page reports it)
and the roofline's per-launch duration.  Events between back-to-back calls
would add about 3 us each, so the step is timed at its two ends only.

Usage:
  python bench.py [--gpus N] [--steps K] [--warmup W]        # this library
  python bench.py --impl reference [--steps K] [--warmup W]  # the oracle on host cores
  python bench.py --crossover                                 # single/multi-CTA sweep
For N > 1 launch one process per GPU with torch.distributed.run; each rank
runs the same workload on its own GPU (replicas: the path has no exchange
step between GPUs) and rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "all-gather / all-reduce GB/s and us per call vs size at 1 GB300; % HBM roofline"
UNIT = "GB/s"
WORKLOAD = ("all-gather sweep: P=8 and P=2 simulated ranks x {1, 8, 32, 64, 128 KiB, 1 MiB, "
            "4 MiB} per rank of BF16 bit patterns, 16-byte aligned; one step = the 14 gathers")
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0  # the ~8 TB/s HBM3e figure: a second denominator beside the measured copy rate
KIB = 1024
MIB = 1024 * KIB


def workload_config(world: int) -> dict:
    """The `config` of the JSON line, the same dict for both arms."""
    return {"workload": WORKLOAD, "P": [8, 2], "bytes_per_rank": W.CONFIG2_SIZES,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["dc", "reference"], default="dc")
    ap.add_argument("--no-reductions", action="store_true",
                    help="skip the all_reduce / reduce_scatter / all_gather_many block")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-comparators", action="store_true",
                    help="skip the torch comparators and the warm back-to-back latency graphs")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU time budget of the oracle baseline sample")
    ap.add_argument("--crossover", action="store_true", help="run the single/multi-CTA sweep")
    ap.add_argument("--skew", action="store_true",
                    help="rank-skew calibration of all_reduce on simulated ranks (one JSON line "
                         "per mode, P, shape and requested delay)")
    ap.add_argument("--skew-shapes", nargs="+", default=["8x8192", "8627x8192", "16384x8192"])
    ap.add_argument("--skew-delays-us", nargs="+", type=float, default=[0.0, 50.0, 250.0, 1000.0])
    ap.add_argument("--skew-ranks", nargs="+", type=int, default=[2, 4],
                    help="simulated rank counts P")
    ap.add_argument("--skew-rank", type=int, default=None,
                    help="the delayed rank (default: the last one)")
    ap.add_argument("--skew-modes", nargs="+", choices=["graph", "eager"], default=["graph", "eager"])
    ap.add_argument("--skew-trials", type=int, default=50)
    ap.add_argument("--skew-warmup", type=int, default=10)
    ap.add_argument("--ipc", action="store_true",
                    help="the staged collectives across processes: one process per rank on this "
                         "GPU, staging buffers shared by CUDA IPC, host handshakes (one JSON "
                         "line per operation, rank count, handshake and size)")
    ap.add_argument("--ipc-ranks", nargs="+", type=int, default=[2, 4])
    ap.add_argument("--ipc-sizes", nargs="+", type=int, default=[4096, 1 << 20, 4 << 20])
    ap.add_argument("--ipc-handshakes", nargs="+", choices=["shm", "gloo"], default=["shm", "gloo"])
    ap.add_argument("--ipc-ops", nargs="+", choices=["all_gather", "all_reduce", "reduce_scatter"],
                    default=["all_gather", "all_reduce", "reduce_scatter"])
    ap.add_argument("--out", default=None, help="also write the JSON line to this file")
    ap.add_argument("--case", default=None, metavar="OP:P:BYTES:REPS",
                    help="profiling helper: run one call REPS times and exit, e.g. "
                         "gather:8:4194304:3, ugather:8:4194305:3 (unaligned), "
                         "allreduce:8:268435456:2, allreduce_mis:8:67108864:2 (rank 1 one "
                         "element off; BYTES per rank), "
                         "many:8:0:3 (the all_gather_many workload), manytiny:8:0:3 (120 tiny "
                         "tensors), gatherbulk:8:4194304:3 (the opt-in bulk-copy gather) or "
                         "fused:8:4194304:3 (the staged protocol), manymid:4:0:2 (250 tensors of 4-64 KiB at +1 B), "
                         "fill:8:33554432:2 (a write-only "
                         "stream of P * BYTES, a comparator)")
    args = ap.parse_args(argv)
    if args.warmup < 0 or args.steps < 1:
        ap.error("--steps must be >= 1 and --warmup >= 0")
    return args


# ------------------------------------------------------------ workload ---

def sweep_cases():
    """(P, bytes_per_rank, seed) of the 14 gathers, in step order."""
    return [(c.P, c.bytes_per_rank, c.seed) for c in W.config2_cases()]


def algorithmic_bytes(P: int, B: int) -> int:
    """Bytes read plus bytes written by one gather: P*B read, P*B written."""
    return 2 * P * B


# ------------------------------------------------------------- helpers ---

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def strip_comments(src: str) -> str:
    """C/C++ source without its comments and blank lines (string and
    character literals kept as they are), so that the digest below follows
    the code, not its commentary."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "\n".join(ln.rstrip() for ln in "".join(out).splitlines() if ln.strip())


def kernel_source_digest() -> str:
    """Digest of the code (comments left out) of every file under
    reduce_copy_rank_gb300/csrc."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "reduce_copy_rank_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, f), encoding="utf-8") as fh:
                h.update(f.encode() + b"\0" + strip_comments(fh.read()).encode())
    return h.hexdigest()[:16]


def load_traffic(kernel: str) -> dict:
    """Per-launch figures of `kernel` from the committed ncu summary (DRAM
    bytes, and the serialised cold-cache duration of ncu's launch list), if
    they were taken from the current kernel sources (else {})."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return {}
    for ln in lines:
        if ln.startswith("#") or not ln.strip():
            continue
        parts = dict(kv.split("=", 1) for kv in ln.split() if "=" in kv)
        if parts.get("kernel") == kernel and parts.get("source") == kernel_source_digest():
            out = {}
            for key in ("bytes_per_launch", "ncu_us_per_launch"):
                try:
                    out[key] = float(parts[key])
                except (KeyError, ValueError):
                    pass
            return out
    return {}


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.file = tempfile.NamedTemporaryFile(mode="w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(device_index), "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [ln.split(",") for ln in self.file.read().splitlines() if ln.count(",") >= 8]
        os.unlink(self.file.name)
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------- the oracle arm ---

_ARM_PARTS = {"0xd0c": "Neoverse-N1", "0xd40": "Neoverse-V1", "0xd49": "Neoverse-N2",
              "0xd4f": "Neoverse-V2", "0xd8e": "Neoverse-N3", "0xd84": "Neoverse-V3"}


def cpu_model() -> str:
    """The host CPU's model as /proc/cpuinfo gives it (x86: the model name;
    Arm: implementer and part, named where the part is a known Neoverse)."""
    import platform

    fields = {}
    try:
        with open("/proc/cpuinfo") as fh:
            for ln in fh:
                k, _, v = ln.partition(":")
                fields.setdefault(k.strip(), v.strip())
    except OSError:
        pass
    if fields.get("model name"):
        return fields["model name"]
    part = fields.get("CPU part")
    if part:
        return (f"{platform.machine()} implementer {fields.get('CPU implementer', '?')} part {part}"
                + (f" ({_ARM_PARTS[part]})" if part in _ARM_PARTS else ""))
    return platform.processor() or platform.machine()


def cpu_oracle_sample(seconds: float):
    """Time the oracle (single-threaded C byte-loop gather) on the host over
    whole passes of the sweep until `seconds` have elapsed (at least one)."""
    import oracle

    cases = sweep_cases()
    host = [[W.random_bf16_patterns(seed, r, B // 2).view(np.uint8) for r in range(P)]
            for (P, B, seed) in cases]
    step_bytes = sum(algorithmic_bytes(P, B) for (P, B, _s) in cases)
    oracle.all_gather(host[0])  # load the library outside the timing
    passes, t0 = 0, time.perf_counter()
    while True:
        for peers in host:
            oracle.all_gather(peers)
        passes += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return {"value": step_bytes * passes / el / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"{passes} full passes of the 14-gather sweep ({step_bytes} algorithmic bytes "
                      f"each) through the single-threaded C oracle, {el:.1f} s"}


def cpu_oracle_threaded(seconds: float):
    """The same oracle sweep run by one thread per host core, each thread
    doing whole passes (the C calls release the GIL), for `seconds`."""
    import threading

    import oracle

    cases = sweep_cases()
    host = [[W.random_bf16_patterns(seed, r, B // 2).view(np.uint8) for r in range(P)]
            for (P, B, seed) in cases]
    step_bytes = sum(algorithmic_bytes(P, B) for (P, B, _s) in cases)
    oracle.all_gather(host[0])
    nthreads = len(os.sched_getaffinity(0))
    done = [0] * nthreads
    t0 = time.perf_counter()

    def work(i):
        while time.perf_counter() - t0 < seconds:
            for peers in host:
                oracle.all_gather(peers)
            done[i] += 1

    th = [threading.Thread(target=work, args=(i,)) for i in range(nthreads)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    el = time.perf_counter() - t0
    return {"value": step_bytes * sum(done) / el / 1e9, "unit": UNIT, "cores": nthreads,
            "kind": "oracle, one thread per core", "cpu_model": cpu_model(),
            "sample": f"{sum(done)} full passes of the 14-gather sweep over {nthreads} threads, "
                      f"{el:.1f} s"}


def run_reference(args) -> int:
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle

    cases = sweep_cases()
    host = [[W.random_bf16_patterns(seed, r, B // 2).view(np.uint8) for r in range(P)]
            for (P, B, seed) in cases]
    step_bytes = sum(algorithmic_bytes(P, B) for (P, B, _s) in cases)
    for _ in range(args.warmup):
        for peers in host:
            oracle.all_gather(peers)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        for peers in host:
            oracle.all_gather(peers)
    el = time.perf_counter() - t0
    value = step_bytes * args.steps / el / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
        "data": "synthetic (seeded random BF16 bit patterns)",
        "config": workload_config(int(os.environ.get("WORLD_SIZE", "1"))),
        "timing": "host oracle on the host cores: whole passes of the sweep, wall clock",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "cpu_model": cpu_model(),
                         "sample": f"{args.steps} full passes of the 14-gather sweep through the "
                                   "single-threaded C oracle"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    emit(line, args)
    return 0


# ----------------------------------------------------------- GPU arm ---

class Flusher:
    """Writes, then reads, a buffer four times the L2 size: afterwards L2 holds
    only clean lines of this buffer, so the next call's inputs come from HBM
    and no dirty line of ours is left to be written back inside its timing."""

    def __init__(self, torch, device):
        l2 = getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 128 << 20)
        n = max(4 * l2, 256 << 20)
        self.buf = torch.empty(n // 4, dtype=torch.int32, device=device)

    def __call__(self):
        self.buf.zero_()
        self.buf.sum()


def timed_calls(torch, stream, flush, calls, reps):
    """Run each call `reps` times, each preceded by a flush outside its
    events; return per-call lists of microseconds."""
    evs = []
    for _ in range(reps):
        for fn in calls:
            flush()
            s = torch.cuda.Event(enable_timing=True)
            e = torch.cuda.Event(enable_timing=True)
            s.record(stream)
            fn()
            e.record(stream)
            evs.append((s, e))
    torch.cuda.synchronize()
    out = [[] for _ in calls]
    for i, (s, e) in enumerate(evs):
        out[i % len(calls)].append(s.elapsed_time(e) * 1e3)
    return out


def build_gather_calls(torch, dc, device, cases):
    calls, keep = [], []
    for (P, B, seed) in cases:
        peers = [torch.from_numpy(W.random_bf16_patterns(seed, r, B // 2).view(np.uint8)).to(device)
                 for r in range(P)]
        out = torch.empty(P * B, dtype=torch.uint8, device=device)
        keep.append((peers, out))
        calls.append(lambda peers=peers, out=out: dc.all_gather(peers, out))
    return calls, keep


def reductions_block(torch, dc, device, stream, flush, peak):
    """The other paths, each measured like the sweep (flush, CUDA events,
    median of 5): all_reduce at the five per-rank sizes, reduce_scatter
    16384x8192 per rank, the typed, tree and batched reductions, an
    all_reduce with one rank's input realigned, unaligned gathers of 4 MiB+1 B
    and 32 MiB+1 B per rank, all_gather_many of the six mixed tensors and of
    120 tiny tensors (P=8), and the staged protocol over 8 ranks x 4 MiB."""
    rows = []
    P = W.CONFIG4_P
    for name, n in W.CONFIG4_COUNTS.items():
        seed = W.seed_for(4, list(W.CONFIG4_COUNTS).index(name))
        ins = [W.normal_bf16_device(seed, r, n, device) for r in range(P)]
        outs = [torch.empty_like(x) for x in ins]
        us = statistics.median(timed_calls(torch, stream, flush, [lambda: dc.all_reduce(ins, outs)], 11)[0])
        nbytes = 4 * P * n
        rows.append({"op": "all_reduce_bf16", "P": P, "count": n, "shape": name, "us": us,
                     "gbs": nbytes / us / 1e3, "frac": nbytes / us / 1e3 / peak, "bytes": nbytes})
        del ins, outs
    c = W.CONFIG5_RS
    n = c["rows"] * c["cols"]
    ins = [W.normal_bf16_device(W.seed_for(5, 0), r, n, device) for r in range(c["P"])]
    outs = [torch.empty(n // c["P"], dtype=torch.bfloat16, device=device) for _ in range(c["P"])]
    us = statistics.median(timed_calls(torch, stream, flush, [lambda: dc.reduce_scatter(ins, outs)], 11)[0])
    nbytes = 2 * c["P"] * n + 2 * n
    rows.append({"op": "reduce_scatter_bf16", "P": c["P"], "count": n, "shape": "16384x8192",
                 "us": us, "gbs": nbytes / us / 1e3, "frac": nbytes / us / 1e3 / peak, "bytes": nbytes})
    del ins, outs
    # one rank's share (dc_reduce), as a rank that is its own process
    # computes it: rank 3's output of the 8627x8192 all_reduce, P = 8
    n = W.CONFIG4_COUNTS["8627x8192"]
    ins = [W.normal_bf16_device(W.seed_for(4, 9930), r, n, device) for r in range(P)]
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    us = statistics.median(timed_calls(torch, stream, flush, [lambda: dc.reduce(ins, out)], 11)[0])
    nbytes = 2 * P * n + 2 * n
    rows.append({"op": "reduce_one_rank_bf16", "P": P, "count": n,
                 "shape": "8627x8192: P inputs folded into one output", "us": us,
                 "gbs": nbytes / us / 1e3, "frac": nbytes / us / 1e3 / peak, "bytes": nbytes})
    del ins, out
    rows.extend(typed_rows(torch, dc, device, stream, flush, peak))
    # all_reduce with rank 1's input one element past the others' alignment
    # (8627x8192 per rank, P=8): the realigning path
    n = W.CONFIG4_COUNTS["8627x8192"]
    store = [W.normal_bf16_device(W.seed_for(4, 9920), r, n + 8, device) for r in range(P)]
    ins = [store[r][(1 if r == 1 else 0):(1 if r == 1 else 0) + n] for r in range(P)]
    outs = [torch.empty(n, dtype=torch.bfloat16, device=device) for _ in range(P)]
    us = statistics.median(timed_calls(torch, stream, flush, [lambda: dc.all_reduce(ins, outs)], 11)[0])
    nbytes = 4 * P * n
    rows.append({"op": "all_reduce_bf16_realigned", "P": P, "count": n,
                 "shape": "8627x8192, rank 1's input one element off 16 bytes", "us": us,
                 "gbs": nbytes / us / 1e3, "frac": nbytes / us / 1e3 / peak, "bytes": nbytes})
    del store, ins, outs
    for B in (4 * 1024 * 1024 + 1, 32 * 1024 * 1024 + 1):  # unaligned: payloads +1, output +3
        peers = [W.random_bytes_device(W.seed_for(3, 9000), r, B + 1, device)[1:] for r in range(8)]
        out = torch.empty(8 * B + 3, dtype=torch.uint8, device=device)[3:]
        us = statistics.median(timed_calls(torch, stream, flush, [lambda: dc.all_gather(peers, out)], 11)[0])
        nbytes = 2 * 8 * B
        rows.append({"op": "all_gather_unaligned", "P": 8, "count": B,
                     "shape": f"{B} B per rank, payloads at +1 B, output at +3 B", "us": us,
                     "gbs": nbytes / us / 1e3, "frac": nbytes / us / 1e3 / peak, "bytes": nbytes})
        del peers, out
    P = W.CONFIG5_MANY_P
    tens = [[W.random_bytes_device(W.seed_for(5, 1), r, B, device, tensor=t) for r in range(P)]
            for t, B in enumerate(W.CONFIG5_MANY_SIZES)]
    outs = [torch.empty(P * B, dtype=torch.uint8, device=device) for B in W.CONFIG5_MANY_SIZES]
    us = statistics.median(timed_calls(torch, stream, flush, [lambda: dc.all_gather_many(tens, outs)], 11)[0])
    nbytes = 2 * P * sum(W.CONFIG5_MANY_SIZES)
    rows.append({"op": "all_gather_many", "P": P, "count": len(W.CONFIG5_MANY_SIZES),
                 "shape": "{3 B, 4 KiB, 100000 B, 1 MiB, 7 MiB+5 B, 32 MiB}", "us": us,
                 "gbs": nbytes / us / 1e3, "frac": nbytes / us / 1e3 / peak, "bytes": nbytes})
    del tens, outs
    # many tiny tensors: 120 tensors x 8 ranks of 3..100 B at odd offsets
    rng = np.random.default_rng(W.seed_for(5, 9005))
    sizes = [int(x) for x in rng.integers(3, 101, 120)]
    tens = [[W.random_bytes_device(W.seed_for(5, 2), r, B + 1, device, tensor=t)[1:] for r in range(8)]
            for t, B in enumerate(sizes)]
    outs = [torch.empty(8 * B, dtype=torch.uint8, device=device) for B in sizes]
    # (timed from CUDA graphs: flush, event, the call -- or 20 of them back
    # to back --, event; the binding's host-side marshalling of a thousand
    # tensors takes longer than the flush, so an eager call's events would
    # count host time)
    def graph_us(fn, n):
        g, evs = build_step_graph(torch, flush, [fn] * n)
        t = []
        for _ in range(5):
            g.replay()
            torch.cuda.synchronize()
            t.append(evs[0].elapsed_time(evs[1]) * 1e3 / n)
        del g
        return statistics.median(t)

    many = lambda: dc.all_gather_many(tens, outs)  # noqa: E731
    us, b2b = graph_us(many, 1), graph_us(many, 20)
    nbytes = 2 * 8 * sum(sizes)
    rows.append({"op": "all_gather_many_tiny", "P": 8, "count": len(sizes),
                 "shape": "120 tensors of 3..100 B per rank, payloads at +1 B; call alone after a "
                          "flush, from a CUDA graph", "us": us, "back_to_back_us": b2b,
                 "gbs": nbytes / us / 1e3, "frac": nbytes / us / 1e3 / peak, "bytes": nbytes})
    del tens, outs
    # many mid-size tensors: 250 tensors x 4 ranks of 128..4096 B at +1 B
    # (the realigning part with a long job table)
    sizes = [int(x) for x in rng.integers(128, 4097, 250)]
    tens = [[W.random_bytes_device(W.seed_for(5, 3), r, B + 1, device, tensor=t)[1:] for r in range(4)]
            for t, B in enumerate(sizes)]
    outs = [torch.empty(4 * B, dtype=torch.uint8, device=device) for B in sizes]
    us, b2b = graph_us(many, 1), graph_us(many, 20)
    nbytes = 2 * 4 * sum(sizes)
    rows.append({"op": "all_gather_many_mid", "P": 4, "count": len(sizes),
                 "shape": "250 tensors of 128..4096 B per rank, payloads at +1 B; call alone after a "
                          "flush, and 20 back to back, from CUDA graphs", "us": us, "back_to_back_us": b2b,
                 "gbs": nbytes / us / 1e3, "frac": nbytes / us / 1e3 / peak, "bytes": nbytes,
                 "back_to_back_gbs": nbytes / b2b / 1e3})
    del tens, outs
    # the staged protocol (stage -> gather -> complete), P = 8 ranks x 4 MiB:
    # P*B read + P*B written to stage, P*P*B read + P*P*B written to gather
    P, B = 8, 4 << 20
    ins = [W.random_bytes_device(W.seed_for(2, 990), r, B, device) for r in range(P)]
    stg = [torch.empty(B, dtype=torch.uint8, device=device) for _ in range(P)]
    outs = [torch.empty(P * B, dtype=torch.uint8, device=device) for _ in range(P)]
    ws = dc.fused_workspace(P, device)
    epoch = [0]

    def fused():
        epoch[0] += 1
        dc.fused_all_gather(ins, stg, outs, ws, epoch[0])

    us = statistics.median(timed_calls(torch, stream, flush, [fused], 11)[0])
    dc.check_device()
    # its DRAM traffic is mostly writes (P*P*B of outputs + P*B of staging):
    # a write-only stream of as many bytes, timed the same way, beside it --
    # torch's zero_ of a float32 view (16-byte stores; a uint8 fill writes 4
    # bytes per thread and runs at about half that rate on this GPU)
    fill = torch.empty(P * P * B // 4, dtype=torch.float32, device=device)
    fill_us = statistics.median(timed_calls(torch, stream, flush, [fill.zero_], 11)[0])
    del fill
    nbytes = 2 * P * B + 2 * P * P * B
    rows.append({"op": "fused_all_gather", "P": P, "count": B,
                 "shape": "4 MiB per rank, every rank's own output (stage, gather, complete)", "us": us,
                 "gbs": nbytes / us / 1e3, "frac": nbytes / us / 1e3 / peak, "bytes": nbytes,
                 "written_bytes": P * P * B + P * B,
                 "write_only_stream_us": fill_us,
                 "write_gbs": (P * P * B + P * B) / us / 1e3,
                 "write_only_stream_gbs": P * P * B / fill_us / 1e3})
    return rows


def typed_rows(torch, dc, device, stream, flush, peak):
    """FP16 / FP32 and tree-order all_reduce at full size, and the batched
    all_reduce_many / reduce_scatter_many over the five per-rank sizes of the
    all_reduce workload (P=8), each timed like the sweep."""
    rows = []
    P = W.CONFIG4_P
    tdt = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}
    for dt, order, shape in (("bf16", "tree", "16384x8192"), ("f16", "tree", "8627x8192"),
                             ("f32", "linear", "8627x8192")):
        n = W.CONFIG4_COUNTS[shape]
        ins = [W.normal_device(W.seed_for(4, 9900), r, n, device, tdt[dt]) for r in range(P)]
        outs = [torch.empty_like(x) for x in ins]
        us = statistics.median(timed_calls(
            torch, stream, flush, [lambda: dc.all_reduce(ins, outs, order=order)], 5)[0])
        nbytes = 2 * P * n * ins[0].element_size()
        rows.append({"op": f"all_reduce_{dt}_{order}", "P": P, "count": n, "shape": shape, "us": us,
                     "gbs": nbytes / us / 1e3, "frac": nbytes / us / 1e3 / peak, "bytes": nbytes})
        del ins, outs
    counts = list(W.CONFIG4_COUNTS.values())
    ins = [[W.normal_bf16_device(W.seed_for(4, 9910), r, n, device, tensor=t) for r in range(P)]
           for t, n in enumerate(counts)]
    outs = [[torch.empty_like(x) for x in t] for t in ins]
    us = statistics.median(timed_calls(
        torch, stream, flush, [lambda: dc.all_reduce_many(ins, outs)], 5)[0])
    nbytes = 4 * P * sum(counts)
    rows.append({"op": "all_reduce_many_bf16_linear", "P": P, "count": len(counts),
                 "shape": "{" + ", ".join(W.CONFIG4_COUNTS) + "}", "us": us,
                 "gbs": nbytes / us / 1e3, "frac": nbytes / us / 1e3 / peak, "bytes": nbytes})
    outs = [[torch.empty(n // P, dtype=torch.bfloat16, device=device) for _ in range(P)]
            for n in counts]
    us = statistics.median(timed_calls(
        torch, stream, flush, [lambda: dc.reduce_scatter_many(ins, outs, order="tree")], 5)[0])
    nbytes = 2 * P * sum(counts) + 2 * sum(counts)
    rows.append({"op": "reduce_scatter_many_bf16_tree", "P": P, "count": len(counts),
                 "shape": "{" + ", ".join(W.CONFIG4_COUNTS) + "}", "us": us,
                 "gbs": nbytes / us / 1e3, "frac": nbytes / us / 1e3 / peak, "bytes": nbytes})
    return rows


def alternating(torch, stream, flush, fns, reps):
    """Time the callables of `fns` after a flush each, alternating which one
    goes first from sample to sample (as the page's benchmark does);
    returns per-callable medians in microseconds."""
    samples = [[] for _ in fns]
    for i in range(reps):
        order = list(range(len(fns)))
        if i % 2:
            order.reverse()
        got = timed_calls(torch, stream, flush, [fns[j] for j in order], 1)
        for k, j in enumerate(order):
            samples[j].extend(got[k])
    return [statistics.median(x) for x in samples]


def comparators_block(torch, dc, device, stream, flush, reps=10):
    """torch comparators beside this library, same inputs, alternating
    order per sample: torch.cat(peers, out=out) for every gather of the
    sweep, and a torch loop (acc = x0.float(); acc = acc + xq.float() for
    q = 1..P-1; one cast to BF16, copied to the P outputs) for the all_reduce
    sizes.  Bits of both are compared, for the record."""
    gathers = []
    for (P, B, seed) in sweep_cases():
        peers = [torch.from_numpy(W.random_bf16_patterns(seed, r, B // 2).view(np.uint8)).to(device)
                 for r in range(P)]
        out_dc = torch.empty(P * B, dtype=torch.uint8, device=device)
        out_t = torch.empty_like(out_dc)
        ours, theirs = alternating(torch, stream, flush,
                                   [lambda: dc.all_gather(peers, out_dc),
                                    lambda: torch.cat(peers, out=out_t)], reps)
        gathers.append({"P": P, "bytes_per_rank": B, "us": ours, "torch_cat_us": theirs,
                        "speedup": theirs / ours, "bits_equal": bool(torch.equal(out_dc, out_t))})
    reduces = []
    P = W.CONFIG4_P
    for name, n in W.CONFIG4_COUNTS.items():
        ins = [W.normal_bf16_device(W.seed_for(4, list(W.CONFIG4_COUNTS).index(name)), r, n, device)
               for r in range(P)]
        outs = [torch.empty_like(x) for x in ins]
        touts = [torch.empty_like(x) for x in ins]

        def torch_loop():
            acc = ins[0].float()
            for q in range(1, P):
                acc = acc + ins[q].float()
            y = acc.bfloat16()
            for o in touts:
                o.copy_(y)

        ours, theirs = alternating(torch, stream, flush,
                                   [lambda: dc.all_reduce(ins, outs), torch_loop], reps)
        reduces.append({"P": P, "shape": name, "count": n, "us": ours, "torch_loop_us": theirs,
                        "speedup": theirs / ours,
                        "bits_equal": bool(torch.equal(outs[0].view(torch.int16),
                                                       touts[0].view(torch.int16)))})
        del ins, outs, touts
    return {"all_gather_vs_torch_cat": gathers, "all_reduce_bf16_vs_torch_loop": reduces}


def back_to_back_block(torch, dc, device, flush, per_size=14, replays=10):
    """Per-call time of each sweep size in the back-to-back regime: one CUDA
    graph of `per_size` calls of that size on distinct buffers (so every
    call reads inputs no kernel has touched since the L2 flush that opens
    the graph), timed by events around the calls; median over replays.
    14 calls per graph, as many as the step has, so the first call's launch
    (which nothing overlaps) weighs as much as in the step."""
    rows = []
    for (P, B, seed) in sweep_cases():
        bufs = []
        for i in range(per_size):
            peers = [torch.from_numpy(W.random_bf16_patterns(seed, r, B // 2, tensor=i).view(np.uint8))
                     .to(device) for r in range(P)]
            bufs.append((peers, torch.empty(P * B, dtype=torch.uint8, device=device)))
        calls = [lambda p=p, o=o: dc.all_gather(p, o) for (p, o) in bufs]
        g, evs = build_step_graph(torch, flush, calls)
        t = []
        for _ in range(replays):
            g.replay()
            torch.cuda.synchronize()
            t.append(evs[0].elapsed_time(evs[1]) * 1e3 / per_size)
        us = statistics.median(t)
        rows.append({"P": P, "bytes_per_rank": B, "us": us,
                     "gbs": algorithmic_bytes(P, B) / us / 1e3})
        del g, bufs
    return rows


def call_kernel(dc, P: int, B: int) -> str:
    """The kernel that runs a 16-byte aligned gather of P x B bytes under the
    library's current options (the planner's rule for one aligned tensor)."""
    total = P * B
    if total <= dc.get_option("gather_single_max_bytes"):
        return "dc_gather_single_kernel<1,64,2>"
    if dc.get_option("gather_bulk") and total >= dc.get_option("gather_bulk_min_bytes"):
        return "dc_gather_bulk_kernel"
    return "dc_gather_kernel<1,64,3>" if dc.get_option("gather_staged") else "dc_gather_kernel<1,64,2>"


def by_size_rows(table, back_to_back, peak):
    """The 4 MiB and 1 MiB per-rank gathers of the sweep (P = 8 and 2): the
    call alone after a flush (median of the timed region's samples) and back
    to back (per_call_back_to_back), each against the measured copy rate and
    the nominal 8 TB/s."""
    rows = []
    for P in (8, 2):
        for B in (4 * MIB, 1 * MIB):
            iso = [r for r in table if r["P"] == P and r["bytes_per_rank"] == B]
            b2b = [r for r in back_to_back if r["P"] == P and r["bytes_per_rank"] == B]
            if not iso or not b2b:
                continue
            nbytes = algorithmic_bytes(P, B)
            iso_us, b2b_us = iso[0]["us_median"], b2b[0]["us"]
            rows.append({"P": P, "bytes_per_rank": B, "kernel": iso[0]["kernel"],
                         "alone_us": iso_us, "alone_gbs": nbytes / iso_us / 1e3,
                         "alone_frac_measured": nbytes / iso_us / 1e3 / peak,
                         "alone_frac_nominal": nbytes / iso_us / 1e3 / NOMINAL_HBM_GBS,
                         "back_to_back_us": b2b_us, "back_to_back_gbs": nbytes / b2b_us / 1e3,
                         "back_to_back_frac_measured": nbytes / b2b_us / 1e3 / peak,
                         "back_to_back_frac_nominal": nbytes / b2b_us / 1e3 / NOMINAL_HBM_GBS})
    return rows


def warm_latency_block(torch, dc, device, calls_per_graph=1000, replays=3):
    """Per-call latency of back-to-back calls with warm caches: for each
    gather of the sweep whose inputs and output fit in a quarter of L2, one
    CUDA graph of `calls_per_graph` identical calls, timed by events around
    its replay (median of `replays`), for this library and torch.cat."""
    l2 = getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 128 << 20)
    rows = []
    for (P, B, seed) in sweep_cases():
        if 2 * P * B > l2 // 4:
            continue
        peers = [torch.from_numpy(W.random_bf16_patterns(seed, r, B // 2).view(np.uint8)).to(device)
                 for r in range(P)]
        out = torch.empty(P * B, dtype=torch.uint8, device=device)
        rows.append({"P": P, "bytes_per_rank": B,
                     "us": warm_per_call(torch, lambda: dc.all_gather(peers, out),
                                         calls_per_graph, replays),
                     "torch_cat_us": warm_per_call(torch, lambda: torch.cat(peers, out=out),
                                                   calls_per_graph, replays)})
    return rows


def build_step_graph(torch, flush, calls):
    """Capture flush, an event, the calls back to back and an event into one
    CUDA graph (events recorded as graph nodes)."""
    evs = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # first use of every call outside the capture
        flush()
        for fn in calls:
            fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        flush()
        evs[0].record()
        for fn in calls:
            fn()
        evs[1].record()
    torch.cuda.synchronize()
    return g, evs


def e2e_groups(cases, small=1 << 20):
    """Consecutive calls of under `small` bytes per rank share one host copy
    each way; larger calls have their own.  Returns lists of case indices."""
    groups, cur = [], []
    for i, (P, B, _s) in enumerate(cases):
        if B < small:
            cur.append(i)
            continue
        if cur:
            groups.append(cur)
            cur = []
        groups.append([i])
    if cur:
        groups.append(cur)
    return groups


def e2e_measure(torch, dc, device, stream, cases, steps):
    """The same sweep through the public API with host buffers.  Each step
    copies the inputs from pinned host memory to the device (copy stream),
    gathers on `stream` as soon as a call's inputs are in, and copies the
    outputs back to pinned host memory (a second copy stream), so the two
    copy directions and the kernels overlap.  Calls under 1 MiB per rank
    share one copy each way with their neighbours (e2e_groups: six copies
    per direction instead of fourteen; a copy has a fixed cost of a few
    microseconds).  The step starts and ends on `stream`; all copies are
    inside the timed region."""
    groups = e2e_groups(cases)
    host_in, dev_in, dev_out, host_out, views, outs = [], [], [], [], {}, {}
    for g in groups:
        total = sum(cases[i][0] * cases[i][1] for i in g)
        h = torch.empty(total, dtype=torch.uint8).pin_memory()
        di = torch.empty(total, dtype=torch.uint8, device=device)
        do = torch.empty(total, dtype=torch.uint8, device=device)
        off = 0
        for i in g:
            P, B, seed = cases[i]
            for r in range(P):
                h[off + r * B:off + (r + 1) * B].copy_(
                    torch.from_numpy(W.random_bf16_patterns(seed, r, B // 2).view(np.uint8)))
            views[i] = [di[off + r * B:off + (r + 1) * B] for r in range(P)]
            outs[i] = do[off:off + P * B]
            off += P * B
        host_in.append(h)
        dev_in.append(di)
        dev_out.append(do)
        host_out.append(torch.empty(total, dtype=torch.uint8).pin_memory())
    h2d = sum(P * B for (P, B, _s) in cases)
    up, down = torch.cuda.Stream(device=device), torch.cuda.Stream(device=device)
    ev_in = [torch.cuda.Event() for _ in groups]
    ev_g = [torch.cuda.Event() for _ in groups]

    def step():
        up.wait_stream(stream)  # the previous step is over before its inputs are overwritten
        with torch.cuda.stream(up):
            for gi in range(len(groups)):
                dev_in[gi].copy_(host_in[gi], non_blocking=True)
                ev_in[gi].record(up)
        for gi, g in enumerate(groups):
            stream.wait_event(ev_in[gi])
            for i in g:
                dc.all_gather(views[i], outs[i], stream=stream)
            ev_g[gi].record(stream)
            down.wait_event(ev_g[gi])
            with torch.cuda.stream(down):
                host_out[gi].copy_(dev_out[gi], non_blocking=True)
        stream.wait_stream(down)

    step()
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(steps):
        step()
    e.record(stream)
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / steps
    for gi in range(len(groups)):  # the round trip really happened
        assert torch.equal(host_out[gi], host_in[gi]), "e2e output differs from its input payloads"
    step_bytes = sum(algorithmic_bytes(P, B) for (P, B, _s) in cases)
    return {"value": step_bytes / ms / 1e6, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": h2d, "ms_per_step": ms, "steps": steps,
            "copies_per_direction": len(groups),
            "pipeline": "H2D copy stream -> gathers on the compute stream -> D2H copy stream, per copy "
                        "group (calls under 1 MiB per rank share one copy each way), joined by events"}


def rank_max(value: float, dist=None, device=None) -> float:
    """The largest `value` over all ranks (the slowest replica sets the
    job's time); the local value when there is no process group."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    import torch

    dev = device if (device is not None and dist.get_backend() == "nccl") else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, bytes_per_rank_step: int, slowest_ms_per_step: float) -> float:
    """GB/s of the whole job: every replica moves `bytes_per_rank_step` per
    step, and the job's step takes as long as its slowest replica's."""
    return world * bytes_per_rank_step / slowest_ms_per_step / 1e6


def stats(xs):
    return {"us_mean": float(np.mean(xs)), "us_median": float(np.median(xs)),
            "us_p10": float(np.percentile(xs, 10)), "us_p90": float(np.percentile(xs, 90))}


def run_dc(args) -> int:
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (this arm times the library's kernels)")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=device)

    import reduce_copy_rank_gb300 as dc

    dc.lib()
    stream = torch.cuda.current_stream()
    flush = Flusher(torch, device)
    peak, peak_src = load_peaks()
    cases = sweep_cases()
    calls, _keep = build_gather_calls(torch, dc, device, cases)
    single_max = dc.get_option("gather_single_max_bytes")
    paths = [call_kernel(dc, P, B) for (P, B, _s) in cases]
    step_bytes = sum(algorithmic_bytes(P, B) for (P, B, _s) in cases)

    launches0 = dc.launch_count()
    graph, evs = build_step_graph(torch, flush, calls)
    kernels_per_step = dc.launch_count() - launches0 - len(calls)  # launches captured in the graph
    # one more graph per kernel (path): that kernel's calls of the step back to
    # back after a flush, for its average launch duration in the roofline
    path_graphs = {}
    for path in sorted(set(paths)):
        idx = [i for i, p in enumerate(paths) if p == path]
        if idx:
            launches0 = dc.launch_count()
            g, e = build_step_graph(torch, flush, [calls[i] for i in idx])
            kernels_per_step += dc.launch_count() - launches0 - len(idx)
            path_graphs[path] = (idx, g, e)
    for _ in range(max(args.warmup, 0)):
        graph.replay()
        for (_idx, g, _e) in path_graphs.values():
            g.replay()
        timed_calls(torch, stream, flush, calls, 1)
    torch.cuda.synchronize()

    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    launches0 = dc.launch_count()
    t_wall = time.perf_counter()
    step_ms, per_call = [], [[] for _ in calls]
    path_ms = {path: [] for path in path_graphs}
    for _ in range(args.steps):
        graph.replay()
        for (_idx, g, _e) in path_graphs.values():
            g.replay()
        iso = timed_calls(torch, stream, flush, calls, 1)  # synchronizes
        step_ms.append(evs[0].elapsed_time(evs[1]))
        for path, (_idx, _g, e) in path_graphs.items():
            path_ms[path].append(e[0].elapsed_time(e[1]))
        for i in range(len(calls)):
            per_call[i].extend(iso[i])
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    eager_launches = dc.launch_count() - launches0
    if dist:
        dist.barrier()
    clocks = sampler.stop()

    gpu_ms_total = rank_max(float(sum(step_ms)), dist, device)
    ms_per_step = gpu_ms_total / args.steps
    value = job_throughput(world, step_bytes, ms_per_step)  # GB/s over all ranks

    table = []
    kern_time = {path: 0.0 for path in paths}
    kern_bytes = {path: 0 for path in paths}
    kern_launches = {path: 0 for path in paths}
    for (P, B, _s), path, us_list in zip(cases, paths, per_call):
        nbytes = algorithmic_bytes(P, B)
        st = stats(us_list)
        table.append({"P": P, "bytes_per_rank": B, "kernel": path, **st,
                      "gbs": nbytes / st["us_mean"] / 1e3, "frac": nbytes / st["us_mean"] / 1e3 / peak})
        kern_time[path] += sum(us_list)
        kern_bytes[path] += nbytes * len(us_list)
        kern_launches[path] += len(us_list)
    # the dominant kernel: the larger share of the per-path graphs' time
    graph_ms = {path: float(sum(v)) for path, v in path_ms.items()}
    dom = max(graph_ms, key=graph_ms.get)
    kname = dom
    dom_idx = path_graphs[dom][0]
    dom_bytes = sum(algorithmic_bytes(cases[i][0], cases[i][1]) for i in dom_idx)
    us_per_launch = graph_ms[dom] * 1e3 / (args.steps * len(dom_idx))
    achieved = dom_bytes / len(dom_idx) / us_per_launch / 1e3  # GB/s
    iso_achieved = kern_bytes[dom] / kern_time[dom] / 1e3
    ncu = load_traffic(kname)
    big = [row for row in table if row["P"] == 8 and row["bytes_per_rank"] == 4 << 20][0]

    extra = None
    if not args.no_reductions:
        extra = reductions_block(torch, dc, device, stream, flush, peak)
    comparators = latency = None
    if not args.no_comparators:
        comparators = comparators_block(torch, dc, device, stream, flush)
        latency = warm_latency_block(torch, dc, device)
    back_to_back = back_to_back_block(torch, dc, device, flush)
    by_size = by_size_rows(table, back_to_back, peak)
    # the floor of every "alone" figure: a 16-byte one-rank gather timed the
    # same way (flush, event, launch, event)
    tiny_in = [torch.zeros(16, dtype=torch.uint8, device=device)]
    tiny_out = torch.empty(16, dtype=torch.uint8, device=device)
    alone_floor_us = statistics.median(
        timed_calls(torch, stream, flush, [lambda: dc.all_gather(tiny_in, tiny_out)], 21)[0])
    e2e = e2e_measure(torch, dc, device, stream, cases, min(args.steps, 20))
    e2e["value"] = job_throughput(world, step_bytes, rank_max(e2e["ms_per_step"], dist, device))

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8",
        "data": "synthetic (seeded random BF16 bit patterns, resident in HBM)",
        "config": workload_config(world),
        "timing": "value: one CUDA graph per step (L2 flush, event, the 14 calls back to back, "
                  "event); roofline: per kernel one more graph per step with that kernel's calls "
                  "of the step back to back (L2 flush, event, the calls, event); per_call and "
                  "roofline.isolated: each call alone (L2 flush, event, the launch, event); all in "
                  "the same timed region",
        "l2": "flushed before every step and before every separately timed call (write + read of "
              "4x L2); each call's inputs are untouched since",
        "library": {"source_digest": kernel_source_digest(),
                    "bounds_checked_build": bool(dc.lib().dc_bounds_checked()),
                    "programmatic_dependent_launch": bool(dc.get_option("pdl")),
                    "gather_single_max_bytes": single_max,
                    "gather_bulk": dc.get_option("gather_bulk"),
                    "gather_bulk_min_bytes": dc.get_option("gather_bulk_min_bytes"),
                    "kernel_of_call": [{"P": P, "bytes_per_rank": B, "kernel": k}
                                       for (P, B, _s), k in zip(cases, paths)]},
        "roofline": {"bound": "hbm", "kernel": kname, "achieved": achieved, "peak": peak,
                     "peak_source": peak_src, "unit": "GB/s", "frac": achieved / peak,
                     "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
                     "traffic": ncu.get("bytes_per_launch"), "launches": args.steps * len(dom_idx),
                     "us_per_launch": us_per_launch,
                     "us_per_launch_regime": "back to back: that kernel's calls of the step in one "
                                             "CUDA graph after an L2 flush, launched with "
                                             "programmatic dependent launch (each launch overlaps "
                                             "the previous one's tail); the average per launch",
                     "ncu_us_per_launch": ncu.get("ncu_us_per_launch"),
                     "ncu_regime": "ncu launch list of the bench command (gpu__time_duration, "
                                   "--clock-control none): each launch serialised, caches flushed",
                     "share": graph_ms[dom] / sum(graph_ms.values()),
                     "algorithmic_bytes_per_launch": dom_bytes / len(dom_idx),
                     "isolated": {"achieved": iso_achieved, "frac": iso_achieved / peak,
                                  "us_per_launch": kern_time[dom] / max(kern_launches[dom], 1),
                                  "share": kern_time[dom] / sum(kern_time.values())},
                     "by_size": by_size, "alone_event_floor_us": alone_floor_us,
                     "alone_event_floor_note": "a 16-byte one-rank gather timed like the alone figures (flush, "
                                               "event, launch, event): the fixed cost every alone figure includes; "
                                               "this GPU's event clock advances in 2.05 us steps"},
        "headline_4MiB_P8": {"us": big["us_mean"], "gbs": big["gbs"], "frac": big["frac"]},
        "per_call": table,
        "per_call_back_to_back": back_to_back,
        "gpu_launches": kernels_per_step * args.steps + eager_launches,
        "wall_s_timed_region": t_wall,
        "clocks": clocks,
        "e2e": e2e,
    }
    if extra is not None:
        line["other_ops"] = extra
    if comparators is not None:
        line["comparators"] = comparators
        line["warm_latency_graph_1000_calls"] = latency
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_sample(args.cpu_seconds)
        line["cpu_oracle_all_cores"] = cpu_oracle_threaded(args.cpu_seconds)
    if rank == 0:
        emit(line, args)
    if dist:
        dist.destroy_process_group()
    return 0


def warm_per_call(torch, fn, calls=200, replays=3):
    """Microseconds per call of `calls` back-to-back calls of `fn` captured in
    one CUDA graph (caches warm), median over `replays` replays."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(calls):
            fn()
    g.replay()
    torch.cuda.synchronize()
    t = []
    for _ in range(replays):
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record()
        g.replay()
        e.record()
        torch.cuda.synchronize()
        t.append(s.elapsed_time(e) * 1e3 / calls)
    return statistics.median(t)


def run_crossover(args) -> int:
    """Single-CTA vs multi-CTA time per call across sizes, for the gather
    (P=2 and P=8) and the all_reduce (P=8).  Each point is timed two ways:
    warm (200 back-to-back calls in a CUDA graph) and cold (L2 flush, event,
    the call, event; median of 30).  The event clock ticks in steps of about
    2 us, which hides differences between the two paths when each call is
    timed alone, so the threshold is the largest size at which the single
    CTA is not slower warm, within the 3 % that repeated warm runs differ by.
    Prints one JSON line per point and the result."""
    NOISE = 0.03
    import torch

    import reduce_copy_rank_gb300 as dc

    device = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    flush = Flusher(torch, device)
    result = {"gather": {}, "all_reduce": {}}
    sizes = [256, 512, 1 * KIB, 2 * KIB, 4 * KIB, 8 * KIB, 16 * KIB, 32 * KIB, 64 * KIB,
             128 * KIB, 256 * KIB]

    def both(fn):
        t = {}
        for path in (1, 2):
            with dc.options(force_path=path):
                t[path] = (warm_per_call(torch, fn),
                           statistics.median(timed_calls(torch, stream, flush, [fn], 30)[0]))
        return t

    for P in (2, 8):
        best, going = 0, True
        for B in sizes:
            if P * B > 256 * KIB:
                continue
            peers = [torch.randint(0, 256, (B,), dtype=torch.uint8, device=device) for _ in range(P)]
            out = torch.empty(P * B, dtype=torch.uint8, device=device)
            t = both(lambda: dc.all_gather(peers, out))
            print(json.dumps({"op": "all_gather", "P": P, "out_bytes": P * B,
                              "single_warm_us": t[1][0], "multi_warm_us": t[2][0],
                              "single_cold_us": t[1][1], "multi_cold_us": t[2][1]}), flush=True)
            going = going and t[1][0] <= t[2][0] * (1 + NOISE)
            if going:
                best = P * B
        result["gather"][P] = best
    P = 8
    best, going = 0, True
    for B in sizes:
        n = B // 2
        ins = [torch.randn(n, device=device).to(torch.bfloat16) for _ in range(P)]
        outs = [torch.empty_like(x) for x in ins]
        t = both(lambda: dc.all_reduce(ins, outs))
        print(json.dumps({"op": "all_reduce", "P": P, "in_bytes_per_rank": B,
                          "single_warm_us": t[1][0], "multi_warm_us": t[2][0],
                          "single_cold_us": t[1][1], "multi_cold_us": t[2][1]}), flush=True)
        going = going and t[1][0] <= t[2][0] * (1 + NOISE)
        if going:
            best = B
    result["all_reduce"][P] = best
    print(json.dumps({"crossover": result, "rule": "largest size up to which every point has "
                      f"the single CTA within {NOISE:.0%} of the grid warm"}), flush=True)
    return 0


def _ipc_worker(rank, world, port, ops, sizes, handshakes, steps, warmup, outfile):
    """One rank of `--ipc` (a spawned process).  For each operation,
    handshake and payload size B (bytes per rank; BF16 for the reductions):
    warm-up, `steps` timed epochs, a bit check against the single-process
    entry point on local copies, and the kernel alone over the mapped
    staging buffers."""
    import torch
    import torch.distributed as dist

    import reduce_copy_rank_gb300 as dc
    from reduce_copy_rank_gb300.ipc import CudaIpcTransport, StagedAllGather, StagedAllReduce, StagedReduceScatter

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    lines = []
    for op, hs, B in [(o, h, b) for o in ops for h in handshakes for b in sizes]:
        if op == "all_gather":
            coll = StagedAllGather(None, B, CudaIpcTransport(), timeout=60.0, handshake=hs)
            payloads = [W.random_bytes_device(W.seed_for(2, 950), q, B, "cuda") for q in range(world)]
            expect = torch.cat(payloads)
            out = torch.empty(world * B, dtype=torch.uint8, device="cuda")
            run = lambda: coll.all_gather(payloads[rank], out)  # noqa: E731
            kernel = lambda views: dc.all_gather(views, out)  # noqa: E731
            alg = algorithmic_bytes(world, B)
        else:
            n = B // 2
            payloads = [W.normal_bf16_device(W.seed_for(4, 950), q, n, "cuda") for q in range(world)]
            if op == "all_reduce":
                coll = StagedAllReduce(None, n, "bf16", CudaIpcTransport(), timeout=60.0, handshake=hs)
                outs = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
                dc.all_reduce(payloads, outs)
                expect = outs[rank]
                out = torch.empty(n, dtype=torch.bfloat16, device="cuda")
                run = lambda: coll.all_reduce(payloads[rank], out)  # noqa: E731
                offset, alg = 0, (world + 1) * B
            else:
                C = n // world
                coll = StagedReduceScatter(None, C, "bf16", CudaIpcTransport(), timeout=60.0, handshake=hs)
                payloads = [x[:world * C] for x in payloads]
                outs = [torch.empty(C, dtype=torch.bfloat16, device="cuda") for _ in range(world)]
                dc.reduce_scatter(payloads, outs)
                expect = outs[rank]
                out = torch.empty(C, dtype=torch.bfloat16, device="cuda")
                run = lambda: coll.reduce_scatter(payloads[rank], out)  # noqa: E731
                offset, alg = rank * C, world * C * 2 + C * 2
            nbytes = payloads[0].nbytes
            kernel = lambda views: dc.reduce([v.view(torch.bfloat16) for v in views], out, offset=offset)  # noqa: E731
        for _ in range(warmup):
            run()
        coll.seconds = dict.fromkeys(coll.seconds, 0.0)
        dist.barrier()
        t0 = time.perf_counter()
        for _ in range(steps):
            run()
        epoch_s = (time.perf_counter() - t0) / steps
        exact = bool(torch.equal(out.view(torch.uint8), expect.view(torch.uint8)))
        # the kernel alone over the mapped staging buffers, one rank at a
        # time: a CUDA graph of 20 back-to-back calls (eager calls from Python
        # would time the host's launch rate instead)
        kernel_us = 0.0
        for q in range(world):
            dist.barrier()
            if q == rank:
                views = [b[:(B if op == "all_gather" else nbytes)] for b in coll.peers]
                side = torch.cuda.Stream()
                with torch.cuda.stream(side):
                    kernel(views)
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=side):
                        for _ in range(20):
                            kernel(views)
                torch.cuda.synchronize()
                times = []
                for _ in range(5):
                    s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    s_ev.record()
                    g.replay()
                    e_ev.record()
                    torch.cuda.synchronize()
                    times.append(s_ev.elapsed_time(e_ev) * 1e3 / 20)
                kernel_us = statistics.median(times)
                del g, views
        dist.barrier()
        vals = torch.tensor([epoch_s] + [coll.seconds[k] / steps for k in coll.seconds] + [kernel_us, float(not exact)],
                            dtype=torch.float64)
        dist.all_reduce(vals, op=dist.ReduceOp.MAX)
        del payloads, expect, out, run, kernel
        coll.close()
        if rank == 0:
            v = vals.tolist()
            lines.append({
                "metric": f"staged {op} across processes on one GPU: us per epoch",
                "impl": "dc-ipc", "op": op, "P": world, "bytes_per_rank": B, "epochs": steps, "warmup": warmup,
                "us_per_epoch": v[0] * 1e6,
                "phases_us": {k: x * 1e6 for k, x in zip(coll.seconds, v[1:5])},
                "kernel_us": v[5],
                "kernel_gbs": alg / (v[5] * 1e3) if v[5] > 0 else None,
                "bit_exact_vs_single_process_entry_point": v[6] == 0.0,
                "timing": "host clock around each epoch (max over ranks); the kernel by CUDA events "
                          "around a graph of 20 back-to-back calls over the mapped buffers, one rank "
                          "at a time (median of 5 replays; buffers L2-resident)",
                "handshake": {"shm": "node-local shared-memory arrival counters, bounded",
                              "gloo": "gloo monitored_barrier, bounded"}[hs],
            })
    if rank == 0:
        with open(outfile, "w") as fh:
            for ln in lines:
                fh.write(json.dumps(ln) + "\n")
    dist.destroy_process_group()


def run_ipc(args) -> int:
    """`--ipc`: the staged collectives across processes, ranks as processes
    sharing this GPU (CUDA IPC staging buffers, host handshakes)."""
    import socket
    import tempfile

    import torch.multiprocessing as mp

    steps = min(args.steps, 200)
    warmup = max(args.warmup, 3)
    for world in args.ipc_ranks:
        with socket.socket() as so:
            so.bind(("127.0.0.1", 0))
            port = so.getsockname()[1]
        with tempfile.TemporaryDirectory() as td:
            path = os.path.join(td, "ipc.jsonl")
            mp.spawn(_ipc_worker, args=(world, port, list(args.ipc_ops), list(args.ipc_sizes),
                                        list(args.ipc_handshakes), steps, warmup, path),
                     nprocs=world, join=True)
            with open(path) as fh:
                for ln in fh:
                    print(ln.strip(), flush=True)
    return 0


def run_skew(args) -> int:
    """Rank-skew calibration (the page "[Benchmark] Add all-reduce rank-skew
    calibration", section "Test Plan"): BF16 all_reduce of each shape per
    rank on P simulated ranks, one rank delayed on the GPU by each requested
    delay, eager and CUDA-graph mode; one JSON line of medians per point."""
    import torch

    import reduce_copy_rank_gb300 as dc
    from reduce_copy_rank_gb300.skew import SkewTrial

    device = torch.device("cuda", 0)
    lines = []
    for P in args.skew_ranks:
        inj = P - 1 if args.skew_rank is None else args.skew_rank
        for shape in args.skew_shapes:
            n = W.CONFIG4_COUNTS[shape]
            ins = [W.normal_bf16_device(W.seed_for(4, 9990), r, n, device) for r in range(P)]
            outs = [torch.empty_like(x) for x in ins]
            for mode in args.skew_modes:
                cal = SkewTrial(P=P, collective=lambda st: dc.all_reduce(ins, outs, stream=st),
                                injected_rank=inj, mode=mode)
                for d in args.skew_delays_us:
                    res = cal.run(d, trials=args.skew_trials, warmup=args.skew_warmup)
                    res.pop("trials_detail")
                    res.update({"op": "all_reduce_bf16", "shape": shape, "count": n})
                    print(json.dumps(res), flush=True)
                    lines.append(res)
            del ins, outs
    if args.out:
        with open(args.out, "w") as fh:
            for ln in lines:
                fh.write(json.dumps(ln) + "\n")
    return 0


def run_case(args) -> int:
    """Run one operation a few times with nothing else on the GPU (for ncu)."""
    import torch

    import reduce_copy_rank_gb300 as dc

    op, P, nbytes, reps = args.case.split(":")
    P, nbytes, reps = int(P), int(nbytes), int(reps)
    device = torch.device("cuda", 0)
    if op == "gather":
        peers = [torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device=device) for _ in range(P)]
        out = torch.empty(P * nbytes, dtype=torch.uint8, device=device)
        fn = lambda: dc.all_gather(peers, out)  # noqa: E731
    elif op == "ugather":  # unaligned: every payload starts 1 byte, the output 3 bytes past 16
        peers = [torch.randint(0, 256, (nbytes + 1,), dtype=torch.uint8, device=device)[1:]
                 for _ in range(P)]
        out = torch.empty(P * nbytes + 3, dtype=torch.uint8, device=device)[3:]
        fn = lambda: dc.all_gather(peers, out)  # noqa: E731
    elif op == "allreduce":
        ins = [torch.randn(nbytes // 2, device=device).to(torch.bfloat16) for _ in range(P)]
        outs = [torch.empty_like(x) for x in ins]
        fn = lambda: dc.all_reduce(ins, outs)  # noqa: E731
    elif op == "many":  # the all_gather_many workload (six mixed tensors); BYTES unused
        tens = [[W.random_bytes_device(W.seed_for(5, 1), r, B, device, tensor=t) for r in range(P)]
                for t, B in enumerate(W.CONFIG5_MANY_SIZES)]
        outs = [torch.empty(P * B, dtype=torch.uint8, device=device) for B in W.CONFIG5_MANY_SIZES]
        fn = lambda: dc.all_gather_many(tens, outs)  # noqa: E731
    elif op == "allreduce_mis":  # rank 1's input one element past the others' alignment
        store = [torch.randn(nbytes // 2 + 8, device=device).to(torch.bfloat16) for _ in range(P)]
        ins = [store[r][(1 if r == 1 else 0):(1 if r == 1 else 0) + nbytes // 2] for r in range(P)]
        outs = [torch.empty(nbytes // 2, dtype=torch.bfloat16, device=device) for _ in range(P)]
        fn = lambda: dc.all_reduce(ins, outs)  # noqa: E731
    elif op == "gatherbulk":  # the opt-in TMA bulk-copy path of the aligned gather
        peers = [torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device=device) for _ in range(P)]
        out = torch.empty(P * nbytes, dtype=torch.uint8, device=device)
        dc.set_option("gather_bulk", 1)
        fn = lambda: dc.all_gather(peers, out)  # noqa: E731
    elif op == "manytiny":  # 120 tensors of 3..100 B per rank at +1 B (BYTES unused)
        rng = np.random.default_rng(W.seed_for(5, 9005))
        sizes = [int(x) for x in rng.integers(3, 101, 120)]
        tens = [[torch.randint(0, 256, (B + 1,), dtype=torch.uint8, device=device)[1:] for _ in range(P)]
                for B in sizes]
        outs = [torch.empty(P * B, dtype=torch.uint8, device=device) for B in sizes]
        fn = lambda: dc.all_gather_many(tens, outs)  # noqa: E731
    elif op == "manymid":  # 250 tensors of 4..64 KiB per rank at +1 B (BYTES unused)
        rng = np.random.default_rng(W.seed_for(5, 9011))
        sizes = [int(x) for x in rng.integers(4096, 65537, 250)]
        tens = [[torch.randint(0, 256, (B + 1,), dtype=torch.uint8, device=device)[1:] for _ in range(P)]
                for B in sizes]
        outs = [torch.empty(P * B, dtype=torch.uint8, device=device) for B in sizes]
        fn = lambda: dc.all_gather_many(tens, outs)  # noqa: E731
    elif op == "fused":  # the staged all-gather protocol, P ranks x BYTES
        ins = [torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device=device) for _ in range(P)]
        stg = [torch.empty(nbytes, dtype=torch.uint8, device=device) for _ in range(P)]
        outs = [torch.empty(P * nbytes, dtype=torch.uint8, device=device) for _ in range(P)]
        ws = dc.fused_workspace(P, device)
        epoch = [0]

        def fn():
            epoch[0] += 1
            dc.fused_all_gather(ins, stg, outs, ws, epoch[0])
    elif op == "fill":  # a write-only stream of P * BYTES bytes (torch zero_ of float32; a comparator)
        buf = torch.empty(P * nbytes // 4, dtype=torch.float32, device=device)
        fn = buf.zero_
    elif op == "reducescatter":
        ins = [torch.randn(nbytes // 2, device=device).to(torch.bfloat16) for _ in range(P)]
        outs = [torch.empty(nbytes // 2 // P, dtype=torch.bfloat16, device=device) for _ in range(P)]
        fn = lambda: dc.reduce_scatter(ins, outs)  # noqa: E731
    else:
        raise SystemExit(f"unknown op {op}")
    for _ in range(reps):
        fn()
    torch.cuda.synchronize()
    dc.check_device()
    print(f"ran {op} P={P} bytes_per_rank={nbytes} x{reps}")
    return 0


def emit(line, args):
    s = json.dumps(line)
    print(s, flush=True)
    if args.out:
        with open(args.out, "w") as fh:
            fh.write(s + "\n")


def main(argv=None) -> int:
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.crossover:
        return run_crossover(args)
    if args.case:
        return run_case(args)
    if args.skew:
        return run_skew(args)
    if args.ipc:
        return run_ipc(args)
    return run_dc(args)


if __name__ == "__main__":
    sys.exit(main())
