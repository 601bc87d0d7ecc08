"""Rank-skew calibration on simulated ranks.

Page, by title: "[Benchmark] Add all-reduce rank-skew calibration" (vLLM
pull request 57037).  Section "Purpose": a collective's duration includes
the time spent waiting for late ranks; the calibration delays one rank on
the GPU and reports per-rank timings for BF16 shapes, eagerly or as a CUDA
graph, with the maximum residence, the injected rank's residence, the
measured delay and the gap between the two residences per trial.  The
review (calvin-fei) adds the residence of the rank that actually arrived
last (at zero requested delay the injected rank need not be last) and asks
that the measured delay, not the requested one, be used.

Here the P ranks are P CUDA streams of one GPU, each owning its buffers.  A
trial, after a host synchronisation (the CPU barrier of the page's design):

    start event (main stream)
    every rank stream waits for it          -- all ranks begin together
    injected rank: delay_begin event, a GPU delay of the requested length
                   (library kernel), delay_end event
    every rank: arrival event               -- the rank reaches the collective
    the main stream waits for every arrival, runs the collective, done event

Rank r's residence = done - arrival_r: the time rank r spends inside the
collective, waiting for later ranks included (the page's GPU residence
includes peer waiting).  All times come from CUDA events of one device, so
no clocks of different GPUs are compared.  In graph mode the whole trial is
captured once per requested delay and replayed.
"""
from __future__ import annotations

import statistics
from dataclasses import dataclass, field
from typing import Callable, Sequence

from . import inject_delay

SUMMARY_FIELDS = ("max_residence_ms", "injected_rank_residence_ms", "last_arriving_residence_ms",
                  "measured_delay_ms", "residence_gap_ms", "collective_ms")


def summarize_trial(arrival_ms: Sequence[float], done_ms: float, delay_ms: float,
                    injected_rank: int, collective_start_ms: float | None = None) -> dict:
    """One trial's figures from event times (ms since the trial's start event).

    arrival_ms[r]: when rank r reached the collective; done_ms: when the
    collective finished; delay_ms: the injected delay as measured (its own
    events); collective_start_ms: when the collective kernel began (None if
    not recorded)."""
    P = len(arrival_ms)
    if P == 0:
        raise ValueError("need at least one rank")
    if not 0 <= injected_rank < P:
        raise ValueError(f"injected rank {injected_rank} is outside 0..{P - 1}")
    residence = [done_ms - a for a in arrival_ms]
    last = max(range(P), key=lambda r: (arrival_ms[r], r))
    out = {
        "residence_ms": residence,
        "arrival_ms": list(arrival_ms),
        "max_residence_ms": max(residence),
        "injected_rank": injected_rank,
        "injected_rank_residence_ms": residence[injected_rank],
        "last_arriving_rank": last,
        "last_arriving_residence_ms": residence[last],
        "measured_delay_ms": delay_ms,
        "residence_gap_ms": max(residence) - residence[injected_rank],
        "collective_ms": (done_ms - collective_start_ms) if collective_start_ms is not None else None,
    }
    return out


def summarize(trials: Sequence[dict]) -> dict:
    """Medians over trials of every scalar figure, how often the injected
    rank arrived last, and the trial count."""
    if not trials:
        raise ValueError("no trials")
    s = {"trials": len(trials)}
    for k in SUMMARY_FIELDS:
        xs = [t[k] for t in trials if t.get(k) is not None]
        s[f"median_{k}"] = statistics.median(xs) if xs else None
    s["injected_arrived_last_fraction"] = sum(
        t["last_arriving_rank"] == t["injected_rank"] for t in trials) / len(trials)
    return s


@dataclass
class SkewTrial:
    """A calibration harness for one collective call on P simulated ranks.

    collective(stream) must enqueue the collective on `stream` (the main
    stream of the trial) and nothing else.  Rank streams, events and CUDA
    graphs are created once; `run(delay_us, trials, warmup)` returns the
    per-trial figures and their summary."""

    P: int
    collective: Callable
    injected_rank: int = 0
    mode: str = "eager"
    device: object = None
    _graphs: dict = field(default_factory=dict, init=False, repr=False)

    def __post_init__(self):
        import torch

        if self.mode not in ("eager", "graph"):
            raise ValueError(f"mode must be 'eager' or 'graph', not {self.mode!r}")
        if not 0 <= self.injected_rank < self.P:
            raise ValueError(f"injected rank {self.injected_rank} is outside 0..{self.P - 1}")
        self._t = torch
        self.device = torch.device("cuda", torch.cuda.current_device()) if self.device is None \
            else torch.device(self.device)
        self.main = torch.cuda.Stream(device=self.device)
        self.ranks = [torch.cuda.Stream(device=self.device) for _ in range(self.P)]
        ext = self.mode == "graph"  # events recorded inside a graph must be external
        mk = lambda: torch.cuda.Event(enable_timing=True, external=ext)  # noqa: E731
        self.ev_start, self.ev_done, self.ev_coll = mk(), mk(), mk()
        self.ev_d0, self.ev_d1 = mk(), mk()
        self.ev_arrive = [mk() for _ in range(self.P)]
        # ordering between streams uses plain events (inside a capture they
        # become graph edges); the timing events above are timestamps only
        self.sync_start = torch.cuda.Event()
        self.sync_arrive = [torch.cuda.Event() for _ in range(self.P)]

    def _enqueue(self, delay_ns: int):
        main = self.main
        self.ev_start.record(main)
        self.sync_start.record(main)
        for r, s in enumerate(self.ranks):
            s.wait_event(self.sync_start)
            if r == self.injected_rank:
                self.ev_d0.record(s)
                inject_delay(delay_ns, s)
                self.ev_d1.record(s)
            self.ev_arrive[r].record(s)
            self.sync_arrive[r].record(s)
        for r in range(self.P):
            main.wait_event(self.sync_arrive[r])
        self.ev_coll.record(main)
        self.collective(main)
        self.ev_done.record(main)

    def _graph(self, delay_ns: int):
        torch = self._t
        g = self._graphs.get(delay_ns)
        if g is None:
            g = torch.cuda.CUDAGraph()
            torch.cuda.synchronize(self.device)
            with torch.cuda.graph(g, stream=self.main):
                self._enqueue(delay_ns)
            torch.cuda.synchronize(self.device)
            self._graphs[delay_ns] = g
        return g

    def trial(self, delay_us: float) -> dict:
        torch = self._t
        ns = int(round(delay_us * 1000.0))
        torch.cuda.synchronize(self.device)  # host barrier before each trial
        if self.mode == "graph":
            self._graph(ns).replay()
        else:
            self._enqueue(ns)
        torch.cuda.synchronize(self.device)
        t0 = self.ev_start
        arrival = [t0.elapsed_time(e) for e in self.ev_arrive]
        rec = summarize_trial(arrival, t0.elapsed_time(self.ev_done),
                              self.ev_d0.elapsed_time(self.ev_d1), self.injected_rank,
                              t0.elapsed_time(self.ev_coll))
        rec["requested_delay_us"] = delay_us
        return rec

    def run(self, delay_us: float, trials: int = 50, warmup: int = 10) -> dict:
        if trials < 1 or warmup < 0:
            raise ValueError("need trials >= 1 and warmup >= 0")
        if self.mode == "graph":
            self._graph(int(round(delay_us * 1000.0)))
        for _ in range(warmup):
            self.trial(delay_us)
        recs = [self.trial(delay_us) for _ in range(trials)]
        return {"requested_delay_us": delay_us, "mode": self.mode, "P": self.P,
                "injected_rank": self.injected_rank, **summarize(recs), "trials_detail": recs}
