"""CPU checks of bench.py's host logic: workload accounting, statistics,
clock parsing, the ncu traffic record, the reference arm's rank handling,
and the multi-rank (replica) aggregation with world_size 2 over gloo."""
from __future__ import annotations

import json
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench
import workloads as W


def test_sweep_is_the_results_table_sizes():
    cases = bench.sweep_cases()
    assert len(cases) == 14
    assert [(P, B) for P, B, _ in cases][:7] == [(8, b) for b in W.CONFIG2_SIZES]
    assert {P for P, _, _ in cases} == {8, 2}
    step = sum(bench.algorithmic_bytes(P, B) for P, B, _ in cases)
    assert step == 2 * 10 * sum(W.CONFIG2_SIZES)  # P=8 and P=2: read + write
    assert len({s for _, _, s in cases}) == 14  # every call has its own seed


def test_stats_and_throughput():
    st = bench.stats([1.0, 2.0, 3.0, 4.0])
    assert st["us_mean"] == 2.5 and st["us_median"] == 2.5
    assert bench.job_throughput(1, 1_000_000, 1.0) == pytest.approx(1.0)  # 1 MB per ms = 1 GB/s
    assert bench.job_throughput(4, 1_000_000, 2.0) == pytest.approx(2.0)


def test_parse_args_defaults_and_errors():
    a = bench.parse_args([])
    assert a.gpus == 1 and a.steps >= 1 and a.warmup >= 3 and a.impl == "dc"
    with pytest.raises(SystemExit):
        bench.parse_args(["--steps", "0"])


def test_clock_sampler_parses_nvidia_smi_rows(tmp_path, monkeypatch):
    rows = ["0, 2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Active",
            "0, 1965, 2070, 1200.0, 0x4, Not Active, Not Active, Not Active, Not Active",
            "0, 2070, 2070, 1300.0, 0x0, Not Active, Not Active, Not Active, Not Active"]
    s = bench.ClockSampler.__new__(bench.ClockSampler)

    class FakeProc:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    s.proc = FakeProc()
    f = tmp_path / "c.csv"
    f.write_text("\n".join(rows) + "\n")
    s.file = open(f, "r+")
    monkeypatch.setattr(bench.time, "sleep", lambda _x: None)
    res = s.stop()
    assert res["sm_mhz"] == 2070 and res["sm_max_mhz"] == 2070 and res["samples"] == 3
    assert res["reasons"] == ["sw_power_cap"]


def test_traffic_record_matches_only_current_sources(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    digest = bench.kernel_source_digest()
    (prof / "traffic.txt").write_text(
        "# comment\n"
        f"kernel=k1 source={digest} bytes_per_launch=123.5 ncu_us_per_launch=4.25\n"
        "kernel=k2 source=0000 bytes_per_launch=99\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_digest", lambda: digest)
    assert bench.load_traffic("k1") == {"bytes_per_launch": 123.5, "ncu_us_per_launch": 4.25}
    assert bench.load_traffic("k2") == {}  # taken from other kernel sources
    assert bench.load_traffic("k3") == {}


def test_reference_arm_nonzero_rank_does_no_work(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    assert bench.run_reference(bench.parse_args(["--impl", "reference", "--steps", "1"])) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_line(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "0")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"]) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["config"]["workload"] == bench.WORKLOAD
    assert line["config"] == bench.workload_config(1)  # the GPU arm prints the same dict


def test_by_size_rows_fractions():
    MiB = 1 << 20
    table = [{"P": P, "bytes_per_rank": B, "kernel": "k", "us_median": 10.0}
             for P in (8, 2) for B in (MiB, 4 * MiB)]
    b2b = [{"P": P, "bytes_per_rank": B, "us": 5.0} for P in (8, 2) for B in (MiB, 4 * MiB)]
    rows = bench.by_size_rows(table, b2b, 6000.0)
    assert [(r["P"], r["bytes_per_rank"]) for r in rows] == [(8, 4 * MiB), (8, MiB), (2, 4 * MiB), (2, MiB)]
    r = rows[0]
    assert r["alone_gbs"] == 2 * 8 * 4 * MiB / 10.0 / 1e3
    assert r["alone_frac_measured"] == r["alone_gbs"] / 6000.0
    assert r["back_to_back_frac_nominal"] == r["back_to_back_gbs"] / 8000.0


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _replica(rank, world, port, out_dir):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [3.0, 5.0][rank]  # rank 1 is the slow replica
    slow = bench.rank_max(local_ms, dist)
    value = bench.job_throughput(world, 10_000_000, slow)
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as fh:
        json.dump({"slow": slow, "value": value}, fh)
    dist.barrier()
    dist.destroy_process_group()


def test_replica_aggregation_world_size_2_gloo(tmp_path):
    mp.spawn(_replica, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(2)]
    for r in res:
        assert r["slow"] == 5.0  # every rank sees the slowest replica's time
        assert r["value"] == pytest.approx(2 * 10_000_000 / 5.0 / 1e6)


def test_rank_max_without_process_group():
    assert bench.rank_max(7.5) == 7.5


class _FakeClock:
    """A scripted device clock for the timing helpers: events read `now`
    when recorded; calls and flushes advance it."""

    def __init__(self):
        self.now = 0.0  # ms
        self.log = []

    def torch(self):
        clock = self

        class Event:
            def __init__(self, enable_timing=False, external=False):
                self.t = None

            def record(self, stream=None):
                self.t = clock.now

            def elapsed_time(self, other):
                return other.t - self.t

        class _Cuda:
            pass

        cuda = _Cuda()
        cuda.Event = Event
        cuda.synchronize = lambda *a, **k: None
        ns = type("FakeTorch", (), {})()
        ns.cuda = cuda
        return ns

    def call(self, name, ms):
        def fn():
            self.log.append(name)
            self.now += ms
        return fn


def test_timed_calls_attribute_each_call_and_exclude_the_flush():
    clk = _FakeClock()

    def flush():
        clk.log.append("flush")
        clk.now += 50.0  # never inside a call's events

    out = bench.timed_calls(clk.torch(), None, flush, [clk.call("a", 0.002), clk.call("b", 0.010)], 3)
    assert [round(x, 6) for x in out[0]] == [2.0] * 3  # microseconds
    assert [round(x, 6) for x in out[1]] == [10.0] * 3
    assert clk.log == ["flush", "a", "flush", "b"] * 3


def test_alternating_swaps_order_and_takes_medians():
    clk = _FakeClock()
    durations = {"a": [0.001, 0.003, 0.002, 0.100], "b": [0.005, 0.004, 0.006, 0.005]}
    counters = {"a": 0, "b": 0}

    def make(name):
        def fn():
            clk.log.append(name)
            clk.now += durations[name][counters[name]]
            counters[name] += 1
        return fn

    med = bench.alternating(clk.torch(), None, lambda: None, [make("a"), make("b")], 4)
    assert clk.log == ["a", "b", "b", "a", "a", "b", "b", "a"]
    assert round(med[0], 6) == 2.5  # median of 1, 3, 2, 100 us
    assert round(med[1], 6) == 5.0


def test_source_digest_follows_code_not_comments():
    """The traffic record stays valid across comment edits of the kernel
    sources, and goes stale on any change of the code."""
    code = 'int f(int a) {  // one\n  /* two */ const char* s = "x // not a comment";\n  return a; }\n'
    stripped = bench.strip_comments(code)
    assert "one" not in stripped and "two" not in stripped
    assert '"x // not a comment"' in stripped
    assert bench.strip_comments(code.replace("// one", "// other words")) == stripped
    assert bench.strip_comments(code.replace("return a;", "return a + 1;")) != stripped
