"""GPU tests of the rank-skew calibration on simulated ranks: the injected
delay's accuracy, the residence figures in eager and graph mode, and the
collective's bits under skew (the fixed order does not depend on which rank
arrives last).

Page, by title: "[Benchmark] Add all-reduce rank-skew calibration" (vLLM pull
request 57037), sections "Purpose" and "Test Plan" (shapes 8x8192 and
8627x8192 per rank, requested delays 0 / 50 / 250 / 1000 us, eager and CUDA
graph), and the review's tables (the late rank's residence stays flat, the
maximum grows by the measured delay).
"""
import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import assert_bf16_equal, bits_of

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import reduce_copy_rank_gb300 as dc  # noqa: E402
from reduce_copy_rank_gb300.skew import SkewTrial  # noqa: E402


def test_delay_is_at_least_requested_and_close():
    s = torch.cuda.current_stream()
    for us in (0, 50, 250, 1000, 5000):
        got = []
        for _ in range(5):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(s)
            dc.inject_delay(us * 1000, s)
            b.record(s)
            torch.cuda.synchronize()
            got.append(a.elapsed_time(b) * 1e3)
        med = sorted(got)[2]
        assert med >= us - 1.0, (us, got)
        assert med <= us * 1.02 + 20.0, (us, got)


def test_delay_rejects_above_limit():
    with pytest.raises(dc.DCError) as e:
        dc.inject_delay(dc.MAX_DELAY_NS + 1)
    assert e.value.name == "DC_ERR_INVALID"


@pytest.mark.parametrize("mode", ["eager", "graph"])
@pytest.mark.parametrize("P,shape", [(2, "8627x8192"), (4, "8x8192")])
def test_calibration_residences(mode, P, shape):
    n = W.CONFIG4_COUNTS[shape]
    seed = W.seed_for(4, 9990)
    ins = [W.normal_bf16_device(seed, r, n, "cuda") for r in range(P)]
    outs = [torch.empty_like(x) for x in ins]
    want = oracle.all_reduce_bf16([bits_of(x) for x in ins])
    inj = P - 1
    cal = SkewTrial(P=P, collective=lambda s: dc.all_reduce(ins, outs, stream=s),
                    injected_rank=inj, mode=mode)
    base = cal.run(0.0, trials=10, warmup=3)
    late = cal.run(1000.0, trials=10, warmup=3)
    coll = base["median_collective_ms"]
    # the injected delay is measured, about as requested
    assert 1.0 <= late["median_measured_delay_ms"] <= 1.05
    # with 1 ms of skew the injected rank arrives last and its residence stays
    # near the collective alone, while the earliest rank waits for it
    assert late["injected_arrived_last_fraction"] == 1.0
    assert late["median_injected_rank_residence_ms"] <= coll + 0.1
    grow = late["median_max_residence_ms"] - base["median_max_residence_ms"]
    assert abs(grow - late["median_measured_delay_ms"]) <= 0.1
    assert abs(late["median_residence_gap_ms"] - late["median_measured_delay_ms"]) <= 0.1
    for t in late["trials_detail"]:
        assert t["residence_ms"][inj] <= min(t["residence_ms"]) + 1e-9
    torch.cuda.synchronize()
    for r in range(P):
        assert_bf16_equal(bits_of(outs[r]), want, f"{mode} P={P} rank {r} under skew")


def test_skew_never_changes_bits():
    """Every rank takes a turn as the late one; the outputs stay identical."""
    P, n = 8, 1 << 20
    ins = [W.normal_bf16_device(W.seed_for(4, 9991), r, n, "cuda") for r in range(P)]
    want = oracle.all_reduce_bf16([bits_of(x) for x in ins])
    for inj in range(P):
        outs = [torch.empty_like(x) for x in ins]
        cal = SkewTrial(P=P, collective=lambda s: dc.all_reduce(ins, outs, stream=s),
                        injected_rank=inj, mode="eager")
        cal.run(100.0, trials=1, warmup=0)
        torch.cuda.synchronize()
        for r in range(P):
            assert_bf16_equal(bits_of(outs[r]), want, f"late rank {inj}, output {r}")
