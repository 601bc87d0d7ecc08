"""Host arithmetic of the rank-skew calibration summaries (no GPU).

Page, by title: "[Benchmark] Add all-reduce rank-skew calibration" (vLLM pull
request 57037): per trial the maximum residence, the injected rank's
residence, the measured delay and their gap; the review's table (pynccl
graph, 8627x8192) shows the delayed rank's residence flat while the maximum
grows by the measured delay, and asks for the last-arriving rank's residence
because the injected rank need not arrive last.
"""
import pytest

from reduce_copy_rank_gb300.skew import summarize, summarize_trial


def test_residence_is_done_minus_arrival():
    t = summarize_trial([0.010, 0.012, 1.020, 0.011], done_ms=1.500, delay_ms=1.009, injected_rank=2,
                        collective_start_ms=1.030)
    assert t["residence_ms"] == pytest.approx([1.490, 1.488, 0.480, 1.489])
    assert t["max_residence_ms"] == pytest.approx(1.490)
    assert t["injected_rank_residence_ms"] == pytest.approx(0.480)
    assert t["last_arriving_rank"] == 2
    assert t["last_arriving_residence_ms"] == pytest.approx(0.480)
    # the gap between the waiting and the late rank is the waiting time
    assert t["residence_gap_ms"] == pytest.approx(1.010)
    assert t["measured_delay_ms"] == 1.009
    assert t["collective_ms"] == pytest.approx(0.470)


def test_injected_rank_need_not_arrive_last():
    # zero requested delay: rank 1 happens to arrive after the injected rank 0
    t = summarize_trial([0.004, 0.006, 0.005], done_ms=0.500, delay_ms=0.003, injected_rank=0)
    assert t["last_arriving_rank"] == 1
    assert t["last_arriving_residence_ms"] == pytest.approx(0.494)
    assert t["injected_rank_residence_ms"] == pytest.approx(0.496)
    assert t["residence_gap_ms"] == pytest.approx(0.0)
    assert t["collective_ms"] is None


def test_ties_pick_the_highest_rank_as_last():
    t = summarize_trial([0.1, 0.1], done_ms=0.3, delay_ms=0.0, injected_rank=0)
    assert t["last_arriving_rank"] == 1


def test_summary_medians_and_fraction():
    trials = [summarize_trial([0.0, d], done_ms=d + 0.3, delay_ms=d, injected_rank=1)
              for d in (1.0, 1.1, 0.9)]
    trials.append(summarize_trial([0.2, 0.0], done_ms=0.5, delay_ms=0.0, injected_rank=1))
    s = summarize(trials)
    assert s["trials"] == 4
    assert s["injected_arrived_last_fraction"] == 0.75
    assert s["median_measured_delay_ms"] == pytest.approx(0.95)
    assert s["median_injected_rank_residence_ms"] == pytest.approx(0.3)
    assert s["median_collective_ms"] is None


@pytest.mark.parametrize("bad", [dict(arrival_ms=[], done_ms=1.0, delay_ms=0.0, injected_rank=0),
                                 dict(arrival_ms=[0.0], done_ms=1.0, delay_ms=0.0, injected_rank=1),
                                 dict(arrival_ms=[0.0], done_ms=1.0, delay_ms=0.0, injected_rank=-1)])
def test_bad_arguments(bad):
    with pytest.raises(ValueError):
        summarize_trial(**bad)
    with pytest.raises(ValueError):
        summarize([])
