"""bench.py's host-side choices: which bf16 peak a tensor-core kernel is measured
against, and which end-to-end run is reported."""

import bench

PEAKS = {"bf16_tflops": 1961.8, "bf16_tflops_sustained": 1770.3, "hbm_gbs": 6655.3}


def test_short_step_at_full_clock_uses_the_burst_peak():
    assert bench.tensor_peak(1.02, [], PEAKS) == (1961.8, "burst")


def test_long_step_uses_the_sustained_peak():
    assert bench.tensor_peak(bench.LONG_STEP_MS, [], PEAKS) == (1770.3, "sustained")
    assert bench.tensor_peak(310.0, [], PEAKS) == (1770.3, "sustained")


def test_power_cap_in_the_timed_region_uses_the_sustained_peak():
    assert bench.tensor_peak(1.0, ["sw_power_cap"], PEAKS) == (1770.3, "sustained")


def test_median_trial_takes_the_longer_clock_of_each_run():
    # (device ms, wall ms) of five runs of 20 steps; the middle one by max() is (40, 46)
    trials = [(36.0, 30.0), (55.0, 40.0), (40.0, 46.0), (38.0, 44.0), (60.0, 70.0)]
    per_step, chosen = bench.median_trial(trials, 20)
    assert per_step == [1.8, 2.2, 2.3, 2.75, 3.5]
    assert chosen == (40.0, 46.0)


def test_median_trial_of_one_run_is_that_run():
    assert bench.median_trial([(10.0, 12.0)], 4) == ([3.0], (10.0, 12.0))
