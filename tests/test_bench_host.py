"""Host-side helpers of bench.py, on CPU: the quantiles reported for the
isolated (L2-flushed) calls, linear interpolation between order statistics."""
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def test_isolated_call_quantiles():
    ms = [0.010, 0.002, 0.004, 0.008, 0.006]            # 2..10 us, unsorted
    assert bench.quantile_us(ms, 0.5) == 6.0
    assert bench.quantile_us(ms, 0.0) == 2.0 and bench.quantile_us(ms, 1.0) == 10.0
    assert bench.quantile_us(ms, 0.1) == 2.8            # 0.4 of the way from 2 to 4
    assert bench.quantile_us(ms, 0.9) == 9.2
    assert bench.quantile_us([0.003], 0.9) == 3.0
