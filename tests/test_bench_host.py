"""Host-side helpers of bench.py, on CPU: the quantiles reported for the
isolated (L2-flushed) calls, linear interpolation between order statistics;
how the timed calls are split into captured CUDA graphs."""
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


def test_graph_plan_keeps_graphs_long_and_rounds_whole():
    """Captured graphs hold whole rounds over the buffer copies and at least
    64 calls (a boundary between graph replays breaks the dependent-launch
    overlap), and together they run exactly the requested calls."""
    for copies in (1, 4, 15, 16, 23, 33, 64, 100):
        for steps in (1, 3, 20, 40, 64, 100, 200, 1000):
            per, full, tail = bench.graph_plan(steps, copies)
            assert full * per + tail == steps and 0 <= tail < per
            assert per == steps or (per % copies == 0 and per >= bench.GRAPH_CALLS)
    assert bench.graph_plan(20, 4) == (20, 1, 0)          # the default bench: one graph of 20 calls
    assert bench.graph_plan(200, 15) == (75, 2, 50)
    assert bench.graph_plan(200, 1) == (64, 3, 8)         # an L2-resident layer: 64 calls a graph, not 1

