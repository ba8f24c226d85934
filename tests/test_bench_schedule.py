"""bench.py's timed region runs exactly K decode steps whatever K is: full
graphs of STEPS_PER_GRAPH consecutive steps, then one graph of the
remaining steps, every step number once and in order within each graph."""
import pytest

import bench


@pytest.mark.parametrize("steps", [1, 3, 7, 8, 9, 20, 127, 128, 129, 20000])
def test_schedule_runs_exactly_k_steps(steps):
    g, n = bench.STEPS_PER_GRAPH, bench.N_SLOTS
    sched = bench.graph_schedule(steps, g, n)
    counted = [st for _, _, sts in sched for st in sts]
    assert len(counted) == steps
    full = [e for e in sched if e[0] == "full"]
    rest = [e for e in sched if e[0] == "rest"]
    assert len(full) == steps // g and len(rest) == (1 if steps % g else 0)
    assert sched == full + rest  # full graphs first
    for kind, j, sts in full:
        assert 0 <= j < n and sts == list(range(j * g, j * g + g))  # graph j's own consecutive steps
    # the remainder's step numbers continue after the full graphs' count
    assert [s for _, _, sts in rest for s in sts] == list(range((steps // g) * g, steps))
