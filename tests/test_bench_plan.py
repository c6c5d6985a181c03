"""Host logic of the benchmark's timed region (no GPU): which steps run as
graph replays and which eagerly, and how the replays are spread in front of
the eager kernel groups."""
import pytest

import bench


@pytest.mark.parametrize("steps,every,chunk", [(200, 4, 8), (20, 4, 8), (5, 4, 8), (200, 4, 12),
                                               (60, 4, 12), (7, 1, 8), (200, 4, 0), (3, 4, 2)])
def test_step_plan_covers_every_step_once(steps, every, chunk):
    plan = bench.StepPlan(steps, every, chunk)
    # the replayed steps come first in index, then the eager ones, no gap or overlap
    assert plan.replays * chunk + len(plan.eager_steps) == steps
    assert plan.eager_steps == list(range(plan.replays * chunk, steps))
    if chunk == 0:
        assert plan.replays == 0
    else:
        # at least the requested share of the steps runs eagerly (per-kernel timing)
        assert len(plan.eager_steps) >= (steps + every - 1) // every


@pytest.mark.parametrize("replays,groups", [(18, 28), (12, 28), (28, 28), (1, 5), (0, 6), (7, 3), (5, 0),
                                            (0, 0), (144, 7)])
def test_replay_schedule_spreads_all_replays_evenly(replays, groups):
    sched = bench.replay_schedule(replays, groups)
    assert sum(sched) == replays
    assert len(sched) == max(groups, 1)
    assert max(sched) - min(sched) <= 1
    assert min(sched) >= 0
