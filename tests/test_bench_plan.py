"""The benchmark's loop plans on CPU: the device-timed graphs time exactly
the requested steps, and the end-to-end loop's input slots are never
overwritten while a step that reads them may still run."""
import pytest

import bench


@pytest.mark.parametrize("steps", [1, 2, 63, 64, 65, 2000])
@pytest.mark.parametrize("nrep", [1, 2, 3, 15, 64])
def test_timed_plan_times_exactly_the_requested_steps(steps, nrep):
    per_graph, full, rem = bench.timed_plan(steps, nrep)
    assert full * per_graph + rem == steps
    assert 0 <= rem < per_graph
    assert per_graph % nrep == 0                 # every graph is whole rounds
    assert per_graph >= bench.TIMED_MIN_STEPS
    assert per_graph < bench.TIMED_MIN_STEPS + nrep


def _replay(per_graph, grp, groups, nrep):
    """Walk the plan in stream order: returns, per slot, the steps that read
    it and the group that wrote it, checking each group's dependencies."""
    assert [i for _, idx, _, _ in groups for i in idx] == list(range(per_graph))
    readers = {}          # slot -> [(group, step)]
    for n, idx, slot0, free_after in groups:
        assert 1 <= len(idx) <= grp
        assert slot0 == (n % 2) * grp
        slots = [slot0 + i - idx[0] for i in idx]
        assert all(0 <= s < 2 * grp for s in slots)
        # Every earlier reader of these slots must be at or before the step
        # whose completion this group's copy waits for.
        earlier = [st for s in slots for (_, st) in readers.get(s, [])]
        if earlier:
            assert free_after is not None and max(earlier) <= free_after < idx[0]
        else:
            assert free_after is None or free_after < idx[0]
        for s, i in zip(slots, idx):
            readers.setdefault(s, []).append((n, i))
    return readers


@pytest.mark.parametrize("nrep", [1, 2, 3, 9, 16, 64])
@pytest.mark.parametrize("input_bytes", [73984, 98560, 1319168, 2064640, 14164224])
def test_e2e_schedule_slots_are_free_before_they_are_rewritten(nrep, input_bytes):
    per_graph, grp, groups = bench.e2e_schedule(nrep, input_bytes, 1 << 20)
    assert per_graph % nrep == 0 and per_graph >= 2 * nrep
    assert per_graph >= bench.E2E_MIN_STEPS       # 1 MB results: no cap applies
    assert grp * input_bytes <= max(input_bytes, bench.E2E_GROUP_BYTES)
    assert grp <= max(1, per_graph // 8)         # groups overlap each other
    _replay(per_graph, grp, groups, nrep)


def test_e2e_schedule_bounds_the_result_spans():
    # 12 MB of results per step: the graph shrinks to two rounds, no fewer.
    per_graph, _, _ = bench.e2e_schedule(9, 14164224, 12681216)
    assert per_graph == 18
    per_graph, _, _ = bench.e2e_schedule(2, 2064640, 1597440)
    assert per_graph == 64 and per_graph * 1597440 <= bench.E2E_MAX_RESULT_BYTES


def test_a_planted_slot_reuse_is_caught():
    # The checker itself: a plan whose third group does not wait for the
    # first must fail.
    per_graph, grp, groups = bench.e2e_schedule(2, 2064640, 1 << 20)
    n, idx, slot0, _ = groups[2]
    bad = list(groups)
    bad[2] = (n, idx, slot0, None)
    with pytest.raises(AssertionError):
        _replay(per_graph, grp, bad, 2)
