"""The per-unit collective schedule of a step against the counts the pages measured
(host logic, no GPU).

"NCCL ZeRO/FSDP state sharding" profiles a model of 8 Linear layers, each its own
FSDP unit, and counts the collectives of one steady step: SHARD_GRAD_OP ("ZeRO-2
方向") issues 8 forward all-gathers, no backward all-gather and 8 reduce-scatters;
FULL_SHARD ("ZeRO-3 方向") 8 forward and 8 backward all-gathers (16 in all) and 8
reduce-scatters."""
import pytest

from fsdp_sharded_state_gb300 import step_schedule

PAGE_COUNTS = {   # strategy -> (forward all-gathers, backward all-gathers, reduce-scatters), 8 units
    "shard_grad_op": (8, 0, 8),
    "full_shard": (8, 8, 8),
}


@pytest.mark.parametrize("strategy", sorted(PAGE_COUNTS))
def test_counts_match_the_pages(strategy):
    sched = step_schedule(8, strategy)
    fwd, bwd, rs = PAGE_COUNTS[strategy]
    first_rs = next(i for i, (k, _) in enumerate(sched) if k == "reduce_scatter")
    n_ag = sum(k == "all_gather" for k, _ in sched)
    assert sum(k == "all_gather" for k, _ in sched[:first_rs]) >= fwd
    assert n_ag == fwd + bwd
    assert sum(k == "reduce_scatter" for k, _ in sched) == rs
    if strategy == "full_shard":
        assert n_ag == 16


@pytest.mark.parametrize("strategy", sorted(PAGE_COUNTS))
@pytest.mark.parametrize("U", [1, 2, 5, 8])
def test_schedule_order(strategy, U):
    sched = step_schedule(U, strategy)
    # forward: every unit gathered once, in order, before any reduce-scatter
    assert sched[:U] == [("all_gather", u) for u in range(U)]
    back = sched[U:]
    # backward: units in reverse; each reduce-scatter once, after the unit's re-gather (FULL_SHARD)
    rs_units = [u for k, u in back if k == "reduce_scatter"]
    assert rs_units == list(reversed(range(U)))
    for u in range(U):
        i = back.index(("reduce_scatter", u))
        if strategy == "full_shard":
            assert back[i - 1] == ("all_gather", u)
        else:
            assert ("all_gather", u) not in back


def test_unknown_strategy():
    with pytest.raises(ValueError):
        step_schedule(8, "no_shard")
