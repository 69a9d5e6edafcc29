"""Independent steps in one launch, checked on the CPU.

The library merges runs of consecutive steps that touch disjoint bytes into
one launch (vc_set_merge_steps), and splits a step whose operations outgrow
the kernel parameter block into several.  Here both passes are re-derived
from the described plan alone (tests/plan_replay.py: launch_groups,
launches_of) and the launch count vc_plan_form reports for per-step execution
must equal the re-derived one, for every collective and schedule, rank
counts 2..16, fp32, bf16 and int32, with merging on and off.  A merge of two
dependent steps (a race: the second would read or overwrite what the first
is still writing) would show as fewer launches than the re-derivation finds.

In-place calls alias buffers the pass compares by kind: an AllReduce in
place runs its out-of-place plan with each rank's send and receive buffer
one, and a Broadcast or Reduce in place shares the root's.  The grouping
re-derived with those buffers made one must equal the plain grouping, so no
merge depends on the buffers being distinct.
"""
import pytest

import collective_communication_algorithms_virtual_gb300 as vc

from .plan_replay import Memory, get_plan, launch_groups, launches_of

CASES = [("allreduce", a, 0) for a in ("ring", "rhd", "dbt", "mesh", "ring_hop", "fused")] + \
    [("reduce_scatter", a, 0) for a in ("ring", "fused")] + [("allgather", a, 0) for a in ("ring", "fused")] + \
    [("broadcast", a, 0) for a in ("binomial", "scatter_allgather", "fused")] + \
    [("broadcast", "pipe_chain", 3), ("broadcast", "pipe_tree", 3), ("broadcast", "pipe_tree", 0)] + \
    [("scatter", a, 0) for a in ("binomial", "fused")] + [("gather", a, 0) for a in ("binomial", "fused")] + \
    [("reduce", a, 0) for a in ("binomial", "fused")] + \
    [("alltoall", a, 0) for a in ("pairwise", "bruck", "ring", "fused")]


@pytest.fixture(autouse=True)
def _per_step():
    saved = (vc.vc_get_slice_limit(), vc.vc_get_single_launch(), vc.vc_get_merge_steps())
    vc.vc_set_slice_limit(0)
    vc.vc_set_single_launch(0)
    yield
    vc.vc_set_slice_limit(saved[0])
    vc.vc_set_single_launch(saved[1])
    vc.vc_set_merge_steps(saved[2])


def _plain(N, scratch):
    return Memory([None] * N, [0] * N, scratch).ident


@pytest.mark.parametrize("merge", [True, False])
@pytest.mark.parametrize("N", [2, 3, 4, 5, 7, 8, 16])
def test_launch_count_equals_the_rederived_groups(N, merge):
    vc.vc_set_merge_steps(merge)
    merged_somewhere = split_somewhere = False
    for dtype in ("f32", "bf16", "i32"):
        for coll, algo, k in CASES:
            for count in (N * 64 + 16, 1000 + 3):
                root = N - 1
                try:
                    plan, scratch = get_plan(coll, algo, N, count, dtype, root=root, nchunks=k)
                except Exception:
                    continue  # a shape the schedule does not define
                assert all(plan), (coll, algo, N, count, "a step without operations")
                groups = launch_groups(plan, _plain(N, scratch)) if merge else [(s, s + 1) for s in range(len(plan))]
                want = sum(launches_of([op for st in plan[s:e] for op in st]) for s, e in groups)
                form, launches, _ = vc.vc_plan_form(coll, algo, N, count, dtype, root, False, k)
                what = (coll, algo, N, count, dtype, merge, groups)
                assert form == "steps" and launches == want, (what, form, launches, want)
                merged_somewhere |= any(e > s + 1 for s, e in groups)
                split_somewhere |= want > len(groups)
    assert merged_somewhere == merge
    if N == 16:
        assert split_somewhere


@pytest.mark.parametrize("N", [2, 3, 4, 5, 7, 8, 16])
def test_in_place_aliases_change_no_grouping(N):
    for dtype in ("f32", "bf16"):
        for coll, algo, k in CASES:
            if coll not in ("allreduce", "broadcast", "reduce"):
                continue
            for root in sorted({0, N - 1}):
                if coll == "allreduce" and root:
                    continue
                # an AllReduce in place runs the out-of-place plan (one rank in place excepted)
                plan_inplace = coll != "allreduce"
                try:
                    plan, scratch = get_plan(coll, algo, N, 1000 + 3, dtype, root=root, inplace=plan_inplace,
                                             nchunks=k)
                except Exception:
                    continue
                ranks = range(N) if coll == "allreduce" else [root]
                one = Memory([None] * N, [0] * N, scratch, inplace_ranks=ranks).ident
                assert launch_groups(plan, one) == launch_groups(plan, _plain(N, scratch)), (coll, algo, N, root)


def test_a_merge_across_a_dependency_is_caught():
    """Planted in the re-derivation: every operand taken as its own buffer, so
    no dependency is seen and each run of same-kind steps merges.  Its launch
    count must then differ from the library's wherever steps depend on one
    another (the Ring AllReduce and AllGather, Bruck), and agree where they do
    not (Pairwise AllToAll)."""
    vc.vc_set_merge_steps(True)
    blind = lambda k, o: object()  # noqa: E731
    for coll, algo, same in (("allreduce", "ring", False), ("allgather", "ring", False),
                             ("alltoall", "bruck", False), ("alltoall", "pairwise", True)):
        plan, _ = get_plan(coll, algo, 8, 1000 + 3, "f32")
        want = sum(launches_of([op for st in plan[s:e] for op in st]) for s, e in launch_groups(plan, blind))
        assert (vc.vc_plan_form(coll, algo, 8, 1000 + 3, "f32")[1] == want) == same, (coll, algo, want)
