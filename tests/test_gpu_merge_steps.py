"""Independent steps in one launch (vc_set_merge_steps), against the oracle.

Pairwise AllToAll's rounds read only the send buffers and write their own
output blocks, and the Ring AllToAll's local copy touches nothing its first
round does, so those steps share a launch by default (as do the Mesh
AllReduce's result copies and some binomial steps at rank counts that are not
powers of 2, which the randomised sweep covers).  With the setting on
and off, every result must equal the C++ oracle's simulation bit for bit, the
launch trace must show the shared launch (or one launch per round), and canary
bands catch stray writes.  Schedules whose every step depends on the one
before (Ring AllReduce) keep one launch per step either way.
"""
import pytest
import torch

import collective_communication_algorithms_virtual_gb300 as vc
from oracle import cxx
from synthetic_inputs import rank_buffers

from .gpu_util import Guarded, first_diff, same_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from collective_communication_algorithms_virtual_gb300 import build

    build.build()
    vc.lib()
    saved = (vc.vc_get_merge_steps(), vc.vc_get_single_launch(), vc.vc_get_slice_limit())
    vc.vc_set_single_launch(0)  # one launch per step otherwise (small calls would take one cluster)
    vc.vc_set_slice_limit(0)
    yield
    vc.vc_set_merge_steps(saved[0])
    vc.vc_set_single_launch(saved[1])
    vc.vc_set_slice_limit(saved[2])
    assert vc.vc_device_errors() == 0


def _traced(fn):
    vc.vc_trace_enable(True)
    try:
        fn()
        torch.cuda.synchronize()
        return vc.vc_trace_read()
    finally:
        vc.vc_trace_enable(False)


@pytest.mark.parametrize("merge", [True, False])
@pytest.mark.parametrize("N", [2, 3, 5, 8, 16])
@pytest.mark.parametrize("dtype", ["bf16", "i32"])
def test_pairwise_and_ring_alltoall(N, dtype, merge):
    vc.vc_set_merge_steps(merge)
    assert vc.vc_get_merge_steps() == merge
    kind = {"bf16": "normal_bf16", "i32": "int32_bits"}[dtype]
    for B in (1, 7, 4096 + 3):
        xs = rank_buffers(kind, 9100 + N + B, N, N * B)
        for algo, nsteps in (("pairwise", N), ("ring", N)):
            want = cxx.alltoall(xs, algo, dtype, want_log=False).outputs
            sends = [Guarded(N * B, dtype, fill=x) for x in xs]
            recvs = [Guarded(N * B, dtype) for _ in range(N)]
            recs = _traced(lambda: vc.vc_alltoall([g.t for g in sends], [g.t for g in recvs], algo=algo))
            assert all(g.guards_intact() for g in sends + recvs)
            for r in range(N):
                got = recvs[r].host()
                assert same_bits(got, want[r]), (algo, N, B, merge, r, first_diff(got, want[r]))
            steps = sorted({rec["step"] for rec in recs})
            if algo == "pairwise":
                assert steps == ([0] if merge else list(range(nsteps))), (N, steps)
            elif N > 1:  # the local copy joins round 1; later rounds read the forwarding buffers
                assert steps == ([0] + list(range(2, nsteps)) if merge else list(range(nsteps))), (N, steps)


def test_merged_plan_skips_the_cluster_form():
    """With one-launch plans allowed (the default limit), a Pairwise AllToAll
    whose rounds all merge runs as that one merged launch, not as a cluster
    with a barrier per round; with merging off it runs a launch per round
    (AllToAlls never take the cluster form)."""
    N, B = 8, 2048  # 64 KiB per rank of fp32-sized int32
    xs = rank_buffers("int32_bits", 9150, N, N * B)
    want = cxx.alltoall(xs, "pairwise", "i32", want_log=False).outputs
    vc.vc_set_single_launch(vc.VC_SINGLE_LAUNCH_DEFAULT)
    try:
        for merge in (True, False):
            vc.vc_set_merge_steps(merge)
            sends = [Guarded(N * B, "i32", fill=x) for x in xs]
            recvs = [Guarded(N * B, "i32") for _ in range(N)]
            recs = _traced(lambda: vc.vc_alltoall([g.t for g in sends], [g.t for g in recvs], algo="pairwise"))
            assert len(recs) == (1 if merge else N), (merge, recs)
            assert not any(r["kernel"].endswith("_single_launch") or r["step"] == -1 for r in recs), (merge, recs)
            assert all(g.guards_intact() for g in sends + recvs)
            for r in range(N):
                assert same_bits(recvs[r].host(), want[r]), (merge, r)
    finally:
        vc.vc_set_single_launch(0)


def test_dependent_steps_keep_their_launches():
    vc.vc_set_merge_steps(True)
    N, count = 8, 65536
    xs = rank_buffers("uniform_f32", 9200, N, count)
    sends = [Guarded(count, "f32", fill=x) for x in xs]
    recvs = [Guarded(count, "f32") for _ in range(N)]
    for algo in ("ring", "rhd", "dbt"):
        recs = _traced(lambda: vc.vc_allreduce([g.t for g in sends], [g.t for g in recvs], algo=algo))
        nsteps = vc.vc_plan_describe("allreduce", algo, N, count)[2]
        assert sorted({r["step"] for r in recs}) == list(range(nsteps)), (algo, recs)
        want = cxx.allreduce(xs, algo, "f32", want_log=False).outputs
        assert all(same_bits(recvs[r].host(), want[r]) for r in range(N)), algo
