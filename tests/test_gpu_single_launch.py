"""Single-launch execution against the oracle and against per-step launches.

A schedule whose steps are small enough runs all of them in one launch of one
thread-block cluster, with a cluster barrier between consecutive steps
(vc_set_single_launch).  Every collective, algorithm, data type and op runs
here with it forced on and switched off; both must equal the oracle's
simulation of the same schedule bit for bit, the launch trace must show one
launch for the whole call (step -1) or one per step, and canary bands around
every buffer catch stray writes.  Also covered: in place, unaligned pointers
and a description too large for the kernel (both fall back to per-step
launches), the default size limit, and capture into a CUDA graph.
"""
import numpy as np
import pytest
import torch

import collective_communication_algorithms_virtual_gb300 as vc
from oracle import cxx
from synthetic_inputs import int32_bits, rank_buffers

from .gpu_util import Guarded, first_diff, same_bits, to_dev

pytestmark = pytest.mark.gpu
ALWAYS = vc.SINGLE_LAUNCH_ALWAYS


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from collective_communication_algorithms_virtual_gb300 import build

    build.build()
    vc.lib()
    yield


@pytest.fixture(autouse=True)
def _restore_limit():
    old, old_slice, old_merge = vc.vc_get_single_launch(), vc.vc_get_slice_limit(), vc.vc_get_merge_steps()
    # the cluster form is the one under test here: not the sliced form (test_gpu_sliced.py), and not
    # the one launch that a plan whose steps all merge takes instead (test_gpu_merge_steps.py)
    vc.vc_set_slice_limit(0)
    vc.vc_set_merge_steps(False)
    yield
    vc.vc_set_single_launch(old)
    vc.vc_set_slice_limit(old_slice)
    vc.vc_set_merge_steps(old_merge)


def _inputs(dtype, seed, N, n):
    if dtype == "f16":
        return [(x * 4).astype(np.float16) for x in rank_buffers("uniform_f32", seed, N, n)]
    kind = {"f32": "uniform_f32", "bf16": "normal_bf16", "i32": "int32_bits"}[dtype]
    return rank_buffers(kind, seed, N, n)


def _traced(fn):
    vc.vc_trace_enable(True)
    try:
        fn()
        torch.cuda.synchronize()
        return vc.vc_trace_read()
    finally:
        vc.vc_trace_enable(False)


def _check_launches(recs, limit, nsteps, what):
    if limit == ALWAYS and nsteps >= 2:
        assert len(recs) == 1 and recs[0]["step"] == -1 and recs[0]["kernel"].endswith("_single_launch"), (what, recs)
    else:
        assert recs and all(r["step"] >= 0 for r in recs), (what, recs)


def _nsteps(coll, algo, N, count, dtype="f32", root=0, nchunks=0, op="sum"):
    return vc.vc_plan_describe(coll, algo, N, count, dtype, root, nchunks=nchunks, op=op)[2]


@pytest.mark.parametrize("op", ["sum", "max"])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32", "f16"])
@pytest.mark.parametrize("N", [2, 3, 5, 8, 16])
def test_allreduce_single_launch(N, dtype, op):
    for count in (1, 13, 4096 + 5, 65536 + 37):
        xs = _inputs(dtype, 7000 + N + count, N, count)
        for algo in cxx.ALGOS["allreduce"]:
            want = cxx.allreduce(xs, algo, dtype, op=op).outputs
            nsteps = _nsteps("allreduce", algo, N, count, dtype, op=op)
            for limit in (ALWAYS, 0):
                vc.vc_set_single_launch(limit)
                sends = [Guarded(count, dtype, fill=x) for x in xs]
                recvs = [Guarded(count, dtype) for _ in range(N)]
                recs = _traced(lambda: vc.vc_allreduce([g.t for g in sends], [g.t for g in recvs], algo=algo, op=op))
                assert all(g.guards_intact() for g in sends + recvs)
                for r in range(N):
                    got = recvs[r].host()
                    assert same_bits(got, want[r]), (algo, N, count, dtype, op, limit, r, first_diff(got, want[r]))
                _check_launches(recs, limit, nsteps, (algo, N, count))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [3, 8])
def test_allreduce_in_place_single_launch(N, dtype):
    vc.vc_set_single_launch(ALWAYS)
    for count in (7, 4096 + 5, 30001):
        xs = _inputs(dtype, 7100 + N + count, N, count)
        for algo in cxx.ALGOS["allreduce"]:
            want = cxx.allreduce(xs, algo, dtype).outputs
            bufs = [Guarded(count, dtype, fill=x) for x in xs]
            recs = _traced(lambda: vc.vc_allreduce([g.t for g in bufs], [g.t for g in bufs], algo=algo))
            assert all(g.guards_intact() for g in bufs)
            for r in range(N):
                assert same_bits(bufs[r].host(), want[r]), (algo, N, count, r)
            _check_launches(recs, ALWAYS, _nsteps("allreduce", algo, N, count, dtype), (algo, N, count))


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
@pytest.mark.parametrize("N", [2, 5, 8])
def test_reduce_scatter_allgather_alltoall_single_launch(N, dtype):
    for limit in (ALWAYS, 0):
        vc.vc_set_single_launch(limit)
        for rc in (1, 3, 1024 + 3, 20001):
            xs = _inputs(dtype, 7200 + N + rc, N, N * rc)
            for algo in cxx.ALGOS["reduce_scatter"]:
                want = cxx.reduce_scatter(xs, algo, dtype).outputs
                sends = [Guarded(N * rc, dtype, fill=x) for x in xs]
                recvs = [Guarded(rc, dtype) for _ in range(N)]
                recs = _traced(lambda: vc.vc_reduce_scatter([g.t for g in sends], [g.t for g in recvs], algo=algo))
                assert all(g.guards_intact() for g in sends + recvs)
                for r in range(N):
                    assert same_bits(recvs[r].host(), want[r]), ("rs", algo, N, rc, limit, r)
                _check_launches(recs, limit, _nsteps("reduce_scatter", algo, N, rc, dtype), ("rs", algo))
            ins = [x[:rc] for x in xs]
            for algo in cxx.ALGOS["allgather"]:
                want = cxx.allgather(ins, algo, dtype).outputs
                sends = [Guarded(rc, dtype, fill=x) for x in ins]
                recvs = [Guarded(N * rc, dtype) for _ in range(N)]
                recs = _traced(lambda: vc.vc_allgather([g.t for g in sends], [g.t for g in recvs], algo=algo))
                assert all(g.guards_intact() for g in sends + recvs)
                for r in range(N):
                    assert same_bits(recvs[r].host(), want[r]), ("ag", algo, N, rc, limit, r)
                _check_launches(recs, limit, _nsteps("allgather", algo, N, rc, dtype), ("ag", algo))
            for algo in cxx.ALGOS["alltoall"]:
                want = cxx.alltoall(xs, algo, dtype).outputs
                sends = [Guarded(N * rc, dtype, fill=x) for x in xs]
                recvs = [Guarded(N * rc, dtype) for _ in range(N)]
                recs = _traced(lambda: vc.vc_alltoall([g.t for g in sends], [g.t for g in recvs], algo=algo))
                assert all(g.guards_intact() for g in sends + recvs)
                for r in range(N):
                    assert same_bits(recvs[r].host(), want[r]), ("a2a", algo, N, rc, limit, r)
                # AllToAll runs per step whatever the limit (faster than one cluster)
                _check_launches(recs, 0, _nsteps("alltoall", algo, N, rc, dtype), ("a2a", algo))


@pytest.mark.parametrize("N", [2, 3, 8, 16])
def test_rooted_collectives_single_launch(N):
    dtype = "i32"
    for limit in (ALWAYS, 0):
        vc.vc_set_single_launch(limit)
        for root in sorted({0, N - 1}):
            for count in (1, 7, 4096 + 5, 30001):
                A = int32_bits(7300 + root, N, count)
                for algo in cxx.ALGOS["broadcast"]:
                    for inplace in (False, True):
                        want = cxx.broadcast(A, N, root, algo, dtype, inplace=inplace).outputs
                        recvs = [Guarded(count, dtype) for _ in range(N)]
                        if inplace:
                            recvs[root].t.copy_(to_dev(A))
                            src = recvs[root].t
                        else:
                            src = Guarded(count, dtype, fill=A).t
                        recs = _traced(lambda: vc.vc_broadcast(src, [g.t for g in recvs], root=root, algo=algo))
                        assert all(g.guards_intact() for g in recvs)
                        for r in range(N):
                            assert same_bits(recvs[r].host(), want[r]), ("bcast", algo, N, root, count, inplace, r)
                        _check_launches(recs, limit, _nsteps("broadcast", algo, N, count, dtype, root), ("bcast", algo))
                for algo in ("pipe_chain", "pipe_tree"):
                    want = cxx.broadcast_pipelined(A, N, root, algo, dtype, 3).outputs
                    recvs = [Guarded(count, dtype) for _ in range(N)]
                    src = Guarded(count, dtype, fill=A).t
                    recs = _traced(lambda: vc.vc_broadcast_pipelined(src, [g.t for g in recvs], root=root,
                                                                     algo=algo, nchunks=3))
                    assert all(g.guards_intact() for g in recvs)
                    for r in range(N):
                        assert same_bits(recvs[r].host(), want[r]), (algo, N, root, count, r)
                    _check_launches(recs, limit, _nsteps("broadcast", algo, N, count, dtype, root, nchunks=3), algo)
                S = int32_bits(7400 + root, N, N * count)
                for algo in cxx.ALGOS["scatter"]:
                    want = cxx.scatter(S, N, root, algo, dtype).outputs
                    src_g = Guarded(N * count, dtype, fill=S)
                    recvs = [Guarded(count, dtype) for _ in range(N)]
                    recs = _traced(lambda: vc.vc_scatter(src_g.t, [g.t for g in recvs], root=root, algo=algo))
                    assert src_g.guards_intact() and all(g.guards_intact() for g in recvs)
                    for r in range(N):
                        assert same_bits(recvs[r].host(), want[r]), ("scatter", algo, N, root, count, r)
                    _check_launches(recs, limit, _nsteps("scatter", algo, N, count, dtype, root), ("scatter", algo))
                xs = _inputs("f32", 7500 + root + count, N, count)
                for algo in cxx.ALGOS_EXTRA["gather"]:
                    want = cxx.gather(xs, root, algo, "f32").outputs[0]
                    sends = [Guarded(count, "f32", fill=x) for x in xs]
                    out = Guarded(N * count, "f32")
                    recs = _traced(lambda: vc.vc_gather([g.t for g in sends], out.t, root=root, algo=algo))
                    assert out.guards_intact() and same_bits(out.host(), want), ("gather", algo, N, root, count)
                    _check_launches(recs, limit, _nsteps("gather", algo, N, count, "f32", root), ("gather", algo))
                for algo in cxx.ALGOS_EXTRA["reduce"]:
                    for op in ("sum", "min"):
                        want = cxx.reduce(xs, root, algo, "f32", op=op).outputs[0]
                        sends = [Guarded(count, "f32", fill=x) for x in xs]
                        out = Guarded(count, "f32")
                        recs = _traced(lambda: vc.vc_reduce([g.t for g in sends], out.t, root=root, algo=algo, op=op))
                        assert out.guards_intact() and same_bits(out.host(), want), ("reduce", algo, op, N, root, count)
                        _check_launches(recs, limit, _nsteps("reduce", algo, N, count, "f32", root, op=op),
                                        ("reduce", algo))


def test_unaligned_pointers_fall_back_to_per_step_launches():
    vc.vc_set_single_launch(ALWAYS)
    N, count = 4, 4096 + 3
    xs = _inputs("f32", 7600, N, count)
    for algo in ("ring", "rhd", "dbt"):
        want = cxx.allreduce(xs, algo, "f32").outputs
        sends = [Guarded(count, "f32", shift=1, fill=x) for x in xs]
        recvs = [Guarded(count, "f32", shift=1) for _ in range(N)]
        recs = _traced(lambda: vc.vc_allreduce([g.t for g in sends], [g.t for g in recvs], algo=algo))
        assert all(r["step"] >= 0 for r in recs)
        for r in range(N):
            assert same_bits(recvs[r].host(), want[r]), (algo, r)


def test_description_too_large_falls_back_to_per_step_launches():
    # 64 ranks: the ring AllReduce has 126 steps of 64 operations
    vc.vc_set_single_launch(ALWAYS)
    N, count = 64, 640
    xs = _inputs("f32", 7700, N, count)
    want = cxx.allreduce(xs, "ring", "f32").outputs
    sends = [Guarded(count, "f32", fill=x) for x in xs]
    recvs = [Guarded(count, "f32") for _ in range(N)]
    recs = _traced(lambda: vc.vc_allreduce([g.t for g in sends], [g.t for g in recvs], algo="ring"))
    assert len(recs) == 126 and all(r["step"] >= 0 for r in recs)
    for r in range(N):
        assert same_bits(recvs[r].host(), want[r]), r


def test_default_limit_splits_small_and_large_calls():
    vc.vc_set_single_launch(vc.vc_get_single_launch())  # the default, restored by the fixture
    assert vc.vc_get_single_launch() == 768 << 10
    N = 8
    for count, single in ((16384, True), (1 << 18, False)):
        x = [torch.rand(count, device="cuda") for _ in range(N)]
        y = [torch.empty(count, device="cuda") for _ in range(N)]
        recs = _traced(lambda: vc.vc_allreduce(x, y, algo="ring"))
        assert (len(recs) == 1 and recs[0]["step"] == -1) == single, (count, recs)
        want = torch.stack(x).sum(0)
        assert torch.allclose(y[3], want, rtol=1e-5, atol=1e-5)


def test_single_launch_inside_a_cuda_graph():
    vc.vc_set_single_launch(ALWAYS)
    N, count = 8, 4096 + 5
    sends = [torch.empty(count, device="cuda") for _ in range(N)]
    recvs = [torch.empty(count, device="cuda") for _ in range(N)]
    fresh = [torch.empty(count + 16, device="cuda") for _ in range(N)]
    fresh_out = [torch.empty(count + 16, device="cuda") for _ in range(N)]
    vc.vc_allreduce(sends, recvs, algo="dbt")  # resident before capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        vc.vc_allreduce(sends, recvs, algo="dbt")
        vc.vc_allreduce(fresh, fresh_out, algo="rhd")  # a shape first seen under capture: per-step launches
    for seed in (1, 2):
        xs = _inputs("f32", 7800 + seed, N, count)
        ys = _inputs("f32", 7900 + seed, N, count + 16)
        for r in range(N):
            sends[r].copy_(to_dev(xs[r]))
            fresh[r].copy_(to_dev(ys[r]))
        g.replay()
        torch.cuda.synchronize()
        want = cxx.allreduce(xs, "dbt", "f32").outputs
        want2 = cxx.allreduce(ys, "rhd", "f32").outputs
        for r in range(N):
            assert same_bits(recvs[r].cpu().numpy(), want[r]), (seed, r)
            assert same_bits(fresh_out[r].cpu().numpy(), want2[r]), (seed, r)
