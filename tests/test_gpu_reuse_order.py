"""The L2 reuse order (vc_set_reuse_order) forced onto small calls.

By default only steps after one writing at least 16 MiB are reordered (the
step walked backwards, its operations listed by when their inputs were
written, results the next step reads stored with the default L2 policy), so
the randomised sweep's small calls never reach it.  Here the minimum is 0:
every schedule of every collective, at sizes with ragged tails and many
tiles, in per-step launches (with and without the bulk-copy pipeline) and in
one launch, must equal the oracle bit for bit with the canary bands intact.
"""
import numpy as np
import pytest
import torch

import collective_communication_algorithms_virtual_gb300 as vc
from oracle import cxx
from synthetic_inputs import int32_bits, rank_buffers

from .gpu_util import Guarded, first_diff, same_bits

pytestmark = pytest.mark.gpu
ALWAYS = vc.SINGLE_LAUNCH_ALWAYS


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from collective_communication_algorithms_virtual_gb300 import build

    build.build()
    vc.lib()
    saved = (vc.vc_get_reuse_order(), vc.vc_get_single_launch(), vc.vc_get_copy_pipeline(), vc.vc_get_slice_limit())
    vc.vc_set_reuse_order(0)
    vc.vc_set_slice_limit(0)  # the per-step and cluster forms are the ones ordered for reuse
    yield
    vc.vc_set_reuse_order(saved[0])
    vc.vc_set_single_launch(saved[1])
    vc.vc_set_copy_pipeline(saved[2])
    vc.vc_set_slice_limit(saved[3])
    assert vc.vc_device_errors() == 0


FORMS = {"per_step": (0, vc.COPY_PIPELINE_NEVER), "per_step_pipeline": (0, 0), "single": (ALWAYS, vc.COPY_PIPELINE_NEVER)}


def _inputs(dtype, seed, N, n):
    if dtype == "f16":
        return [(x * 4).astype(np.float16) for x in rank_buffers("uniform_f32", seed, N, n)]
    return rank_buffers({"f32": "uniform_f32", "bf16": "normal_bf16", "i32": "int32_bits"}[dtype], seed, N, n)


@pytest.mark.parametrize("form", list(FORMS))
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [3, 8])
def test_reduction_schedules_with_the_reuse_order(N, dtype, form):
    vc.vc_set_single_launch(FORMS[form][0])
    vc.vc_set_copy_pipeline(FORMS[form][1])
    assert vc.vc_get_reuse_order() == 0
    for count in (1000, 65536 + 40):
        xs = _inputs(dtype, 9600 + N + count, N, count)
        for algo in cxx.ALGOS["allreduce"]:
            want = cxx.allreduce(xs, algo, dtype).outputs
            sends = [Guarded(count, dtype, fill=x) for x in xs]
            recvs = [Guarded(count, dtype) for _ in range(N)]
            vc.vc_allreduce([g.t for g in sends], [g.t for g in recvs], algo=algo)
            torch.cuda.synchronize()
            assert all(g.guards_intact() for g in sends + recvs)
            for r in range(N):
                got = recvs[r].host()
                assert same_bits(got, want[r]), ("ar", algo, N, count, dtype, form, r, first_diff(got, want[r]))
        rc = count // N + 1
        xr = _inputs(dtype, 9700 + N + count, N, N * rc)
        for algo in cxx.ALGOS["reduce_scatter"]:
            want = cxx.reduce_scatter(xr, algo, dtype).outputs
            sends = [Guarded(N * rc, dtype, fill=x) for x in xr]
            recvs = [Guarded(rc, dtype) for _ in range(N)]
            vc.vc_reduce_scatter([g.t for g in sends], [g.t for g in recvs], algo=algo)
            torch.cuda.synchronize()
            assert all(g.guards_intact() for g in sends + recvs)
            for r in range(N):
                assert same_bits(recvs[r].host(), want[r]), ("rs", algo, N, rc, dtype, form, r)


@pytest.mark.parametrize("form", list(FORMS))
@pytest.mark.parametrize("N", [5, 8])
def test_data_movement_schedules_with_the_reuse_order(N, form):
    vc.vc_set_single_launch(FORMS[form][0])
    vc.vc_set_copy_pipeline(FORMS[form][1])
    dtype = "bf16"
    for rc in (1024, 20000):  # whole 16-byte groups (the pipeline) and many tiles
        xs = _inputs(dtype, 9800 + N + rc, N, N * rc)
        ins = [x[:rc] for x in xs]
        for algo in cxx.ALGOS["allgather"]:
            want = cxx.allgather(ins, algo, dtype).outputs
            sends = [Guarded(rc, dtype, fill=x) for x in ins]
            recvs = [Guarded(N * rc, dtype) for _ in range(N)]
            vc.vc_allgather([g.t for g in sends], [g.t for g in recvs], algo=algo)
            torch.cuda.synchronize()
            assert all(g.guards_intact() for g in sends + recvs)
            for r in range(N):
                assert same_bits(recvs[r].host(), want[r]), ("ag", algo, N, rc, form, r)
        for algo in cxx.ALGOS["alltoall"]:
            want = cxx.alltoall(xs, algo, dtype).outputs
            sends = [Guarded(N * rc, dtype, fill=x) for x in xs]
            recvs = [Guarded(N * rc, dtype) for _ in range(N)]
            vc.vc_alltoall([g.t for g in sends], [g.t for g in recvs], algo=algo)
            torch.cuda.synchronize()
            assert all(g.guards_intact() for g in sends + recvs)
            for r in range(N):
                assert same_bits(recvs[r].host(), want[r]), ("a2a", algo, N, rc, form, r)
    count = 30000
    A = int32_bits(9900 + N, N, count)
    for algo in cxx.ALGOS["broadcast"]:
        want = cxx.broadcast(A, N, 1, algo, "i32").outputs
        src = Guarded(count, "i32", fill=A)
        recvs = [Guarded(count, "i32") for _ in range(N)]
        vc.vc_broadcast(src.t, [g.t for g in recvs], root=1, algo=algo)
        torch.cuda.synchronize()
        assert src.guards_intact() and all(g.guards_intact() for g in recvs)
        for r in range(N):
            assert same_bits(recvs[r].host(), want[r]), ("bcast", algo, N, form, r)


def test_setting_round_trips_and_clears_the_plan_cache():
    for v in (vc.REUSE_ORDER_NEVER, 16 << 20, 0):
        vc.vc_set_reuse_order(v)
        assert vc.vc_get_reuse_order() == v
