"""The bulk-copy (TMA) pipeline that runs aligned copy steps.

Copy launches whose operations are 16-byte aligned with no element tail, and
that write at least the set minimum, go through a pipeline of bulk loads into
shared memory (mbarrier completion) and bulk stores to every destination.
Checked here, with the minimum set to 0 so that small cases take it: those
launches take it (the launch trace names them), their results equal the
oracle bit for bit on copy-heavy collectives at sizes that give many tiles per
block and strided multi-run operations, the device error word stays clear, the
default minimum and the setting that turns it off keep small copies on the
register kernel, and a launch whose wait is made to run out (a load announced
but never issued) reports it and returns, leaving the context usable.
"""
import numpy as np
import pytest
import torch

import collective_communication_algorithms_virtual_gb300 as vc
from oracle import cxx
from synthetic_inputs import int32_bits, rank_buffers

from .gpu_util import Guarded, same_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from collective_communication_algorithms_virtual_gb300 import build

    build.build()
    vc.lib()
    old_sl = vc.vc_get_single_launch()
    old_cp = vc.vc_get_copy_pipeline()
    old_slice = vc.vc_get_slice_limit()
    vc.vc_set_single_launch(0)  # every step its own launch, so copy steps take the step kernels
    vc.vc_set_slice_limit(0)
    vc.vc_set_copy_pipeline(0)
    yield
    vc.vc_set_single_launch(old_sl)
    vc.vc_set_slice_limit(old_slice)
    vc.vc_set_copy_pipeline(old_cp)


def _traced(fn):
    vc.vc_trace_enable(True)
    try:
        fn()
        torch.cuda.synchronize()
        return vc.vc_trace_read()
    finally:
        vc.vc_trace_enable(False)


@pytest.mark.parametrize("N", [2, 3, 8])
def test_copy_heavy_collectives_take_the_pipeline_and_match(N):
    dtype = "bf16"
    for rc in (4096, 333 * 8, 1 << 18):  # aligned: whole 16-byte groups
        xs = rank_buffers("normal_bf16", 9100 + N + rc, N, N * rc)
        ins = [x[:rc] for x in xs]
        for algo in cxx.ALGOS["allgather"]:
            want = cxx.allgather(ins, algo, dtype).outputs
            sends = [Guarded(rc, dtype, fill=x) for x in ins]
            recvs = [Guarded(N * rc, dtype) for _ in range(N)]
            recs = _traced(lambda: vc.vc_allgather([g.t for g in sends], [g.t for g in recvs], algo=algo))
            assert all(g.guards_intact() for g in sends + recvs)
            for r in range(N):
                assert same_bits(recvs[r].host(), want[r]), ("ag", algo, N, rc, r)
            assert recs and all(r["kernel"].endswith("_tma") for r in recs), (algo, recs[:2])
        for algo in cxx.ALGOS["alltoall"]:
            want = cxx.alltoall(xs, algo, dtype).outputs
            sends = [Guarded(N * rc, dtype, fill=x) for x in xs]
            recvs = [Guarded(N * rc, dtype) for _ in range(N)]
            recs = _traced(lambda: vc.vc_alltoall([g.t for g in sends], [g.t for g in recvs], algo=algo))
            assert all(g.guards_intact() for g in sends + recvs)
            for r in range(N):
                assert same_bits(recvs[r].host(), want[r]), ("a2a", algo, N, rc, r)
            assert recs and all(r["kernel"].endswith("_tma") for r in recs), (algo, recs[:2])
    for count in (8192, 1 << 20):
        A = int32_bits(9200, N, count)
        for algo in cxx.ALGOS["broadcast"] + ("pipe_chain", "pipe_tree"):
            if algo.startswith("pipe"):
                want = cxx.broadcast_pipelined(A, N, 0, algo, "i32", 4).outputs
            else:
                want = cxx.broadcast(A, N, 0, algo, "i32").outputs
            src = Guarded(count, "i32", fill=A)
            recvs = [Guarded(count, "i32") for _ in range(N)]
            if algo.startswith("pipe"):
                vc.vc_broadcast_pipelined(src.t, [g.t for g in recvs], root=0, algo=algo, nchunks=4)
            else:
                vc.vc_broadcast(src.t, [g.t for g in recvs], root=0, algo=algo)
            torch.cuda.synchronize()
            assert src.guards_intact() and all(g.guards_intact() for g in recvs)
            for r in range(N):
                assert same_bits(recvs[r].host(), want[r]), ("bcast", algo, N, count, r)
    assert vc.vc_device_errors() == 0


def test_unaligned_copies_take_the_register_kernel():
    N, rc = 4, 1001  # 1001 bf16 per block: blocks are not whole 16-byte groups
    xs = rank_buffers("normal_bf16", 9300, N, N * rc)
    want = cxx.alltoall(xs, "pairwise", "bf16").outputs
    sends = [Guarded(N * rc, "bf16", fill=x) for x in xs]
    recvs = [Guarded(N * rc, "bf16") for _ in range(N)]
    recs = _traced(lambda: vc.vc_alltoall([g.t for g in sends], [g.t for g in recvs], algo="pairwise"))
    assert recs and not any(r["kernel"].endswith("_tma") for r in recs), recs[:2]
    for r in range(N):
        assert same_bits(recvs[r].host(), want[r]), r


def test_the_minimum_size_and_the_off_switch_keep_small_copies_on_the_register_kernel():
    N, rc = 4, 1 << 16  # aligned: the pipeline would take it at minimum 0
    xs = rank_buffers("normal_bf16", 9400, N, N * rc)
    want = cxx.alltoall(xs, "pairwise", "bf16").outputs
    try:
        for setting in (vc.COPY_PIPELINE_NEVER, 128 << 20, 0):
            vc.vc_set_copy_pipeline(setting)
            assert vc.vc_get_copy_pipeline() == setting
            sends = [Guarded(N * rc, "bf16", fill=x) for x in xs]
            recvs = [Guarded(N * rc, "bf16") for _ in range(N)]
            recs = _traced(lambda: vc.vc_alltoall([g.t for g in sends], [g.t for g in recvs], algo="pairwise"))
            assert recs and all(r["kernel"].endswith("_tma") == (setting == 0) for r in recs), (setting, recs[:2])
            for r in range(N):
                assert same_bits(recvs[r].host(), want[r]), (setting, r)
    finally:
        vc.vc_set_copy_pipeline(0)


def test_calls_with_16_bit_reductions_keep_their_copies_on_the_register_kernel():
    N, count = 4, 1 << 16
    for dtype, pipelined in (("bf16", False), ("f16", False), ("f32", True)):
        xs = rank_buffers({"bf16": "normal_bf16", "f16": "uniform_f32", "f32": "uniform_f32"}[dtype], 9500, N, count)
        if dtype == "f16":
            xs = [x.astype(np.float16) for x in xs]
        want = cxx.allreduce(xs, "ring", dtype).outputs
        sends = [Guarded(count, dtype, fill=x) for x in xs]
        recvs = [Guarded(count, dtype) for _ in range(N)]
        recs = _traced(lambda: vc.vc_allreduce([g.t for g in sends], [g.t for g in recvs], algo="ring"))
        copies = [r for r in recs if r["kernel"].startswith("copy")]
        assert copies and all(r["kernel"].endswith("_tma") == pipelined for r in copies), (dtype, copies[:2])
        for r in range(N):
            assert same_bits(recvs[r].host(), want[r]), (dtype, r)


def test_a_copy_wait_that_runs_out_is_reported_and_the_launch_returns():
    assert vc.vc_copy_selftest() == 2
    assert vc.vc_device_errors() == 0  # the self-test clears the word it used
    x = [torch.arange(4096, dtype=torch.int32, device="cuda") for _ in range(3)]
    y = [torch.empty(3 * 4096, dtype=torch.int32, device="cuda") for _ in range(3)]
    vc.vc_allgather(x, y, algo="ring")
    torch.cuda.synchronize()
    assert torch.equal(y[1], torch.arange(4096, dtype=torch.int32, device="cuda").repeat(3))
    assert vc.vc_device_errors() == 0
