"""Many virtual ranks (up to VC_MAX_RANKS = 64) against the oracle.

Every collective and schedule at 24, 33, 63 and 64 ranks, ragged counts,
fp32 / bf16 / int32, non-zero roots: the long rings (126 steps at 64 ranks),
RHD with a 31-pair fold-in (63 ranks), deep heaps, Bruck with 6 rounds,
Pairwise with 64 rounds merged into launches of at most 128 operations.
Bit for bit against the C++ oracle's simulation of the same schedule, with
canary bands around every buffer.
"""
import pytest
import torch

import collective_communication_algorithms_virtual_gb300 as vc
from oracle import cxx
from synthetic_inputs import int32_bits, rank_buffers

from .gpu_util import Guarded, first_diff, same_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from collective_communication_algorithms_virtual_gb300 import build

    build.build()
    vc.lib()
    yield
    assert vc.vc_device_errors() == 0


def _inputs(dtype, seed, N, n):
    kind = {"f32": "uniform_f32", "bf16": "normal_bf16", "i32": "int32_bits"}[dtype]
    return rank_buffers(kind, seed, N, n)


def _check(outs, want, what):
    for r, (g, w) in enumerate(zip(outs, want)):
        got = g.host()
        assert same_bits(got, w), (what, r, first_diff(got, w))


@pytest.mark.parametrize("N", [24, 33, 63, 64])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
def test_allreduce_reduce_scatter_allgather(N, dtype):
    for count in (N * 8 + 5, 4099):
        xs = _inputs(dtype, 9700 + N + count, N, count)
        for algo in cxx.ALGOS["allreduce"]:
            want = cxx.allreduce(xs, algo, dtype, want_log=False).outputs
            sends = [Guarded(count, dtype, fill=x) for x in xs]
            recvs = [Guarded(count, dtype) for _ in range(N)]
            vc.vc_allreduce([g.t for g in sends], [g.t for g in recvs], algo=algo)
            torch.cuda.synchronize()
            assert all(g.guards_intact() for g in sends + recvs), algo
            _check(recvs, want, ("allreduce", algo, N, dtype, count))
    rc = 37
    xs = _inputs(dtype, 9800 + N, N, N * rc)
    for algo in cxx.ALGOS["reduce_scatter"]:
        want = cxx.reduce_scatter(xs, algo, dtype, want_log=False).outputs
        sends = [Guarded(N * rc, dtype, fill=x) for x in xs]
        recvs = [Guarded(rc, dtype) for _ in range(N)]
        vc.vc_reduce_scatter([g.t for g in sends], [g.t for g in recvs], algo=algo)
        torch.cuda.synchronize()
        _check(recvs, want, ("reduce_scatter", algo, N, dtype))
    ins = [x[:rc] for x in xs]
    for algo in cxx.ALGOS["allgather"]:
        want = cxx.allgather(ins, algo, dtype, want_log=False).outputs
        sends = [Guarded(rc, dtype, fill=x) for x in ins]
        recvs = [Guarded(N * rc, dtype) for _ in range(N)]
        vc.vc_allgather([g.t for g in sends], [g.t for g in recvs], algo=algo)
        torch.cuda.synchronize()
        _check(recvs, want, ("allgather", algo, N, dtype))


@pytest.mark.parametrize("N", [24, 33, 63, 64])
def test_rooted_collectives_and_alltoall(N):
    root = N // 3
    count = 3001
    A = int32_bits(9900, N, count)
    for algo in cxx.ALGOS["broadcast"] + cxx.ALGOS_EXTRA["broadcast"]:
        if algo.startswith("pipe_"):
            want = cxx.broadcast_pipelined(A, N, root, algo, "i32", 5, want_log=False).outputs
        else:
            want = cxx.broadcast(A, N, root, algo, "i32", want_log=False).outputs
        src = Guarded(count, "i32", fill=A)
        recvs = [Guarded(count, "i32") for _ in range(N)]
        if algo.startswith("pipe_"):
            vc.vc_broadcast_pipelined(src.t, [g.t for g in recvs], root=root, algo=algo, nchunks=5)
        else:
            vc.vc_broadcast(src.t, [g.t for g in recvs], root=root, algo=algo)
        torch.cuda.synchronize()
        _check(recvs, want, ("broadcast", algo, N))
    rc = 41
    A = int32_bits(9901, N, N * rc)
    for algo in cxx.ALGOS["scatter"]:
        want = cxx.scatter(A, N, root, algo, "i32", want_log=False).outputs
        src = Guarded(N * rc, "i32", fill=A)
        recvs = [Guarded(rc, "i32") for _ in range(N)]
        vc.vc_scatter(src.t, [g.t for g in recvs], root=root, algo=algo)
        torch.cuda.synchronize()
        _check(recvs, want, ("scatter", algo, N))
    xs = [int32_bits(9902, r, rc) for r in range(N)]
    for algo in cxx.ALGOS_EXTRA["gather"]:
        want = cxx.gather(xs, root, algo, "i32", want_log=False).outputs[0]
        sends = [Guarded(rc, "i32", fill=x) for x in xs]
        out = Guarded(N * rc, "i32")
        vc.vc_gather([g.t for g in sends], out.t, root=root, algo=algo)
        torch.cuda.synchronize()
        assert same_bits(out.host(), want), ("gather", algo, N)
    xf = rank_buffers("uniform_f32", 9903, N, 777)
    for algo in cxx.ALGOS_EXTRA["reduce"]:
        want = cxx.reduce(xf, root, algo, "f32", want_log=False).outputs[0]
        sends = [Guarded(777, "f32", fill=x) for x in xf]
        out = Guarded(777, "f32")
        vc.vc_reduce([g.t for g in sends], out.t, root=root, algo=algo)
        torch.cuda.synchronize()
        assert same_bits(out.host(), want), ("reduce", algo, N)
    B = 13
    xb = rank_buffers("normal_bf16", 9904, N, N * B)
    for algo in cxx.ALGOS["alltoall"]:
        want = cxx.alltoall(xb, algo, "bf16", want_log=False).outputs
        sends = [Guarded(N * B, "bf16", fill=x) for x in xb]
        recvs = [Guarded(N * B, "bf16") for _ in range(N)]
        vc.vc_alltoall([g.t for g in sends], [g.t for g in recvs], algo=algo)
        torch.cuda.synchronize()
        _check(recvs, want, ("alltoall", algo, N))
