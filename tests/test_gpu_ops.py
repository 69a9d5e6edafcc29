"""MAX / MIN and fp16 on the GPU against the oracle, bit for bit, for every
reducing collective and algorithm (Mesh AllReduce and Ring AllToAll are
covered with the other algorithms in test_gpu_parity.py)."""
import numpy as np
import pytest
import torch

import collective_communication_algorithms_virtual_gb300 as vc
from oracle import cxx
from synthetic_inputs import rank_buffers

from .gpu_util import Guarded, first_diff, same_bits, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from collective_communication_algorithms_virtual_gb300 import build

    build.build()
    vc.lib()


def _inputs(dtype, seed, N, n):
    if dtype == "f16":
        return [(x * 4).astype(np.float16) for x in rank_buffers("uniform_f32", seed, N, n)]
    kind = {"f32": "uniform_f32", "bf16": "normal_bf16", "i32": "int32_bits"}[dtype]
    return rank_buffers(kind, seed, N, n)


@pytest.mark.parametrize("op", ["sum", "max", "min"])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32", "f16"])
@pytest.mark.parametrize("N", [2, 3, 8])
def test_reductions_with_ops_match_oracle(N, dtype, op):
    for count in (13, 4099 * 2, 300007):
        xs = _inputs(dtype, 50 + N + count, N, count)
        for algo in cxx.ALGOS["allreduce"]:
            want = cxx.allreduce(xs, algo, dtype, op=op).outputs
            sends = [Guarded(count, dtype, fill=x) for x in xs]
            recvs = [Guarded(count, dtype) for _ in range(N)]
            vc.vc_allreduce([g.t for g in sends], [g.t for g in recvs], algo=algo, op=op)
            torch.cuda.synchronize()
            assert all(g.guards_intact() for g in sends + recvs)
            for r in range(N):
                got = recvs[r].host()
                assert same_bits(got, want[r]), ("ar", algo, op, dtype, N, count, r, first_diff(got, want[r]))
        rc = count // N + 1
        xr = _inputs(dtype, 60 + N + count, N, N * rc)
        for algo in cxx.ALGOS["reduce_scatter"]:
            want = cxx.reduce_scatter(xr, algo, dtype, op=op).outputs
            sends = [to_dev(x) for x in xr]
            recvs = [torch.empty(rc, dtype=sends[0].dtype, device="cuda") for _ in range(N)]
            vc.vc_reduce_scatter(sends, recvs, algo=algo, op=op)
            torch.cuda.synchronize()
            for r in range(N):
                assert same_bits(to_host(recvs[r]), want[r]), ("rs", algo, op, dtype, N, r)
        for algo in cxx.ALGOS_EXTRA["reduce"]:
            want = cxx.reduce(xs, N - 1, algo, dtype, op=op).outputs[0]
            sends = [to_dev(x) for x in xs]
            out = torch.empty_like(sends[0])
            vc.vc_reduce(sends, out, root=N - 1, algo=algo, op=op)
            torch.cuda.synchronize()
            assert same_bits(to_host(out), want), ("reduce", algo, op, dtype, N)


def test_max_min_nan_and_signed_zero_on_gpu():
    nan = float("nan")
    cases = [((nan, 1.0, nan, 2.0), 2.0, 1.0), ((-0.0, 0.0, 0.0, 0.0), -0.0, -0.0), ((0.0, -0.0, -0.0, -0.0), 0.0, 0.0)]
    for vals, mx, mn in cases:
        xs = [torch.full((9,), v, device="cuda") for v in vals]
        out = [torch.empty(9, device="cuda") for _ in range(4)]
        for op, want in (("max", mx), ("min", mn)):
            vc.vc_allreduce(xs, out, algo="fused", op=op)
            torch.cuda.synchronize()
            got = out[0].cpu().numpy().view(np.uint32)
            assert np.array_equal(got, np.full(9, want, dtype=np.float32).view(np.uint32)), (vals, op)


@pytest.mark.parametrize("N", [2, 5, 8])
def test_fp16_data_movement(N):
    rc = 4099
    xs = _inputs("f16", 70 + N, N, N * rc)
    for algo in cxx.ALGOS["alltoall"]:
        want = cxx.alltoall(xs, algo, "f16").outputs
        sends = [to_dev(x) for x in xs]
        recvs = [torch.empty_like(s) for s in sends]
        vc.vc_alltoall(sends, recvs, algo=algo)
        torch.cuda.synchronize()
        for j in range(N):
            assert same_bits(to_host(recvs[j]), want[j]), (algo, j)
    for algo in cxx.ALGOS["allgather"]:
        ins = [to_dev(x[:rc]) for x in xs]
        outs = [torch.empty(N * rc, dtype=torch.float16, device="cuda") for _ in range(N)]
        vc.vc_allgather(ins, outs, algo=algo)
        torch.cuda.synchronize()
        want = cxx.allgather([x[:rc] for x in xs], algo, "f16").outputs
        for r in range(N):
            assert same_bits(to_host(outs[r]), want[r])


@pytest.mark.parametrize("single", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_fp32_partials_at_offsets_that_are_16_but_not_32_byte_aligned(dtype, single):
    # 16-bit reductions keep fp32 partial sums in scratch.  With 100 or 1004
    # elements per rank a rank's scratch region starts 16 bytes past a
    # 32-byte boundary: the vector path takes it (16-byte aligned) and must
    # not use a 32-byte access there.  Checked in per-step and one-launch form.
    old = vc.vc_get_single_launch()
    vc.vc_set_single_launch(vc.SINGLE_LAUNCH_ALWAYS if single else 0)
    try:
        for N, rc in ((4, 100), (5, 1004), (8, 1004)):
            entries, _, _ = vc.vc_plan_describe("reduce_scatter", "ring", N, rc, dtype)
            f32 = [e for e in entries if e.dtype == 0]
            assert any(e.byte_off % 32 == 16 for e in f32), (N, rc)
            xr = _inputs(dtype, 70 + N + rc, N, N * rc)
            want = cxx.reduce_scatter(xr, "ring", dtype).outputs
            sends = [Guarded(N * rc, dtype, fill=x) for x in xr]
            recvs = [Guarded(rc, dtype) for _ in range(N)]
            vc.vc_reduce_scatter([g.t for g in sends], [g.t for g in recvs], algo="ring")
            torch.cuda.synchronize()
            assert all(g.guards_intact() for g in sends + recvs)
            for r in range(N):
                got = recvs[r].host()
                assert same_bits(got, want[r]), (dtype, single, N, rc, r, first_diff(got, want[r]))
    finally:
        vc.vc_set_single_launch(old)
