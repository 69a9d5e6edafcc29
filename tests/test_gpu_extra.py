"""Pipelined Broadcasts, Gather and Tree Reduce on the GPU against the oracle
(bit for bit; canary bands around every buffer)."""
import pytest
import torch

import collective_communication_algorithms_virtual_gb300 as vc
from oracle import cxx
from synthetic_inputs import int32_bits, rank_buffers

from .gpu_util import Guarded, first_diff, same_bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from collective_communication_algorithms_virtual_gb300 import build

    build.build()
    vc.lib()


@pytest.mark.parametrize("N", [1, 2, 3, 5, 8, 16])
def test_pipelined_broadcast_matches_oracle(N):
    for root in sorted({0, N - 1}):
        for count in (1, 4099, 300001):
            A = int32_bits(10 + root, N, count)
            for algo in ("pipe_chain", "pipe_tree"):
                for k in (1, 4, 13):
                    for inplace in (False, True):
                        want = cxx.broadcast_pipelined(A, N, root, algo, "i32", k, inplace=inplace).outputs
                        recvs = [Guarded(count, "i32") for _ in range(N)]
                        if inplace:
                            recvs[root].t.copy_(to_dev(A))
                            src = recvs[root].t
                        else:
                            sg = Guarded(count, "i32", fill=A)
                            src = sg.t
                        vc.vc_broadcast_pipelined(src, [g.t for g in recvs], root=root, algo=algo, nchunks=k)
                        torch.cuda.synchronize()
                        assert all(g.guards_intact() for g in recvs)
                        for r in range(N):
                            assert same_bits(recvs[r].host(), want[r]), (algo, N, root, count, k, inplace, r)
    # nchunks = 0 takes the cost model's k; the result is the same Broadcast
    A = int32_bits(3, 0, 1 << 20)
    recvs = [torch.empty(1 << 20, dtype=torch.int32, device="cuda") for _ in range(N)]
    src = to_dev(A)
    for algo in ("pipe_chain", "pipe_tree"):
        vc.vc_broadcast_pipelined(src, recvs, root=0, algo=algo)
        torch.cuda.synchronize()
        assert all(torch.equal(r, src) for r in recvs)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
@pytest.mark.parametrize("N", [1, 2, 3, 5, 8, 16])
def test_gather_reduce_match_oracle(N, dtype):
    kind = {"f32": "uniform_f32", "bf16": "normal_bf16", "i32": "int32_bits"}[dtype]
    for root in sorted({0, N - 1, N // 2}):
        for rc in (1, 5, 4096, 70001):
            xs = rank_buffers(kind, 20 + root + rc, N, rc)
            for algo in cxx.ALGOS_EXTRA["gather"]:
                want = cxx.gather(xs, root, algo, dtype).outputs[0]
                sends = [Guarded(rc, dtype, fill=x) for x in xs]
                out = Guarded(N * rc, dtype)
                vc.vc_gather([g.t for g in sends], out.t, root=root, algo=algo)
                torch.cuda.synchronize()
                assert out.guards_intact() and all(g.guards_intact() for g in sends)
                assert same_bits(out.host(), want), ("gather", algo, N, root, rc)
            for algo in cxx.ALGOS_EXTRA["reduce"]:
                for inplace in (False, True):
                    want = cxx.reduce(xs, root, algo, dtype, inplace=inplace).outputs[0]
                    sends = [Guarded(rc, dtype, fill=x) for x in xs]
                    out = sends[root] if inplace else Guarded(rc, dtype)
                    vc.vc_reduce([g.t for g in sends], out.t, root=root, algo=algo)
                    torch.cuda.synchronize()
                    assert out.guards_intact() and all(g.guards_intact() for g in sends)
                    got = out.host()
                    assert same_bits(got, want), ("reduce", algo, N, root, rc, inplace, first_diff(got, want))


def test_reduce_witness_on_gpu():
    """Balanced tree from the root: x = (0, 2^24, 1, -2^24) gives 1 at root 0
    and 0 at root 1; the rank-order fold gives 0."""
    xs = [torch.full((8,), v, device="cuda") for v in (0.0, 2.0 ** 24, 1.0, -(2.0 ** 24))]
    out = torch.empty(8, device="cuda")
    for root, algo, want in ((0, "binomial", 1.0), (1, "binomial", 0.0), (0, "fused", 0.0)):
        vc.vc_reduce(xs, out, root=root, algo=algo)
        torch.cuda.synchronize()
        assert bool((out == want).all()), (root, algo, out)
