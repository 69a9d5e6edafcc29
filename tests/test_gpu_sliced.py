"""The sliced form of the AllReduce, ReduceScatter, AllGather, Broadcast,
Scatter, Gather and Reduce schedules, against the oracle.

In the sliced form (vc_set_slice_limit) one launch over the whole GPU runs
every step of the plan, each thread carrying its 16-byte group of every rank
buffer (and, for bf16 / fp16, of the fp32 partial sums in scratch) through
the steps in order.  Forced on for every eligible call here: Ring, RHD (any
rank count, with the fold-in), DBT, Mesh and the per-hop ring on fp32, int32,
bf16 and fp16 with every op, ragged counts whose last group is partial,
sizes from one element to 64 MiB per rank, in place.  Every result must equal
the C++ oracle's simulation of the same schedule bit for bit, and the launch
trace must show one sliced launch for the call.  Also: calls that do not
qualify (an 8-rank 16-bit Ring whose fp32 partial sums take more than 16
MiB per rank and alternate between two chunk slots, unaligned pointers,
single-step plans, the AllToAlls) take the other forms and stay exact; the
default size limit; a sliced call captured in a CUDA graph; canary bands
around every buffer.
"""
import numpy as np
import pytest
import torch

import collective_communication_algorithms_virtual_gb300 as vc
from oracle import cxx
from synthetic_inputs import rank_buffers

from .gpu_util import Guarded, first_diff, same_bits, to_dev, to_host

pytestmark = pytest.mark.gpu
SLICED_ALGOS = ("ring", "rhd", "dbt", "mesh", "ring_hop")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from collective_communication_algorithms_virtual_gb300 import build

    build.build()
    vc.lib()
    old = vc.vc_get_slice_limit()
    yield
    vc.vc_set_slice_limit(old)
    assert vc.vc_device_errors() == 0


def _inputs(dtype, seed, N, n):
    if dtype == "f16":
        return [x.astype(np.float16) for x in rank_buffers("normal_f32", seed, N, n)]
    return rank_buffers({"f32": "uniform_f32", "i32": "int32_bits", "bf16": "normal_bf16"}[dtype], seed, N, n)


def _traced(fn):
    vc.vc_trace_enable(True)
    try:
        fn()
        torch.cuda.synchronize()
        return vc.vc_trace_read()
    finally:
        vc.vc_trace_enable(False)


def _run(xs, algo, dtype, op="sum", shift=0, inplace=False):
    N, count = len(xs), len(xs[0])
    sends = [Guarded(count, dtype, shift, fill=x) for x in xs]
    recvs = sends if inplace else [Guarded(count, dtype, shift) for _ in range(N)]
    recs = _traced(lambda: vc.vc_allreduce([g.t for g in sends], [g.t for g in recvs], algo=algo, op=op))
    assert all(g.guards_intact() for g in sends + recvs)
    return [g.host() for g in recvs], recs


@pytest.mark.parametrize("op", ["sum", "max", "min"])
@pytest.mark.parametrize("dtype", ["f32", "i32"])
@pytest.mark.parametrize("N", [2, 3, 4, 5, 7, 8, 9, 16])
def test_sliced_allreduce_matches_oracle(N, dtype, op):
    vc.vc_set_slice_limit(vc.SLICE_ALWAYS)
    for count in (1, 3, 4, 13, 1023, 4096 + 5, 65536 + 37) + ((300_001,) if op == "sum" else ()):
        xs = _inputs(dtype, 8100 + N + count, N, count)
        for algo in SLICED_ALGOS:
            want = cxx.allreduce(xs, algo, dtype, op=op, want_log=False).outputs
            got, recs = _run(xs, algo, dtype, op)
            assert len(recs) == 1 and recs[0]["kernel"].endswith("_sliced"), (algo, N, count, recs)
            for r in range(N):
                assert same_bits(got[r], want[r]), (algo, N, dtype, op, count, r, first_diff(got[r], want[r]))


@pytest.mark.parametrize("op", ["sum", "max", "min"])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("N", [2, 3, 5, 8, 16])
def test_sliced_16bit_allreduce_matches_oracle(N, dtype, op):
    """bf16 / fp16: fp32 partial sums in scratch, rounded once into the
    receive buffers; every launch shape (1, 2 and 4 groups a thread)."""
    vc.vc_set_slice_limit(vc.SLICE_ALWAYS)
    counts = (1, 7, 8, 13, 1023, 4096 + 5, 65536 + 37) + ((300_001, 1_500_003) if op == "sum" else ())
    for count in counts:
        xs = _inputs(dtype, 8700 + N + count, N, count)
        for algo in SLICED_ALGOS:
            want = cxx.allreduce(xs, algo, dtype, op=op, want_log=False).outputs
            got, recs = _run(xs, algo, dtype, op)
            assert len(recs) == 1 and recs[0]["kernel"].endswith("_sliced"), (algo, N, count, recs)
            for r in range(N):
                assert same_bits(got[r], want[r]), (algo, N, dtype, op, count, r, first_diff(got[r], want[r]))


@pytest.mark.parametrize("N", [4, 8])
def test_sliced_in_place(N):
    vc.vc_set_slice_limit(vc.SLICE_ALWAYS)
    for count in (777, 100_000):
        for dtype in ("f32", "bf16"):
            xs = _inputs(dtype, 8200 + N + count, N, count)
            for algo in SLICED_ALGOS:
                want = cxx.allreduce(xs, algo, dtype, want_log=False).outputs
                got, recs = _run(xs, algo, dtype, inplace=True)
                assert recs[0]["kernel"].endswith("_sliced"), (algo, recs)
                for r in range(N):
                    assert same_bits(got[r], want[r]), (algo, N, dtype, count, r)


def test_sliced_large_messages():
    """64 MiB per rank, 8 ranks: every element of rank 0 and every rank equal."""
    vc.vc_set_slice_limit(vc.SLICE_ALWAYS)
    N, count = 8, (64 << 20) // 4
    xs = _inputs("f32", 8300, N, count)
    sends = [to_dev(x) for x in xs]
    recvs = [torch.empty_like(s) for s in sends]
    for algo in ("ring", "rhd", "dbt"):
        recs = _traced(lambda: vc.vc_allreduce(sends, recvs, algo=algo))
        assert recs[0]["kernel"].endswith("_sliced"), recs
        for r in range(1, N):
            assert torch.equal(recvs[r], recvs[0]), (algo, r)
        want = cxx.allreduce(xs, algo, "f32", want_log=False, keep=(0,)).outputs[0]
        got = to_host(recvs[0])
        assert same_bits(got, want), (algo, first_diff(got, want))


def test_sliced_16bit_at_8_mib():
    """bf16 at 8 MiB per rank, 8 ranks (16 MiB of fp32 partials: the largest
    flat Ring): every element of rank 0 equal to the oracle's, every rank equal."""
    vc.vc_set_slice_limit(vc.SLICE_ALWAYS)
    N, count = 8, (8 << 20) // 2
    xs = _inputs("bf16", 8310, N, count)
    sends = [to_dev(x) for x in xs]
    recvs = [torch.empty_like(s) for s in sends]
    for algo in ("ring", "rhd", "dbt"):
        recs = _traced(lambda: vc.vc_allreduce(sends, recvs, algo=algo))
        assert recs[0]["kernel"].endswith("_sliced"), recs
        for r in range(1, N):
            assert torch.equal(recvs[r], recvs[0]), (algo, r)
        want = cxx.allreduce(xs, algo, "bf16", want_log=False, keep=(0,)).outputs[0]
        got = to_host(recvs[0])
        assert same_bits(got, want), (algo, first_diff(got, want))


def _rs_ag_counts(dtype):
    G = 16 // {"f32": 4, "i32": 4, "bf16": 2, "f16": 2}[dtype]
    # whole groups a block (sliced), and a block of 5 elements, whose blocks are
    # not 16-byte aligned in the send buffer (the other forms)
    return ((G, True), (64 * G + G, True), (4096, True), (5, False))


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32", "f16"])
@pytest.mark.parametrize("N", [2, 3, 5, 8, 16])
def test_sliced_reduce_scatter_allgather(N, dtype):
    """Ring ReduceScatter and AllGather: positions counted within a block."""
    vc.vc_set_slice_limit(vc.SLICE_ALWAYS)
    for rc, aligned in _rs_ag_counts(dtype):
        sliced = aligned and N > 2  # at 2 ranks the ring is one step
        xs = _inputs(dtype, 8800 + N + rc, N, N * rc)
        want = cxx.reduce_scatter(xs, "ring", dtype, want_log=False).outputs
        sends = [Guarded(N * rc, dtype, fill=x) for x in xs]
        recvs = [Guarded(rc, dtype) for _ in range(N)]
        recs = _traced(lambda: vc.vc_reduce_scatter([g.t for g in sends], [g.t for g in recvs], algo="ring"))
        assert (len(recs) == 1 and recs[0]["kernel"].endswith("_sliced")) == sliced, ("rs", N, rc, recs)
        assert all(g.guards_intact() for g in sends + recvs)
        for r in range(N):
            got = recvs[r].host()
            assert same_bits(got, want[r]), ("rs", N, dtype, rc, r, first_diff(got, want[r]))
        ins = _inputs(dtype, 8900 + N + rc, N, rc)
        want = cxx.allgather(ins, "ring", dtype, want_log=False).outputs
        sends = [Guarded(rc, dtype, fill=x) for x in ins]
        recvs = [Guarded(N * rc, dtype) for _ in range(N)]
        recs = _traced(lambda: vc.vc_allgather([g.t for g in sends], [g.t for g in recvs], algo="ring"))
        assert (len(recs) == 1 and recs[0]["kernel"].endswith("_sliced")) == sliced, ("ag", N, rc, recs)
        assert all(g.guards_intact() for g in sends + recvs)
        for r in range(N):
            got = recvs[r].host()
            assert same_bits(got, want[r]), ("ag", N, dtype, rc, r, first_diff(got, want[r]))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [2, 3, 5, 8, 16])
def test_sliced_broadcast(N, dtype):
    """Binomial and pipelined Broadcasts (absolute positions), every root:
    every rank ends with the root's message, bit for bit; in place at the
    root takes the other forms."""
    vc.vc_set_slice_limit(vc.SLICE_ALWAYS)
    for count in (1, 1000 + 3, 65536 + 5):
        A = _inputs(dtype, 9000 + N + count, 1, count)[0]
        for root in sorted({0, N // 2, N - 1}):
            for algo, k in (("binomial", 0), ("pipe_chain", 4), ("pipe_tree", 3), ("pipe_chain", 0)):
                for inplace in (False, True):
                    recvs = [Guarded(count, dtype) for _ in range(N)]
                    if inplace:
                        recvs[root].t.copy_(to_dev(A))
                        src = recvs[root].t
                    else:
                        src = to_dev(A)
                    if algo.startswith("pipe"):
                        fn = lambda: vc.vc_broadcast_pipelined(src, [g.t for g in recvs], root=root, algo=algo,
                                                               nchunks=k)
                    else:
                        fn = lambda: vc.vc_broadcast(src, [g.t for g in recvs], root=root, algo=algo)
                    recs = _traced(fn)
                    steps = vc.vc_plan_describe("broadcast", algo, N, count, dtype, root, inplace, k)[2]
                    sliced = steps >= 2 and not inplace
                    assert (len(recs) == 1 and recs[0]["kernel"].endswith("_sliced")) == sliced, (
                        algo, k, N, count, root, inplace, recs)
                    assert all(g.guards_intact() for g in recvs)
                    for r in range(N):
                        assert same_bits(recvs[r].host(), A), (algo, k, N, count, root, inplace, r)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [3, 5, 8, 16])
def test_sliced_scatter_gather_reduce_and_scatter_allgather(N, dtype):
    """Binomial Scatter and Gather (positions: the root's buffer), tree
    Reduce, Scatter+AllGather Broadcast: every root, against the oracle."""
    vc.vc_set_slice_limit(vc.SLICE_ALWAYS)
    G = 16 // (4 if dtype == "f32" else 2)
    for rc in (G, 64 * G + G):
        for root in sorted({0, N // 2, N - 1}):
            B = _inputs(dtype, 9100 + N + rc + root, 1, N * rc)[0]
            recvs = [Guarded(rc, dtype) for _ in range(N)]
            recs = _traced(lambda: vc.vc_scatter(to_dev(B), [g.t for g in recvs], root=root, algo="binomial"))
            assert len(recs) == 1 and recs[0]["kernel"].endswith("_sliced"), ("scatter", N, rc, root, recs)
            for r in range(N):
                assert same_bits(recvs[r].host(), B[r * rc:(r + 1) * rc]), ("scatter", N, rc, root, r)
            xs = _inputs(dtype, 9200 + N + rc + root, N, rc)
            out = Guarded(N * rc, dtype)
            recs = _traced(lambda: vc.vc_gather([to_dev(x) for x in xs], out.t, root=root, algo="binomial"))
            assert len(recs) == 1 and recs[0]["kernel"].endswith("_sliced"), ("gather", N, rc, root, recs)
            assert same_bits(out.host(), np.concatenate(xs)), ("gather", N, rc, root)
            want = cxx.reduce(xs, root, "binomial", dtype, want_log=False).outputs[0]
            out = Guarded(rc, dtype)
            recs = _traced(lambda: vc.vc_reduce([to_dev(x) for x in xs], out.t, root=root, algo="binomial"))
            assert len(recs) == 1 and recs[0]["kernel"].endswith("_sliced"), ("reduce", N, rc, root, recs)
            got = out.host()
            assert same_bits(got, want), ("reduce", N, rc, root, first_diff(got, want))
            A = _inputs(dtype, 9300 + N + rc + root, 1, N * rc + 3)[0]
            bout = [Guarded(len(A), dtype) for _ in range(N)]
            recs = _traced(lambda: vc.vc_broadcast(to_dev(A), [g.t for g in bout], root=root, algo="scatter_allgather"))
            assert len(recs) == 1 and recs[0]["kernel"].endswith("_sliced"), ("sag", N, rc, root, recs)
            assert all(g.guards_intact() for g in recvs + bout + [out])
            for r in range(N):
                assert same_bits(bout[r].host(), A), ("sag", N, rc, root, r)


def test_calls_that_do_not_qualify_take_other_forms():
    vc.vc_set_slice_limit(vc.SLICE_ALWAYS)
    # a 16-bit Ring with more than 16 MiB of fp32 partials per rank: they
    # alternate between two chunk slots (at 8 ranks six steps write partials,
    # so each slot holds three chunks in turn; at 4 ranks or fewer each slot
    # holds one and stays positional)
    N, count = 8, (16 << 20) // 4 + 8 * 3 + 5
    xb = _inputs("bf16", 8400, N, count)
    want = cxx.allreduce(xb, "ring", "bf16", want_log=False).outputs
    got, recs = _run(xb, "ring", "bf16")
    assert not any(r["kernel"].endswith("_sliced") for r in recs), recs
    assert all(same_bits(got[r], want[r]) for r in range(N))
    # unaligned pointers, a single-step plan
    N, count = 8, 4096 + 3
    xs = _inputs("f32", 8401, N, count)
    for algo in ("ring", "fused"):
        want = cxx.allreduce(xs, algo, "f32", want_log=False).outputs
        got, recs = _run(xs, algo, "f32", shift=1 if algo == "ring" else 0)
        assert not any(r["kernel"].endswith("_sliced") for r in recs), (algo, recs)
        assert all(same_bits(got[r], want[r]) for r in range(N)), algo
    # AllToAll (blocks move between offsets that differ by rank)
    B = np.arange(N * N * 1024, dtype=np.int32).reshape(N, N * 1024)
    ins = [to_dev(B[r]) for r in range(N)]
    outs = [torch.empty(N * 1024, dtype=torch.int32, device="cuda") for _ in range(N)]
    for algo in ("bruck", "ring"):
        recs = _traced(lambda: vc.vc_alltoall(ins, outs, algo=algo))
        assert not any(r["kernel"].endswith("_sliced") for r in recs), (algo, recs)
        for j in range(N):
            got = to_host(outs[j]).reshape(N, 1024)
            assert all(np.array_equal(got[i], B[i, j * 1024:(j + 1) * 1024]) for i in range(N)), (algo, j)


def test_default_limit():
    """Every eligible schedule takes the sliced form up to the default limit."""
    vc.vc_set_slice_limit(vc.VC_SLICE_DEFAULT)
    assert vc.vc_get_slice_limit() == vc.VC_SLICE_DEFAULT
    N = 8
    for nbytes, sliced in ((1 << 20, True), (vc.VC_SLICE_DEFAULT, True), (2 * vc.VC_SLICE_DEFAULT, False)):
        count = nbytes // 4
        x = [torch.rand(count, device="cuda") for _ in range(N)]
        y = [torch.empty_like(t) for t in x]
        s = torch.stack(x).sum(0)
        for algo in ("ring", "dbt", "mesh", "rhd"):
            recs = _traced(lambda: vc.vc_allreduce(x, y, algo=algo))
            want = sliced
            assert any(r["kernel"].endswith("_sliced") for r in recs) == want, (algo, nbytes, recs)
            assert torch.allclose(y[0], s, atol=1e-5), (algo, nbytes)
        del x, y
    # 16-bit data: the limit counts the fp32 partial sums, 4 bytes per element
    for nbytes, sliced in ((1 << 20, True), (vc.VC_SLICE_DEFAULT // 2, True), (vc.VC_SLICE_DEFAULT, False)):
        count = nbytes // 2
        x = [torch.randn(count, device="cuda").to(torch.bfloat16) for _ in range(N)]
        y = [torch.empty_like(t) for t in x]
        s = torch.stack(x).float().sum(0)
        for algo in ("ring", "dbt", "mesh", "rhd"):
            recs = _traced(lambda: vc.vc_allreduce(x, y, algo=algo))
            assert any(r["kernel"].endswith("_sliced") for r in recs) == sliced, (algo, nbytes, recs)
            assert torch.allclose(y[0].float(), s, rtol=1e-2, atol=1e-2), (algo, nbytes)
        del x, y


def test_sliced_inside_a_cuda_graph():
    """A shape seen before capture runs sliced inside the graph; a shape first
    seen under capture takes the per-step path (its description is uploaded
    only outside a capture).  Both replay exactly, twice, on new data."""
    vc.vc_set_slice_limit(vc.VC_SLICE_DEFAULT)
    N, count = 8, 65536 + 12
    sends = [torch.empty(count, device="cuda") for _ in range(N)]
    recvs = [torch.empty(count, device="cuda") for _ in range(N)]
    fresh = [torch.empty(count + 16, device="cuda") for _ in range(N)]
    fresh_out = [torch.empty(count + 16, device="cuda") for _ in range(N)]
    recs = _traced(lambda: vc.vc_allreduce(sends, recvs, algo="ring"))  # resident before capture
    assert recs[0]["kernel"].endswith("_sliced"), recs
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        vc.vc_allreduce(sends, recvs, algo="ring")
        vc.vc_allreduce(fresh, fresh_out, algo="dbt")
    for seed in (1, 2):
        xs = _inputs("f32", 8500 + seed, N, count)
        ys = _inputs("f32", 8600 + seed, N, count + 16)
        for r in range(N):
            sends[r].copy_(to_dev(xs[r]))
            fresh[r].copy_(to_dev(ys[r]))
        g.replay()
        torch.cuda.synchronize()
        want = cxx.allreduce(xs, "ring", "f32", want_log=False).outputs
        want2 = cxx.allreduce(ys, "dbt", "f32", want_log=False).outputs
        for r in range(N):
            assert same_bits(to_host(recvs[r]), want[r]), (seed, r)
            assert same_bits(to_host(fresh_out[r]), want2[r]), (seed, r)
