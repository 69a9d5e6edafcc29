"""The C++ oracle (oracle/sim.cpp) against the numpy oracle (oracle/schedules.py).

The two are independent restatements of the same schedules.  They must agree
on every output bit, every transfer-log record (step, sender, receiver,
elements, reduce or store, wire element size, offsets, chunks, phase), the
algorithmic HBM bytes and the local steps, over every collective, algorithm,
dtype, op, rank count, root, ragged size and in-place flag below.  The pins in
test_oracle_pins.py then hold for both.  fp16 NaN payloads are the one known
difference (numpy's cast keeps the payload bits, the C++ oracle also sets the
quiet bit), so fp16 data here has no NaN.
"""
import numpy as np
import pytest

from oracle import cxx, schedules
from synthetic_inputs import int32_bits, normal_f32, rank_buffers


def _data(dtype, seed, N, n):
    if dtype == "f16":
        return [normal_f32(seed, r, n).astype(np.float16) for r in range(N)]
    kind = {"f32": "uniform_f32", "bf16": "normal_bf16", "i32": "int32_bits"}[dtype]
    return rank_buffers(kind, seed, N, n)


def same(a, b):
    a, b = np.ascontiguousarray(a), np.ascontiguousarray(b)
    return a.shape == b.shape and a.dtype.itemsize == b.dtype.itemsize and np.array_equal(
        a.view(np.uint8), b.view(np.uint8))


def check(rn, rc, what):
    assert len(rn.outputs) == len(rc.outputs), what
    for i, (a, b) in enumerate(zip(rn.outputs, rc.outputs)):
        assert same(a, b), (what, "output", i)
    assert rn.hbm_bytes == rc.hbm_bytes, (what, rn.hbm_bytes, rc.hbm_bytes)
    assert rn.local_steps == rc.local_steps, what
    assert len(rn.log.records) == len(rc.log.records), what
    for t, u in zip(rn.log.records, rc.log.records):
        assert t == u, (what, t, u)


def call_both(fn_name, *args, **kw):
    outs = []
    for mod in (schedules, cxx):
        try:
            outs.append(getattr(mod, fn_name)(*args, **kw))
        except (schedules.Unsupported, cxx.Unsupported) as e:
            outs.append(type(e).__name__)
    return outs


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 6, 7, 8, 9, 12, 16])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32", "f16"])
def test_allreduce_agrees(N, dtype):
    for count in (0, 1, 7, N * 8 + 3, 203, 1000):
        xs = _data(dtype, 100 + N + count, N, count)
        for algo in schedules.ALGOS["allreduce"]:
            for op in ("sum", "max", "min"):
                for inplace in (False, True):
                    rn, rc = call_both("allreduce", xs, algo, dtype, inplace=inplace, op=op)
                    check(rn, rc, ("allreduce", algo, N, dtype, count, op, inplace))


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 7, 8, 16])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32", "f16"])
def test_reduce_scatter_allgather_agree(N, dtype):
    for rc_ in (0, 1, 5, 13, 64):
        xs = _data(dtype, 200 + N + rc_, N, N * rc_)
        for algo in schedules.ALGOS["reduce_scatter"]:
            for op in ("sum", "max"):
                rn, rc = call_both("reduce_scatter", xs, algo, dtype, op=op)
                check(rn, rc, ("reduce_scatter", algo, N, dtype, rc_, op))
        ins = [x[:rc_] for x in xs]
        for algo in schedules.ALGOS["allgather"]:
            rn, rc = call_both("allgather", ins, algo, dtype)
            check(rn, rc, ("allgather", algo, N, dtype, rc_))


@pytest.mark.parametrize("N", [1, 2, 3, 5, 8, 16])
def test_rooted_collectives_agree(N):
    for root in sorted({0, 1 % N, N - 1}):
        for count in (0, 1, 5, 37, 160):
            A = int32_bits(300 + N, root, count)
            for algo in schedules.ALGOS["broadcast"]:
                for inplace in (False, True):
                    rn, rc = call_both("broadcast", A, N, root, algo, "i32", inplace=inplace)
                    check(rn, rc, ("broadcast", algo, N, root, count, inplace))
            for algo in schedules.ALGOS_EXTRA["broadcast"]:
                for k in (1, 2, 3, 7):
                    rn, rc = call_both("broadcast_pipelined", A, N, root, algo, "i32", k)
                    check(rn, rc, ("broadcast", algo, N, root, count, k))
        for rc_ in (0, 1, 3, 8):
            A = int32_bits(310 + N, root, N * rc_)
            for algo in schedules.ALGOS["scatter"]:
                rn, rc = call_both("scatter", A, N, root, algo, "i32")
                check(rn, rc, ("scatter", algo, N, root, rc_))
            xs = [int32_bits(320 + N, r, rc_) for r in range(N)]
            for algo in schedules.ALGOS_EXTRA["gather"]:
                rn, rc = call_both("gather", xs, root, algo, "i32")
                check(rn, rc, ("gather", algo, N, root, rc_))
        for dtype in ("f32", "bf16", "f16", "i32"):
            xs = _data(dtype, 330 + N + root, N, 77)
            for algo in schedules.ALGOS_EXTRA["reduce"]:
                for op in ("sum", "min"):
                    for inplace in (False, True):
                        rn, rc = call_both("reduce", xs, root, algo, dtype, inplace=inplace, op=op)
                        check(rn, rc, ("reduce", algo, N, root, dtype, op, inplace))


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 6, 7, 8, 11, 16])
@pytest.mark.parametrize("dtype", ["bf16", "i32"])
def test_alltoall_agrees(N, dtype):
    for B in (0, 1, 3, 8):
        xs = _data(dtype, 400 + N + B, N, N * B)
        for algo in schedules.ALGOS["alltoall"]:
            rn, rc = call_both("alltoall", xs, algo, dtype)
            check(rn, rc, ("alltoall", algo, N, dtype, B))


def test_unsupported_agrees():
    xs = _data("f32", 1, 4, 16)
    for fn, args in [("allreduce", (xs, "bruck", "f32")), ("reduce_scatter", (xs, "rhd", "f32")),
                     ("allgather", (xs, "dbt", "f32")), ("alltoall", (xs, "rhd", "f32")),
                     ("broadcast", (xs[0], 4, 0, "ring", "f32")), ("scatter", (xs[0], 4, 0, "ring", "f32")),
                     ("reduce", (xs, 0, "ring", "f32")), ("gather", (xs, 0, "ring", "f32"))]:
        rn, rc = call_both(fn, *args)
        assert rn == rc == "Unsupported", (fn, rn, rc)


@pytest.mark.parametrize("N", [2, 3, 5, 6, 7, 8, 12, 16])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_closed_form_trees_agree(N, dtype):
    from oracle import orders

    count = N * 8 * 3 + 5
    xs = _data(dtype, 500 + N, N, count)
    idx = np.arange(count)
    for algo in schedules.ALGOS["allreduce"]:
        a = orders.allreduce_at(xs, algo, count, dtype, idx)
        b = cxx.allreduce_at(xs, algo, count, dtype, idx)
        assert same(a, b), (algo, N, dtype)
    rc_ = 13
    xr = _data(dtype, 510 + N, N, N * rc_)
    for algo in schedules.ALGOS["reduce_scatter"]:
        a = orders.reduce_scatter_at(xr, algo, rc_, dtype, np.arange(N * rc_))
        b = cxx.reduce_scatter_at(xr, algo, rc_, dtype, np.arange(N * rc_))
        assert same(a, b), (algo, N, dtype)
