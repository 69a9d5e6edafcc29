"""Randomized sweep (fixed seed) over the whole call space on the CPU: every
collective and algorithm, N in 1..16, ragged counts, roots, dtypes, ops,
in-place and chunk counts.  Each plan the library would launch is replayed
and must match the oracle bit for bit, move data between the same ranks in
the same steps, read and write the oracle's algorithmic bytes, and have no
intra-step hazards.  The execution form the library reports for it
(vc_plan_form) must be the one predicted from the plan's positions."""
import random

import numpy as np
import pytest

from oracle import numerics, schedules
from synthetic_inputs import rank_buffers

from .plan_replay import (DT, ESZ, NPT, Memory, get_plan, hazards, oracle_transfers, predict_sliced, run_plan,
                          transfers)

import collective_communication_algorithms_virtual_gb300 as vc

ALL = {c: tuple(schedules.ALGOS.get(c, ())) + tuple(a for a in schedules.ALGOS_EXTRA.get(c, ())
                                                     if a not in schedules.ALGOS.get(c, ()))
       for c in ("allreduce", "reduce_scatter", "allgather", "broadcast", "scatter", "alltoall", "gather", "reduce")}
REDUCING = ("allreduce", "reduce_scatter", "reduce")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from collective_communication_algorithms_virtual_gb300 import build

    build.build()


def _inputs(dtype, seed, N, n):
    if dtype == "f16":
        return [x.astype(np.float16) for x in rank_buffers("uniform_f32", seed, N, n)]
    kind = {"f32": "uniform_f32", "bf16": "uniform_bf16", "i32": "int32_bits"}[dtype]
    return rank_buffers(kind, seed, N, n)


def _case(rng):
    coll = rng.choice(sorted(ALL))
    algo = rng.choice(ALL[coll])
    N = rng.randint(1, 16)
    dtype = rng.choice(["f32", "bf16", "i32", "f16"])
    op = rng.choice(["sum", "max", "min"]) if coll in REDUCING else "sum"
    root = rng.randrange(N)
    count = rng.choice([0, 1, rng.randint(2, 40), rng.randint(41, 700)])
    inplace = rng.random() < 0.3 and coll in ("allreduce", "broadcast", "reduce")
    k = rng.randint(1, 9)
    return coll, algo, N, dtype, op, root, count, inplace, k


def _oracle(coll, algo, N, dtype, op, root, count, inplace, k, seed):
    if coll == "allreduce":
        xs = _inputs(dtype, seed, N, count)
        return xs, schedules.allreduce(xs, algo, dtype, inplace=inplace, op=op)
    if coll == "reduce_scatter":
        xs = _inputs(dtype, seed, N, N * count)
        return xs, schedules.reduce_scatter(xs, algo, dtype, op=op)
    if coll == "allgather":
        xs = _inputs(dtype, seed, N, count)
        return xs, schedules.allgather(xs, algo, dtype)
    if coll == "broadcast":
        A = _inputs(dtype, seed, 1, count)[0]
        if algo.startswith("pipe_"):
            return A, schedules.broadcast_pipelined(A, N, root, algo, dtype, k, inplace=inplace)
        return A, schedules.broadcast(A, N, root, algo, dtype, inplace=inplace)
    if coll == "scatter":
        A = _inputs(dtype, seed, 1, N * count)[0]
        return A, schedules.scatter(A, N, root, algo, dtype)
    if coll == "gather":
        xs = _inputs(dtype, seed, N, count)
        return xs, schedules.gather(xs, root, algo, dtype)
    if coll == "reduce":
        xs = _inputs(dtype, seed, N, count)
        return xs, schedules.reduce(xs, root, algo, dtype, inplace=inplace, op=op)
    xs = _inputs(dtype, seed, N, N * count)
    return xs, schedules.alltoall(xs, algo, dtype)


@pytest.mark.parametrize("batch", range(8))
def test_random_calls_replay_to_oracle(batch):
    rng = random.Random(1000 + batch)
    for i in range(50):
        coll, algo, N, dtype, op, root, count, inplace, k = _case(rng)
        es = ESZ[DT[dtype]]
        data, res = _oracle(coll, algo, N, dtype, op, root, count, inplace, k, 7 * batch + i)
        plan, scratch = get_plan(coll, algo, N, count, dtype, root, inplace, k, op)
        ctx = (coll, algo, N, dtype, op, root, count, inplace, k)
        # buffers as the library sees them
        if coll in ("broadcast", "scatter"):
            send = [None] * N
            send[root] = data
        else:
            send = data
        out_elems = {"allreduce": count, "reduce_scatter": count, "allgather": N * count, "broadcast": count,
                     "scatter": count, "alltoall": N * count, "gather": N * count, "reduce": count}[coll]
        sizes = [out_elems * es] * N
        if coll in ("gather", "reduce"):
            sizes = [out_elems * es if r == root else 0 for r in range(N)]
        inplace_ranks = ()
        if inplace:
            inplace_ranks = range(N) if coll == "allreduce" else [root]
        mem = Memory(send, sizes, scratch, inplace_ranks=inplace_ranks)
        run_plan(plan, mem)
        assert not hazards(plan, mem), ctx
        outs = [mem.recv[root]] if coll in ("gather", "reduce") else mem.recv
        for got, want in zip(outs, res.outputs):
            assert numerics.same_bits(got.view(NPT[DT[dtype]]), want), ctx
        assert transfers(plan) == oracle_transfers(res.log), ctx
        entries = vc.vc_plan_describe(coll, algo, N, count, dtype, root, inplace, k, op)[0]
        assert sum(e.n * e.nb * ESZ[e.dtype] for e in entries) == res.hbm_bytes, ctx
        # the library's form against the prediction from the plan's positions
        form, launches, host_ranges = vc.vc_plan_form(coll, algo, N, count, dtype, root, inplace, k, op)
        sliced, want_hr = predict_sliced(coll, algo, N, count, dtype, root, inplace, k, op)
        assert (form == "sliced") == sliced, (ctx, form)
        assert not sliced or (launches, host_ranges) == (1, want_hr), (ctx, launches, host_ranges)
        assert coll != "alltoall" or form == "steps", (ctx, form)


def test_corner_cases_replay_to_oracle():
    """Single rank in place, empty buffers, one element, every algorithm."""
    for coll, algos in ALL.items():
        for algo in algos:
            for N, count, inplace in ((1, 5, True), (1, 5, False), (2, 0, False), (3, 1, False), (16, 1, False)):
                if inplace and coll not in ("allreduce", "broadcast", "reduce"):
                    continue
                data, res = _oracle(coll, algo, N, "f32", "sum", 0, count, inplace, 3, 5)
                entries, scratch, _ = vc.vc_plan_describe(coll, algo, N, count, "f32", 0, inplace, 3)
                assert sum(e.n * e.nb * 4 for e in entries) == res.hbm_bytes, (coll, algo, N, count, inplace)
