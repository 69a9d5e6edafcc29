"""MAX / MIN reductions, fp16, Mesh AllReduce and Ring AllToAll (CPU): the
oracle against library routines, hand-derived cases and the pages; the
library's plans replayed against the oracle."""
import numpy as np
import pytest

from oracle import cost_model as cm
from oracle import numerics, orders, schedules
from synthetic_inputs import rank_buffers

from .plan_replay import DT, ESZ, NPT, Memory, get_plan, hazards, oracle_transfers, run_plan, transfers


@pytest.fixture(scope="module", autouse=True)
def _built():
    from collective_communication_algorithms_virtual_gb300 import build

    build.build()


def _kind(dtype):
    return {"f32": "uniform_f32", "bf16": "uniform_bf16", "i32": "int32_bits"}[dtype]


def _inputs(dtype, seed, N, n):
    if dtype == "f16":
        return [x.astype(np.float16) for x in rank_buffers("uniform_f32", seed, N, n)]
    return rank_buffers(_kind(dtype), seed, N, n)


@pytest.mark.parametrize("N", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32", "f16"])
def test_max_min_equal_library_max_min(N, dtype):
    """No zeros or NaNs in these inputs, so every association gives numpy's
    elementwise max / min of the stacked ranks."""
    count = 203
    xs = _inputs(dtype, 1 + N, N, count)
    lanes = np.stack([numerics.widen(x, dtype) for x in xs])
    if dtype == "i32":
        lanes = lanes.view(np.int32)
    for op, f in (("max", np.max), ("min", np.min)):
        want = f(lanes, axis=0)
        want = numerics.narrow(want.view(np.uint32) if dtype == "i32" else want, dtype)
        for algo in schedules.ALGOS["allreduce"]:
            out = schedules.allreduce(xs, algo, dtype, op=op).outputs
            for o in out:
                assert numerics.same_bits(o, want), (op, algo, N, dtype)
        for algo in schedules.ALGOS_EXTRA["reduce"]:
            assert numerics.same_bits(schedules.reduce(xs, N - 1, algo, dtype, op=op).outputs[0], want)
        rc = 7
        xr = _inputs(dtype, 9 + N, N, N * rc)
        lr = np.stack([numerics.widen(x, dtype) for x in xr])
        if dtype == "i32":
            lr = lr.view(np.int32)
        wr = f(lr, axis=0)
        wr = numerics.narrow(wr.view(np.uint32) if dtype == "i32" else wr, dtype)
        for algo in schedules.ALGOS["reduce_scatter"]:
            out = schedules.reduce_scatter(xr, algo, dtype, op=op).outputs
            assert numerics.same_bits(np.concatenate(out), wr), (op, algo, N, dtype)


def test_max_min_nan_and_signed_zero():
    """Hand-derived: max keeps the first operand unless the second is larger
    or the first is NaN.  Rank order 0..3 (fused):
      NaN, 1, NaN, 2  -> max 2, min 1 (NaN passed over)
      -0, +0          -> max -0, min -0 (equal: the first kept)
      +0, -0          -> +0 both
      NaN everywhere  -> NaN."""
    nan = np.float32(np.nan)
    rows = [((nan, 1.0, nan, 2.0), 2.0, 1.0), ((-0.0, 0.0, 0.0, 0.0), -0.0, -0.0),
            ((0.0, -0.0, -0.0, -0.0), 0.0, 0.0)]
    for vals, mx, mn in rows:
        xs = [np.full(4, v, dtype=np.float32) for v in vals]
        for op, want in (("max", mx), ("min", mn)):
            got = schedules.allreduce(xs, "fused", "f32", op=op).outputs[0]
            assert np.array_equal(got.view(np.uint32), np.full(4, want, dtype=np.float32).view(np.uint32)), (vals, op)
    xs = [np.full(4, nan, dtype=np.float32) for _ in range(4)]
    assert np.all(np.isnan(schedules.allreduce(xs, "ring", "f32", op="max").outputs[0]))


def test_fp16_sum_rounds_once():
    N, count = 8, 4096
    xs = _inputs("f16", 3, N, count)
    direct = xs[0].astype(np.float32)
    for x in xs[1:]:
        direct = direct + x.astype(np.float32)
    assert np.array_equal(schedules.allreduce(xs, "fused", "f16").outputs[0], direct.astype(np.float16))
    for algo in schedules.ALGOS["allreduce"]:
        out = schedules.allreduce(xs, algo, "f16").outputs[0]
        assert np.max(np.abs(out.astype(np.float32) - direct.astype(np.float16).astype(np.float32))) <= \
            np.max(np.abs(direct)) * 2.0 ** -10
        want = orders.allreduce_at(xs, algo, count, "f16", np.arange(count))
        assert numerics.same_bits(out, want), algo


def test_mesh_steps_follow_the_article():
    """Root 0 receives from 1, 2, ..., N-1 one per step, then sends to 1, ...,
    N-1 one per step: 2(N-1) steps, each carrying the whole message."""
    N, count = 5, 64
    res = schedules.allreduce(rank_buffers("uniform_f32", 4, N, count), "mesh", "f32")
    assert res.log.table() == [(t, t + 1, 0) for t in range(N - 1)] + [(N - 1 + t, 0, t + 1) for t in range(N - 1)]
    assert res.nsteps == 2 * (N - 1)
    assert all(t.nbytes == count * 4 for t in res.log.records)


def test_ring_alltoall_traffic_contradicts_the_printed_formula():
    """Store and forward: round k carries N-k blocks per rank, (N-1)/2 * M in
    all per rank; eq. model-algo-a2a-ring prints Pairwise's (N-1)/N * M."""
    N, B = 8, 4
    M = N * B * 4
    res = schedules.alltoall(rank_buffers("uniform_f32", 5, N, N * B), "ring", "f32")
    assert res.nsteps == N - 1
    per = res.log.max_message_bytes_per_step()
    assert [per[k] for k in range(1, N)] == [(N - k) * B * 4 for k in range(1, N)]
    assert res.log.bandwidth_bytes() == (N - 1) * M // 2
    assert res.log.bandwidth_bytes() != (N - 1) * M // N
    for t in res.log.records:
        assert t.dst == (t.src + 1) % N  # neighbours only
    assert cm.t_a2a_ring(N, M, 1e-6, 1e9) == pytest.approx(cm.t_a2a_pairwise(N, M, 1e-6, 1e9))


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("op", ["max", "min", "sum"])
@pytest.mark.parametrize("dtype", ["f32", "f16", "i32"])
def test_op_and_fp16_plans_replay(N, op, dtype):
    count = 57
    xs = _inputs(dtype, 20 + N, N, count)
    es = ESZ[DT[dtype]]
    for algo in schedules.ALGOS["allreduce"]:
        res = schedules.allreduce(xs, algo, dtype, op=op)
        plan, scratch = get_plan("allreduce", algo, N, count, dtype, op=op)
        mem = Memory(xs, [count * es] * N, scratch)
        run_plan(plan, mem)
        assert not hazards(plan, mem)
        for r in range(N):
            assert numerics.same_bits(mem.recv[r].view(NPT[DT[dtype]]), res.outputs[r]), (algo, op, dtype, r)
        assert transfers(plan) == oracle_transfers(res.log)
    rc = 9
    xr = _inputs(dtype, 30 + N, N, N * rc)
    for algo in schedules.ALGOS["reduce_scatter"]:
        res = schedules.reduce_scatter(xr, algo, dtype, op=op)
        plan, scratch = get_plan("reduce_scatter", algo, N, rc, dtype, op=op)
        mem = Memory(xr, [rc * es] * N, scratch)
        run_plan(plan, mem)
        for r in range(N):
            assert numerics.same_bits(mem.recv[r].view(NPT[DT[dtype]]), res.outputs[r]), (algo, op, dtype, r)
    for algo in schedules.ALGOS_EXTRA["reduce"]:
        res = schedules.reduce(xs, N // 2, algo, dtype, op=op)
        plan, scratch = get_plan("reduce", algo, N, count, dtype, root=N // 2, op=op)
        mem = Memory(xs, [count * es if r == N // 2 else 0 for r in range(N)], scratch)
        run_plan(plan, mem)
        assert numerics.same_bits(mem.recv[N // 2].view(NPT[DT[dtype]]), res.outputs[0]), (algo, op, dtype)


def test_rhd_fold_in_for_n_not_a_power_of_2():
    """N = 6: P = 4, r = 2.  Step 0: 1->0 and 3->2 fold in (whole buffer);
    then halving / doubling among real ranks 0, 2, 4, 5 (2 log2 4 steps);
    last step 0->1 and 2->3 hand the result back: 2 + 2 log2 P steps."""
    N, count = 6, 64
    res = schedules.allreduce(rank_buffers("small_ints_f32", 7, N, count), "rhd", "f32")
    table = res.log.table()
    assert [t for t in table if t[0] == 0] == [(0, 1, 0), (0, 3, 2)]
    assert [t for t in table if t[0] == 5] == [(5, 0, 1), (5, 2, 3)]
    mid = {t[1] for t in table if 1 <= t[0] <= 4} | {t[2] for t in table if 1 <= t[0] <= 4}
    assert mid == {0, 2, 4, 5}
    assert res.nsteps == 2 + 2 * 2
    for o in res.outputs:
        assert numerics.same_bits(o, res.outputs[0])
