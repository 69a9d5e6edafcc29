"""The sliced form's precondition and its execution order, on the CPU.

In the sliced form one thread owns a group of element positions (16 bytes
of the data type: 4 fp32 / int32 elements, 8 bf16 / fp16 ones) of every
buffer and walks every step of the AllReduce plan for them alone.  That is
exact only if each byte an operation touches belongs to one position: every
operand holds position elem0 + i at a fixed place of its buffer.  Here, from
the plan the library describes (no GPU):

- every AllReduce schedule in every data type and op meets that condition
  while the partial sums take at most 16 MiB per rank (the 16-bit Ring keeps
  one fp32 partial per position), writes no send buffer, and reads a receive
  buffer or scratch only where an earlier step wrote (the sliced kernels
  read those through L1: the reading thread stored them itself);
- running the plan group by group -- each group to the end before the next,
  and the groups' steps randomly interleaved -- gives the oracle's result bit
  for bit;
- a planted layout that reuses partial-sum slots across chunks (still exact
  step by step) fails the condition and breaks an interleaved run, so both
  checks can fail;
- above 16 MiB of fp32 partial sums per rank the 16-bit Ring's alternating
  slots fail the condition at 8 ranks (at 4 or fewer each slot holds one
  chunk and the condition holds).
"""
import numpy as np
import pytest

from collective_communication_algorithms_virtual_gb300 import build
from oracle import schedules
from synthetic_inputs import rank_buffers

from .plan_replay import (DT, ESZ, NPT, SCRATCH, Memory, get_plan, hazards, one_after_another, position_places,
                          reads_before_writes, run_plan, run_plan_sliced, shuffled)

ALGOS = tuple(a for a in schedules.ALGOS["allreduce"] if a != "fused")  # multi-step schedules


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def _inputs(dtype, seed, N, n):
    if dtype == "f16":
        return [x.astype(np.float16) for x in rank_buffers("uniform_f32", seed, N, n)]
    kind = {"f32": "uniform_f32", "bf16": "uniform_bf16", "i32": "int32_bits"}[dtype]
    return rank_buffers(kind, seed, N, n)


def _group(dtype):
    return 16 // ESZ[DT[dtype]]


def _outputs(mem, N, dtype):
    return [mem.recv[r].view(NPT[DT[dtype]]) for r in range(N)]


def _same(got, want):
    return np.array_equal(np.ascontiguousarray(got).view(np.uint8), np.ascontiguousarray(want).view(np.uint8))


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16", "i32"])
@pytest.mark.parametrize("N", [2, 3, 5, 8, 16])
def test_allreduce_plans_keep_positions(N, dtype):
    for count in (1, 13, 1000, 4096 + 5):
        for algo in ALGOS:
            for op in ("sum", "max"):
                plan, scratch = get_plan("allreduce", algo, N, count, dtype, op=op)
                mem = Memory([None] * N, [0] * N, scratch)
                bad = position_places(plan, mem, _group(dtype))
                assert not bad, (algo, N, count, dtype, op, bad[:3])
                for inplace in (False, True):
                    plan_i = get_plan("allreduce", algo, N, count, dtype, op=op, inplace=inplace)[0]
                    bad = reads_before_writes(plan_i, mem)
                    assert not bad, (algo, N, count, dtype, op, inplace, bad[:3])


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16", "i32"])
@pytest.mark.parametrize("N,count", [(2, 203), (3, 1000), (5, 517), (8, 1024 + 9), (16, 999)])
def test_group_by_group_runs_equal_the_oracle(N, count, dtype):
    xs = _inputs(dtype, 900 + N + count, N, count)
    G = _group(dtype)
    groups = (count + G - 1) // G
    rng = np.random.default_rng(N * 1000 + count)
    for algo in ALGOS:
        for op in ("sum", "min"):
            if dtype == "i32" and op == "min":
                continue
            want = schedules.allreduce(xs, algo, dtype, op=op).outputs
            plan, scratch = get_plan("allreduce", algo, N, count, dtype, op=op)
            for sched in (one_after_another(groups, len(plan)), shuffled(groups, len(plan), rng)):
                mem = Memory(xs, [count * ESZ[DT[dtype]]] * N, scratch)
                run_plan_sliced(plan, mem, count, G, sched)
                for r, got in enumerate(_outputs(mem, N, dtype)):
                    assert _same(got, want[r]), (algo, op, N, count, dtype, r)


def _alternating_slots(plan, N, count):
    """The 8-rank bf16 Ring plan with its fp32 partial sums moved into two
    chunk-sized slots per rank, by chunk parity (neighbouring chunks, which
    one step writes and reads, take different slots): exact step by step,
    but positions ce apart share bytes."""
    ce = (count + N - 1) // N
    ce = (ce + 7) // 8 * 8
    base = {}
    for ops in plan:
        for op in ops:
            for (k, o, dt, off, stride) in op["src"] + op["dst"]:
                if k == SCRATCH:
                    base[o] = min(base.get(o, off), off - op["elem0"] * 4)
    out = []
    for ops in plan:
        new_ops = []
        for op in ops:
            op = dict(op)
            for role in ("src", "dst"):
                moved = []
                for (k, o, dt, off, stride) in op[role]:
                    if k == SCRATCH:
                        c = (off - base[o]) // 4 // ce
                        off = base[o] + (c % 2) * ce * 4
                    moved.append((k, o, dt, off, stride))
                op[role] = moved
            new_ops.append(op)
        out.append(new_ops)
    return out


def test_reads_before_writes_catches_a_planted_early_read():
    """A read of a receive buffer moved one step before the write it needs:
    in the bf16 Ring (partials in scratch) AllGather step 2 copies the chunk
    that step 1 stored, and nothing wrote those bytes before."""
    N, count = 4, 4 * 64
    plan, scratch = get_plan("allreduce", "ring", N, count, "bf16")
    mem = Memory([None] * N, [0] * N, scratch)
    assert not reads_before_writes(plan, mem)
    planted = plan[:N] + [plan[-1]] + plan[N:-1]  # AllGather steps 0, 2, 1
    assert reads_before_writes(planted, mem)


def test_planted_slot_reuse_fails_both_checks():
    N, count = 8, 8 * 64
    xs = _inputs("bf16", 77, N, count)
    want = schedules.allreduce(xs, "ring", "bf16").outputs
    plan, scratch = get_plan("allreduce", "ring", N, count, "bf16")
    planted = _alternating_slots(plan, N, count)
    # step by step the planted layout is still exact and race-free ...
    mem = Memory(xs, [count * 2] * N, scratch)
    run_plan(planted, mem)
    assert not hazards(planted, mem)
    assert all(_same(g, w) for g, w in zip(_outputs(mem, N, "bf16"), want))
    # ... but positions share bytes: the condition fails, and interleaved it breaks
    assert position_places(planted, mem, 8)
    sched = shuffled(count // 8, len(plan), np.random.default_rng(5))
    mem = Memory(xs, [count * 2] * N, scratch)
    run_plan_sliced(planted, mem, count, 8, sched)
    assert not all(_same(g, w) for g, w in zip(_outputs(mem, N, "bf16"), want))
    # the library's own layout passes both
    assert not position_places(plan, mem, 8)
    mem = Memory(xs, [count * 2] * N, scratch)
    run_plan_sliced(plan, mem, count, 8, sched)
    assert all(_same(g, w) for g, w in zip(_outputs(mem, N, "bf16"), want))


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_ring_partials_above_16_mib_alternate(dtype):
    limit = (16 << 20) // 4  # elements whose fp32 partials take 16 MiB
    for N, count, positional in ((8, limit, True), (8, limit + 8, False), (4, limit + 8, True), (3, limit + 8, True)):
        plan, scratch = get_plan("allreduce", "ring", N, count, dtype)
        mem = Memory([None] * N, [0] * N, scratch)
        assert (not position_places(plan, mem, 8)) == positional, (N, count)
        # flat: one fp32 partial per position and rank; above: two chunk slots per rank
        ce = ((count + N - 1) // N + 7) // 8 * 8
        per_rank = count * 4 if count <= limit else 2 * ce * 4
        assert scratch == N * ((per_rank + 255) // 256 * 256), (N, count, scratch)
