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
                          predict_sliced, reads_before_writes, run_plan, run_plan_sliced, shuffled)

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


# ---- the other collectives whose schedules keep positions ---------------------------------
# Positions are the elements of the message: the ring ReduceScatter's input
# (its partial sums keep one slot per block while they take at most 16 MiB per
# rank), the ring AllGather's output, the Broadcasts' message, the binomial
# Scatter's input and Gather's output at the root, the tree Reduce's buffer.

def _rs_ag_bcast_cases(N, dtype):
    G = _group(dtype)
    rc = 8 * G + (G if dtype != "bf16" else 0)  # whole groups a block; every block 16-byte aligned
    xs = _inputs(dtype, 1300 + N, N, N * rc)
    yield ("reduce_scatter", "ring", rc, 0, 0,
           lambda: schedules.reduce_scatter(xs, "ring", dtype).outputs, xs, [rc * ESZ[DT[dtype]]] * N, N * rc)
    ins = _inputs(dtype, 1400 + N, N, rc)
    yield ("allgather", "ring", rc, 0, 0,
           lambda: schedules.allgather(ins, "ring", dtype).outputs, ins, [N * rc * ESZ[DT[dtype]]] * N, N * rc)
    count = 1000 + 3
    A = _inputs(dtype, 1500 + N, 1, count)[0]
    for root in (0, N - 1):
        send = [None] * N
        send[root] = A
        for algo, k in (("binomial", 0), ("scatter_allgather", 0), ("pipe_chain", 5), ("pipe_tree", 3)):
            if k:
                want = lambda root=root, algo=algo, k=k: schedules.broadcast_pipelined(A, N, root, algo, dtype, k).outputs
            else:
                want = lambda root=root, algo=algo: schedules.broadcast(A, N, root, algo, dtype).outputs
            yield ("broadcast", algo, count, root, k, want, send, [count * ESZ[DT[dtype]]] * N, count)
        # binomial Scatter / Gather (blocks of rc) and tree Reduce, at the root only
        B = _inputs(dtype, 1600 + N + root, 1, N * rc)[0]
        sendB = [None] * N
        sendB[root] = B
        yield ("scatter", "binomial", rc, root, 0, lambda root=root: schedules.scatter(B, N, root, "binomial", dtype).outputs,
               sendB, [rc * ESZ[DT[dtype]]] * N, N * rc)
        root_only = lambda nbytes, root=root: [nbytes if r == root else 0 for r in range(N)]
        yield ("gather", "binomial", rc, root, 0,
               lambda root=root: _at_root(schedules.gather(ins, root, "binomial", dtype).outputs[0], root, N),
               ins, root_only(N * rc * ESZ[DT[dtype]]), N * rc)
        if dtype != "i32":
            yield ("reduce", "binomial", rc, root, 0,
                   lambda root=root: _at_root(schedules.reduce(ins, root, "binomial", dtype).outputs[0], root, N),
                   ins, root_only(rc * ESZ[DT[dtype]]), rc)


def _at_root(out, root, N):
    """A root-only output as a per-rank list (other ranks: empty)."""
    return [out if r == root else np.zeros(0, out.dtype) for r in range(N)]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
@pytest.mark.parametrize("N", [2, 3, 5, 8])
def test_other_collective_plans_keep_positions_and_run_group_by_group(N, dtype):
    G = _group(dtype)
    rng = np.random.default_rng(31 + N)
    for coll, algo, count, root, k, want_fn, send, recv_bytes, positions in _rs_ag_bcast_cases(N, dtype):
        plan, scratch = get_plan(coll, algo, N, count, dtype, root=root, nchunks=k)
        mem = Memory(send, recv_bytes, scratch)
        assert not position_places(plan, mem, G), (coll, algo, N, dtype, position_places(plan, mem, G)[:3])
        assert not reads_before_writes(plan, mem), (coll, algo, N, dtype)
        want = want_fn()
        groups = (positions + G - 1) // G
        for sched in (one_after_another(groups, len(plan)), shuffled(groups, len(plan), rng)):
            mem = Memory(send, recv_bytes, scratch)
            run_plan_sliced(plan, mem, positions, G, sched)
            for r in range(N):
                got = mem.recv[r].view(NPT[DT[dtype]])
                assert _same(got, want[r]), (coll, algo, N, dtype, root, r)


def test_alltoall_plans_do_not_keep_positions():
    """AllToAll's rounds move blocks between offsets that differ by rank: the
    library leaves them to the other forms (operations without elem0)."""
    for algo in ("pairwise", "bruck", "ring"):
        plan, _ = get_plan("alltoall", algo, 8, 1024, "f32")
        assert any(op["elem0"] < 0 for ops in plan for op in ops), algo


def test_reduce_scatter_partials_flat_up_to_16_mib():
    """One partial slot per block and rank while the partials take at most
    16 MiB per rank (positional), two above (not); the scratch sizes say so."""
    N = 8
    for dtype, acc in (("f32", 4), ("bf16", 4)):
        limit = (16 << 20) // (N * acc)  # block size at which N blocks of partials take 16 MiB
        for rc, flat in ((limit, True), (limit + 8, False)):
            plan, scratch = get_plan("reduce_scatter", "ring", N, rc, dtype)
            mem = Memory([None] * N, [0] * N, scratch)
            assert (not position_places(plan, mem, _group(dtype))) == flat, (dtype, rc)
            per_rank = (N if flat else 2) * rc * acc
            assert scratch == N * ((per_rank + 255) // 256 * 256), (dtype, rc, scratch)


# ---- the library's choice of form, against these checks ------------------------------------
# vc_plan_form reports the form a call takes (host only).  The sliced form is
# predicted here from the plan alone, with the checks above: two or more
# steps, every operation keeping positions (one run; a copy from one source),
# each byte at one position, origins aligned, write-before-read, within the
# size limit and not in place (AllReduce excepted).  Its kernel derives
# operation ranges only where every origin is 0 (else "host ranges").

FORM_CASES = [("allreduce", a, 0) for a in ("ring", "rhd", "dbt", "mesh", "ring_hop", "fused")] + \
    [("reduce_scatter", a, 0) for a in ("ring", "fused")] + [("allgather", a, 0) for a in ("ring", "fused")] + \
    [("broadcast", a, 0) for a in ("binomial", "scatter_allgather", "fused")] + \
    [("broadcast", "pipe_chain", 3), ("broadcast", "pipe_tree", 3)] + \
    [("scatter", a, 0) for a in ("binomial", "fused")] + [("gather", a, 0) for a in ("binomial", "fused")] + \
    [("reduce", a, 0) for a in ("binomial", "fused")] + \
    [("alltoall", a, 0) for a in ("pairwise", "bruck", "ring", "fused")]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
@pytest.mark.parametrize("N", [2, 3, 5, 8])
def test_library_form_matches_the_independent_checks(N, dtype):
    import collective_communication_algorithms_virtual_gb300 as vc

    for coll, algo, k in FORM_CASES:
        for count in (1, 5, 64, 1000 + 3):
            for root in sorted({0, N - 1}):
                for inplace in (False, True):
                    if inplace and coll not in ("allreduce", "broadcast", "reduce"):
                        continue
                    sliced, hr = predict_sliced(coll, algo, N, count, dtype, root, inplace, k)
                    form, launches, got_hr = vc.vc_plan_form(coll, algo, N, count, dtype, root, inplace, k)
                    what = (coll, algo, N, count, dtype, root, inplace)
                    assert (form == "sliced") == sliced, (what, form)
                    if sliced:
                        assert launches == 1 and got_hr == hr, (what, launches, got_hr, hr)
                    elif coll == "alltoall":
                        assert form == "steps", (what, form)


def test_library_form_above_the_limit_and_for_merged_rounds():
    import collective_communication_algorithms_virtual_gb300 as vc

    # 8 Mi fp32 elements: 32 MiB carried per rank, above the 16 MiB default
    assert vc.vc_plan_form("allreduce", "ring", 8, 8 << 20, "f32") == ("steps", 14, False)
    assert vc.vc_plan_form("allreduce", "ring", 8, 4 << 20, "f32")[0] == "sliced"
    # Pairwise AllToAll: its rounds share one launch; Bruck runs a launch per step
    assert vc.vc_plan_form("alltoall", "pairwise", 8, 1024, "f32") == ("steps", 1, False)
    assert vc.vc_plan_form("alltoall", "bruck", 8, 128, "f32") == ("steps", 3, False)
    # 16 ranks: 16 rounds of 16 two-operand copies, over the 128 operations of
    # the large parameter block: two launches
    assert vc.vc_plan_form("alltoall", "pairwise", 16, 1024, "f32") == ("steps", 2, False)
    # Mesh AllReduce, 16 ranks, 20 MiB per rank: 15 reduce steps into the root,
    # then its 15 copies of the result, independent, in one launch
    assert vc.vc_plan_form("allreduce", "mesh", 16, 5 << 20, "f32") == ("steps", 16, False)
    # binomial Broadcast of 64 MiB over 5 ranks (above the slice limit): 0 -> 4
    # and 0 -> 2 touch different ranks (rank 4 forwards nothing), then 0 -> 1, 2 -> 3
    assert vc.vc_plan_form("broadcast", "binomial", 5, 16 << 20, "f32") == ("steps", 2, False)
    old = vc.vc_get_slice_limit()
    try:
        vc.vc_set_slice_limit(0)
        assert vc.vc_plan_form("allreduce", "ring", 8, 1024, "f32")[0] == "cluster"
    finally:
        vc.vc_set_slice_limit(old)


def test_library_form_of_degenerate_calls_and_bad_arguments():
    import ctypes

    import collective_communication_algorithms_virtual_gb300 as vc
    from collective_communication_algorithms_virtual_gb300.binding import (VC_ERR_INVALID_ARG, VC_ERR_UNSUPPORTED,
                                                                           VCError)

    # nothing to do: no launch (an empty message; one rank in place)
    assert vc.vc_plan_form("allreduce", "ring", 8, 0, "f32") == ("steps", 0, False)
    assert vc.vc_plan_form("allreduce", "ring", 1, 1000, "f32", inplace=True) == ("steps", 0, False)
    # one rank out of place: its copy, one launch
    assert vc.vc_plan_form("allreduce", "ring", 1, 1000, "f32") == ("steps", 1, False)
    # RHD folds 6 ranks into 4 and still keeps positions; DBT at 16 ranks, bf16: host ranges
    assert vc.vc_plan_form("allreduce", "rhd", 6, 1000, "f32") == ("sliced", 1, False)
    assert vc.vc_plan_form("allreduce", "dbt", 16, 1 << 20, "bf16") == ("sliced", 1, True)
    for args in (("allreduce", "ring", 0, 10), ("allreduce", "ring", 65, 10), ("broadcast", "binomial", 4, 10, "f32", 4)):
        with pytest.raises(VCError) as e:
            vc.vc_plan_form(*args)
        assert e.value.status == VC_ERR_INVALID_ARG, args
    with pytest.raises(VCError) as e:
        vc.vc_plan_form("reduce_scatter", "rhd", 4, 10, "f32")
    assert e.value.status == VC_ERR_UNSUPPORTED
    # chunk counts as vc_broadcast_pipelined takes them: 0 (the optimum) to 1024; ignored by other algorithms
    for k in (-1, 1025):
        with pytest.raises(VCError) as e:
            vc.vc_plan_form("broadcast", "pipe_tree", 8, 4096, "f32", 0, False, k)
        assert e.value.status == VC_ERR_INVALID_ARG
    assert vc.vc_plan_form("broadcast", "binomial", 8, 4096, "f32", 0, False, -1)[0] == "sliced"
    # in place as the calls allow it: AllReduce, Broadcast and Reduce only
    for coll, algo in (("allgather", "ring"), ("reduce_scatter", "ring"), ("scatter", "binomial"),
                       ("gather", "binomial"), ("alltoall", "pairwise")):
        with pytest.raises(VCError) as e:
            vc.vc_plan_form(coll, algo, 8, 64, "f32", 0, True)
        assert e.value.status == VC_ERR_INVALID_ARG, coll
    assert vc.vc_plan_form("reduce", "binomial", 8, 1000, "f32", 3, True)[0] == "cluster"
    # a null output through the C ABI itself
    L = vc.lib()
    i = ctypes.c_int()
    assert L.vc_plan_form(0, 1, 8, 1024, 0, 0, 0, 0, 0, None, ctypes.byref(i), ctypes.byref(i)) == VC_ERR_INVALID_ARG


def test_library_form_keeps_positions_below_2_pow_29():
    """The sliced kernels keep element and byte offsets in 32 bits: with no
    size limit, a call runs sliced only while its positions stay below 2^29
    (AllGather, Gather and Scatter: N x count of them)."""
    import collective_communication_algorithms_virtual_gb300 as vc

    old = vc.vc_get_slice_limit()
    try:
        vc.vc_set_slice_limit((1 << 64) - 1)
        assert vc.vc_plan_form("allgather", "ring", 8, 1 << 26, "f32")[0] == "sliced"  # last position 2^29 - 1
        assert vc.vc_plan_form("allgather", "ring", 8, (1 << 26) + 4, "f32") == ("steps", 7, False)
        assert vc.vc_plan_form("gather", "binomial", 8, (1 << 26) + 4, "f32")[0] == "steps"
        assert vc.vc_plan_form("allreduce", "ring", 8, (1 << 29) - 8, "f32")[0] == "sliced"
        assert vc.vc_plan_form("allreduce", "ring", 8, 1 << 29, "f32") == ("steps", 14, False)
        # ReduceScatter partials above 16 MiB per rank: two slots a rank, positional at 4 ranks, not at 8
        assert vc.vc_plan_form("reduce_scatter", "ring", 4, (1 << 27) - 4, "f32")[0] == "sliced"
        assert vc.vc_plan_form("reduce_scatter", "ring", 8, 1 << 26, "f32")[0] == "steps"
    finally:
        vc.vc_set_slice_limit(old)


def test_library_form_needs_the_description_in_shared_memory():
    """Past 18 ranks the Ring AllReduce's description (2(N-1) steps of N
    operations) with the sliced kernel's range and address tables outgrows a
    block's 96 KB of shared memory: the call keeps positions, but runs as one
    cluster, whose kernel holds the description alone, up to 21 ranks, and per
    step beyond."""
    import collective_communication_algorithms_virtual_gb300 as vc

    assert vc.vc_plan_form("allreduce", "ring", 18, 1024, "f32")[0] == "sliced"
    assert predict_sliced("allreduce", "ring", 19, 1024, "f32")[0]
    assert vc.vc_plan_form("allreduce", "ring", 19, 1024, "f32")[0] == "cluster"
    assert vc.vc_plan_form("allreduce", "ring", 21, 1024, "f32")[0] == "cluster"
    assert vc.vc_plan_form("allreduce", "ring", 22, 1024, "f32") == ("steps", 42, False)
    # the tree schedules' descriptions stay small up to 64 ranks
    assert vc.vc_plan_form("allreduce", "dbt", 64, 1024, "f32")[0] == "sliced"
