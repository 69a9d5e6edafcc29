"""Pipelined Broadcasts, Gather and Tree Reduce on the CPU: the oracle
against the pages, and the library's plans replayed against the oracle."""
import numpy as np
import pytest

from oracle import cost_model as cm
from oracle import numerics, schedules, selection
from synthetic_inputs import int32_bits, rank_buffers, small_ints_f32

from .plan_replay import ESZ, Memory, get_plan, hazards, oracle_transfers, run_plan, transfers

import collective_communication_algorithms_virtual_gb300 as vc


@pytest.fixture(scope="module", autouse=True)
def _built():
    from collective_communication_algorithms_virtual_gb300 import build

    build.build()


# ---------------------------------------------------------------------------
# oracle pins
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("N", [2, 3, 5, 8, 16])
@pytest.mark.parametrize("k", [1, 2, 4, 7])
def test_pipelined_step_counts_and_formula(N, k):
    """N + k - 2 steps along the chain, ceil(log2 N) + k - 1 down the tree, each
    moving one chunk of M/k: summing (alpha + largest message / beta) over the
    log's steps gives eqs. pipe-chain-bcast and pipe-tree-bcast exactly."""
    count = k * 16 * 4
    M = count * 4
    A = int32_bits(1, 0, count)
    a, b = 5e-6, 450e9
    for algo, steps, f in (("pipe_chain", N + k - 2, cm.t_pipe_chain_bcast),
                           ("pipe_tree", cm.ceil_log2(N) + k - 1, cm.t_pipe_tree_bcast)):
        res = schedules.broadcast_pipelined(A, N, 0, algo, "i32", k)
        assert res.nsteps == steps, (algo, res.nsteps)
        assert all(t.nbytes == M // k for t in res.log.records)
        per = res.log.max_message_bytes_per_step()
        assert sum(a + per[s] / b for s in res.log.steps()) == pytest.approx(f(N, M, a, b, k), rel=1e-12)
        for o in res.outputs:
            assert np.array_equal(o, A)


def test_pipelined_k1_reduces_to_chain_and_binomial(golden):
    A = np.arange(64, dtype=np.int32)
    chain = schedules.broadcast_pipelined(A, 8, 0, "pipe_chain", "i32", 1)
    assert chain.log.table() == [(s, s, s + 1) for s in range(7)]   # eq. chain-bcast: N-1 steps
    assert cm.t_chain_bcast(8, 256, 5e-6, 450e9) == pytest.approx(cm.t_pipe_chain_bcast(8, 256, 5e-6, 450e9, 1))
    tree = schedules.broadcast_pipelined(A, 8, 0, "pipe_tree", "i32", 1)
    want = sorted((int(s) - 1, int(a), int(b)) for s, a, b in golden("binomial_broadcast_n8.txt"))
    assert tree.log.table() == want


def test_gather_is_the_reversed_scatter_table(golden):
    """Reversing the 8-node Scatter table's data flow (duality section): step 1
    1->0, 3->2, 5->4, 7->6 (M/8 each); step 2 2->0 [A2,A3], 6->4 [A6,A7] (M/4);
    step 3 4->0 [A4..A7] (M/2)."""
    rows = golden("binomial_scatter_n8.txt")
    rc = 16
    M = 8 * rc * 4
    xs = [np.full(rc, r, dtype=np.int32) for r in range(8)]
    res = schedules.gather(xs, 0, "binomial", "i32")
    got = sorted((t.step, t.src, t.dst, tuple(sorted(t.chunks)), t.nbytes) for t in res.log.records)
    want = sorted((3 - int(s), int(b), int(a), tuple(int(c) for c in ch.split(",")), M // int(den))
                  for s, a, b, ch, den in rows)
    assert got == want
    assert res.log.bandwidth_bytes() == (8 - 1) * M // 8
    assert cm.t_gather(8, M, 5e-6, 450e9) == cm.t_binomial_scatter(8, M, 5e-6, 450e9)
    assert np.array_equal(res.outputs[0], np.repeat(np.arange(8, dtype=np.int32), rc))


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 7, 8, 13])
def test_gather_reduce_bruteforce(N):
    for root in sorted({0, N - 1, N // 2}):
        for rc in (0, 1, 5, 33):
            xs = [int32_bits(2, r, rc) for r in range(N)]
            for algo in schedules.ALGOS_EXTRA["gather"]:
                out = schedules.gather(xs, root, algo, "i32").outputs[0]
                assert np.array_equal(out, np.concatenate(xs)), (algo, N, root, rc)
            fs = [small_ints_f32(3, r, rc) for r in range(N)]
            exact = np.sum(np.stack([f.astype(np.int64) for f in fs]), axis=0).astype(np.float32) if rc else fs[0]
            wrap = (np.sum(np.stack([x.astype(np.int64) for x in xs]), axis=0) & 0xFFFFFFFF).astype(np.uint32).view(np.int32) if rc else xs[0]
            for algo in schedules.ALGOS_EXTRA["reduce"]:
                assert np.array_equal(schedules.reduce(fs, root, algo, "f32").outputs[0], exact), (algo, N, root)
                assert np.array_equal(schedules.reduce(xs, root, algo, "i32").outputs[0], wrap), (algo, N, root)


def test_tree_reduce_levels_and_association():
    """log2 N steps, each carrying the whole message (eq. model-algo-reduce-tree);
    the association is the balanced tree over adjacent ranks counted from the
    root: with x = (0, 2^24, 1, -2^24) at root 0 that is (0 + 2^24) + (1 - 2^24)
    = 1, while the rank-order fold gives ((0 + 2^24) + 1) - 2^24 = 0 (2^24 + 1
    rounds to 2^24).  From root 1 the relative order is (x1 + x2) + (x3 + x0):
    (2^24 + 1) + (-2^24 + 0) = 0."""
    xs = [np.full(8, v, dtype=np.float32) for v in (0.0, 2.0 ** 24, 1.0, -(2.0 ** 24))]
    assert schedules.reduce(xs, 0, "binomial", "f32").outputs[0][0] == 1.0
    assert schedules.reduce(xs, 0, "fused", "f32").outputs[0][0] == 0.0
    assert schedules.reduce(xs, 1, "binomial", "f32").outputs[0][0] == 0.0
    N, count = 8, 64
    res = schedules.reduce(rank_buffers("uniform_f32", 4, N, count), 0, "binomial", "f32")
    assert res.nsteps == 3 and res.log.bandwidth_bytes() == 3 * count * 4
    assert all(t.reduce for t in res.log.records)


def test_bf16_reduce_rounds_once():
    N, count = 8, 2048
    xs = rank_buffers("normal_bf16", 5, N, count, sigma=1e-3)
    fused = schedules.reduce(xs, 3, "fused", "bf16").outputs[0]
    direct = numerics.bf16_to_f32(xs[0]).copy()
    for x in xs[1:]:
        direct = direct + numerics.bf16_to_f32(x)
    assert np.array_equal(fused, numerics.f32_to_bf16(direct))


# ---------------------------------------------------------------------------
# the library's plans replayed against the oracle
# ---------------------------------------------------------------------------

def _check(plan, mem, want, got):
    assert not hazards(plan, mem)
    assert np.array_equal(np.ascontiguousarray(got).view(np.uint8), np.ascontiguousarray(want).view(np.uint8))


@pytest.mark.parametrize("N", [1, 2, 3, 5, 8, 11, 16])
def test_pipelined_broadcast_plans_replay(N):
    for root in sorted({0, N - 1}):
        for count in (1, 37, 640):
            A = int32_bits(6, root, count)
            for algo in ("pipe_chain", "pipe_tree"):
                for k in (1, 3, 8):
                    for inplace in (False, True):
                        res = schedules.broadcast_pipelined(A, N, root, algo, "i32", k, inplace=inplace)
                        plan, scratch = get_plan("broadcast", algo, N, count, "i32", root, inplace, k)
                        send = [None] * N
                        send[root] = A
                        mem = Memory(send, [count * 4] * N, scratch, inplace_ranks=[root] if inplace else ())
                        run_plan(plan, mem)
                        for r in range(N):
                            _check(plan, mem, res.outputs[r], mem.recv[r].view(np.int32))
                        assert transfers(plan) == oracle_transfers(res.log), (algo, N, root, count, k)
                        assert sum(e.n * e.nb * 4 for e in vc.vc_plan_describe(
                            "broadcast", algo, N, count, "i32", root, inplace, k)[0]) == res.hbm_bytes


@pytest.mark.parametrize("N", [1, 2, 3, 5, 8, 11, 16])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
def test_gather_reduce_plans_replay(N, dtype):
    kind = {"f32": "uniform_f32", "bf16": "uniform_bf16", "i32": "int32_bits"}[dtype]
    es = ESZ[{"f32": 0, "bf16": 1, "i32": 2}[dtype]]
    npt = {"f32": np.float32, "bf16": np.uint16, "i32": np.int32}[dtype]
    for root in sorted({0, N - 1, N // 2}):
        for rc in (1, 13, 100):
            xs = rank_buffers(kind, 7 + root, N, rc)
            for algo in schedules.ALGOS_EXTRA["gather"]:
                res = schedules.gather(xs, root, algo, dtype)
                plan, scratch = get_plan("gather", algo, N, rc, dtype, root)
                sizes = [N * rc * es if r == root else 0 for r in range(N)]
                mem = Memory(xs, sizes, scratch)
                run_plan(plan, mem)
                _check(plan, mem, res.outputs[0], mem.recv[root].view(npt))
                assert transfers(plan) == oracle_transfers(res.log), ("gather", algo, N, root)
            for algo in schedules.ALGOS_EXTRA["reduce"]:
                for inplace in (False, True):
                    res = schedules.reduce(xs, root, algo, dtype, inplace=inplace)
                    plan, scratch = get_plan("reduce", algo, N, rc, dtype, root, inplace)
                    sizes = [rc * es if r == root else 0 for r in range(N)]
                    mem = Memory(xs, sizes, scratch, inplace_ranks=[root] if inplace else ())
                    run_plan(plan, mem)
                    _check(plan, mem, res.outputs[0], mem.recv[root].view(npt))
                    assert transfers(plan) == oracle_transfers(res.log), ("reduce", algo, N, root)
                    assert sum(e.n * e.nb * ESZ[e.dtype] for e in vc.vc_plan_describe(
                        "reduce", algo, N, rc, dtype, root, inplace)[0]) == res.hbm_bytes


# ---------------------------------------------------------------------------
# AUTO over the new collectives
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("policy", ["link", "hbm"])
def test_selection_new_collectives(policy):
    try:
        for alpha, beta in ((5e-6, 450e9), (1.9e-6, 6.6e12)):
            vc.vc_set_cost_model(policy, alpha, beta)
            for N in (2, 5, 8, 16):
                for coll in ("broadcast", "gather", "reduce"):
                    for count in (64, 1 << 14, 1 << 18):
                        got, t = vc.vc_select_algo(coll, N, count, "f32")
                        if policy == "link":
                            want, tw = selection.select_link(coll, N, count, "f32", alpha, beta)
                        else:
                            want, tw = selection.select_hbm(coll, N, count, "f32", alpha, beta)
                        assert got == want, (policy, coll, N, count, got, want)
                        assert t == pytest.approx(tw, rel=1e-12)
    finally:
        vc.vc_set_cost_model("hbm")
