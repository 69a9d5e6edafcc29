"""Dataflow plans on the host: tiles and their dependency lists.

``vc_flow_describe`` cuts a call into the tiles a launch over the whole GPU
uses and lists, for each, the tiles of earlier steps it must follow.  Without
a GPU these tests check that

* every dependency points to an earlier step;
* every pair of tiles of different steps that touch the same bytes, one of
  them writing, is ordered through the lists (small plans, full closure);
* executing the tiles with numpy in random orders that respect the lists,
  and in the order that runs the latest steps first, gives the oracle's
  results bit for bit (in place included).
"""
import numpy as np
import pytest

import collective_communication_algorithms_virtual_gb300 as vc
from collective_communication_algorithms_virtual_gb300 import build as vcbuild
from oracle import schedules
from synthetic_inputs import int32_bits, rank_buffers

from .plan_replay import DT, ESZ, NPT, Memory, get_plan, run_tile, tile_order, tile_touches


@pytest.fixture(scope="module", autouse=True)
def built():
    vcbuild.build()
    yield


def _inputs(dtype, seed, N, n):
    kind = {"f32": "uniform_f32", "bf16": "uniform_bf16", "i32": "int32_bits"}[dtype]
    return rank_buffers(kind, seed, N, n)


def _replay(plan, tiles, deps, make_mem, want, read, ctx, orders=3):
    rng = np.random.default_rng(7)
    for k in range(orders + 1):
        mem = make_mem()
        for t in tile_order(tiles, deps, rng if k < orders else None):
            run_tile(plan, tiles[t], mem)
        for r, w in enumerate(want):
            got = read(mem, r)
            assert np.array_equal(got.view(np.uint8), np.ascontiguousarray(w).view(np.uint8)), (ctx, k, r)


def _closure(plan, tiles, deps, mem, ctx):
    """Every conflicting pair of tiles of different steps is ordered."""
    reach = [0] * len(tiles)
    for t, tile in enumerate(tiles):  # tiles are numbered in step order
        r = 0
        for d in deps[tile.dep_begin:tile.dep_end]:
            r |= reach[d] | (1 << d)
        reach[t] = r
    touches = [tile_touches(plan, t, mem) for t in tiles]
    for t in range(len(tiles)):
        for u in range(t):
            if tiles[u].step == tiles[t].step:
                continue
            conflict = any(a[0] == b[0] and a[1] < b[2] and b[1] < a[2] and (a[3] or b[3])
                           for a in touches[t] for b in touches[u])
            if conflict:
                assert (reach[t] >> u) & 1, (ctx, "unordered", u, t)


AR = [(N, c) for N in (1, 2, 3, 5, 8) for c in (1, 13, 1000, 4099)] + [(16, 3000)]


@pytest.mark.parametrize("workers", [1, 1000])
@pytest.mark.parametrize("N,count", AR)
@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
def test_allreduce_tiles_replay_to_oracle(N, count, dtype, workers):
    xs = _inputs(dtype, 700 + N, N, count)
    for algo in schedules.ALGOS["allreduce"]:
        res = schedules.allreduce(xs, algo, dtype)
        for inplace in (False, True):
            plan, scratch = get_plan("allreduce", algo, N, count, dtype, inplace=inplace and N == 1)
            tiles, deps = vc.vc_flow_describe("allreduce", algo, N, count, dtype, inplace=inplace, workers=workers)
            nb = count * ESZ[DT[dtype]]
            mk = lambda: Memory(xs, [nb] * N, scratch, inplace_ranks=range(N) if inplace else ())
            ctx = (algo, N, count, dtype, inplace, workers)
            if len(tiles) <= 400:
                _closure(plan, tiles, deps, mk(), ctx)
            _replay(plan, tiles, deps, mk, res.outputs, lambda m, r: m.recv[r].view(NPT[DT[dtype]]), ctx)


@pytest.mark.parametrize("N", [2, 3, 5, 8])
@pytest.mark.parametrize("dtype", ["bf16", "i32"])
def test_rs_ag_a2a_tiles_replay_to_oracle(N, dtype):
    for rc in (1, 5, 700):
        xs = _inputs(dtype, 800 + N, N, N * rc)
        es = ESZ[DT[dtype]]
        for coll, algos in (("reduce_scatter", schedules.ALGOS["reduce_scatter"]),
                            ("allgather", schedules.ALGOS["allgather"]),
                            ("alltoall", schedules.ALGOS["alltoall"])):
            for algo in algos:
                ins = [x[:rc] for x in xs] if coll == "allgather" else xs
                res = getattr(schedules, coll)(ins, algo, dtype)
                plan, scratch = get_plan(coll, algo, N, rc, dtype)
                tiles, deps = vc.vc_flow_describe(coll, algo, N, rc, dtype, workers=1000)
                out_bytes = rc * es if coll == "reduce_scatter" else N * rc * es
                mk = lambda: Memory(ins, [out_bytes] * N, scratch)
                ctx = (coll, algo, N, rc, dtype)
                if len(tiles) <= 400:
                    _closure(plan, tiles, deps, mk(), ctx)
                _replay(plan, tiles, deps, mk, res.outputs, lambda m, r: m.recv[r].view(NPT[DT[dtype]]), ctx)


@pytest.mark.parametrize("N", [2, 3, 5, 8, 16])
def test_rooted_tiles_replay_to_oracle(N):
    dtype = "i32"
    for root in sorted({0, N - 1}):
        for count in (1, 7, 3000):
            A = int32_bits(900 + root, N, count)
            send = [None] * N
            send[root] = A
            for algo in schedules.ALGOS["broadcast"] + ("pipe_chain", "pipe_tree"):
                for inplace in (False, True):
                    if algo.startswith("pipe"):
                        res = schedules.broadcast_pipelined(A, N, root, algo, dtype, 3, inplace=inplace)
                    else:
                        res = schedules.broadcast(A, N, root, algo, dtype, inplace=inplace)
                    plan, scratch = get_plan("broadcast", algo, N, count, dtype, root=root, inplace=inplace, nchunks=3)
                    tiles, deps = vc.vc_flow_describe("broadcast", algo, N, count, dtype, root, inplace, nchunks=3,
                                                      workers=1000)
                    mk = lambda: Memory(send, [count * 4] * N, scratch, inplace_ranks=[root] if inplace else ())
                    ctx = ("bcast", algo, N, root, count, inplace)
                    _replay(plan, tiles, deps, mk, res.outputs, lambda m, r: m.recv[r].view(np.int32), ctx, orders=2)
            S = int32_bits(950 + root, N, N * count)
            ssend = [None] * N
            ssend[root] = S
            for algo in schedules.ALGOS["scatter"]:
                res = schedules.scatter(S, N, root, algo, dtype)
                plan, scratch = get_plan("scatter", algo, N, count, dtype, root=root)
                tiles, deps = vc.vc_flow_describe("scatter", algo, N, count, dtype, root, workers=1000)
                mk = lambda: Memory(ssend, [count * 4] * N, scratch)
                _replay(plan, tiles, deps, mk, res.outputs, lambda m, r: m.recv[r].view(np.int32),
                        ("scatter", algo, N, root, count), orders=2)
            xs = _inputs("f32", 990 + root, N, count)
            for algo in schedules.ALGOS_EXTRA["reduce"]:
                for inplace in (False, True):
                    res = schedules.reduce(xs, root, algo, "f32", inplace=inplace)
                    plan, scratch = get_plan("reduce", algo, N, count, "f32", root=root, inplace=inplace)
                    tiles, deps = vc.vc_flow_describe("reduce", algo, N, count, "f32", root, inplace, workers=1000)
                    recv_bytes = [0] * N
                    recv_bytes[root] = count * 4
                    mk = lambda: Memory(xs, recv_bytes, scratch, inplace_ranks=[root] if inplace else ())
                    _replay(plan, tiles, deps, mk, res.outputs, lambda m, r: m.recv[root].view(np.float32),
                            ("reduce", algo, N, root, count, inplace), orders=2)
            for algo in schedules.ALGOS_EXTRA["gather"]:
                res = schedules.gather(xs, root, algo, "f32")
                plan, scratch = get_plan("gather", algo, N, count, "f32", root=root)
                tiles, deps = vc.vc_flow_describe("gather", algo, N, count, "f32", root, workers=1000)
                recv_bytes = [0] * N
                recv_bytes[root] = N * count * 4
                mk = lambda: Memory(xs, recv_bytes, scratch)
                _replay(plan, tiles, deps, mk, res.outputs, lambda m, r: m.recv[root].view(np.float32),
                        ("gather", algo, N, root, count), orders=2)


def test_tile_limit_is_reported():
    with pytest.raises(vc.VCError):
        vc.vc_flow_describe("allreduce", "ring", 8, 1 << 28, "f32", workers=760)
