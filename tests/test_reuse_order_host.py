"""The L2 reuse order, checked on the host against its definition.

vc_plan_exec_order reports the order the library executes a plan in.  With
the minimum forced to 0 (every step ordered) and for plans of every kind,
recomputed here from vc_plan_describe's operand ranges:
  - every step's operations are a permutation of the built ones;
  - step 0 walks forward and every later step opposite to the one before;
  - an operation is kept exactly when one of its destinations overlaps a
    source of the next step (never in the last step);
  - walked in the step's direction, the operations come in the order of
    when the previous step wrote their inputs, latest first (operations
    whose inputs it did not write last).
With the default minimum a small call is not reordered at all and a large
one is; with REUSE_ORDER_NEVER nothing is.
"""
import pytest

import collective_communication_algorithms_virtual_gb300 as vc

ESZ = {0: 4, 1: 2, 2: 4, 3: 2}


@pytest.fixture(autouse=True)
def _restore():
    old = vc.vc_get_reuse_order()
    yield
    vc.vc_set_reuse_order(old)


def _spans(entries):
    """(step, op) -> {"src": [...], "dst": [...]} of (buf, owner, lo, hi)."""
    out = {}
    for e in entries:
        last = e.byte_off + (e.nb - 1) * e.stride_bytes
        lo, hi = min(e.byte_off, last), max(e.byte_off, last) + e.n * ESZ[e.dtype]
        owner = -1 if e.buf == 2 else e.owner
        out.setdefault((e.step, e.op), {"src": [], "dst": []})["src" if e.role == 0 else "dst"].append((e.buf, owner, lo, hi))
    return out


def _overlap(a, b):
    return a[0] == b[0] and a[1] == b[1] and a[2] < b[3] and b[2] < a[3]


PLANS = [("allreduce", a, N, c, dt) for a in ("ring", "rhd", "dbt", "mesh") for N in (4, 8) for c in (1000, 4096)
         for dt in ("f32", "bf16")] + \
        [("allreduce", "ring", 5, 333, "f16"), ("allreduce", "dbt", 6, 777, "f32")] + \
        [("reduce_scatter", "ring", N, 513, dt) for N in (3, 8) for dt in ("f32", "bf16")] + \
        [("allgather", "ring", N, 100, "i32") for N in (3, 8)] + \
        [("broadcast", a, N, 1000, "i32") for a in ("binomial", "scatter_allgather") for N in (5, 8)] + \
        [("alltoall", a, N, 64, "bf16") for a in ("pairwise", "bruck", "ring") for N in (4, 7)]


@pytest.mark.parametrize("coll,algo,N,count,dtype", PLANS)
def test_forced_order_follows_its_definition(coll, algo, N, count, dtype):
    vc.vc_set_reuse_order(0)
    entries, _, nsteps = vc.vc_plan_describe(coll, algo, N, count, dtype)
    order, keep, rev = vc.vc_plan_exec_order(coll, algo, N, count, dtype)
    sp = _spans(entries)
    nops = [len(o) for o in order]
    assert len(order) == nsteps == len(rev)
    for s in range(nsteps):
        assert sorted(order[s]) == list(range(nops[s])), (s, order[s])
    assert rev[0] == 0
    for s in range(1, nsteps):
        assert rev[s] == 1 - rev[s - 1], (s, rev)
    for s in range(nsteps):
        for k, i in enumerate(order[s]):
            want = s + 1 < nsteps and any(_overlap(d, r) for d in sp[(s, i)]["dst"]
                                          for j in range(nops[s + 1]) for r in sp[(s + 1, j)]["src"])
            assert keep[s][k] == int(want), (coll, algo, s, i)
    for s in range(1, nsteps):
        prev = order[s - 1]
        # when each operation of the previous step ran, in its walk direction
        when_prev = {i: (len(prev) - 1 - k if rev[s - 1] else k) for k, i in enumerate(prev)}
        def when(i):
            w = -1
            for j in range(nops[s - 1]):
                if any(_overlap(d, r) for d in sp[(s - 1, j)]["dst"] for r in sp[(s, i)]["src"]):
                    w = max(w, when_prev[j])
            return w
        walk = order[s][::-1] if rev[s] else order[s]
        ws = [when(i) for i in walk]
        assert ws == sorted(ws, reverse=True), (coll, algo, s, ws)


def test_default_minimum_orders_large_calls_only():
    vc.vc_set_reuse_order(vc.vc_get_reuse_order())  # the default, restored after
    assert vc.vc_get_reuse_order() == 16 << 20
    order, keep, rev = vc.vc_plan_exec_order("allreduce", "ring", 8, 1 << 18, "f32")  # 1 MiB per rank
    assert all(o == sorted(o) for o in order) and not any(map(any, keep)) and not any(rev)
    order, keep, rev = vc.vc_plan_exec_order("allreduce", "ring", 8, 64 << 20, "f32")  # 256 MiB per rank
    assert rev == [0] + [1, 0] * 6 + [1]
    assert all(all(k) for k in keep[:-1]) and not any(keep[-1])


def test_never_leaves_the_built_order():
    vc.vc_set_reuse_order(vc.REUSE_ORDER_NEVER)
    order, keep, rev = vc.vc_plan_exec_order("allreduce", "rhd", 8, 64 << 20, "bf16")
    assert all(o == list(range(len(o))) for o in order) and not any(map(any, keep)) and not any(rev)
