"""Every collective schedule of the pages as a message-passing simulation.

Model: N ranks, each holding its own numpy arrays.  A step is a set of
messages; every payload is copied from its sender before any message of the
step is delivered, so all messages of one step travel at the same time (the
alpha-beta model of the [Latency-formula page], section "本文是集合通信算法的
alpha-beta 延迟公式手册").  A receiver either stores a payload (copy) or adds it
to its own data (reduce), in the order the messages are listed.  Each schedule
returns its outputs, a ``TransferLog`` of every message, and its algorithmic
HBM bytes: what one execution on a single device must read and write when the
N ranks are N buffers in one memory (see ``_Bytes``).

Arithmetic is that of ``oracle.numerics`` (fp32 RNE adds in the schedule's own
association, int32 wrap-around, bf16 widened to fp32 and rounded once at the
end).

Parity status: every schedule is pinned by brute force on integer data (any
association is exact there), by the definitions in ``oracle.orders`` on order
witnesses, by the printed tables and formulas of the pages (binomial tables,
step counts, bandwidth terms), and by library routines for the data-movement
collectives.  The association of the Double Binary Tree and the block route of
Bruck rest on readings (see their docstrings); their data results are pinned
by the definitions.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable

import numpy as np

from .numerics import ACC_ESIZE, ESIZE, combine, narrow, storage_dtype, widen
from .partition import chunk_range
from .translog import TransferLog

ALGOS = {
    "allreduce": ("fused", "ring", "rhd", "dbt", "mesh", "ring_hop"),
    "reduce_scatter": ("fused", "ring"),
    "allgather": ("fused", "ring"),
    "broadcast": ("fused", "binomial", "scatter_allgather"),
    "scatter": ("fused", "binomial"),
    "alltoall": ("fused", "pairwise", "bruck", "ring"),
}

# Test-only fault injection: {"drop_step": s} loses every message of step s,
# {"dup_step": s} delivers every message of step s twice.  Never set outside tests.
_FAULT: dict | None = None


class Unsupported(ValueError):
    """The schedule is not defined for these arguments (e.g. RHD with N not a power of 2)."""


@dataclass
class Result:
    outputs: list
    log: TransferLog
    hbm_bytes: int
    local_steps: int = 0  # steps that only copy within a rank (no message)

    @property
    def nsteps(self) -> int:
        """Steps that carry messages: the coefficient of alpha."""
        return len(self.log.steps())

    @property
    def launch_steps(self) -> int:
        """Steps that move any data on one device (messages or local copies)."""
        if self.nsteps == 0:
            return 1 if self.hbm_bytes > 0 else 0
        return self.nsteps + self.local_steps


@dataclass
class _Msg:
    src: int
    dst: int
    n: int
    reduce: bool
    esize: int
    payload: object
    deliver: Callable
    phase: str = ""
    src_off: int | None = None
    dst_off: int | None = None
    chunks: tuple = ()


def _run_step(log: TransferLog, step: int, msgs: list) -> None:
    if _FAULT and _FAULT.get("drop_step") == step:
        return
    for m in msgs:
        log.add(step=step, phase=m.phase, src=m.src, dst=m.dst, n=m.n, reduce=m.reduce,
                esize=m.esize, src_off=m.src_off, dst_off=m.dst_off, chunks=m.chunks)
        m.deliver(m.payload)
        if _FAULT and _FAULT.get("dup_step") == step:
            m.deliver(m.payload)


def _reduce_into(buf: np.ndarray, lo: int, hi: int, op: str = "sum"):
    def f(p):
        buf[lo:hi] = combine(buf[lo:hi], p, op)
    return f


def _store_into(buf: np.ndarray, lo: int, hi: int):
    def f(p):
        buf[lo:hi] = p
    return f


class _Bytes:
    """Algorithmic HBM bytes: every operand read and every result written once
    per step, with storage sizes e_in (inputs), e_acc (partial sums: fp32 for
    bf16 inputs) and e_out (results)."""

    def __init__(self, dtype: str):
        self.e_in = ESIZE[dtype]
        self.e_out = ESIZE[dtype]
        self.e_acc = ACC_ESIZE[dtype]
        self.total = 0

    def rw(self, n: int, *sizes: int) -> None:
        self.total += n * sum(sizes)


def _ceil_log2(n: int) -> int:
    return (n - 1).bit_length()


def _check_same(inputs, dtype):
    want = storage_dtype(dtype)
    assert len(inputs) >= 1
    n = len(inputs[0])
    for x in inputs:
        assert x.dtype == want and x.ndim == 1 and len(x) == n, (x.dtype, want, x.shape)
    return len(inputs), n


# --------------------------------------------------------------------------
# AllReduce
# --------------------------------------------------------------------------

def allreduce(inputs, algo: str, dtype: str, inplace: bool = False, op: str = "sum") -> Result:
    """out_r = elementwise sum of all ranks' inputs, on every rank
    ([Latency-formula page], section "Ring AllReduce"; [hccl article] section
    "集合通信vs点对点" -- every rank ends with the same reduced data)."""
    N, count = _check_same(inputs, dtype)
    if algo not in ALGOS["allreduce"]:
        raise Unsupported(f"allreduce/{algo}")
    if N == 1 and inplace:  # one rank, in place: the result is already there
        return Result([np.array(inputs[0], copy=True)], TransferLog(), 0)
    if algo == "fused":
        return _allreduce_fused(inputs, dtype, op)
    if algo == "ring":
        return _allreduce_ring(inputs, dtype, op)
    if algo == "rhd":
        return _allreduce_rhd(inputs, dtype, op)
    if algo == "dbt":
        return _allreduce_dbt(inputs, dtype, op)
    if algo == "mesh":
        return _allreduce_mesh(inputs, dtype, op)
    if algo == "ring_hop":
        return _allreduce_ring(inputs, dtype, op, round_each_hop=True)
    raise Unsupported(f"allreduce/{algo}")


def _self_copy_result(inputs, dtype, bm: _Bytes):
    bm.rw(len(inputs[0]), bm.e_in, bm.e_out)
    return [np.array(x, copy=True) for x in inputs]


def _allreduce_fused(inputs, dtype, op="sum"):
    """One pass: every rank's element e is read once and summed in rank order,
    ((x0 + x1) + x2) + ... -- the order in which the Mesh root of the
    [hccl article] (section "Mesh算法：全连接广播") folds ranks 0..N-1 into its
    buffer -- and the sum is written to all N outputs.  Every rank "sends" its
    data to every other rank in the single step."""
    N, count = len(inputs), len(inputs[0])
    bm = _Bytes(dtype)
    log = TransferLog()
    acc = widen(inputs[0], dtype)
    for q in range(1, N):
        acc = combine(acc, widen(inputs[q], dtype), op)
    if N > 1:
        for q in range(N):
            for r in range(N):
                if q != r:
                    log.add(step=0, phase="fused", src=q, dst=r, n=count, reduce=True,
                            esize=bm.e_in, src_off=0, dst_off=0)
    bm.rw(count, *([bm.e_in] * N), *([bm.e_out] * N))
    out = narrow(acc, dtype)
    return Result([out.copy() for _ in range(N)], log, bm.total)


def _allreduce_mesh(inputs, dtype, op="sum"):
    """Mesh AllReduce of the [hccl article] (section "Mesh算法：全连接广播"),
    taken step for step from its code: the root receives every other rank's
    buffer in rank order and folds each into its own (N-1 steps of one
    message), then sends the result to every other rank in rank order (N-1
    steps).  The article's AllReduce has a root argument; an AllReduce call
    here has none, and the reading taken is root 0.  The fold is the rank
    order ((x0 + x1) + x2) + ..., the fused kernel's."""
    N, count = len(inputs), len(inputs[0])
    bm = _Bytes(dtype)
    log = TransferLog()
    if N == 1:
        return Result(_self_copy_result(inputs, dtype, bm), log, bm.total)
    acc = [widen(x, dtype) for x in inputs]
    root, step = 0, 0
    others = [i for i in range(N) if i != root]
    for t, i in enumerate(others):
        wire_own = bm.e_in if t == 0 else bm.e_acc
        _run_step(log, step, [_Msg(src=i, dst=root, n=count, reduce=True, esize=bm.e_in,
                                   payload=acc[i].copy(), deliver=_reduce_into(acc[root], 0, count, op),
                                   phase="mesh_reduce", src_off=0, dst_off=0)])
        bm.rw(count, wire_own, bm.e_in, bm.e_out if t == N - 2 else bm.e_acc)
        step += 1
    for i in others:
        _run_step(log, step, [_Msg(src=root, dst=i, n=count, reduce=False, esize=bm.e_out,
                                   payload=acc[root].copy(), deliver=_store_into(acc[i], 0, count),
                                   phase="mesh_bcast", src_off=0, dst_off=0)])
        bm.rw(count, bm.e_out, bm.e_out)
        step += 1
    return Result([narrow(a, dtype) for a in acc], log, bm.total)


def _allreduce_ring(inputs, dtype, op="sum", round_each_hop=False):
    """Ring AllReduce = Ring ReduceScatter (N-1 steps) then Ring AllGather
    (N-1 steps) ([hccl article] section "Ring算法：环形流水线传输";
    [Latency-formula page] eqs. model-algo-ring-rs, -ag, -ar).

    ReduceScatter step s: rank r sends chunk (r - s) mod N to rank r + 1 and
    adds chunk (r - s - 1) mod N received from rank r - 1 to its own copy.
    After N - 1 steps rank r holds chunk (r + 1) mod N fully reduced, summed in
    the order x_c + x_{c+1} + ... + x_{c+N-1} for chunk c.

    AllGather step s: rank r forwards the chunk it obtained in the previous
    step, chunk (r + 1 - s) mod N, and stores chunk (r - s) mod N from rank
    r - 1.  (The article's pseudo-code prints the AllGather indices as r+s+1 /
    r+s, which agree with this only at s = 0: from s = 1 on they would forward
    chunks not yet received and never deliver chunk r - 1.  The reading taken
    is the forwarding the article's prose and the formula page describe.)

    bf16 / fp16: partial sums travel and are stored as fp32; the last
    ReduceScatter step writes the rounded result, which the AllGather copies.
    ``round_each_hop`` (algorithm "ring_hop"): every hop instead rounds the
    partial sum to the data type and stores it there, as a ring that sends
    its partials in the data type would -- half the partial traffic of
    16-bit data, one rounding per hop; for fp32 and int32 nothing changes."""
    N, count = len(inputs), len(inputs[0])
    e = ESIZE[dtype]
    bm = _Bytes(dtype)
    log = TransferLog()
    if N == 1:
        return Result(_self_copy_result(inputs, dtype, bm), log, bm.total)
    acc = [widen(x, dtype) for x in inputs]
    e_part = bm.e_in if round_each_hop else bm.e_acc

    def reduce_and_round(buf, lo, hi):
        plain = _reduce_into(buf, lo, hi, op)
        if not round_each_hop:
            return plain

        def f(p):
            plain(p)
            buf[lo:hi] = widen(narrow(buf[lo:hi], dtype), dtype)
        return f

    step = 0
    for s in range(N - 1):
        msgs = []
        for r in range(N):
            c = (r - s) % N
            lo, hi = chunk_range(c, count, N, e)
            dst = (r + 1) % N
            wire = bm.e_in if s == 0 else e_part
            msgs.append(_Msg(src=r, dst=dst, n=hi - lo, reduce=True, esize=wire,
                             payload=acc[r][lo:hi].copy(), deliver=reduce_and_round(acc[dst], lo, hi),
                             phase="rs", src_off=lo, dst_off=lo, chunks=(c,)))
            bm.rw(hi - lo, bm.e_in, wire, bm.e_out if s == N - 2 else e_part)
        _run_step(log, step, msgs)
        step += 1
    for s in range(N - 1):
        msgs = []
        for r in range(N):
            c = (r + 1 - s) % N
            lo, hi = chunk_range(c, count, N, e)
            dst = (r + 1) % N
            msgs.append(_Msg(src=r, dst=dst, n=hi - lo, reduce=False, esize=bm.e_out,
                             payload=acc[r][lo:hi].copy(), deliver=_store_into(acc[dst], lo, hi),
                             phase="ag", src_off=lo, dst_off=lo, chunks=(c,)))
            bm.rw(hi - lo, bm.e_out, bm.e_out)
        _run_step(log, step, msgs)
        step += 1
    return Result([narrow(a, dtype) for a in acc], log, bm.total)


def rhd_virtual_ranks(N: int):
    """(P, r, real): RHD runs on P = 2**floor(log2 N) virtual ranks; the first
    2r real ranks (r = N - P) fold in pairwise beforehand, virtual rank v < r
    being real rank 2v and v >= r real rank v + r."""
    P = 1 << (N.bit_length() - 1)
    r = N - P
    return P, r, [2 * v if v < r else v + r for v in range(P)]


def _allreduce_rhd(inputs, dtype, op="sum"):
    """Recursive Halving-Doubling (Rabenseifner) AllReduce ([Latency-formula
    page] section "Recursive Halving-Doubling", eqs. model-algo-rhd-rs, -ag,
    -ar, which ask for N a power of 2).

    Halving round k = 0 .. log2(P)-1: virtual rank v pairs with v XOR 2**k;
    both hold the same segment (a run of chunks); the one whose bit k is 0
    keeps the lower half, the other the upper half; each sends the half it
    gives up and adds the half it keeps.  Round k moves M / 2**(k+1).
    Afterwards rank v holds chunk bitreverse(v) fully reduced; every element
    was summed as the balanced tree over adjacent rank pairs,
    ((x0+x1)+(x2+x3)) + ....  Doubling: the reverse process; round j pairs v
    with v XOR 2**(log2P-1-j), each sends its whole segment (M * 2**j / P) and
    stores the partner's.  Which half is kept and the order of the doubling
    distances are readings; the reduced values do not depend on them.

    N not a power of 2 (the page leaves it out; the reading taken is
    Rabenseifner's own fold-in): with P the largest power of 2 below N and
    r = N - P, odd rank 2i+1 first hands its whole buffer to rank 2i (i < r),
    which adds it; RHD runs on the P remaining ranks; rank 2i finally hands
    the whole result back to 2i+1.  For N a power of 2 there is no such step."""
    N, count = len(inputs), len(inputs[0])
    e = ESIZE[dtype]
    bm = _Bytes(dtype)
    log = TransferLog()
    if N == 1:
        return Result(_self_copy_result(inputs, dtype, bm), log, bm.total)
    P, rr, real = rhd_virtual_ranks(N)
    L = P.bit_length() - 1
    acc = [widen(x, dtype) for x in inputs]
    folded = set()  # real ranks holding a partial sum before the halving
    step = 0
    if rr:
        msgs = []
        for i in range(rr):
            msgs.append(_Msg(src=2 * i + 1, dst=2 * i, n=count, reduce=True, esize=bm.e_in,
                             payload=acc[2 * i + 1].copy(), deliver=_reduce_into(acc[2 * i], 0, count, op),
                             phase="fold", src_off=0, dst_off=0))
            bm.rw(count, bm.e_in, bm.e_in, bm.e_acc)
            folded.add(2 * i)
        _run_step(log, step, msgs)
        step += 1
    seg = [(0, P)] * P  # chunk index range [c0, c1) each virtual rank is responsible for

    def elems(c0, c1):
        return chunk_range(c0, count, P, e)[0], chunk_range(c1 - 1, count, P, e)[1]

    for k in range(L):
        msgs = []
        new_seg = list(seg)
        for v in range(P):
            w = v ^ (1 << k)
            c0, c1 = seg[v]
            h = (c1 - c0) // 2
            if (v >> k) & 1 == 0:
                keep, give = (c0, c0 + h), (c0 + h, c1)
            else:
                keep, give = (c0 + h, c1), (c0, c0 + h)
            new_seg[v] = keep
            lo, hi = elems(*give)
            wire = bm.e_acc if (k > 0 or real[v] in folded) else bm.e_in
            msgs.append(_Msg(src=real[v], dst=real[w], n=hi - lo, reduce=True, esize=wire,
                             payload=acc[real[v]][lo:hi].copy(), deliver=_reduce_into(acc[real[w]], lo, hi, op),
                             phase="halving", src_off=lo, dst_off=lo,
                             chunks=tuple(range(*give))))
            own = bm.e_acc if (k > 0 or real[w] in folded) else bm.e_in
            bm.rw(hi - lo, own, wire, bm.e_out if k == L - 1 else bm.e_acc)
        _run_step(log, step, msgs)
        seg = new_seg
        step += 1
    for j in range(L):
        d = 1 << (L - 1 - j)
        msgs = []
        new_seg = list(seg)
        for v in range(P):
            w = v ^ d
            c0, c1 = seg[v]
            lo, hi = elems(c0, c1)
            msgs.append(_Msg(src=real[v], dst=real[w], n=hi - lo, reduce=False, esize=bm.e_out,
                             payload=acc[real[v]][lo:hi].copy(), deliver=_store_into(acc[real[w]], lo, hi),
                             phase="doubling", src_off=lo, dst_off=lo,
                             chunks=tuple(range(c0, c1))))
            bm.rw(hi - lo, bm.e_out, bm.e_out)
            pc0, pc1 = seg[w]
            new_seg[v] = (min(c0, pc0), max(c1, pc1))
        _run_step(log, step, msgs)
        seg = new_seg
        step += 1
    if rr:
        msgs = []
        for i in range(rr):
            msgs.append(_Msg(src=2 * i, dst=2 * i + 1, n=count, reduce=False, esize=bm.e_out,
                             payload=acc[2 * i].copy(), deliver=_store_into(acc[2 * i + 1], 0, count),
                             phase="unfold", src_off=0, dst_off=0))
            bm.rw(count, bm.e_out, bm.e_out)
        _run_step(log, step, msgs)
    return Result([narrow(a, dtype) for a in acc], log, bm.total)


def dbt_trees(N: int, count: int, esize: int):
    """The two complementary binary trees and the half of the data each one
    carries.  Tree A: heap numbering on the ranks, parent (i-1)/2, children
    2i+1 and 2i+2 ([hccl article] section "Tree算法：层次化规约").  Tree B:
    the mirror, heap index i on rank N-1-i; every rank is an interior node in
    at most one of the two ([Latency-formula page] section "Double Binary
    Tree" asks for two trees with different parent/child relations; how to
    build them is a reading).  Tree A reduces chunk 0 of a two-way split of
    the buffer, tree B chunk 1 (the partition rule of ``oracle.partition``)."""
    a = chunk_range(0, count, 2, esize)
    b = chunk_range(1, count, 2, esize)
    return [("A", (lambda i: i), a), ("B", (lambda i, N=N: N - 1 - i), b)]


def heap_depth(i: int) -> int:
    return (i + 1).bit_length() - 1


def _allreduce_dbt(inputs, dtype, op="sum"):
    """Double Binary Tree AllReduce ([Latency-formula page] section "Double
    Binary Tree", eq. model-algo-dbt-ar): each tree reduces its half up to the
    root (one tree level per step, deepest first) and broadcasts it back down
    (root first).  A node adds its left child's subtree sum, then its right
    child's, to its own value: S(i) = (x_i + S(2i+1)) + S(2i+2), as in the
    [hccl article] Tree pseudo-code.  The two trees run their levels in the
    same steps.  (The article's pseudo-code broadcasts its receive buffer,
    which at the root holds the last child's data; the reading taken is that
    the root broadcasts its sum.)"""
    N, count = len(inputs), len(inputs[0])
    e = ESIZE[dtype]
    bm = _Bytes(dtype)
    log = TransferLog()
    if N == 1:
        return Result(_self_copy_result(inputs, dtype, bm), log, bm.total)
    acc = [widen(x, dtype) for x in inputs]
    D = heap_depth(N - 1)
    trees = dbt_trees(N, count, e)
    step = 0
    for t in range(D):
        depth = D - 1 - t
        msgs = []
        for name, rank_of, (lo, hi) in trees:
            for i in range(N):
                if heap_depth(i) != depth:
                    continue
                kids = [c for c in (2 * i + 1, 2 * i + 2) if c < N]
                if not kids:
                    continue
                v = rank_of(i)
                reads = [bm.e_in]
                for c in kids:
                    leaf = 2 * c + 1 >= N
                    wire = bm.e_in if leaf else bm.e_acc
                    reads.append(wire)
                    u = rank_of(c)
                    msgs.append(_Msg(src=u, dst=v, n=hi - lo, reduce=True, esize=wire,
                                     payload=acc[u][lo:hi].copy(), deliver=_reduce_into(acc[v], lo, hi, op),
                                     phase="reduce" + name, src_off=lo, dst_off=lo))
                bm.rw(hi - lo, *reads, bm.e_out if i == 0 else bm.e_acc)
        _run_step(log, step, msgs)
        step += 1
    for t in range(D):
        depth = t + 1
        msgs = []
        for name, rank_of, (lo, hi) in trees:
            for i in range(N):
                if heap_depth(i) != depth:
                    continue
                u, v = rank_of((i - 1) // 2), rank_of(i)
                msgs.append(_Msg(src=u, dst=v, n=hi - lo, reduce=False, esize=bm.e_out,
                                 payload=acc[u][lo:hi].copy(), deliver=_store_into(acc[v], lo, hi),
                                 phase="bcast" + name, src_off=lo, dst_off=lo))
                bm.rw(hi - lo, bm.e_out, bm.e_out)
        _run_step(log, step, msgs)
        step += 1
    return Result([narrow(a, dtype) for a in acc], log, bm.total)


# --------------------------------------------------------------------------
# ReduceScatter and AllGather alone
# --------------------------------------------------------------------------

def reduce_scatter(inputs, algo: str, dtype: str, op: str = "sum") -> Result:
    """Each input holds N blocks of rc elements; rank r ends with block r of
    the elementwise sum ([Latency-formula page] section "Ring ReduceScatter",
    eq. model-algo-ring-reducescatter: every node ends with 1/N of the reduced
    result)."""
    N, total = _check_same(inputs, dtype)
    assert total % N == 0
    rc = total // N
    e = ESIZE[dtype]
    bm = _Bytes(dtype)
    log = TransferLog()
    if algo == "fused":
        outs = []
        for r in range(N):
            acc = widen(inputs[0][r * rc:(r + 1) * rc], dtype)
            for q in range(1, N):
                acc = combine(acc, widen(inputs[q][r * rc:(r + 1) * rc], dtype), op)
            for q in range(N):
                if q != r:
                    log.add(step=0, phase="fused", src=q, dst=r, n=rc, reduce=True, esize=e,
                            src_off=r * rc, dst_off=0)
            outs.append(narrow(acc, dtype))
            bm.rw(rc, *([bm.e_in] * N), bm.e_out)
        return Result(outs, log, bm.total)
    if algo != "ring":
        raise Unsupported(f"reduce_scatter/{algo}")
    if N == 1:
        bm.rw(rc, bm.e_in, bm.e_out)
        return Result([np.array(inputs[0], copy=True)], log, bm.total)
    # Standalone ring: the AllReduce ReduceScatter shifted by one chunk, so that
    # rank r ends with block r (the pages leave block ownership open): at step
    # s rank r sends block (r - s - 1) and adds block (r - s - 2) from r - 1.
    # Block c is summed x_{c+1} + x_{c+2} + ... + x_{c+N} (indices mod N).
    acc = [widen(x, dtype) for x in inputs]
    for s in range(N - 1):
        msgs = []
        for r in range(N):
            c = (r - s - 1) % N
            lo, hi = c * rc, (c + 1) * rc
            dst = (r + 1) % N
            wire = bm.e_in if s == 0 else bm.e_acc
            msgs.append(_Msg(src=r, dst=dst, n=rc, reduce=True, esize=wire,
                             payload=acc[r][lo:hi].copy(), deliver=_reduce_into(acc[dst], lo, hi, op),
                             phase="rs", src_off=lo, dst_off=lo, chunks=(c,)))
            bm.rw(rc, bm.e_in, wire, bm.e_out if s == N - 2 else bm.e_acc)
        _run_step(log, s, msgs)
    outs = [narrow(acc[r][r * rc:(r + 1) * rc], dtype) for r in range(N)]
    return Result(outs, log, bm.total)


def allgather(inputs, algo: str, dtype: str) -> Result:
    """Each rank contributes sc elements; every rank ends with all N blocks,
    block q from rank q ([Latency-formula page] section "Ring AllGather", eq.
    model-algo-ring-allgather)."""
    N, sc = _check_same(inputs, dtype)
    bm = _Bytes(dtype)
    log = TransferLog()
    if algo == "fused":
        outs = [np.concatenate([np.array(x, copy=True) for x in inputs]) for _ in range(N)]
        for q in range(N):
            for r in range(N):
                if q != r:
                    log.add(step=0, phase="fused", src=q, dst=r, n=sc, reduce=False,
                            esize=bm.e_in, src_off=0, dst_off=q * sc)
        bm.rw(sc * N, bm.e_in)
        bm.rw(sc * N * N, bm.e_out)
        return Result(outs, log, bm.total)
    if algo != "ring":
        raise Unsupported(f"allgather/{algo}")
    # Each rank first places its own block (a local copy), then N-1 ring
    # steps: at step s rank r forwards block (r - s) and stores block
    # (r - s - 1) from rank r - 1.
    out = [np.zeros(N * sc, dtype=storage_dtype(dtype)) for _ in range(N)]
    for r in range(N):
        out[r][r * sc:(r + 1) * sc] = inputs[r]
        bm.rw(sc, bm.e_in, bm.e_out)
    for s in range(N - 1):
        msgs = []
        for r in range(N):
            c = (r - s) % N
            lo, hi = c * sc, (c + 1) * sc
            dst = (r + 1) % N
            msgs.append(_Msg(src=r, dst=dst, n=sc, reduce=False, esize=bm.e_out,
                             payload=out[r][lo:hi].copy(), deliver=_store_into(out[dst], lo, hi),
                             phase="ag", src_off=lo, dst_off=lo, chunks=(c,)))
            bm.rw(sc, bm.e_out, bm.e_out)
        _run_step(log, s, msgs)
    return Result(out, log, bm.total)


# --------------------------------------------------------------------------
# Broadcast and Scatter
# --------------------------------------------------------------------------

def binomial_rounds(N: int):
    """Distances of the binomial tree, one per step: 2**(L-1), ..., 2, 1 with
    L = ceil(log2 N) ([Bcast/Scatter page] section "二叉树（Binomial Tree）",
    the 8-node table: 0->4; 0->2, 4->6; 0->1, 2->3, 4->5, 6->7).  At distance
    d every relative rank v with v mod 2d == 0 and v + d < N sends to v + d."""
    L = _ceil_log2(N)
    return [1 << (L - 1 - s) for s in range(L)]


def broadcast(root_input, N: int, root: int, algo: str, dtype: str, inplace: bool = False) -> Result:
    """B_i = A_root on every rank ([Bcast/Scatter page] eq.
    onetoall-bcast-semantic).  Ranks are renumbered relative to the root,
    v = (r - root) mod N, for the tree schedules."""
    _check_same([root_input], dtype)
    assert 0 <= root < N
    count = len(root_input)
    e = ESIZE[dtype]
    bm = _Bytes(dtype)
    log = TransferLog()
    if algo == "fused":
        out = [np.array(root_input, copy=True) for _ in range(N)]
        for r in range(N):
            if r != root:
                log.add(step=0, phase="fused", src=root, dst=r, n=count, reduce=False,
                        esize=e, src_off=0, dst_off=0)
        ndst = N - 1 if inplace else N
        if ndst:  # read once, written to every destination (none: nothing moves)
            bm.rw(count, bm.e_in, *([bm.e_out] * ndst))
        return Result(out, log, bm.total)
    if algo == "binomial":
        return _broadcast_binomial(root_input, N, root, dtype, inplace)
    if algo == "scatter_allgather":
        return _broadcast_scatter_allgather(root_input, N, root, dtype, inplace)
    raise Unsupported(f"broadcast/{algo}")


def _broadcast_binomial(A, N, root, dtype, inplace):
    """Binomial-tree Broadcast: ceil(log2 N) steps, each holder sends the whole
    message to one new rank per step ([Bcast/Scatter page] eq. binomial-bcast;
    [Latency-formula page] eq. model-algo-bcast-tree)."""
    count = len(A)
    bm = _Bytes(dtype)
    log = TransferLog()
    have = {root: np.array(A, copy=True)}
    if not inplace:
        bm.rw(count, bm.e_in, bm.e_out)
    for s, d in enumerate(binomial_rounds(N)):
        msgs = []
        for v in range(0, N, 2 * d):
            if v + d >= N:
                continue
            src, dst = (v + root) % N, (v + d + root) % N

            def deliver(p, dst=dst):
                have[dst] = p
            msgs.append(_Msg(src=src, dst=dst, n=count, reduce=False, esize=bm.e_in,
                             payload=have[src].copy(), deliver=deliver, phase="bcast",
                             src_off=0, dst_off=0))
            bm.rw(count, bm.e_out, bm.e_out)
        _run_step(log, s, msgs)
    return Result([have[r] for r in range(N)], log, bm.total)


def _binomial_scatter_steps(N, root, chunk_lo_hi, log, bm, holdings, step0=0):
    """Shared step loop of the binomial Scatter.  At distance d, relative rank v
    hands the chunks of relative ranks [v+d, min(v+2d, N)) to v+d, so the step
    moves M/2, M/4, ... ([Bcast/Scatter page] section "二叉树 Scatter" and its
    8-node table: 0->4 [A4..A7]; 0->2 [A2,A3], 4->6 [A6,A7]; then M/8 each).
    Chunk of relative rank v is absolute chunk (v + root) mod N."""
    for s, d in enumerate(binomial_rounds(N)):
        msgs = []
        for v in range(0, N, 2 * d):
            if v + d >= N:
                continue
            src, dst = (v + root) % N, (v + d + root) % N
            chunks = tuple((q + root) % N for q in range(v + d, min(v + 2 * d, N)))
            n = sum(chunk_lo_hi(c)[1] - chunk_lo_hi(c)[0] for c in chunks)
            payload = {c: holdings[src][c].copy() for c in chunks}

            def deliver(p, dst=dst):
                holdings[dst].update(p)
            msgs.append(_Msg(src=src, dst=dst, n=n, reduce=False, esize=bm.e_in,
                             payload=payload, deliver=deliver, phase="scatter", chunks=chunks))
            bm.rw(n, bm.e_in, bm.e_out)
        _run_step(log, step0 + s, msgs)
    return step0 + len(binomial_rounds(N))


def _broadcast_scatter_allgather(A, N, root, dtype, inplace):
    """Broadcast as a binomial Scatter of the message's N chunks followed by a
    Ring AllGather ([Bcast/Scatter page] section "Broadcast 与 Scatter 的关系").
    Rank r receives chunk r (cut by ``oracle.partition``) in the Scatter, then
    the ring forwards chunks: at step s rank r sends chunk (r - s) and stores
    chunk (r - s - 1) from rank r - 1."""
    count = len(A)
    e = ESIZE[dtype]
    bm = _Bytes(dtype)
    log = TransferLog()

    def lohi(c):
        return chunk_range(c, count, N, e)

    holdings = {r: {} for r in range(N)}
    holdings[root] = {c: A[slice(*lohi(c))].copy() for c in range(N)}
    lo, hi = lohi(root)
    if not inplace:
        bm.rw(hi - lo, bm.e_in, bm.e_out)
    step = _binomial_scatter_steps(N, root, lohi, log, bm, holdings)
    out = [np.zeros(count, dtype=storage_dtype(dtype)) for _ in range(N)]
    for r in range(N):
        lo, hi = lohi(r)
        out[r][lo:hi] = holdings[r][r]
    if inplace:
        out[root][:] = A
    for s in range(N - 1):
        msgs = []
        for r in range(N):
            c = (r - s) % N
            lo, hi = lohi(c)
            dst = (r + 1) % N
            msgs.append(_Msg(src=r, dst=dst, n=hi - lo, reduce=False, esize=bm.e_out,
                             payload=out[r][lo:hi].copy(), deliver=_store_into(out[dst], lo, hi),
                             phase="ag", src_off=lo, dst_off=lo, chunks=(c,)))
            bm.rw(hi - lo, bm.e_out, bm.e_out)
        _run_step(log, step + s, msgs)
    return Result(out, log, bm.total)


def scatter(root_input, N: int, root: int, algo: str, dtype: str) -> Result:
    """The root holds [A_0, ..., A_{N-1}], rank i receives A_i
    ([Bcast/Scatter page] eq. onetoall-scatter-semantic)."""
    _check_same([root_input], dtype)
    assert 0 <= root < N and len(root_input) % N == 0
    rc = len(root_input) // N
    bm = _Bytes(dtype)
    log = TransferLog()
    if algo == "fused":
        out = [np.array(root_input[r * rc:(r + 1) * rc], copy=True) for r in range(N)]
        for r in range(N):
            if r != root:
                log.add(step=0, phase="fused", src=root, dst=r, n=rc, reduce=False,
                        esize=bm.e_in, src_off=r * rc, dst_off=0, chunks=(r,))
        bm.rw(rc * N, bm.e_in, bm.e_out)
        return Result(out, log, bm.total)
    if algo != "binomial":
        raise Unsupported(f"scatter/{algo}")

    def lohi(c):
        return c * rc, (c + 1) * rc

    holdings = {r: {} for r in range(N)}
    holdings[root] = {c: root_input[c * rc:(c + 1) * rc].copy() for c in range(N)}
    bm.rw(rc, bm.e_in, bm.e_out)  # the root's own block
    _binomial_scatter_steps(N, root, lohi, log, bm, holdings)
    return Result([holdings[r][r] for r in range(N)], log, bm.total)


# --------------------------------------------------------------------------
# AllToAll
# --------------------------------------------------------------------------

def alltoall(inputs, algo: str, dtype: str) -> Result:
    """Every rank sends a different block to every rank: with N blocks of B
    elements per buffer, out_j[block i] = in_i[block j] ([Latency-formula page]
    section "AllToAll 算法怎么选")."""
    N, total = _check_same(inputs, dtype)
    assert total % N == 0
    B = total // N
    bm = _Bytes(dtype)
    log = TransferLog()

    def blk(x, j):
        return x[j * B:(j + 1) * B]

    if algo == "fused":
        out = [np.concatenate([blk(inputs[i], j) for i in range(N)]) for j in range(N)]
        for i in range(N):
            for j in range(N):
                if i != j:
                    log.add(step=0, phase="fused", src=i, dst=j, n=B, reduce=False,
                            esize=bm.e_in, src_off=j * B, dst_off=i * B)
        bm.rw(total * N, bm.e_in, bm.e_out)
        return Result(out, log, bm.total)
    if algo == "pairwise":
        return _alltoall_pairwise(inputs, dtype, B)
    if algo == "bruck":
        return _alltoall_bruck(inputs, dtype, B)
    if algo == "ring":
        return _alltoall_ring(inputs, dtype, B)
    raise Unsupported(f"alltoall/{algo}")


def _alltoall_pairwise(inputs, dtype, B):
    """Pairwise exchange ([Latency-formula page] eq. model-algo-a2a-pairwise):
    in round k = 1 .. N-1 rank i sends its block for rank (i + k) mod N there
    (and so receives from (i - k) mod N).  Round 0 is the local block."""
    N = len(inputs)
    bm = _Bytes(dtype)
    log = TransferLog()
    out = [np.zeros(N * B, dtype=storage_dtype(dtype)) for _ in range(N)]
    for i in range(N):
        out[i][i * B:(i + 1) * B] = inputs[i][i * B:(i + 1) * B]
        bm.rw(B, bm.e_in, bm.e_out)
    for k in range(1, N):
        msgs = []
        for i in range(N):
            j = (i + k) % N
            msgs.append(_Msg(src=i, dst=j, n=B, reduce=False, esize=bm.e_in,
                             payload=inputs[i][j * B:(j + 1) * B].copy(),
                             deliver=_store_into(out[j], i * B, (i + 1) * B), phase="round",
                             src_off=j * B, dst_off=i * B))
            bm.rw(B, bm.e_in, bm.e_out)
        _run_step(log, k, msgs)
    return Result(out, log, bm.total, local_steps=1 if N > 1 else 0)


def _alltoall_ring(inputs, dtype, B):
    """Ring AllToAll ([Latency-formula page] eq. model-algo-a2a-ring: N-1
    rounds, each rank talking only to its ring neighbours).  Reading: store
    and forward -- in round k every rank passes to rank i+1 every block it
    holds that is not addressed to itself, and keeps the one that is; a block
    from rank s for rank d travels (d - s) mod N hops.  Round 0 is the local
    block.  Round k carries N-k blocks per rank, so a rank sends
    (N-1)/2 * M in all, not the (N-1)/N * M the page's formula charges (it
    writes Pairwise's bandwidth term for the ring as well)."""
    N = len(inputs)
    bm = _Bytes(dtype)
    log = TransferLog()
    out = [np.zeros(N * B, dtype=storage_dtype(dtype)) for _ in range(N)]
    for i in range(N):
        out[i][i * B:(i + 1) * B] = inputs[i][i * B:(i + 1) * B]
        bm.rw(B, bm.e_in, bm.e_out)
    # in transit at rank i: {(source, destination): block}
    transit = {i: {(i, d): inputs[i][d * B:(d + 1) * B].copy() for d in range(N) if d != i} for i in range(N)}
    for k in range(1, N):
        msgs = []
        nxt = {i: {} for i in range(N)}
        for i in range(N):
            dst = (i + 1) % N
            keys = sorted(transit[i], key=lambda sd: (sd[1] - dst) % N)
            payload = {key: transit[i][key] for key in keys}

            def deliver(p, dst=dst):
                for (src, d), blk in p.items():
                    if d == dst:
                        out[dst][src * B:(src + 1) * B] = blk
                    else:
                        nxt[dst][(src, d)] = blk
            msgs.append(_Msg(src=i, dst=dst, n=len(keys) * B, reduce=False, esize=bm.e_in,
                             payload=payload, deliver=deliver, phase="ring", chunks=tuple(keys)))
            bm.rw(len(keys) * B, bm.e_in, bm.e_out)
        _run_step(log, k, msgs)
        transit = nxt
    return Result(out, log, bm.total, local_steps=1 if N > 1 else 0)


def _alltoall_bruck(inputs, dtype, B):
    """Bruck AllToAll in ceil(log2 N) rounds ([Latency-formula page] eq.
    model-algo-a2a-bruck; the algorithm of Bruck et al., 1997, which the page
    cites).  Rank i first rotates its blocks so that position p holds its
    block for rank (i + p) mod N.  In round k it sends every position p whose
    bit k is set to rank (i + 2**k) mod N, which stores it at the same
    position.  After all rounds a block has moved sum(bits of p) = p ranks,
    so rank j's position p holds the block from rank (j - p) mod N, and a
    final inverse rotation puts it at block (j - p) mod N.

    Bytes: every round rewrites each rank's working buffer once (blocks with
    bit k set from rank i - 2**k, the rest from itself), with the two
    rotations folded into the first and last rounds' addressing, so
    2 * ceil(log2 N) * N * M bytes move, against the (N-1)/N * M per rank the
    page quotes for the link."""
    N = len(inputs)
    bm = _Bytes(dtype)
    log = TransferLog()
    L = _ceil_log2(N)
    if N == 1:
        bm.rw(B, bm.e_in, bm.e_out)
        return Result([np.array(inputs[0], copy=True)], log, bm.total)
    W = [[inputs[i][((i + p) % N) * B:((i + p) % N + 1) * B].copy() for p in range(N)]
         for i in range(N)]
    for k in range(L):
        msgs = []
        for i in range(N):
            dst = (i + (1 << k)) % N
            pos = tuple(p for p in range(N) if (p >> k) & 1)

            def deliver(payload, dst=dst):
                for p, blkdata in payload.items():
                    W[dst][p] = blkdata
            msgs.append(_Msg(src=i, dst=dst, n=len(pos) * B, reduce=False, esize=bm.e_in,
                             payload={p: W[i][p].copy() for p in pos}, deliver=deliver,
                             phase="round", chunks=pos))
        _run_step(log, k, msgs)
        bm.rw(N * N * B, bm.e_in, bm.e_out)
    out = []
    for j in range(N):
        blocks = [W[j][(j - i) % N] for i in range(N)]
        out.append(np.concatenate(blocks))
    return Result(out, log, bm.total)


# --------------------------------------------------------------------------
# Pipelined Broadcasts, Gather, Tree Reduce
# --------------------------------------------------------------------------

ALGOS_EXTRA = {
    "broadcast": ("pipe_chain", "pipe_tree"),
    "gather": ("fused", "binomial"),
    "reduce": ("fused", "binomial"),
}


def broadcast_pipelined(root_input, N: int, root: int, algo: str, dtype: str, k: int,
                        inplace: bool = False) -> Result:
    """Chunked (pipelined) Broadcasts of the [Bcast/Scatter page]: the message
    is cut into k chunks (``oracle.partition``) and chunk j runs the
    unpipelined schedule delayed by j steps.

    * pipe_chain (section "分块链式流水线", eq. pipe-chain-bcast): relative
      rank v forwards chunk j to v + 1 at step v + j; N + k - 2 steps.
    * pipe_tree (section "分块二叉树流水线", eq. pipe-tree-bcast): chunk j
      takes binomial step s at step j + s; ceil(log2 N) + k - 1 steps.

    That each chunk follows the unpipelined route shifted by its index is the
    reading taken; the pages give only the step counts and chunk sizes."""
    _check_same([root_input], dtype)
    assert 0 <= root < N and k >= 1
    count = len(root_input)
    e = ESIZE[dtype]
    bm = _Bytes(dtype)
    log = TransferLog()
    have = {r: {} for r in range(N)}
    have[root] = {j: root_input[slice(*chunk_range(j, count, k, e))].copy() for j in range(k)}
    if not inplace:
        bm.rw(count, bm.e_in, bm.e_out)
    if algo == "pipe_chain":
        nsteps = N + k - 2 if N > 1 else 0
        route = [[(v, v + 1) for v in range(N - 1)]]  # one hop per step
        hops = lambda t, j: [route[0][t - j]] if 0 <= t - j < N - 1 else []
    elif algo == "pipe_tree":
        rounds = binomial_rounds(N)
        nsteps = len(rounds) + k - 1 if N > 1 else 0

        def hops(t, j):
            s = t - j
            if not 0 <= s < len(rounds):
                return []
            d = rounds[s]
            return [(v, v + d) for v in range(0, N, 2 * d) if v + d < N]
    else:
        raise Unsupported(f"broadcast/{algo}")
    for t in range(nsteps):
        msgs = []
        for j in range(k):
            lo, hi = chunk_range(j, count, k, e)
            for v, w in hops(t, j):
                src, dst = (v + root) % N, (w + root) % N

                def deliver(p, dst=dst, j=j):
                    have[dst][j] = p
                msgs.append(_Msg(src=src, dst=dst, n=hi - lo, reduce=False, esize=bm.e_in,
                                 payload=have[src][j].copy(), deliver=deliver, phase=algo,
                                 src_off=lo, dst_off=lo, chunks=(j,)))
                bm.rw(hi - lo, bm.e_out, bm.e_out)
        _run_step(log, t, msgs)
    outs = []
    for r in range(N):
        outs.append(np.concatenate([have[r][j] for j in range(k)]) if k else np.array(root_input[:0]))
    return Result(outs, log, bm.total)


def gather(inputs, root: int, algo: str, dtype: str) -> Result:
    """The dual of Scatter: the root ends with [A_0, ..., A_{N-1}], A_i being
    rank i's input ([Bcast/Scatter page] section "对偶性：Scatter 与 Gather",
    eq. onetoall-gather-scatter-duality: reverse the Scatter's data flow).

    binomial: distances 1, 2, 4, ...; at distance d relative rank v with
    v mod 2d == d hands everything it holds -- the chunks of relative ranks
    [v, min(v+d, N)) -- to v - d."""
    N, rc = _check_same(inputs, dtype)
    assert 0 <= root < N
    bm = _Bytes(dtype)
    log = TransferLog()
    if algo == "fused":
        out = np.concatenate([np.array(x, copy=True) for x in inputs]) if N else None
        for r in range(N):
            if r != root:
                log.add(step=0, phase="fused", src=r, dst=root, n=rc, reduce=False, esize=bm.e_in,
                        src_off=0, dst_off=r * rc, chunks=(r,))
        bm.rw(rc * N, bm.e_in, bm.e_out)
        return Result([out], log, bm.total)
    if algo != "binomial":
        raise Unsupported(f"gather/{algo}")
    holdings = {r: {r: np.array(inputs[r], copy=True)} for r in range(N)}
    bm.rw(rc, bm.e_in, bm.e_out)  # the root's own block
    L = _ceil_log2(N)
    for s in range(L):
        d = 1 << s
        msgs = []
        for u in range(0, N, 2 * d):
            v = u + d
            if v >= N:
                continue
            src, dst = (v + root) % N, (u + root) % N
            chunks = tuple((q + root) % N for q in range(v, min(v + d, N)))
            payload = {c: holdings[src][c].copy() for c in chunks}

            def deliver(p, dst=dst):
                holdings[dst].update(p)
            msgs.append(_Msg(src=src, dst=dst, n=rc * len(chunks), reduce=False, esize=bm.e_in,
                             payload=payload, deliver=deliver, phase="gather", chunks=chunks))
            bm.rw(rc * len(chunks), bm.e_in, bm.e_out)
        _run_step(log, s, msgs)
    out = np.concatenate([holdings[root][c] for c in range(N)])
    return Result([out], log, bm.total)


def reduce(inputs, root: int, algo: str, dtype: str, inplace: bool = False, op: str = "sum") -> Result:
    """Reduce to one root: out_root = elementwise sum of every rank's input
    ([Latency-formula page] section "Broadcast / Reduce 怎么用 Tree 算法", eq.
    model-algo-reduce-tree: the Tree Broadcast run backwards, same cost).

    binomial: distances 1, 2, 4, ...; at distance d relative rank u with
    u mod 2d == 0 adds the partial sum of u + d to its own.  The association
    is the balanced tree over adjacent relative ranks, ((x0+x1)+(x2+x3)) + ...
    fused: rank order ((x_0 + x_1) + x_2) + ..., as the fused AllReduce."""
    N, count = _check_same(inputs, dtype)
    assert 0 <= root < N
    bm = _Bytes(dtype)
    log = TransferLog()
    if algo not in ALGOS_EXTRA["reduce"]:
        raise Unsupported(f"reduce/{algo}")
    if N == 1:  # one rank: the result is its input (copied unless in place)
        if not inplace:
            bm.rw(count, bm.e_in, bm.e_out)
        return Result([np.array(inputs[0], copy=True)], log, bm.total)
    if algo == "fused":
        acc = widen(inputs[0], dtype)
        for q in range(1, N):
            acc = combine(acc, widen(inputs[q], dtype), op)
        for q in range(N):
            if q != root:
                log.add(step=0, phase="fused", src=q, dst=root, n=count, reduce=True, esize=bm.e_in,
                        src_off=0, dst_off=0)
        bm.rw(count, *([bm.e_in] * N), bm.e_out)
        return Result([narrow(acc, dtype)], log, bm.total)
    acc = [widen(x, dtype) for x in inputs]
    partial = [False] * N  # relative rank holds a partial sum (not its raw input)
    L = _ceil_log2(N)
    for s in range(L):
        d = 1 << s
        msgs = []
        for u in range(0, N, 2 * d):
            v = u + d
            if v >= N:
                continue
            src, dst = (v + root) % N, (u + root) % N
            wire = bm.e_acc if partial[v] else bm.e_in
            msgs.append(_Msg(src=src, dst=dst, n=count, reduce=True, esize=wire,
                             payload=acc[src].copy(), deliver=_reduce_into(acc[dst], 0, count, op),
                             phase="reduce", src_off=0, dst_off=0))
            last = u == 0 and s == L - 1
            bm.rw(count, bm.e_acc if partial[u] else bm.e_in, wire, bm.e_out if last else bm.e_acc)
            partial[u] = True
        _run_step(log, s, msgs)
    return Result([narrow(acc[root], dtype)], log, bm.total)
