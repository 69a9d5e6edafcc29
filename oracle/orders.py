"""Closed-form association tree of every reduction schedule, per element.

IEEE addition is commutative, so a schedule's result for one element is fixed
by the shape of its binary tree of adds over the ranks' values.  This module
states that tree for each schedule directly (the table below), evaluates it for
any set of sampled elements, and is checked against the message-passing
simulation of ``oracle.schedules`` on small buffers and on order-witness
inputs.  Large buffers are checked element by element through this module.

AllReduce, element e (chunks cut by ``oracle.partition``):

* fused, mesh:  ((x0 + x1) + x2) + ... + x_{N-1}  -- rank order, the fold
  of the [hccl article]'s Mesh root (section "Mesh算法：全连接广播").
* ring:   chunk c = chunk of e; ((x_c + x_{c+1}) + x_{c+2}) + ... + x_{c+N-1},
  indices mod N ([hccl article] section "Ring算法": at step 0 rank c sends
  chunk c, each later hop adds its own copy).  ring_hop: the same tree with
  every partial sum rounded to the data type.
* rhd:    balanced tree over adjacent rank pairs, ((x0+x1)+(x2+x3)) + ...
  ([Latency-formula page] section "Recursive Halving-Doubling": round k pairs
  ranks at distance 2**k, starting at distance 1); for N not a power of 2
  the leaves are the folded pairs (x_{2i} + x_{2i+1}), i < N - P, and then
  the ranks 2r .. N-1.
* dbt:    S(i) = (x_i + S(2i+1)) + S(2i+2) on the heap of the tree holding e
  (tree A: rank i; tree B: rank N-1-i) ([hccl article] section "Tree算法").

ReduceScatter, element e of the N*rc input (block c = e // rc):

* fused:  rank order, as above.
* ring:   x_{c+1} + x_{c+2} + ... + x_{c+N}, the AllReduce chain shifted by
  one so that it ends on rank c.

Parity status: the fused, ring and rhd trees follow from the pages' step
descriptions; the dbt tree rests on the reading of how the two trees are
built.  Every tree is stated here on its own, with no helper shared with the
simulation in ``oracle.schedules``; hand-derived order witnesses pin them at
N = 4 and 8 (and the RHD fold-in at N = 5, 6, 7).
"""
from __future__ import annotations

import numpy as np

from .numerics import ESIZE, combine, narrow, widen
from .partition import chunk_of, chunk_range


def left_fold(ranks):
    t = ranks[0]
    for r in ranks[1:]:
        t = (t, r)
    return t


def balanced_pairs(ranks):
    if len(ranks) == 1:
        return ranks[0]  # a rank, or an already built subtree
    mid = len(ranks) // 2
    return (balanced_pairs(ranks[:mid]), balanced_pairs(ranks[mid:]))


def halving_leaves(N: int):
    """The participants of the recursive halving, in order: with P the largest
    power of 2 not above N and r = N - P, ranks 2i+1 fold into 2i (i < r)
    first, so the first r leaves are the pairs (2i, 2i+1) and the rest are the
    ranks 2r .. N-1 ([Latency-formula page] section "Recursive
    Halving-Doubling" for N = 2^k; the fold-in is the reading taken for other
    N).  Stated here from that description, apart from the simulation."""
    P = 1
    while 2 * P <= N:
        P *= 2
    extra = N - P
    return [(2 * i, 2 * i + 1) for i in range(extra)] + list(range(2 * extra, N))


def heap_tree(i: int, N: int, rank_of):
    t = rank_of(i)
    for c in (2 * i + 1, 2 * i + 2):
        if c < N:
            t = (t, heap_tree(c, N, rank_of))
    return t


def allreduce_tree(algo: str, N: int, count: int, dtype: str, e: int):
    """Association tree (nested pairs of rank indices) for element e."""
    esz = ESIZE[dtype]
    if algo in ("fused", "mesh"):
        return left_fold(list(range(N)))
    if algo in ("ring", "ring_hop"):
        c = chunk_of(e, count, N, esz)
        return left_fold([(c + j) % N for j in range(N)])
    if algo == "rhd":
        return balanced_pairs(halving_leaves(N))
    if algo == "dbt":
        # the first part of a two-way split on tree A (heap on the ranks), the
        # rest on tree B (heap node i on rank N-1-i)
        lo, hi = chunk_range(0, count, 2, esz)
        if not 0 <= e < count:
            raise IndexError(e)
        return heap_tree(0, N, (lambda i: i) if e < hi else (lambda i: N - 1 - i))
    raise ValueError(algo)


def reduce_scatter_tree(algo: str, N: int, rc: int, e: int):
    if algo == "fused":
        return left_fold(list(range(N)))
    if algo == "ring":
        c = e // rc
        return left_fold([(c + 1 + j) % N for j in range(N)])
    raise ValueError(algo)


def evaluate(tree, cols: dict, op: str = "sum", round_to: str | None = None):
    """Evaluate a tree on lane-type columns (one array per rank).  With
    ``round_to`` every inner node's value is rounded to that storage type (a
    schedule that stores its partial results in the data type)."""
    if isinstance(tree, int):
        return cols[tree]
    a, b = tree
    v = combine(evaluate(a, cols, op, round_to), evaluate(b, cols, op, round_to), op)
    return widen(narrow(v, round_to), round_to) if round_to else v


def _group_key_allreduce(algo, N, count, dtype, e):
    esz = ESIZE[dtype]
    if algo in ("ring", "ring_hop"):
        return chunk_of(e, count, N, esz)
    if algo == "dbt":
        return 0 if e < chunk_range(0, count, 2, esz)[1] else 1
    return 0


def allreduce_at(values_at, algo: str, count: int, dtype: str, idx, op: str = "sum") -> np.ndarray:
    """Expected AllReduce output at element indices ``idx``.

    ``values_at[r]`` holds rank r's stored input values at ``idx``.  Returns
    the stored-type results (identical on every rank)."""
    N = len(values_at)
    idx = np.asarray(idx, dtype=np.int64)
    out = None
    keys = np.array([_group_key_allreduce(algo, N, count, dtype, int(e)) for e in idx])
    for key in np.unique(keys):
        sel = np.nonzero(keys == key)[0]
        tree = allreduce_tree(algo, N, count, dtype, int(idx[sel[0]]))
        cols = {r: widen(np.asarray(values_at[r])[sel], dtype) for r in range(N)}
        res = narrow(evaluate(tree, cols, op, dtype if algo == "ring_hop" else None), dtype)
        if out is None:
            out = np.empty(len(idx), dtype=res.dtype)
        out[sel] = res
    return out


def reduce_scatter_at(values_at, algo: str, rc: int, dtype: str, idx, op: str = "sum") -> np.ndarray:
    """Expected ReduceScatter result for input-space element indices ``idx``
    (element e lands on rank e // rc at offset e % rc)."""
    N = len(values_at)
    idx = np.asarray(idx, dtype=np.int64)
    out = None
    keys = idx // rc if algo == "ring" else np.zeros(len(idx), dtype=np.int64)
    for key in np.unique(keys):
        sel = np.nonzero(keys == key)[0]
        tree = reduce_scatter_tree(algo, N, rc, int(idx[sel[0]]))
        cols = {r: widen(np.asarray(values_at[r])[sel], dtype) for r in range(N)}
        res = narrow(evaluate(tree, cols, op), dtype)
        if out is None:
            out = np.empty(len(idx), dtype=res.dtype)
        out[sel] = res
    return out
