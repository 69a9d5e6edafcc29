"""Choosing an algorithm from a cost model (the AUTO selection) -- oracle side.

Two models, both from the [Latency-formula page]'s alpha-beta framework
(section "本文是集合通信算法的 alpha-beta 延迟公式手册"):

* "link": the pages' own formulas, where M/beta is link time.  AllReduce picks
  among Ring, Recursive Halving-Doubling (N a power of 2) and Double Binary
  Tree by eqs. model-algo-ring-ar, -rhd-ar, -dbt-ar (the comparison and
  crossover of section "三种算法对比与交叉点"); Broadcast between the binomial
  tree (eq. binomial-bcast of the [Bcast/Scatter page]) and Scatter +
  AllGather (eq. binomial-scatter plus eq. model-algo-ring-allgather);
  AllToAll between Pairwise and Bruck (eqs. model-algo-a2a-pairwise, -bruck);
  ReduceScatter, AllGather and Scatter have one page algorithm each.
* "hbm": the same model with the data-movement term taken as what one GPU
  must move through its memory: cost = steps * alpha + algorithmic bytes /
  beta, with steps and bytes from the simulated schedule (``Result``).  Every
  algorithm of the collective, fused one included, is a candidate.

Ties go to the earlier candidate in ``schedules.ALGOS`` order (link: ring,
rhd, dbt / binomial, scatter_allgather / pairwise, bruck).

Parity status: pinned by the crossover the page prints (14.4 MB at N=8,
alpha=5 us, beta=450 GB/s) and by the closed forms it is made of.
"""
from __future__ import annotations

import numpy as np

from . import cost_model as cm
from . import schedules
from .numerics import ESIZE, storage_dtype


def message_bytes(coll: str, N: int, count: int, dtype: str) -> int:
    """M of the formulas: the per-rank message (AllReduce / ReduceScatter:
    the per-rank input; AllGather: the per-rank output; AllToAll: the
    per-rank send; Broadcast / Scatter / Gather: the root's total; Reduce:
    the per-rank input)."""
    e = ESIZE[dtype]
    if coll in ("allreduce", "broadcast", "reduce"):
        return count * e
    return N * count * e


def default_chunks(algo: str, N: int, count: int, dtype: str, alpha: float, beta: float) -> int:
    """Chunks of a pipelined Broadcast when none are given: the optimum of the
    page's formula, dT/dk = 0 on (h + k) (alpha + M/(k beta)) -> k* =
    sqrt(h M / (alpha beta)), with h = N - 2 for the chain (eq.
    pipe-chain-bcast) and ceil(log2 N) - 1 for the tree (eq. pipe-tree-bcast),
    rounded half up, kept within [1, 256] and at most one chunk per 16 bytes."""
    import math

    e = ESIZE[dtype]
    h = N - 2 if algo == "pipe_chain" else cm.ceil_log2(N) - 1
    M = count * e
    k = 1
    if h > 0 and M > 0:
        k = int(math.floor(math.sqrt(h * M / (alpha * beta)) + 0.5))
    return max(1, min(k, 256, max(1, M // 16)))


def link_candidates(coll: str, N: int) -> dict:
    pow2 = N & (N - 1) == 0
    if coll == "allreduce":
        c = {"ring": cm.t_ring_ar}
        if pow2:
            c["rhd"] = cm.t_rhd_ar
        c["dbt"] = cm.t_dbt_ar
        return c
    if coll == "reduce_scatter":
        return {"ring": cm.t_ring_reducescatter}
    if coll == "allgather":
        return {"ring": cm.t_ring_allgather}
    if coll == "broadcast":
        return {"binomial": cm.t_binomial_bcast,
                "scatter_allgather": lambda N, M, a, b: cm.t_binomial_scatter(N, M, a, b) + cm.t_ring_allgather(N, M, a, b),
                "pipe_chain": cm.t_pipe_chain_bcast, "pipe_tree": cm.t_pipe_tree_bcast}
    if coll == "scatter":
        return {"binomial": cm.t_binomial_scatter}
    if coll == "gather":
        return {"binomial": cm.t_gather}
    if coll == "reduce":
        return {"binomial": cm.t_reduce_tree}
    if coll == "alltoall":
        return {"pairwise": cm.t_a2a_pairwise, "bruck": cm.t_a2a_bruck, "ring": cm.t_a2a_ring}
    raise ValueError(coll)


def select_link(coll: str, N: int, count: int, dtype: str, alpha: float, beta: float):
    M = message_bytes(coll, N, count, dtype)
    best, best_t = None, None
    for algo, f in link_candidates(coll, N).items():
        if algo.startswith("pipe_"):
            t = f(N, M, alpha, beta, default_chunks(algo, N, count, dtype, alpha, beta))
        else:
            t = f(N, M, alpha, beta)
        if best_t is None or t < best_t:
            best, best_t = algo, t
    return best, best_t


def _run(coll, algo, N, count, dtype, root, alpha=None, beta=None):
    z = np.zeros
    sd = storage_dtype(dtype)
    if algo.startswith("pipe_"):
        k = default_chunks(algo, N, count, dtype, alpha, beta)
        return schedules.broadcast_pipelined(z(count, sd), N, root, algo, dtype, k)
    if coll == "gather":
        return schedules.gather([z(count, sd) for _ in range(N)], root, algo, dtype)
    if coll == "reduce":
        return schedules.reduce([z(count, sd) for _ in range(N)], root, algo, dtype)
    if coll == "allreduce":
        return schedules.allreduce([z(count, sd) for _ in range(N)], algo, dtype)
    if coll == "reduce_scatter":
        return schedules.reduce_scatter([z(N * count, sd) for _ in range(N)], algo, dtype)
    if coll == "allgather":
        return schedules.allgather([z(count, sd) for _ in range(N)], algo, dtype)
    if coll == "broadcast":
        return schedules.broadcast(z(count, sd), N, root, algo, dtype)
    if coll == "scatter":
        return schedules.scatter(z(N * count, sd), N, root, algo, dtype)
    return schedules.alltoall([z(N * count, sd) for _ in range(N)], algo, dtype)


def select_hbm(coll: str, N: int, count: int, dtype: str, alpha: float, beta: float, root: int = 0):
    best, best_t = None, None
    algos = tuple(schedules.ALGOS.get(coll, ())) + tuple(a for a in schedules.ALGOS_EXTRA.get(coll, ())
                                                          if a not in schedules.ALGOS.get(coll, ()))
    for algo in algos:
        try:
            res = _run(coll, algo, N, count, dtype, root, alpha, beta)
        except schedules.Unsupported:
            continue
        t = res.launch_steps * alpha + res.hbm_bytes / beta
        if best_t is None or t < best_t:
            best, best_t = algo, t
    return best, best_t
