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
    per-rank send; Broadcast / Scatter: the root's total)."""
    e = ESIZE[dtype]
    if coll in ("allreduce", "broadcast"):
        return count * e
    return N * count * e


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
                "scatter_allgather": lambda N, M, a, b: cm.t_binomial_scatter(N, M, a, b) + cm.t_ring_allgather(N, M, a, b)}
    if coll == "scatter":
        return {"binomial": cm.t_binomial_scatter}
    if coll == "alltoall":
        return {"pairwise": cm.t_a2a_pairwise, "bruck": cm.t_a2a_bruck}
    raise ValueError(coll)


def select_link(coll: str, N: int, count: int, dtype: str, alpha: float, beta: float):
    M = message_bytes(coll, N, count, dtype)
    best, best_t = None, None
    for algo, f in link_candidates(coll, N).items():
        t = f(N, M, alpha, beta)
        if best_t is None or t < best_t:
            best, best_t = algo, t
    return best, best_t


def _run(coll, algo, N, count, dtype, root):
    z = np.zeros
    sd = storage_dtype(dtype)
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
    for algo in schedules.ALGOS[coll]:
        try:
            res = _run(coll, algo, N, count, dtype, root)
        except schedules.Unsupported:
            continue
        t = res.launch_steps * alpha + res.hbm_bytes / beta
        if best_t is None or t < best_t:
            best, best_t = algo, t
    return best, best_t
