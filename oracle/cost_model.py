"""alpha-beta (Hockney) cost model of the pages.

Symbols as on the [Latency-formula page]: N ranks, M message bytes, alpha the
start-up latency of one step (seconds here), beta the link bandwidth (B/s).
Each function is one printed formula, cited by its equation label; where a
formula contains a sum, the sum is written out as a loop rather than in closed
form so that the closed form can be checked against it.

Parity status: pinned by the numbers the pages print (the N=8 comparison
table, the 14.4 MB crossover, the N=64 and N=1024 latency terms, the binomial
scatter sum) and by the transfer logs of ``oracle.schedules``.
"""
from __future__ import annotations

import math


def log2(N: int) -> float:
    return math.log2(N)


def ceil_log2(N: int) -> int:
    return (N - 1).bit_length()


# ---- [Latency-formula page] section "Ring AllReduce：带宽最优" -------------

def t_ring_rs(N, M, alpha, beta):  # eq. model-algo-ring-rs
    return (N - 1) * alpha + (N - 1) / N * M / beta


def t_ring_ag(N, M, alpha, beta):  # eq. model-algo-ring-ag
    return (N - 1) * alpha + (N - 1) / N * M / beta


def t_ring_ar(N, M, alpha, beta):  # eq. model-algo-ring-ar
    return 2 * (N - 1) * alpha + 2 * (N - 1) / N * M / beta


# ---- section "Recursive Halving-Doubling" --------------------------------

def t_rhd_rs(N, M, alpha, beta):  # eq. model-algo-rhd-rs, sum written out
    L = int(round(log2(N)))
    return L * alpha + sum(M / 2 ** (k + 1) for k in range(L)) / beta


def t_rhd_ag(N, M, alpha, beta):  # eq. model-algo-rhd-ag, sum written out
    L = int(round(log2(N)))
    return L * alpha + sum(M * 2 ** k / N for k in range(L)) / beta


def t_rhd_ar(N, M, alpha, beta):  # eq. model-algo-rhd-ar
    return 2 * log2(N) * alpha + 2 * (N - 1) / N * M / beta


# ---- section "Double Binary Tree：延迟最优" --------------------------------

def t_dbt_ar(N, M, alpha, beta):  # eq. model-algo-dbt-ar
    return 2 * log2(N) * alpha + log2(N) * M / beta


def allreduce_latency_coeff(algo: str, N: int) -> float:
    """Coefficient of alpha (table tbl-model-algo-allreduce-compare)."""
    return {"ring": 2 * (N - 1), "rhd": 2 * log2(N), "dbt": 2 * log2(N)}[algo]


def allreduce_bandwidth_coeff(algo: str, N: int) -> float:
    """Coefficient of M/beta (same table)."""
    return {"ring": 2 * (N - 1) / N, "rhd": 2 * (N - 1) / N, "dbt": log2(N)}[algo]


def crossover_ring_dbt(N, alpha, beta):  # eq. model-algo-ring-dbt-crossover
    """M* where T_ring = T_dbt; below it DBT is faster, above it Ring."""
    return 2 * alpha * beta * ((N - 1) - log2(N)) / (log2(N) - 2 * (N - 1) / N)


# ---- section "AllGather / ReduceScatter 的公式是什么" ------------------------

def t_ring_allgather(N, M, alpha, beta):  # eq. model-algo-ring-allgather
    return (N - 1) * alpha + (N - 1) / N * M / beta


def t_ring_reducescatter(N, M, alpha, beta):  # eq. model-algo-ring-reducescatter
    return (N - 1) * alpha + (N - 1) / N * M / beta


# ---- section "AllToAll 算法怎么选" -------------------------------------------

def t_a2a_pairwise(N, M, alpha, beta):  # eq. model-algo-a2a-pairwise
    return (N - 1) * (alpha + M / (N * beta))


def t_a2a_bruck(N, M, alpha, beta):  # eq. model-algo-a2a-bruck (as printed)
    return ceil_log2(N) * alpha + (N - 1) / N * M / beta


def t_a2a_ring(N, M, alpha, beta):  # eq. model-algo-a2a-ring
    return (N - 1) * alpha + (N - 1) / N * M / beta


# ---- section "Broadcast / Reduce 怎么用 Tree 算法" ----------------------------

def t_bcast_tree(N, M, alpha, beta):  # eq. model-algo-bcast-tree
    return log2(N) * (alpha + M / beta)


def t_reduce_tree(N, M, alpha, beta):  # eq. model-algo-reduce-tree
    return log2(N) * (alpha + M / beta)


# ---- busbw table (tbl-model-algo-busbw-coef) ------------------------------

def busbw_factor(coll: str, N: int) -> float:
    """busbw = algbw * factor.  Scatter is not in the table; the reading taken
    is (N-1)/N, the class of AllGather (its bandwidth bound is (N-1)M/N)."""
    return {
        "allreduce": 2 * (N - 1) / N,
        "allgather": (N - 1) / N,
        "reduce_scatter": (N - 1) / N,
        "alltoall": (N - 1) / N,
        "scatter": (N - 1) / N,
        "broadcast": 1.0,
        "reduce": 1.0,
    }[coll]


# ---- [Bcast/Scatter page] -------------------------------------------------

def bcast_latency_lower_bound(N, alpha):  # eq. bcast-delay-lb
    return ceil_log2(N) * alpha


def bcast_bandwidth_lower_bound(M, beta, d=1):  # eq. broadcast-bw-lower-bound
    """d is not defined on the page; read as the number of ports per node."""
    return M / (d * beta)


def bcast_lower_bound(N, M, alpha, beta, d=1):  # eq. bcast-combined-lb
    return max(bcast_latency_lower_bound(N, alpha), bcast_bandwidth_lower_bound(M, beta, d))


def t_chain_bcast(N, M, alpha, beta):  # eq. chain-bcast
    return (N - 1) * (alpha + M / beta)


def t_binomial_bcast(N, M, alpha, beta):  # eq. binomial-bcast
    return ceil_log2(N) * (alpha + M / beta)


def t_pipe_chain_bcast(N, M, alpha, beta, k):  # eq. pipe-chain-bcast
    return (N + k - 2) * (alpha + M / (k * beta))


def k_star_chain_printed(N, M, alpha, beta):
    """Optimal chunk count as printed beside eq. pipe-chain-bcast."""
    return math.sqrt((N - 1) * M / (alpha * beta))


def k_star_chain_derived(N, M, alpha, beta):
    """dT/dk = 0 on eq. pipe-chain-bcast: alpha = (N-2) M / (k**2 beta)."""
    return math.sqrt((N - 2) * M / (alpha * beta))


def t_pipe_tree_bcast(N, M, alpha, beta, k):  # eq. pipe-tree-bcast
    return (ceil_log2(N) + k - 1) * (alpha + M / (k * beta))


def scatter_latency_lower_bound(N, alpha):  # eq. onetoall-scatter-delay-lb
    return ceil_log2(N) * alpha


def scatter_bandwidth_lower_bound(N, M, beta, d=1):  # eq. onetoall-scatter-bw-lb
    return (N - 1) * M / (N * d * beta)


def t_scatter_naive(N, M, alpha, beta):  # eq. onetoall-scatter-naive
    return (N - 1) * alpha + (N - 1) * M / (N * beta)


def binomial_scatter_bw_sum(N, M, beta):
    """Left side of eq. onetoall-scatter-binomial-bw-sum, summed term by term."""
    L = ceil_log2(N)
    return sum(M / 2 ** j for j in range(1, L + 1)) / beta


def t_binomial_scatter(N, M, alpha, beta):  # eq. binomial-scatter
    return ceil_log2(N) * alpha + (N - 1) * M / (N * beta)


def t_gather(N, M, alpha, beta):  # eq. onetoall-gather-scatter-duality
    return t_binomial_scatter(N, M, alpha, beta)
