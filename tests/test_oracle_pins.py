"""The oracle against what the pages and mathematics fix (CPU only).

Pins: the printed tables (binomial Broadcast / Scatter, the N=8 AllReduce
comparison, busbw factors, latency examples, the 14.4 MB crossover), closed
forms, brute force on integer data (any association is exact), hand-derived
order witnesses, library routines for data movement and for bf16 / fp16
rounding, and a planted-fault check that the pins catch a broken schedule.

Every pin on a schedule runs against both oracles (the ``sim`` fixture: the
C++ simulation and the numpy one).
"""
import math

import numpy as np
import pytest
import torch

from oracle import cost_model as cm
from oracle import cxx, numerics, orders, schedules
from oracle.partition import chunk_elems, chunk_range
from synthetic_inputs import int32_bits, rank_buffers, small_ints_f32

from . import witness


# ----------------------------------------------------------------------------
# printed tables
# ----------------------------------------------------------------------------

def test_binomial_broadcast_table_n8(golden, sim):
    want = sorted((int(s) - 1, int(a), int(b)) for s, a, b in golden("binomial_broadcast_n8.txt"))
    A = np.arange(64, dtype=np.int32)
    res = sim.broadcast(A, 8, 0, "binomial", "i32")
    assert res.log.table() == want
    assert res.nsteps == 3


def test_binomial_scatter_table_n8(golden, sim):
    rows = golden("binomial_scatter_n8.txt")
    rc = 16
    M = 8 * rc * 4
    A = np.arange(8 * rc, dtype=np.int32)
    res = sim.scatter(A, 8, 0, "binomial", "i32")
    got = sorted((t.step, t.src, t.dst, tuple(sorted(t.chunks)), t.nbytes) for t in res.log.records)
    want = sorted((int(s) - 1, int(a), int(b), tuple(int(c) for c in ch.split(",")), M // int(den))
                  for s, a, b, ch, den in rows)
    assert got == want
    # step j moves M / 2**j per message; the bandwidth term sums to (N-1)M/N
    assert res.log.bandwidth_bytes() == (8 - 1) * M // 8
    assert res.log.bytes_sent_by(0) == (8 - 1) * M // 8


def test_allreduce_compare_table_n8(golden, sim):
    N, count = 8, 8 * 64
    M = count * 4
    xs = rank_buffers("small_ints_f32", 1, N, count)
    for algo, lat, bw in golden("allreduce_compare_n8.txt"):
        res = sim.allreduce(xs, algo, "f32")
        assert res.nsteps == int(lat), algo
        assert res.log.bandwidth_bytes() / M == pytest.approx(float(bw), rel=0, abs=1e-12), algo
        assert cm.allreduce_latency_coeff(algo, N) == pytest.approx(float(lat))
        assert cm.allreduce_bandwidth_coeff(algo, N) == pytest.approx(float(bw))


def test_latency_examples(golden, sim):
    for algo, N, lat in golden("latency_examples.txt"):
        assert cm.allreduce_latency_coeff(algo, int(N)) == pytest.approx(float(lat))
    # the schedules themselves at N = 64 (small buffers)
    xs = [np.full(64 * 4, r, dtype=np.int32) for r in range(64)]
    assert sim.allreduce(xs, "rhd", "i32").nsteps == 12
    assert sim.allreduce(xs, "ring", "i32").nsteps == 126


def test_ring_dbt_crossover(golden):
    (N, a, b, mstar), = golden("ring_dbt_crossover.txt")
    N, a, b, mstar = int(N), float(a), float(b), float(mstar)
    m = cm.crossover_ring_dbt(N, a, b)
    assert m == pytest.approx(mstar, rel=1e-9)
    assert cm.t_ring_ar(N, m, a, b) == pytest.approx(cm.t_dbt_ar(N, m, a, b), rel=1e-12)
    assert cm.t_dbt_ar(N, 0.5 * m, a, b) < cm.t_ring_ar(N, 0.5 * m, a, b)
    assert cm.t_dbt_ar(N, 2.0 * m, a, b) > cm.t_ring_ar(N, 2.0 * m, a, b)


def test_busbw_factors(golden):
    for coll, f in golden("busbw_factors.txt"):
        assert cm.busbw_factor(coll, 8) == pytest.approx(float(f))


# ----------------------------------------------------------------------------
# closed forms and identities of the cost model
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("N", [2, 4, 8, 16, 64, 1024])
def test_cost_identities(N):
    a, b = 3e-6, 1e11
    for M in (1e3, 1e6, 1e9):
        # T_Ring-AR = T_RS + T_AG
        assert cm.t_ring_ar(N, M, a, b) == pytest.approx(cm.t_ring_rs(N, M, a, b) + cm.t_ring_ag(N, M, a, b))
        # the halving / doubling sums equal their printed closed forms
        closed = math.log2(N) * a + (N - 1) / N * M / b
        assert cm.t_rhd_rs(N, M, a, b) == pytest.approx(closed, rel=1e-12)
        assert cm.t_rhd_ag(N, M, a, b) == pytest.approx(closed, rel=1e-12)
        assert cm.t_rhd_ar(N, M, a, b) == pytest.approx(cm.t_rhd_rs(N, M, a, b) + cm.t_rhd_ag(N, M, a, b))
        # binomial scatter: sum_j M/2^j = (N-1)M/N
        assert cm.binomial_scatter_bw_sum(N, M, b) == pytest.approx((N - 1) * M / (N * b), rel=1e-12)
        # binomial scatter meets both scatter lower bounds
        assert cm.t_binomial_scatter(N, M, a, b) == pytest.approx(
            cm.scatter_latency_lower_bound(N, a) + cm.scatter_bandwidth_lower_bound(N, M, b))
        # gather = scatter (duality)
        assert cm.t_gather(N, M, a, b) == cm.t_binomial_scatter(N, M, a, b)
        # the three AllToAll formulas share the bandwidth term
        bw = (N - 1) / N * M / b
        assert cm.t_a2a_pairwise(N, M, a, b) == pytest.approx((N - 1) * a + bw)
        assert cm.t_a2a_bruck(N, M, a, b) == pytest.approx(cm.ceil_log2(N) * a + bw)


def test_pipelined_chain_optimum():
    """dT/dk = 0 on eq. pipe-chain-bcast gives sqrt((N-2)M/(alpha beta)); the
    printed optimum uses N-1 (a reading noted in the design notes)."""
    N, M, a, b = 8, 64e6, 5e-6, 450e9
    ks = np.linspace(1, 400, 400001)
    T = np.array([cm.t_pipe_chain_bcast(N, M, a, b, k) for k in ks[::50]])
    k_num = ks[::50][int(np.argmin(T))]
    assert k_num == pytest.approx(cm.k_star_chain_derived(N, M, a, b), rel=2e-3)
    assert abs(cm.k_star_chain_printed(N, M, a, b) - k_num) > 1.0
    # large messages: T* -> M / beta
    Mbig = 1e13
    kb = cm.k_star_chain_derived(N, Mbig, a, b)
    assert cm.t_pipe_chain_bcast(N, Mbig, a, b, kb) / (Mbig / b) == pytest.approx(1.0, rel=2e-2)
    # the pipelined tree never needs more steps than the pipelined chain
    assert cm.t_pipe_tree_bcast(N, M, a, b, 16) < cm.t_pipe_chain_bcast(N, M, a, b, 16)


def test_bcast_lower_bounds():
    N, M, a, b = 8, 1e6, 5e-6, 450e9
    lb = cm.bcast_lower_bound(N, M, a, b)
    assert cm.t_binomial_bcast(N, M, a, b) >= lb
    assert cm.t_chain_bcast(N, M, a, b) >= cm.t_binomial_bcast(N, M, a, b)
    assert cm.t_bcast_tree(N, M, a, b) == pytest.approx(cm.t_binomial_bcast(N, M, a, b))


@pytest.mark.parametrize("N", [3, 4, 8, 16, 64])
def test_binomial_and_scatter_allgather_broadcast_cross_where_derived(N):
    """The binomial Broadcast (eq. binomial-bcast) and Scatter + AllGather
    (eq. binomial-scatter plus eq. model-algo-ring-allgather) cost the same at
    M* = (N-1) alpha beta / (ceil(log2 N) - 2(N-1)/N), derived by hand from
    L(alpha + M/beta) = (L + N - 1) alpha + 2 (N-1) M / (N beta): 5.6 alpha
    beta at N = 8.  (The Bcast/Scatter page's rule of thumb below its
    comparison table, M* ~ 2 N alpha beta, is context only: 16 alpha beta at
    N = 8.)  Below it the tree is cheaper, above it Scatter + AllGather."""
    a, b = 5e-6, 450e9
    L = (N - 1).bit_length()
    Ms = (N - 1) * a * b / (L - 2 * (N - 1) / N)

    def sag(M):
        return cm.t_binomial_scatter(N, M, a, b) + cm.t_ring_allgather(N, M, a, b)

    assert cm.t_binomial_bcast(N, Ms, a, b) == pytest.approx(sag(Ms), rel=1e-12)
    assert cm.t_binomial_bcast(N, Ms / 2, a, b) < sag(Ms / 2)
    assert cm.t_binomial_bcast(N, Ms * 2, a, b) > sag(Ms * 2)
    if N == 8:
        assert Ms / (a * b) == pytest.approx(5.6)


@pytest.mark.parametrize("N", [2, 4, 8, 64])
def test_naive_scatter_meets_the_bandwidth_bound_not_the_latency_bound(N):
    """The root sending each rank its piece in turn (eq. onetoall-scatter-
    naive): the Bcast/Scatter page notes that its bandwidth term reaches the
    lower bound (eq. onetoall-scatter-bw-lb) while its latency term grows as
    O(N), above the ceil(log2 N) alpha of eq. onetoall-scatter-delay-lb from
    N = 3 on; the binomial Scatter meets both."""
    a, b = 5e-6, 450e9
    for M in (1e3, 1e9):
        assert cm.t_scatter_naive(N, M, 0.0, b) == pytest.approx(cm.scatter_bandwidth_lower_bound(N, M, b))
        latency = cm.t_scatter_naive(N, M, a, b) - cm.t_scatter_naive(N, M, 0.0, b)
        assert latency == pytest.approx((N - 1) * a)
        assert (latency > cm.scatter_latency_lower_bound(N, a) * (1 + 1e-9)) == (N > 2)
        assert cm.t_binomial_scatter(N, M, a, b) <= cm.t_scatter_naive(N, M, a, b) * (1 + 1e-12)


def test_two_rank_broadcast_never_prefers_scatter_allgather():
    """At N = 2 the denominator above is 0: Scatter + AllGather costs one
    more alpha than the tree's single step at every size."""
    a, b = 5e-6, 450e9
    for M in (1.0, 1e4, 1e8, 1e12):
        sag = cm.t_binomial_scatter(2, M, a, b) + cm.t_ring_allgather(2, M, a, b)
        assert sag - cm.t_binomial_bcast(2, M, a, b) == pytest.approx(a)


# ----------------------------------------------------------------------------
# schedules: step counts and bytes against the printed formulas
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("N", [2, 3, 4, 5, 8, 16])
def test_ring_and_rhd_bytes_sent(N, sim):
    count = N * 32
    M = count * 4
    xs = rank_buffers("small_ints_f32", 2, N, count)
    res = sim.allreduce(xs, "ring", "f32")
    assert res.nsteps == 2 * (N - 1)
    for r in range(N):
        assert res.log.bytes_sent_by(r) == 2 * (N - 1) * M // N
    assert res.log.bandwidth_bytes() == 2 * (N - 1) * M // N
    if N & (N - 1) == 0:
        res = sim.allreduce(xs, "rhd", "f32")
        L = N.bit_length() - 1
        assert res.nsteps == 2 * L
        for r in range(N):
            assert res.log.bytes_sent_by(r) == 2 * (N - 1) * M // N
        # round k of the halving moves M / 2^(k+1), doubling round k moves M 2^k / N
        per_step = res.log.max_message_bytes_per_step()
        assert [per_step[k] for k in range(L)] == [M >> (k + 1) for k in range(L)]
        assert [per_step[L + k] for k in range(L)] == [M * (1 << k) // N for k in range(L)]


@pytest.mark.parametrize("N", [2, 4, 8, 16])
def test_dbt_levels_and_bandwidth(N, sim):
    count = N * 32
    M = count * 4
    xs = rank_buffers("small_ints_f32", 3, N, count)
    res = sim.allreduce(xs, "dbt", "f32")
    L = N.bit_length() - 1
    assert res.nsteps == 2 * L
    assert all(t.nbytes == M // 2 for t in res.log.records)
    assert res.log.bandwidth_bytes() == L * M  # log2(N) * M / beta
    # each rank is an interior node of at most one tree
    interior = {"A": set(), "B": set()}
    for t in res.log.records:
        if t.reduce:
            interior[t.phase[-1]].add(t.dst)
    assert not (interior["A"] & interior["B"])


def test_ring_rs_ag_pieces(sim):
    N, rc = 8, 16
    xs = rank_buffers("small_ints_f32", 4, N, N * rc)
    rs = sim.reduce_scatter(xs, "ring", "f32")
    M = N * rc * 4
    assert rs.nsteps == N - 1 and rs.log.bandwidth_bytes() == (N - 1) * M // N
    ag = sim.allgather([np.arange(rc, dtype=np.float32)] * N, "ring", "f32")
    assert ag.nsteps == N - 1 and ag.log.bandwidth_bytes() == (N - 1) * M // N
    ar = sim.allreduce(xs, "ring", "f32")
    assert ar.nsteps == rs.nsteps + ag.nsteps


def test_pairwise_and_bruck_rounds(sim):
    N, B = 8, 16
    M = N * B * 4
    xs = rank_buffers("uniform_f32", 5, N, N * B)
    pw = sim.alltoall(xs, "pairwise", "f32")
    assert pw.nsteps == N - 1
    assert pw.log.bandwidth_bytes() == (N - 1) * M // N
    for i in range(N):
        assert pw.log.bytes_sent_by(i) == (N - 1) * M // N
    br = sim.alltoall(xs, "bruck", "f32")
    assert br.nsteps == 3
    # the page quotes (N-1)/N * M for Bruck's bandwidth term; the rounds carry
    # the blocks with bit k set, 4 of 8 per round at N = 8: 1.5 M, not 0.875 M
    assert br.log.bandwidth_bytes() == 3 * 4 * B * 4
    assert br.log.bandwidth_bytes() != (N - 1) * M // N
    for k, t in enumerate(sorted(br.log.records, key=lambda t: t.step)[::N]):
        assert t.dst == (t.src + (1 << t.step)) % N


def test_binomial_bcast_bandwidth(sim):
    for N in (2, 3, 5, 8, 16):
        A = np.arange(40, dtype=np.int32)
        res = sim.broadcast(A, N, 0, "binomial", "i32")
        assert res.nsteps == cm.ceil_log2(N)
        assert res.log.bandwidth_bytes() == cm.ceil_log2(N) * 160


@pytest.mark.parametrize("N", [2, 4, 8, 16])
def test_printed_times_equal_the_simulated_steps(N, sim):
    """Each schedule's printed time is the alpha-beta model summed over its
    steps: every step costs alpha plus its largest message over beta.  Summed
    over the simulated transfer log that gives the printed formula exactly, for
    the ring AllReduce, ReduceScatter and AllGather (eqs. model-algo-ring-ar,
    -ring-reducescatter, -ring-allgather), RHD and DBT (eqs. model-algo-rhd-ar,
    -dbt-ar), Pairwise AllToAll (eq. model-algo-a2a-pairwise), the binomial
    Broadcast, Scatter and Gather (eqs. binomial-bcast, binomial-scatter,
    onetoall-gather-scatter-duality) and the tree Reduce (eq.
    model-algo-reduce-tree), at powers of 2, where log2 N is whole."""
    a, b = 5e-6, 450e9
    count = N * 64
    M = count * 4

    def logged(res):
        per = res.log.max_message_bytes_per_step()
        return sum(a + per[s] / b for s in per)

    xs = rank_buffers("small_ints_f32", 7, N, count)
    blocks = [x[: count // N] for x in xs]
    cases = [
        (sim.allreduce(xs, "ring", "f32"), cm.t_ring_ar(N, M, a, b)),
        (sim.allreduce(xs, "rhd", "f32"), cm.t_rhd_ar(N, M, a, b)),
        (sim.allreduce(xs, "dbt", "f32"), cm.t_dbt_ar(N, M, a, b)),
        (sim.reduce_scatter(xs, "ring", "f32"), cm.t_ring_reducescatter(N, M, a, b)),
        (sim.allgather(blocks, "ring", "f32"), cm.t_ring_allgather(N, M, a, b)),
        (sim.alltoall(xs, "pairwise", "f32"), cm.t_a2a_pairwise(N, M, a, b)),
        (sim.broadcast(xs[0], N, 0, "binomial", "f32"), cm.t_binomial_bcast(N, M, a, b)),
        (sim.scatter(xs[0], N, 0, "binomial", "f32"), cm.t_binomial_scatter(N, M, a, b)),
        (sim.gather(blocks, 0, "binomial", "f32"), cm.t_gather(N, M, a, b)),
        (sim.reduce(xs, 0, "binomial", "f32"), cm.t_reduce_tree(N, M, a, b)),
    ]
    for i, (res, printed) in enumerate(cases):
        assert logged(res) == pytest.approx(printed, rel=1e-12), (i, logged(res), printed)


def test_ring_and_mesh_toy_example(golden, sim):
    """The hccl article's toy example (100 GB over 100 GB/s links, 32 nodes:
    Ring about 2 s, Mesh about 32 s, the root the bottleneck), against the
    simulated transfer logs scaled to that size: the busiest Ring rank sends
    2 (N-1)/N of the data (1.94 s); the Mesh root takes in the other N-1
    ranks' data (31 s), within N/(N-1) of the page's N x data / bandwidth."""
    rows = {algo: (int(n), float(t)) for algo, n, t in golden("ring_mesh_toy_n32.txt")}
    N = rows["ring"][0]
    count = N * 16
    xs = rank_buffers("small_ints_f32", 9, N, count)
    scale = 1.0 / (count * 4)  # seconds per simulated byte: the page's data takes 1 s at its bandwidth
    ring = sim.allreduce(xs, "ring", "f32").log
    t_ring = max(ring.bytes_sent_by(r) for r in range(N)) * scale
    assert t_ring == pytest.approx(2 * (N - 1) / N)
    assert t_ring == pytest.approx(rows["ring"][1], rel=1.0 / N)
    mesh = sim.allreduce(xs, "mesh", "f32").log
    t_root = max(mesh.bytes_received_by(r) for r in range(N)) * scale
    assert t_root == pytest.approx(N - 1)
    assert t_root == pytest.approx(rows["mesh"][1], rel=1.0 / N)
    # every other Mesh rank takes in one copy of the result: the root is the bottleneck
    assert sorted(mesh.bytes_received_by(r) for r in range(N))[-2] * scale == pytest.approx(1.0)


@pytest.mark.parametrize("N", [8])
def test_hbm_bytes_closed_forms(N, sim):
    """Algorithmic bytes at N = 8, fp32, M per rank."""
    count = N * 64
    M = count * 4
    xs = rank_buffers("small_ints_f32", 6, N, count)
    ar = {a: sim.allreduce(xs, a, "f32").hbm_bytes for a in ("fused", "ring", "rhd", "dbt")}
    assert ar == {"fused": 2 * N * M, "ring": 5 * (N - 1) * M, "rhd": 5 * (N - 1) * M, "dbt": 29 * M}
    assert sim.reduce_scatter(xs, "fused", "f32").hbm_bytes == (N + 1) * M
    assert sim.reduce_scatter(xs, "ring", "f32").hbm_bytes == 3 * (N - 1) * M
    sc = [x[:count // N] for x in xs]
    assert sim.allgather(sc, "ring", "f32").hbm_bytes == 2 * N * M
    assert sim.allgather(sc, "fused", "f32").hbm_bytes == (N + 1) * M
    assert sim.alltoall(xs, "fused", "f32").hbm_bytes == 2 * N * M
    assert sim.alltoall(xs, "pairwise", "f32").hbm_bytes == 2 * N * M
    assert sim.alltoall(xs, "bruck", "f32").hbm_bytes == 2 * 3 * N * M
    A = xs[0]
    assert sim.broadcast(A, N, 0, "fused", "f32").hbm_bytes == (N + 1) * M
    assert sim.broadcast(A, N, 0, "binomial", "f32").hbm_bytes == 2 * N * M
    assert sim.scatter(A, N, 0, "binomial", "f32").hbm_bytes == 3 * M + 2 * M // N
    assert sim.scatter(A, N, 0, "fused", "f32").hbm_bytes == 2 * M
    # bf16 ring with fp32 partials (rounded once on the last ReduceScatter step)
    xb = rank_buffers("small_ints_bf16", 6, N, count)
    Mb = count * 2
    assert sim.allreduce(xb, "ring", "bf16").hbm_bytes == 47 * Mb


# ----------------------------------------------------------------------------
# brute force on integer data: every association is exact
# ----------------------------------------------------------------------------

def _exact_sum(xs):
    return np.sum(np.stack([x.astype(np.int64) for x in xs]), axis=0)


@pytest.mark.parametrize("N", [1, 2, 3, 4])
def test_bruteforce_allreduce(N, sim):
    for count in range(0, 68):
        xs = [small_ints_f32(7, r, count) for r in range(N)]
        want = _exact_sum(xs).astype(np.float32)
        xb = [numerics.f32_to_bf16(small_ints_f32(8, r, count, lim=8)) for r in range(N)]
        wantb = _exact_sum([numerics.bf16_to_f32(x) for x in xb]).astype(np.float32)
        xi = [int32_bits(9, r, count) for r in range(N)]
        wanti = (_exact_sum(xi) & 0xFFFFFFFF).astype(np.uint32).view(np.int32)
        for algo in sim.ALGOS["allreduce"]:
            res = sim.allreduce(xs, algo, "f32")
            for o in res.outputs:
                assert np.array_equal(o, want), (algo, N, count)
            res = sim.allreduce(xb, algo, "bf16")
            for o in res.outputs:
                assert np.array_equal(numerics.bf16_to_f32(o), wantb), (algo, N, count)
            res = sim.allreduce(xi, algo, "i32")
            for o in res.outputs:
                assert np.array_equal(o, wanti), (algo, N, count)


@pytest.mark.parametrize("N", [1, 2, 3, 4])
def test_bruteforce_reduce_scatter_allgather(N, sim):
    for rc in range(0, 18):
        xs = [small_ints_f32(10, r, N * rc) for r in range(N)]
        total = _exact_sum(xs).astype(np.float32)
        for algo in sim.ALGOS["reduce_scatter"]:
            res = sim.reduce_scatter(xs, algo, "f32")
            for r, o in enumerate(res.outputs):
                assert np.array_equal(o, total[r * rc:(r + 1) * rc]), (algo, N, rc)
        ins = [int32_bits(11, r, rc) for r in range(N)]
        for algo in sim.ALGOS["allgather"]:
            res = sim.allgather(ins, algo, "i32")
            for o in res.outputs:
                assert np.array_equal(o, np.concatenate(ins)), (algo, N, rc)


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 7, 8])
def test_bruteforce_broadcast_scatter(N, sim):
    for root in range(N):
        for count in (0, 1, 5, 16, 37, 67):
            A = int32_bits(12, root, count)
            for algo in sim.ALGOS["broadcast"]:
                for inplace in (False, True):
                    res = sim.broadcast(A, N, root, algo, "i32", inplace=inplace)
                    for o in res.outputs:
                        assert np.array_equal(o, A), (algo, N, root, count)
        for rc in (0, 1, 3, 8):
            A = int32_bits(13, root, N * rc)
            parts = np.split(A, N) if rc else [A[:0]] * N
            for algo in sim.ALGOS["scatter"]:
                res = sim.scatter(A, N, root, algo, "i32")
                for r in range(N):
                    assert np.array_equal(res.outputs[r], parts[r]), (algo, N, root, rc)


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 6, 7, 8, 16])
def test_alltoall_against_block_transpose(N, sim):
    for B in (0, 1, 3, 8):
        xs = [int32_bits(14, r, N * B) for r in range(N)]
        # library special case: out_j[block i] = in_i[block j] is a transpose of
        # the (source rank, destination block) grid
        grid = np.stack(xs).reshape(N, N, B)
        want = np.transpose(grid, (1, 0, 2)).reshape(N, N * B)
        for algo in sim.ALGOS["alltoall"]:
            res = sim.alltoall(xs, algo, "i32")
            for j in range(N):
                assert np.array_equal(res.outputs[j], want[j]), (algo, N, B)
            twice = sim.alltoall(res.outputs, algo, "i32")
            for j in range(N):
                assert np.array_equal(twice.outputs[j], xs[j])


# ----------------------------------------------------------------------------
# rounding: bound, order witnesses, closed-form association trees
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("N", [2, 4, 8, 16])
def test_allreduce_within_recursive_summation_bound(N, sim):
    count = 997
    xs = rank_buffers("uniform_f32", 15, N, count)
    exact = np.sum(np.stack([x.astype(np.float64) for x in xs]), axis=0)
    absum = np.sum(np.stack([np.abs(x.astype(np.float64)) for x in xs]), axis=0)
    u = 2.0 ** -24
    gamma = (N - 1) * u / (1 - (N - 1) * u)
    for algo in sim.ALGOS["allreduce"]:
        res = sim.allreduce(xs, algo, "f32")
        for o in res.outputs[1:]:
            assert numerics.same_bits(o, res.outputs[0])
        err = np.abs(res.outputs[0].astype(np.float64) - exact)
        assert np.all(err <= gamma * absum + 1e-30), algo


def _witness_inputs(vals, count=16):
    return [np.full(count, v, dtype=np.float32) for v in vals]


def test_order_witnesses_n4(golden, sim):
    for row in golden("order_witness_n4.txt"):
        vals = [float(v) for v in row[1:5]]
        algo = row[5]
        want = np.repeat(np.array([float(v) for v in row[6:10]], dtype=np.float32), 4)
        xs = _witness_inputs(vals)
        if algo.startswith("rs_"):
            res = sim.reduce_scatter(xs, algo[3:], "f32")
            got = np.concatenate(res.outputs)
        else:
            res = sim.allreduce(xs, algo, "f32")
            got = res.outputs[0]
            for o in res.outputs:
                assert numerics.same_bits(o, got)
        assert np.array_equal(got, want), (row[0], algo, got)


def _witness_results(sim, wid, N, algo, xs):
    if algo.startswith("rs_"):
        res = sim.reduce_scatter(xs, algo[3:], "f32")
        return [np.concatenate(res.outputs)]
    return sim.allreduce(xs, algo, "f32").outputs


def test_order_witnesses_n8_and_foldin(golden, sim):
    """Hand-derived witnesses: the N = 8 Ring, RHD and both Double Binary
    Trees, and RHD's fold-in at N = 5, 6, 7 (every rank's output)."""
    for wid, N, algo, xs, want in witness.rows(golden):
        for r, got in enumerate(_witness_results(sim, wid, N, algo, xs)):
            assert np.array_equal(got, want), (wid, N, algo, r, got)


def test_order_witnesses_n8_and_foldin_closed_forms(golden):
    """The same witnesses against both closed-form statements of the trees."""
    for wid, N, algo, xs, want in witness.rows(golden):
        count = len(xs[0])
        for closed in (orders, cxx):
            if algo.startswith("rs_"):
                got = closed.reduce_scatter_at(xs, algo[3:], count // N, "f32", np.arange(count))
            else:
                got = closed.allreduce_at(xs, algo, count, "f32", np.arange(count))
            assert np.array_equal(got, want), (wid, N, algo, closed.__name__, got)


def test_planted_rhd_mapping_fault_is_caught(monkeypatch, golden):
    """Placing virtual rank 1 on the wrong real rank (a plausible mistake in
    the fold-in's mapping) turns a fold-in witness red."""
    real = schedules.rhd_virtual_ranks

    def swapped(N):
        P, r, m = real(N)
        m = list(m)
        m[1], m[2] = m[2], m[1]
        return P, r, m

    monkeypatch.setattr(schedules, "rhd_virtual_ranks", swapped)
    failed = [wid for wid, N, algo, xs, want in witness.rows(golden)
              if algo == "rhd" and N in (5, 6, 7)
              and not np.array_equal(schedules.allreduce(xs, "rhd", "f32").outputs[0], want)]
    assert failed


def test_planted_dbt_tree_fault_is_caught(monkeypatch, golden):
    """Building tree B as a copy of tree A instead of its mirror, or summing a
    node's children before adding its own value, turns an N = 8 witness red."""
    real = schedules.dbt_trees

    def unmirrored(N, count, esize):
        (na, fa, ra), (nb, fb, rb) = real(N, count, esize)
        return [(na, fa, ra), (nb, fa, rb)]

    monkeypatch.setattr(schedules, "dbt_trees", unmirrored)
    failed = [wid for wid, N, algo, xs, want in witness.rows(golden)
              if algo == "dbt" and not np.array_equal(schedules.allreduce(xs, "dbt", "f32").outputs[0], want)]
    assert failed
    monkeypatch.undo()
    # the right-hand association: children summed first, then the node's own value
    def kids_first(tree):
        if isinstance(tree, int):
            return tree
        a, b = tree
        if isinstance(a, tuple) and isinstance(a[0], int):  # ((own, left), right)
            return (a[0], (kids_first(a[1]), kids_first(b)))
        return (kids_first(a), kids_first(b))

    wrong = 0
    for wid, N, algo, xs, want in witness.rows(golden):
        if algo != "dbt":
            continue
        count = len(xs[0])
        half = count // 2
        for lo, hi in ((0, half), (half, count)):
            t = kids_first(orders.allreduce_tree("dbt", N, count, "f32", lo))
            cols = {r: xs[r][lo:hi] for r in range(N)}
            if not np.array_equal(orders.evaluate(t, cols), want[lo:hi]):
                wrong += 1
    assert wrong


@pytest.mark.parametrize("N", [2, 3, 4, 5, 7, 8, 16])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_closed_form_trees_match_simulation(N, dtype, sim):
    esz = numerics.ESIZE[dtype]
    for count in (N * 8 * 3 + 5, 203):
        kind = "uniform_f32" if dtype == "f32" else "uniform_bf16"
        xs = rank_buffers(kind, 16 + N, N, count)
        idx = np.arange(count)
        for algo in sim.ALGOS["allreduce"]:
            res = sim.allreduce(xs, algo, dtype)
            for closed in (orders, cxx):  # both closed-form statements of the trees
                want = closed.allreduce_at(xs, algo, count, dtype, idx)
                assert numerics.same_bits(res.outputs[0], want), (algo, N, count, closed.__name__)
        rc = 13
        xr = rank_buffers(kind, 30 + N, N, N * rc)
        for algo in sim.ALGOS["reduce_scatter"]:
            res = sim.reduce_scatter(xr, algo, dtype)
            for closed in (orders, cxx):
                want = closed.reduce_scatter_at(xr, algo, rc, dtype, np.arange(N * rc))
                assert numerics.same_bits(np.concatenate(res.outputs), want), (algo, N, closed.__name__)
    assert chunk_elems(0, N, esz) == 0


@pytest.mark.parametrize("N", [3, 5, 8])
def test_witnesses_distinguish_orders(N, sim):
    """Each schedule's tree differs from the rank-order fold on some witness,
    so bit-exact agreement with the oracle pins the association, not just the sum."""
    count = N * 4 * 2
    for algo in ("ring", "dbt", "rhd"):
        if algo == "rhd" and N == 3:
            continue  # folded RHD on 3 ranks is (x0 + x1) + x2, the rank-order fold
        distinct = False
        for a in range(N):
            for b in range(N):
                for c in range(N):
                    if len({a, b, c}) < 3:
                        continue
                    vals = [0.0] * N
                    vals[a], vals[b], vals[c] = 2.0 ** 24, -(2.0 ** 24), 1.0
                    xs = _witness_inputs(vals, count)
                    r1 = sim.allreduce(xs, algo, "f32").outputs[0]
                    r0 = sim.allreduce(xs, "fused", "f32").outputs[0]
                    if not np.array_equal(r1, r0):
                        distinct = True
                        break
                if distinct:
                    break
            if distinct:
                break
        assert distinct, algo


# ----------------------------------------------------------------------------
# partition, bf16 rules
# ----------------------------------------------------------------------------

def test_partition_covers_once():
    for N in range(1, 17):
        for count in list(range(0, 70)) + [4096, 4097, 10 ** 6 + 3]:
            for esz in (2, 4):
                seen = 0
                prev_hi = 0
                for c in range(N):
                    lo, hi = chunk_range(c, count, N, esz)
                    assert lo == prev_hi and hi >= lo
                    assert (lo * esz) % 16 == 0 or lo == count
                    seen += hi - lo
                    prev_hi = hi
                assert seen == count
                if count % (N * 16 // esz) == 0:
                    assert all(chunk_range(c, count, N, esz)[1] - chunk_range(c, count, N, esz)[0]
                               == count // N for c in range(N))


def test_bf16_rounding_matches_library():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(100000).astype(np.float32),
        (rng.standard_normal(10000) * 1e-40).astype(np.float32),   # subnormals
        (rng.uniform(-1, 1, 10000) * 3.3e38).astype(np.float32),    # near overflow
        np.array([0.0, -0.0, np.inf, -np.inf, 3.3895314e38, -3.3895314e38,
                  1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9], dtype=np.float32),
    ])
    # exact ties: the dropped half is 0x8000
    u = rng.integers(0, 2 ** 31, 10000, dtype=np.uint64).astype(np.uint32) & np.uint32(0x7F7F0000)
    x = np.concatenate([x, (u | np.uint32(0x8000)).view(np.float32)])
    lib = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for impl in (numerics, cxx):
        ours = impl.f32_to_bf16(x)
        assert np.array_equal(ours, lib), impl.__name__
        back = impl.bf16_to_f32(ours)
        assert np.array_equal(back, torch.from_numpy(ours.view(np.int16)).view(torch.bfloat16).float().numpy())
        nan = np.array([np.nan, -np.nan], dtype=np.float32)
        assert np.all(np.isnan(impl.bf16_to_f32(impl.f32_to_bf16(nan))))
    # every bf16 pattern widens exactly (NaNs stay NaN)
    allb = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    wide = torch.from_numpy(allb.view(np.int16)).view(torch.bfloat16).float().numpy()
    got = cxx.bf16_to_f32(allb)
    fin = ~np.isnan(wide)
    assert np.array_equal(got[fin].view(np.uint32), wide[fin].view(np.uint32))
    assert np.all(np.isnan(got[~fin]))


def test_f16_conversions_of_the_cxx_oracle_match_library():
    """The C++ oracle writes its binary16 conversions from the format; they
    must equal numpy's (a library routine): every binary16 pattern widens
    exactly, and narrowing rounds to nearest even, including ties, the
    subnormal range, the underflow tie at 2^-25 and overflow at 65520."""
    allh = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    lib_wide = allh.view(np.float16).astype(np.float32)
    got = cxx.f16_bits_to_f32(allh)
    fin = ~np.isnan(lib_wide)
    assert np.array_equal(got[fin].view(np.uint32), lib_wide[fin].view(np.uint32))
    assert np.all(np.isnan(got[~fin]))
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(200000).astype(np.float32) * np.float32(100.0),
        (rng.uniform(-1, 1, 50000) * 7e-5).astype(np.float32),       # around the subnormal halves
        (rng.uniform(-1, 1, 50000) * 7e4).astype(np.float32),        # around overflow
        (rng.uniform(-1, 1, 20000) * 1e-7).astype(np.float32),       # below the smallest subnormal
        np.array([0.0, -0.0, np.inf, -np.inf, 65504.0, 65519.996, 65520.0, -65520.0, 2.0 ** -24, 2.0 ** -25,
                  -(2.0 ** -25), 2.0 ** -25 * 1.0000001, 3 * 2.0 ** -25, 2.0 ** -14, 2.0 ** -14 - 2.0 ** -25],
                 dtype=np.float32),
    ])
    # exact ties of the normal range: the 13 dropped bits are 0x1000
    u = rng.integers(0x38800000, 0x477FE000, 20000, dtype=np.uint64).astype(np.uint32) & np.uint32(0xFFFFE000)
    x = np.concatenate([x, (u | np.uint32(0x1000)).view(np.float32)])
    # every representable half plus and minus a hair, and the midpoints between neighbours
    fin_h = lib_wide[fin & np.isfinite(lib_wide)]
    mids = ((fin_h[:-1].astype(np.float64) + fin_h[1:].astype(np.float64)) / 2).astype(np.float32)
    x = np.concatenate([x, fin_h, np.nextafter(fin_h, np.float32(np.inf)), mids])
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    got = cxx.f32_to_f16_bits(x)
    assert np.array_equal(got, want), np.nonzero(got != want)[0][:5]
    # NaN: quiet NaN, sign kept
    nan = np.array([np.nan, -np.nan], dtype=np.float32)
    h = cxx.f32_to_f16_bits(nan)
    assert np.all((h & 0x7E00) == 0x7E00) and (h[1] & 0x8000) and not (h[0] & 0x8000)


def test_bf16_allreduce_one_rounding(sim):
    """bf16: fp32 accumulation in the schedule's order, one rounding at the end:
    within 1 bf16 ulp of the rounded direct-order fp32 sum, bit-exact to it for
    the fused order."""
    N, count = 8, 4096
    xs = rank_buffers("normal_bf16", 17, N, count, sigma=1e-3)
    wide = [numerics.bf16_to_f32(x) for x in xs]
    direct = wide[0].copy()
    for w in wide[1:]:
        direct = direct + w
    ref = numerics.f32_to_bf16(direct)
    exact = np.sum(np.stack([w.astype(np.float64) for w in wide]), axis=0)
    absum = np.sum(np.stack([np.abs(w.astype(np.float64)) for w in wide]), axis=0)
    for algo in sim.ALGOS["allreduce"]:
        out = sim.allreduce(xs, algo, "bf16").outputs[0]
        if algo == "fused":
            assert np.array_equal(out, ref)
        if algo == "ring_hop":
            # a rounding to bf16 (unit roundoff 2^-8) after each of N-1 hops and at the end
            err = np.abs(numerics.bf16_to_f32(out).astype(np.float64) - exact)
            assert np.all(err <= N * 2.0 ** -8 * absum), algo
            continue
        ordered = lambda b: np.where(b & 0x8000, 0x8000 - (b.astype(np.int64) & 0x7FFF), b.astype(np.int64) + 0x8000)
        assert np.max(np.abs(ordered(out) - ordered(ref))) <= 1, algo


# ----------------------------------------------------------------------------
# planted faults: the pins catch a broken schedule
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("algo", ["ring", "rhd", "dbt"])
def test_planted_schedule_fault_is_caught(monkeypatch, algo):
    """Losing any step's messages, or delivering a reduce step twice, breaks
    the brute-force pin (both oracles)."""
    N, count = 4, 64
    xs = [small_ints_f32(18, r, count) for r in range(N)]
    want = _exact_sum(xs).astype(np.float32)
    clean = schedules.allreduce(xs, algo, "f32")
    for t in clean.log.steps():
        kinds = [("drop_step", t)]
        if any(r.reduce for r in clean.log.records if r.step == t):
            kinds.append(("dup_step", t))
        for kind, step in kinds:
            monkeypatch.setattr(schedules, "_FAULT", {kind: step})
            res = schedules.allreduce(xs, algo, "f32")
            assert not all(np.array_equal(o, want) for o in res.outputs), (algo, kind, step)
            monkeypatch.setattr(schedules, "_FAULT", None)
            with cxx.fault(kind, step):
                res = cxx.allreduce(xs, algo, "f32")
            assert not all(np.array_equal(o, want) for o in res.outputs), ("cxx", algo, kind, step)
    for impl in (schedules, cxx):
        assert all(np.array_equal(o, want) for o in impl.allreduce(xs, algo, "f32").outputs)
