"""The library's host side, without a GPU.

* libvcoll.so loads and exports every function include/vc.h declares;
* argument checks reject bad calls before any CUDA call;
* every step plan the library would launch, replayed on the CPU, gives the
  oracle's results bit for bit, moves data between exactly the ranks the
  oracle's schedule does in the same steps, and has no intra-step hazards.
"""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import collective_communication_algorithms_virtual_gb300 as vc
from collective_communication_algorithms_virtual_gb300 import build as vcbuild
from oracle import cost_model, schedules
from synthetic_inputs import int32_bits, rank_buffers

from .plan_replay import DT, ESZ, NPT, Memory, get_plan, hazards, oracle_transfers, run_plan, transfers

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    vcbuild.build()
    yield


def header_functions():
    text = open(os.path.join(ROOT, "include", "vc.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(vc_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    names = header_functions()
    assert "vc_allreduce" in names and len(names) >= 10
    out = subprocess.run(["nm", "-D", "--defined-only", vc.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (vc_\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    L = vc.lib()
    for n in names:
        assert hasattr(L, n)


def test_status_strings_and_version():
    assert vc.vc_status_string(0) == "VC_SUCCESS"
    assert vc.vc_status_string(2) == "VC_ERR_UNSUPPORTED"
    assert vc.vc_version() >= 100


def test_single_launch_limit_is_settable_without_a_gpu():
    old = vc.vc_get_single_launch()
    try:
        assert old == 768 << 10  # VC_SINGLE_LAUNCH_DEFAULT
        for v in (0, 1, 4096, vc.SINGLE_LAUNCH_ALWAYS):
            vc.vc_set_single_launch(v)
            assert vc.vc_get_single_launch() == v
        assert vc.lib().vc_get_single_launch(None) == 1  # VC_ERR_INVALID_ARG
    finally:
        vc.vc_set_single_launch(old)


def test_busbw_factors_match_cost_model():
    for coll in ("allreduce", "reduce_scatter", "allgather", "alltoall", "broadcast", "scatter"):
        for N in (1, 2, 8, 16, 64):
            assert vc.vc_busbw_factor(coll, N) == pytest.approx(cost_model.busbw_factor(coll, N))
    assert vc.vc_busbw_factor("allreduce", 0) == 0.0


# ----------------------------------------------------------------------------
# argument checks (fake pointer values: these calls must fail before touching them)
# ----------------------------------------------------------------------------

def _arr(vals):
    return (ctypes.c_void_p * len(vals))(*[ctypes.c_void_p(v) for v in vals])


def test_invalid_arguments_rejected_on_host():
    L = vc.lib()
    good = _arr([0x10000 * (i + 1) for i in range(4)])
    outs = _arr([0x1000000 + 0x10000 * i for i in range(4)])
    F32, SUM, RING, FUSED = 0, 0, 1, 0
    assert L.vc_allreduce(None, outs, 4, 16, F32, SUM, RING, None) == vc.binding.VC_ERR_INVALID_ARG
    assert L.vc_allreduce(good, None, 4, 16, F32, SUM, RING, None) == vc.binding.VC_ERR_INVALID_ARG
    assert L.vc_allreduce(good, outs, 0, 16, F32, SUM, RING, None) == vc.binding.VC_ERR_INVALID_ARG
    assert L.vc_allreduce(good, outs, 65, 16, F32, SUM, RING, None) == vc.binding.VC_ERR_INVALID_ARG
    assert L.vc_allreduce(good, outs, 4, 16, 7, SUM, RING, None) == vc.binding.VC_ERR_INVALID_ARG
    assert L.vc_allreduce(good, outs, 4, 16, F32, 7, RING, None) == vc.binding.VC_ERR_INVALID_ARG
    assert L.vc_allreduce(good, outs, 4, 16, F32, SUM, 99, None) == vc.binding.VC_ERR_INVALID_ARG
    # RHD and DBT are not ReduceScatters
    assert L.vc_reduce_scatter(good, outs, 4, 16, F32, SUM, 2, None) == vc.binding.VC_ERR_UNSUPPORTED
    assert "not defined" in vc.vc_last_error()
    assert L.vc_reduce_scatter(good, outs, 4, 16, F32, SUM, 3, None) == vc.binding.VC_ERR_UNSUPPORTED
    assert L.vc_alltoall(good, outs, 4, 16, F32, 3, None) == vc.binding.VC_ERR_UNSUPPORTED  # DBT
    assert L.vc_allgather(good, outs, 4, 16, F32, 11, None) == vc.binding.VC_ERR_UNSUPPORTED  # MESH
    # roots
    assert L.vc_broadcast(ctypes.c_void_p(0x10000), outs, 4, 16, F32, 4, FUSED, None) == vc.binding.VC_ERR_INVALID_ARG
    assert L.vc_scatter(ctypes.c_void_p(0x10000), outs, 4, 16, F32, -1, FUSED, None) == vc.binding.VC_ERR_INVALID_ARG
    # null buffers
    assert L.vc_allreduce(_arr([0x10000, 0, 0x30000, 0x40000]), outs, 4, 16, F32, SUM, RING, None) == 1
    # overlapping outputs, outputs overlapping inputs
    ov = _arr([0x1000000, 0x1000000 + 32, 0x2000000, 0x3000000])
    assert L.vc_allreduce(good, ov, 4, 16, F32, SUM, RING, None) == vc.binding.VC_ERR_INVALID_ARG
    assert "overlap" in vc.vc_last_error()
    cross = _arr([0x10000 * 2, 0x2000000, 0x3000000, 0x4000000])  # recv[0] == send[1]
    assert L.vc_allreduce(good, cross, 4, 16, F32, SUM, RING, None) == vc.binding.VC_ERR_INVALID_ARG
    ag_inplace = _arr([0x10000 * (i + 1) for i in range(4)])
    assert L.vc_allgather(good, ag_inplace, 4, 16, F32, RING, None) == vc.binding.VC_ERR_INVALID_ARG
    # zero count is a no-op success
    assert L.vc_allreduce(good, outs, 4, 0, F32, SUM, RING, None) == vc.binding.VC_SUCCESS
    # counts whose byte sizes overflow: refused by the calls and by every host-side description of them
    huge = 1 << 62
    assert L.vc_allgather(good, outs, 4, huge, F32, RING, None) == vc.binding.VC_ERR_INVALID_ARG
    for fn in (lambda: vc.vc_plan_describe("allgather", "ring", 4, huge, "f32"),
               lambda: vc.vc_plan_form("allgather", "ring", 4, huge, "f32"),
               lambda: vc.vc_select_algo("allgather", 4, huge, "f32")):
        with pytest.raises(vc.VCError) as e:
            fn()
        assert e.value.status == vc.binding.VC_ERR_INVALID_ARG and "too large" in str(e.value)
    # an algorithm the collective does not define is reported first, at any size
    with pytest.raises(vc.VCError) as e:
        vc.vc_plan_form("allgather", "bruck", 4, huge, "f32")
    assert e.value.status == vc.binding.VC_ERR_UNSUPPORTED
    assert vc.vc_plan_form("allgather", "ring", 4, 1 << 40, "f32") == ("steps", 3, False)


# ----------------------------------------------------------------------------
# plan replay against the oracle
# ----------------------------------------------------------------------------

def _inputs(dtype, seed, N, n):
    if dtype == "f32":
        return rank_buffers("uniform_f32", seed, N, n)
    if dtype == "bf16":
        return rank_buffers("uniform_bf16", seed, N, n)
    return rank_buffers("int32_bits", seed, N, n)


def _check(plan, mem, res_outputs, recv_views, ctx):
    hz = hazards(plan, mem)
    assert not hz, (ctx, hz[:3])
    for r, want in enumerate(res_outputs):
        got = recv_views[r]
        assert np.array_equal(got.view(np.uint8), np.ascontiguousarray(want).view(np.uint8)), (ctx, r)


AR_CASES = [(N, c) for N in (1, 2, 3, 4, 5, 8) for c in (0, 1, 13, 64, 203)] + [(16, 1000), (7, 999), (8, 4096)]


@pytest.mark.parametrize("N,count", AR_CASES)
@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
def test_allreduce_plans_replay_to_oracle(N, count, dtype):
    xs = _inputs(dtype, 100 + N, N, count)
    for algo in schedules.ALGOS["allreduce"]:
        res = schedules.allreduce(xs, algo, dtype)
        for inplace in (False, True):
            plan, scratch = get_plan("allreduce", algo, N, count, dtype, inplace=inplace and N == 1)
            nbytes = count * ESZ[DT[dtype]]
            mem = Memory(xs, [nbytes] * N, scratch, inplace_ranks=range(N) if inplace else ())
            run_plan(plan, mem)
            outs = [mem.recv[r].view(NPT[DT[dtype]]) for r in range(N)]
            _check(plan, mem, res.outputs, outs, (algo, N, count, dtype, inplace))
        assert transfers(plan) == oracle_transfers(res.log), (algo, N, count)


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 8, 9, 16])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "i32"])
def test_reduce_scatter_allgather_plans_replay_to_oracle(N, dtype):
    for rc in (0, 1, 5, 16, 33):
        xs = _inputs(dtype, 200 + N, N, N * rc)
        for algo in schedules.ALGOS["reduce_scatter"]:
            res = schedules.reduce_scatter(xs, algo, dtype)
            plan, scratch = get_plan("reduce_scatter", algo, N, rc, dtype)
            mem = Memory(xs, [rc * ESZ[DT[dtype]]] * N, scratch)
            run_plan(plan, mem)
            _check(plan, mem, res.outputs, [mem.recv[r].view(NPT[DT[dtype]]) for r in range(N)], (algo, N, rc))
            assert transfers(plan) == oracle_transfers(res.log), (algo, N, rc)
        ins = _inputs(dtype, 300 + N, N, rc)
        for algo in schedules.ALGOS["allgather"]:
            res = schedules.allgather(ins, algo, dtype)
            plan, scratch = get_plan("allgather", algo, N, rc, dtype)
            mem = Memory(ins, [N * rc * ESZ[DT[dtype]]] * N, scratch)
            run_plan(plan, mem)
            _check(plan, mem, res.outputs, [mem.recv[r].view(NPT[DT[dtype]]) for r in range(N)], (algo, N, rc))
            assert transfers(plan) == oracle_transfers(res.log), (algo, N, rc)


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 6, 7, 8, 11, 16])
def test_broadcast_scatter_plans_replay_to_oracle(N):
    dtype = "i32"
    for root in sorted({0, 1 % N, N - 1, N // 2}):
        for count in (0, 1, 7, 64, 203):
            A = int32_bits(400 + root, N, count)
            for algo in schedules.ALGOS["broadcast"]:
                for inplace in (False, True):
                    res = schedules.broadcast(A, N, root, algo, dtype, inplace=inplace)
                    plan, scratch = get_plan("broadcast", algo, N, count, dtype, root=root, inplace=inplace)
                    send = [None] * N
                    send[root] = A
                    mem = Memory(send, [count * 4] * N, scratch, inplace_ranks=[root] if inplace else ())
                    run_plan(plan, mem)
                    _check(plan, mem, res.outputs, [mem.recv[r].view(np.int32) for r in range(N)],
                           (algo, N, root, count, inplace))
                    assert transfers(plan) == oracle_transfers(res.log), (algo, N, root, count)
        for rc in (0, 1, 5, 16):
            A = int32_bits(500 + root, N, N * rc)
            for algo in schedules.ALGOS["scatter"]:
                res = schedules.scatter(A, N, root, algo, dtype)
                plan, scratch = get_plan("scatter", algo, N, rc, dtype, root=root)
                send = [None] * N
                send[root] = A
                mem = Memory(send, [rc * 4] * N, scratch)
                run_plan(plan, mem)
                _check(plan, mem, res.outputs, [mem.recv[r].view(np.int32) for r in range(N)], (algo, N, root, rc))
                assert transfers(plan) == oracle_transfers(res.log), (algo, N, root, rc)


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 6, 7, 8, 12, 16])
@pytest.mark.parametrize("dtype", ["bf16", "i32"])
def test_alltoall_plans_replay_to_oracle(N, dtype):
    for B in (0, 1, 3, 8, 16):
        xs = _inputs(dtype, 600 + N, N, N * B)
        for algo in schedules.ALGOS["alltoall"]:
            res = schedules.alltoall(xs, algo, dtype)
            plan, scratch = get_plan("alltoall", algo, N, B, dtype)
            mem = Memory(xs, [N * B * ESZ[DT[dtype]]] * N, scratch)
            run_plan(plan, mem)
            _check(plan, mem, res.outputs, [mem.recv[r].view(NPT[DT[dtype]]) for r in range(N)], (algo, N, B))
            assert transfers(plan) == oracle_transfers(res.log), (algo, N, B)


def test_plan_step_counts_match_oracle_at_n8():
    N, count = 8, 8 * 1024
    xs = _inputs("f32", 7, N, count)
    for algo, steps in (("ring", 14), ("rhd", 6), ("dbt", 6), ("fused", 1)):
        plan, _ = get_plan("allreduce", algo, N, count, "f32")
        assert len(plan) == steps == max(1, schedules.allreduce(xs, algo, "f32").nsteps)


def test_scratch_sizes():
    # fp32 ring / rhd / dbt AllReduce keep partial sums in the receive buffers
    for algo in ("ring", "rhd", "dbt", "fused"):
        assert get_plan("allreduce", algo, 8, 1 << 20, "f32")[1] == 0
    # bf16 ring: one fp32 partial per element and rank while they take at most
    # 16 MiB per rank, above that two fp32 chunk slots per rank
    assert get_plan("allreduce", "ring", 8, 1 << 20, "bf16")[1] == 8 * (1 << 20) * 4
    assert get_plan("allreduce", "ring", 8, 1 << 24, "bf16")[1] == 8 * 2 * (1 << 21) * 4
    # Bruck at N = 8 (3 rounds) uses two working buffers of N blocks per rank
    assert get_plan("alltoall", "bruck", 8, 1024, "bf16")[1] == 2 * 8 * 8 * 1024 * 2


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_plan_bytes_equal_oracle_algorithmic_bytes(dtype):
    """The bytes the library's launches read and write are the oracle's
    algorithmic bytes for the schedule (the roofline numerator)."""
    def plan_bytes(coll, algo, N, count, root=0, inplace=False):
        entries, _, _ = vc.vc_plan_describe(coll, algo, N, count, dtype, root, inplace)
        return sum(e.n * e.nb * ESZ[e.dtype] for e in entries)

    for N in (2, 3, 8, 16):
        count = N * 1000 + 8
        xs = _inputs(dtype, 3, N, count)
        for algo in schedules.ALGOS["allreduce"]:
            assert plan_bytes("allreduce", algo, N, count) == schedules.allreduce(xs, algo, dtype).hbm_bytes
        rc = 100
        xr = _inputs(dtype, 4, N, N * rc)
        for algo in schedules.ALGOS["reduce_scatter"]:
            assert plan_bytes("reduce_scatter", algo, N, rc) == schedules.reduce_scatter(xr, algo, dtype).hbm_bytes
        for algo in schedules.ALGOS["allgather"]:
            assert plan_bytes("allgather", algo, N, rc) == schedules.allgather([x[:rc] for x in xr], algo, dtype).hbm_bytes
        for algo in schedules.ALGOS["alltoall"]:
            assert plan_bytes("alltoall", algo, N, rc) == schedules.alltoall(xr, algo, dtype).hbm_bytes
        for root in (0, N - 1):
            for algo in schedules.ALGOS["broadcast"]:
                for inplace in (False, True):
                    assert plan_bytes("broadcast", algo, N, count, root, inplace) == \
                        schedules.broadcast(xs[0], N, root, algo, dtype, inplace=inplace).hbm_bytes
            for algo in schedules.ALGOS["scatter"]:
                assert plan_bytes("scatter", algo, N, rc, root) == \
                    schedules.scatter(xr[0], N, root, algo, dtype).hbm_bytes


def test_step_merging_keeps_the_described_steps():
    """vc_set_merge_steps changes how independent steps are launched, never
    the steps vc_plan_describe reports: Pairwise AllToAll keeps its local
    round and N-1 rounds either way."""
    old = vc.vc_get_merge_steps()
    try:
        for on in (True, False):
            vc.vc_set_merge_steps(on)
            assert vc.vc_get_merge_steps() == on
            for N in (2, 5, 8):
                assert vc.vc_plan_describe("alltoall", "pairwise", N, 64, "bf16")[2] == N
    finally:
        vc.vc_set_merge_steps(old)


@pytest.mark.parametrize("N", [2, 5, 8, 64])
def test_plans_at_the_count_limit_stay_in_their_buffers(N):
    """At the largest count a plan takes (2 N x N x count x 4 bytes within
    int64) every operand of every schedule lies inside its buffer, scratch
    included, with no offset or size wrapped; one more element is refused."""
    limit = (2 ** 63 - 1) // 16 // (N * N)
    colls = {"allreduce": ("fused", "ring", "rhd", "dbt", "mesh", "ring_hop"),
             "reduce_scatter": ("fused", "ring"), "allgather": ("fused", "ring"),
             "broadcast": ("fused", "binomial", "scatter_allgather", "pipe_chain", "pipe_tree"),
             "scatter": ("fused", "binomial"), "gather": ("fused", "binomial"),
             "reduce": ("fused", "binomial"), "alltoall": ("fused", "pairwise", "bruck", "ring")}
    for coll, algos in colls.items():
        for algo in algos:
            for dtype, es in (("f32", 4), ("bf16", 2)):
                entries, scratch, _ = vc.vc_plan_describe(coll, algo, N, limit, dtype, 0, False, 3)
                send = limit * (N if coll in ("reduce_scatter", "scatter", "alltoall") else 1) * es
                recv = limit * (N if coll in ("allgather", "gather", "alltoall") else 1) * es
                size = {0: send, 1: recv, 2: scratch}
                for e in entries:
                    z = {0: 4, 1: 2, 2: 4, 3: 2}[e.dtype]
                    last = e.byte_off + (e.nb - 1) * e.stride_bytes
                    assert 0 <= min(e.byte_off, last) and e.n >= 0 and e.nb >= 1, (coll, algo, dtype, e.byte_off)
                    assert max(e.byte_off, last) + e.n * z <= size[e.buf] < 2 ** 63, (coll, algo, dtype, e.buf)
                with pytest.raises(vc.VCError):
                    vc.vc_plan_describe(coll, algo, N, limit + 1, dtype, 0, False, 3)
