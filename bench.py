#!/usr/bin/env python
"""Benchmark of the virtual-rank AllReduce algorithms on one GB300.

Workload (the AllReduce algorithm sweep): N = 8 virtual ranks, fp32 sum,
inputs uniform[-1, 1).  One step = one AllReduce of 256 MiB per rank with each
of Ring, Recursive Halving-Doubling, Double Binary Tree and the fused one-pass
kernel (out of place, each algorithm into its own output buffers).

value = busbw of the step: sum over the four AllReduces of
M * 2(N-1)/N, divided by the step time (GB/s, 1e9 B/s).  Inputs (2 GiB per
buffer set) are larger than the 129 MB L2, so no flush is needed between
steps.  The JSON line also carries per-algorithm busbw and HBM fractions at
256 MiB, the busbw-vs-message-size sweep (1 KiB .. 256 MiB per rank), the
roofline of the dominant kernel from the library's launch trace (taken over a
second pass of the same steps, so that its per-launch events do not slow the
pass that gives `value`), sampled clocks, an end-to-end number through host
buffers, and the oracle's CPU time.

Multi-GPU: replicas only (every GPU runs the same workload on its own
buffers; nothing crosses GPUs); value = all ranks' bytes / the slowest rank.

``--impl reference`` times the C++ oracle (oracle/sim.cpp, single-threaded) on
the host instead, at the same 256 MiB per rank, one AllReduce per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import shutil
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "busbw GB/s vs message size per algo (N virtual ranks); % of HBM roofline"
WORKLOAD = "allreduce_sweep_n8_f32"
NVR = 8
BYTES_PER_RANK = 256 << 20
ALGOS = ["ring", "rhd", "dbt", "fused"]
NOMINAL_HBM_GBS = 8000.0


# ----------------------------------------------------------------------------
# helpers shared by both arms (and by the multi-rank tests)
# ----------------------------------------------------------------------------

def busbw_factor(N: int) -> float:
    return 2.0 * (N - 1) / N


def step_bus_bytes(bytes_per_rank: int, nalgos: int | None = None, N: int = NVR) -> float:
    return (len(ALGOS) if nalgos is None else nalgos) * bytes_per_rank * busbw_factor(N)


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def dist_init(world: int, backend: str):
    if world > 1:
        import torch.distributed as dist

        if not dist.is_initialized():
            dist.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def reduce_max(x: float, world: int, device=None) -> float:
    """Max over ranks (one scalar, host-side timing only)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x: float, world: int, device=None) -> float:
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


def kernel_source_hash() -> str:
    """Hash of the device code (the traffic summary is valid while it matches)."""
    h = hashlib.sha256()
    with open(os.path.join(ROOT, "collective_communication_algorithms_virtual_gb300", "csrc", "kernels.cuh"), "rb") as f:
        h.update(f.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or None
    when the summary is absent or was taken on different kernel sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("source_hash") != kernel_source_hash():
        return None
    k = d.get("kernels", {}).get(kernel)
    return None if k is None else k.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.proc = None
        self.path = None
        exe = shutil.which("nvidia-smi")
        if not exe:
            return
        fd, self.path = tempfile.mkstemp(prefix="vc_clocks_", suffix=".csv")
        os.close(fd)
        cmd = [exe, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if gpu_id:
            cmd += ["-i", gpu_id]
        self.out = open(self.path, "w")
        self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)

    def stop(self) -> dict | None:
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        sm, smax, reasons = [], [], set()
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, v in zip(self.NAMES, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------
# the oracle on the host: CPU baseline and reference arm
# ----------------------------------------------------------------------------

def oracle_step(xs, algos=None) -> None:
    """One step of the workload through the C++ oracle (single-threaded)."""
    from oracle import cxx

    for algo in (algos or ALGOS):
        cxx.allreduce(xs, algo, "f32", want_log=False, want_outputs=False)


def oracle_inputs(mib_per_rank: float):
    from synthetic_inputs import uniform_pm1_f32

    count = max(4, int(mib_per_rank * (1 << 20)) // 4)
    return [uniform_pm1_f32(2, r, count) for r in range(NVR)], count * 4


ORACLE_KIND = "C++ oracle (oracle/sim.cpp, g++ -O2), single-threaded"


def time_oracle(target_s: float = 15.0, mib: float | None = None) -> dict:
    """The oracle, as it stands, on a bounded sample of the workload: whole
    steps (every algorithm) at a message size sized to the target time."""
    from oracle import cxx

    cxx.build()
    if mib is None:
        xs, _ = oracle_inputs(16)
        oracle_step(xs)  # first touch of the oracle's memory
        t0 = time.perf_counter()
        oracle_step(xs)
        t1 = time.perf_counter() - t0
        mib = int(max(1, min(256, 16 * target_s / 2 / max(t1, 1e-3))))
        del xs
    xs, nbytes = oracle_inputs(mib)
    reps, total, t_start = 0, 0.0, time.perf_counter()
    while True:
        t0 = time.perf_counter()
        oracle_step(xs)
        total += time.perf_counter() - t0
        reps += 1
        if time.perf_counter() - t_start >= target_s or reps >= 50:
            break
    busbw = step_bus_bytes(nbytes) * reps / total / 1e9
    return {"value": busbw, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": (f"{ORACLE_KIND}, 1 thread of nproc={os.cpu_count()}: N={NVR} fp32 AllReduce "
                       f"ring+rhd+dbt+fused at {nbytes / (1 << 20):g} MiB per rank, {reps} step(s), {total:.1f} s")}


def run_reference(args) -> int:
    """The oracle timed on the host cores on the GPU arm's workload: N = 8,
    fp32, 256 MiB per rank (--ref-mib changes it).  A step is one AllReduce
    with one algorithm, the algorithms taken in turn (ring, rhd, dbt, fused,
    ring, ...), so that K steps of the single-threaded oracle end within a few
    minutes; busbw = the bus bytes of the K AllReduces / their time."""
    from oracle import cxx

    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    cxx.build()
    steps, warm = args.steps, args.warmup
    mib = args.ref_mib if args.ref_mib is not None else BYTES_PER_RANK / (1 << 20)
    xs, nbytes = oracle_inputs(mib)
    for i in range(warm):
        oracle_step(xs, [ALGOS[i % len(ALGOS)]])
    t0 = time.perf_counter()
    for i in range(steps):
        oracle_step(xs, [ALGOS[i % len(ALGOS)]])
    el = time.perf_counter() - t0
    value = step_bus_bytes(nbytes, nalgos=1) * steps / el / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": steps, "warmup": warm, "ms_per_step": el / steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": config_block(nbytes),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": (f"{ORACLE_KIND}, 1 thread of nproc={os.cpu_count()}: "
                                    f"{nbytes / (1 << 20):g} MiB per rank, one AllReduce per step, "
                                    f"algorithms in turn {','.join(ALGOS)}")},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_block(bytes_per_rank: int) -> dict:
    return {"workload": WORKLOAD, "virtual_ranks": NVR, "dtype": "f32", "op": "sum",
            "bytes_per_rank": bytes_per_rank, "algos": ALGOS,
            "step": "one out-of-place AllReduce per algorithm",
            "inputs": "uniform[-1,1) fp32, seed 2, PCG64 per (seed, rank)",
            "l2": (f"inputs larger than L2 ({NVR * bytes_per_rank >> 20} MiB per buffer set), no flush"
                   if NVR * bytes_per_rank > (129 << 20) else "inputs fit in L2"),
            "parallelism": "replicas"}


# ----------------------------------------------------------------------------
# the GPU arm
# ----------------------------------------------------------------------------

def run_ours(args) -> int:
    import numpy as np
    import torch

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dist_init(world, "nccl")
    dev = torch.device("cuda", local)
    import __graft_entry__

    if rank == 0:  # one compile per node; the other ranks load what it built
        __graft_entry__.build()
    barrier(world)
    if rank != 0:
        __graft_entry__.build()  # up to date by now: only loads
    import collective_communication_algorithms_virtual_gb300 as vc
    from synthetic_inputs import uniform_pm1_f32

    if args.slice_limit is not None:  # e.g. 0: small calls take the cluster form, for profiling it
        vc.vc_set_slice_limit(args.slice_limit)
    global ALGOS
    ALGOS = [a for a in args.algos.split(",") if a]
    N, M = NVR, int(args.mib_per_rank * (1 << 20)) // 16 * 16
    count = M // 4
    host = [uniform_pm1_f32(2, r, count) for r in range(N)]
    send = [torch.from_numpy(h).to(dev) for h in host]
    recv = {a: [torch.empty_like(send[0]) for _ in range(N)] for a in ALGOS}
    stream = torch.cuda.current_stream(dev)

    def step(sz=None):
        for a in ALGOS:
            if sz is None:
                vc.vc_allreduce(send, recv[a], algo=a)
            else:
                vc.vc_allreduce([s[:sz] for s in send], [r[:sz] for r in recv[a]], algo=a)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    barrier(world)
    torch.cuda.synchronize()
    sampler = ClockSampler(uuid)
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    # The same steps again with the launch trace on, for the per-kernel
    # figures: the trace's events around every launch also keep each launch
    # from starting early behind the previous one, so `value` is timed apart.
    barrier(world)
    vc.vc_trace_enable(True)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    trace = vc.vc_trace_read(1 << 22)
    vc.vc_trace_enable(False)
    clocks = sampler.stop()
    barrier(world)
    ms_local = e0.elapsed_time(e1)
    ms_traced = reduce_max(t0.elapsed_time(t1), world, dev) / args.steps
    ms_max = reduce_max(ms_local, world, dev)
    ms_per_step = ms_max / args.steps
    value = step_bus_bytes(M) * world / (ms_per_step * 1e-3) / 1e9

    peaks = measured_peaks()
    # roofline of the dominant kernel, from the traced launches of the second pass
    by_kernel = {}
    for r in trace:
        k = by_kernel.setdefault(r["kernel"], {"launches": 0, "ms": 0.0, "bytes": 0})
        k["launches"] += 1
        k["ms"] += r["ms"]
        k["bytes"] += r["bytes"]
    dom = max(by_kernel, key=lambda k: by_kernel[k]["ms"])
    d = by_kernel[dom]
    achieved = d["bytes"] / (d["ms"] * 1e-3) / 1e9
    traffic = committed_traffic(dom)
    roofline = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "peak_source": peaks["source"],
                "traffic": traffic, "algorithmic_bytes_per_launch": d["bytes"] / d["launches"],
                "launches": d["launches"], "avg_launch_ms": d["ms"] / d["launches"],
                "frac_of_nominal_8TBs": achieved / NOMINAL_HBM_GBS,
                "kernels": {k: {"launches": v["launches"], "share": v["ms"] / sum(x["ms"] for x in by_kernel.values()),
                                "gbs": v["bytes"] / (v["ms"] * 1e-3) / 1e9} for k, v in by_kernel.items()},
                "measured": "launch trace (CUDA events around each launch on its stream) over a second pass "
                            "of the same steps", "ms_per_step_traced": ms_traced}

    out = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
           "config": config_block(M), "roofline": roofline, "gpu_launches": len(trace),  # per pass of the steps
           "clocks": clocks}

    # per-algorithm figures at 256 MiB and the message-size sweep (rank 0 only)
    if rank == 0 and not args.no_per_algo:
        out["per_algo"] = per_algo(vc, send, recv, stream, M, peaks)
        if not args.no_sweep:
            out["sweep"] = sweep(vc, send, recv, stream)
            out["alpha_beta"] = alpha_beta_fit(
                out["sweep"], auto=lambda M: vc.vc_select_algo("allreduce", N, M // 4, "f32")[0])
            out["sweep_collectives"] = sweep_collectives(vc, send, recv, stream)
        if not args.no_configs:
            out["configs"] = other_configs(vc, dev, peaks)

    # end to end: pinned host inputs -> device -> four AllReduces -> all outputs back
    if not args.no_e2e:
        out["e2e"] = e2e(vc, host, send, recv, stream, args, world, dev, M)

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = time_oracle(args.cpu_seconds)
    if rank == 0:
        emit(out, args.details_out)
    barrier(world)
    return 0


DETAIL_KEYS = ("per_algo", "sweep", "alpha_beta", "sweep_collectives", "configs")
FINAL_LINE_MAX = 2048


def _r(x, nd=4):
    """Round floats for the final line (keeps it short); other values pass."""
    if isinstance(x, float):
        return float(f"{x:.{nd}g}")
    if isinstance(x, dict):
        return {k: _r(v, nd) for k, v in x.items()}
    if isinstance(x, list):
        return [_r(v, nd) for v in x]
    return x


def final_line(out: dict) -> dict:
    """The headline JSON line: the contract's keys, a compact roofline of the
    dominant kernel, clocks, e2e and the CPU baseline, plus one busbw figure per
    algorithm.  The detail sections (per-algorithm figures, the message-size
    sweep, the alpha-beta fit, the other workload configurations) are printed
    on earlier lines; this one stays under FINAL_LINE_MAX bytes."""
    line = {k: out[k] for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config")
            if k in out}
    line["value"] = _r(out["value"], 6)
    line["ms_per_step"] = _r(out["ms_per_step"], 6)
    cfg = dict(out["config"])
    cfg.pop("inputs", None)
    line["config"] = cfg
    rf = out.get("roofline")
    if rf:
        line["roofline"] = _r({k: rf[k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic", "kernel",
                                                   "launches", "avg_launch_ms", "algorithmic_bytes_per_launch",
                                                   "peak_source") if k in rf}, 6)
    for k in ("gpu_launches", "clocks"):
        if k in out:
            line[k] = _r(out[k])
    if "e2e" in out:
        line["e2e"] = _r({k: out["e2e"][k] for k in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step",
                                                     "ms_per_step") if k in out["e2e"]})
    if "cpu_baseline" in out:
        cb = dict(out["cpu_baseline"])
        cb["sample"] = cb.get("sample", "")[:200]
        line["cpu_baseline"] = _r(cb)
    if "per_algo" in out:
        line["busbw_256MiB"] = {a: round(v["busbw"], 1) for a, v in out["per_algo"].items()}
        line["frac_of_measured_256MiB"] = {a: round(v["frac_of_measured"], 3) for a, v in out["per_algo"].items()}
    line["details"] = "earlier stdout lines, one JSON object per section: " + ",".join(
        k for k in DETAIL_KEYS if k in out)
    return line


def emit(out: dict, details_out: str | None = None) -> str:
    """Print every detail section on its own line, then the final line."""
    for k in ("roofline",) + DETAIL_KEYS:
        if k in out:
            print(json.dumps({"detail": k, k: out[k]}), flush=True)
    if details_out:
        os.makedirs(os.path.dirname(os.path.abspath(details_out)), exist_ok=True)
        with open(details_out, "w") as f:
            json.dump(out, f)
    s = json.dumps(final_line(out))
    assert len(s) <= FINAL_LINE_MAX, len(s)
    print(s, flush=True)
    return s


def time_calls(fn, stream, min_ms=20.0, max_reps=2000):
    import torch

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    fn()
    torch.cuda.synchronize()
    reps = 1
    while True:
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        if ms >= min_ms or reps >= max_reps:
            return ms / reps
        reps = min(max_reps, reps * max(2, int(min_ms / max(ms, 1e-3))))


def plan_bytes(vc, algo: str, N: int, count: int) -> int:
    """Algorithmic bytes of one AllReduce: every operand of every operation of
    the library's plan read or written once."""
    entries, _, _ = vc.vc_plan_describe("allreduce", algo, N, count, "f32")
    return sum(e.n * e.nb * 4 for e in entries)


def per_algo(vc, send, recv, stream, M, peaks):
    N = len(send)
    alg_bytes = {a: plan_bytes(vc, a, N, M // 4) for a in ALGOS}
    res = {}
    for a in ALGOS:
        ms = time_calls(lambda: vc.vc_allreduce(send, recv[a], algo=a), stream, min_ms=50.0)
        hbm = alg_bytes[a] / (ms * 1e-3) / 1e9
        res[a] = {"ms": ms, "algbw": M / (ms * 1e-3) / 1e9, "busbw": M * busbw_factor(N) / (ms * 1e-3) / 1e9,
                  "hbm_gbs": hbm, "algorithmic_bytes": alg_bytes[a],
                  "frac_of_measured": hbm / peaks["hbm_gbs"], "frac_of_nominal_8TBs": hbm / NOMINAL_HBM_GBS}
    return res


def time_graph(fn, stream, target_ms=3.0, max_reps=512):
    """Per-call time with the calls captured in a CUDA graph: GPU time only,
    no Python or launch-submission cost between calls."""
    import torch

    per = time_calls(fn, stream, min_ms=2.0, max_reps=64)
    reps = int(max(1, min(max_reps, target_ms / max(per, 1e-4))))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            fn()
    g.replay()
    torch.cuda.synchronize()
    # median of 7 separately timed replays: one stall on a shared host does not move it
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    for _ in range(7):
        e0.record(torch.cuda.current_stream())
        g.replay()
        e1.record(torch.cuda.current_stream())
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) / reps)
    del g
    return sorted(times)[3]


def plan_shape(vc, coll, algo, N, count, dtype="f32", root=0):
    """(algorithmic bytes, launched steps) of one call, from the library's plan."""
    entries, _, _ = vc.vc_plan_describe(coll, algo, N, count, dtype, root)
    return sum(e.n * e.nb * (2 if e.dtype == 1 else 4) for e in entries), len({e.step for e in entries})


def sweep(vc, send, recv, stream):
    N = len(send)
    res = {a: [] for a in ALGOS}
    top = (send[0].numel() * 4).bit_length() - 1
    for lg in range(10, top + 1):
        nbytes = 1 << lg
        sz = nbytes // 4
        for a in ALGOS:
            ins, outs = [s[:sz] for s in send], [r[:sz] for r in recv[a]]
            fn = lambda: vc.vc_allreduce(ins, outs, algo=a)
            ms_eager = time_calls(fn, stream, min_ms=5.0)
            ms = time_graph(fn, stream)
            hbm, steps = plan_shape(vc, "allreduce", a, N, sz)
            res[a].append({"bytes_per_rank": nbytes, "us": ms * 1e3, "us_eager": ms_eager * 1e3,
                           "busbw": nbytes * busbw_factor(N) / (ms * 1e-3) / 1e9,
                           "busbw_eager": nbytes * busbw_factor(N) / (ms_eager * 1e-3) / 1e9,
                           "steps": steps, "algorithmic_bytes": hbm,
                           "l2_resident": 2 * N * nbytes <= (129 << 20)})
    return res


# the other collectives' algorithms, and the busbw factor of the pages' table
# tbl-model-algo-busbw-coef for each (latency-formula page; Scatter and Gather,
# not in it, take (N-1)/N): M is the bytes per rank the table counts --
# ReduceScatter's input, AllGather's output, Broadcast's and Reduce's
# message, AllToAll's buffer, Scatter's input and Gather's output at the root
COLL_SWEEP = {"reduce_scatter": ("ring", "fused"), "allgather": ("ring", "fused"),
              "broadcast": ("binomial", "scatter_allgather", "pipe_chain", "pipe_tree", "fused"),
              "alltoall": ("pairwise", "bruck", "ring", "fused"),
              "scatter": ("binomial", "fused"), "gather": ("binomial", "fused"), "reduce": ("binomial", "fused")}
COLL_SWEEP_SIZES = (4 << 10, 64 << 10, 1 << 20, 16 << 20, 256 << 20)


def coll_busbw_factor(coll: str, N: int) -> float:
    return 1.0 if coll in ("broadcast", "reduce") else (N - 1) / N


def sweep_collectives(vc, send, recv, stream, sizes=COLL_SWEEP_SIZES):
    """busbw versus message size for ReduceScatter, AllGather, Broadcast,
    AllToAll, Scatter, Gather and Reduce, every algorithm, 8 ranks, fp32,
    graph-timed, on the bench's buffers (sends, and the first output set)."""
    N = len(send)
    outs = recv[ALGOS[0]]
    res = {}
    for coll, algos in COLL_SWEEP.items():
        for a in algos:
            rows = []
            for nbytes in sizes:
                cnt = nbytes // 4
                if cnt * 4 > send[0].numel() * 4 or cnt % N:
                    continue
                blk = cnt // N
                if coll == "reduce_scatter":
                    ins, o = [x[:cnt] for x in send], [y[:blk] for y in outs]
                    fn = lambda: vc.vc_reduce_scatter(ins, o, algo=a)
                    shape = plan_shape(vc, coll, a, N, blk)
                elif coll == "allgather":
                    ins, o = [x[:blk] for x in send], [y[:cnt] for y in outs]
                    fn = lambda: vc.vc_allgather(ins, o, algo=a)
                    shape = plan_shape(vc, coll, a, N, blk)
                elif coll == "broadcast":
                    src, o = send[0][:cnt], [y[:cnt] for y in outs]
                    if a.startswith("pipe_"):
                        fn = lambda: vc.vc_broadcast_pipelined(src, o, root=0, algo=a)
                    else:
                        fn = lambda: vc.vc_broadcast(src, o, root=0, algo=a)
                    shape = plan_shape(vc, coll, a, N, cnt)
                elif coll == "alltoall":
                    ins, o = [x[:cnt] for x in send], [y[:cnt] for y in outs]
                    fn = lambda: vc.vc_alltoall(ins, o, algo=a)
                    shape = plan_shape(vc, coll, a, N, blk)
                elif coll == "scatter":
                    src, o = send[0][:cnt], [y[:blk] for y in outs]
                    fn = lambda: vc.vc_scatter(src, o, root=0, algo=a)
                    shape = plan_shape(vc, coll, a, N, blk)
                elif coll == "gather":
                    ins, o = [x[:blk] for x in send], outs[0][:cnt]
                    fn = lambda: vc.vc_gather(ins, o, root=0, algo=a)
                    shape = plan_shape(vc, coll, a, N, blk)
                else:
                    ins, o = [x[:cnt] for x in send], outs[0][:cnt]
                    fn = lambda: vc.vc_reduce(ins, o, root=0, algo=a)
                    shape = plan_shape(vc, coll, a, N, cnt)
                ms = time_graph(fn, stream)
                rows.append({"bytes_per_rank": nbytes, "us": ms * 1e3,
                             "busbw": nbytes * coll_busbw_factor(coll, N) / (ms * 1e-3) / 1e9,
                             "algorithmic_bytes": shape[0], "steps": shape[1]})
            res[f"{coll}_{a}"] = rows
    return res


def _crossover(ta, tb, a: str, b: str, sizes=None):
    """Where two cost lines T = s * alpha + k * M cross, as a record: the
    message size per rank (bytes) or, when they never cross at a positive
    size, which algorithm the model finds faster at every size."""
    (sa, ka), (sb, kb) = ta, tb
    if ka != kb:
        m = (sb - sa) / (ka - kb)
        if m > 0:
            return {"bytes_per_rank": m, "below": a if sa < sb else b, "above": b if sa < sb else a}
    faster = a if (sa, ka) <= (sb, kb) else b
    if sa == sb and ka == kb:
        return {"bytes_per_rank": None, "never": "equal cost at every size"}
    return {"bytes_per_rank": None, "never": f"{faster} faster at every size"}


def measured_crossover(pa: list, pb: list, a: str, b: str):
    """Every swept size at which the faster of the two changes (graph-timed):
    the first of them as ``bytes_per_rank``, all of them in ``switches``."""
    first = pa[0]["us"] < pb[0]["us"]
    cur, switches = first, []
    for x, y in zip(pa, pb):
        now = x["us"] < y["us"]
        if now != cur:
            switches.append({"bytes_per_rank": x["bytes_per_rank"], "faster_from_here": a if now else b})
            cur = now
    if not switches:
        return {"bytes_per_rank": None, "never": f"{a if first else b} faster at every swept size"}
    return {"bytes_per_rank": switches[0]["bytes_per_rank"], "below": a if first else b, "switches": switches}


# The latency-formula page's AllReduce costs (eqs. model-algo-ring-ar, -rhd-ar,
# -dbt-ar) as (alpha coefficient, coefficient of M / beta) at N ranks.
def page_costs(N: int) -> dict:
    import math

    lg = math.log2(N)
    return {"ring": (2 * (N - 1), 2 * (N - 1) / N), "rhd": (2 * lg, 2 * (N - 1) / N), "dbt": (2 * lg, lg)}


def alpha_beta_fit(sw: dict, min_bytes: int = 0, auto=None) -> dict:
    """Least-squares fit of T = steps * alpha + bytes / beta over the graph-timed
    sweep of every algorithm: alpha is the cost of one dependent step on this
    GPU, beta the HBM rate -- the pages' model with a launch for a link
    start-up and HBM for the link.

    For every pair of algorithms it reports three crossover message sizes:
    the one measured in the sweep; the one the fitted HBM model predicts
    (each algorithm's steps and algorithmic bytes per byte of message, from
    the library's plans); and the one the latency-formula page's link
    formulas give with the fitted alpha and beta (eq.
    model-algo-ring-dbt-crossover and its analogues; the fused kernel has no
    formula on the pages).  Where two cost lines never cross the record says
    which algorithm is faster at every size.  ``auto(bytes_per_rank)`` gives
    the algorithm AUTO picks; the sizes where it is not the measured fastest
    are listed."""
    import numpy as np

    rows, ts = [], []
    for a, pts in sw.items():
        for p in pts:
            if p["bytes_per_rank"] >= min_bytes:
                rows.append([p["steps"], p["algorithmic_bytes"]])
                ts.append(p["us"] * 1e-6)
    A, t = np.array(rows, dtype=np.float64), np.array(ts)
    w = 1.0 / t  # relative error
    coef, *_ = np.linalg.lstsq(A * w[:, None], t * w, rcond=None)
    alpha, inv_beta = float(coef[0]), float(coef[1])
    pred = A @ coef
    N = NVR
    out = {"alpha_us": alpha * 1e6, "beta_gbs": 1.0 / inv_beta / 1e9 if inv_beta > 0 else None,
           "median_rel_err": float(np.median(np.abs(pred - t) / t)), "crossovers": {}}
    # each algorithm's (steps, algorithmic bytes per message byte) at the largest swept size
    shape = {a: (pts[-1]["steps"], pts[-1]["algorithmic_bytes"] / pts[-1]["bytes_per_rank"]) for a, pts in sw.items()}
    pc = page_costs(N)
    algos = list(sw)
    for i, a in enumerate(algos):
        for b in algos[i + 1:]:
            hbm = _crossover((shape[a][0] * alpha, shape[a][1] * inv_beta),
                             (shape[b][0] * alpha, shape[b][1] * inv_beta), a, b)
            if a in pc and b in pc:
                link = _crossover((pc[a][0] * alpha, pc[a][1] * inv_beta), (pc[b][0] * alpha, pc[b][1] * inv_beta), a, b)
            else:
                link = {"bytes_per_rank": None, "never": "no formula for the fused kernel on the pages"}
            out["crossovers"][f"{a}/{b}"] = {"measured": measured_crossover(sw[a], sw[b], a, b),
                                             "predicted_hbm_model": hbm, "predicted_page_formula": link}
    if auto is not None:
        diffs, sched = [], [x for x in algos if x in pc]
        for k, p in enumerate(sw[algos[0]]):
            M = p["bytes_per_rank"]
            fastest = min(algos, key=lambda x: sw[x][k]["us"])
            fastest_sched = min(sched, key=lambda x: sw[x][k]["us"]) if sched else None
            pick = auto(M)
            if pick != fastest:
                diffs.append({"bytes_per_rank": M, "auto": pick, "measured_fastest": fastest,
                              "auto_us": sw[pick][k]["us"] if pick in sw else None, "fastest_us": sw[fastest][k]["us"]})
            # among the schedules alone the HBM model always ranks by steps then bytes
            model_sched = min(sched, key=lambda x: (shape[x][0] * alpha + shape[x][1] * inv_beta * M)) if sched else None
            if model_sched != fastest_sched:
                out.setdefault("schedule_model_vs_measured", []).append(
                    {"bytes_per_rank": M, "model": model_sched, "measured_fastest": fastest_sched,
                     "model_us": sw[model_sched][k]["us"], "fastest_us": sw[fastest_sched][k]["us"]})
        out["auto_vs_measured"] = {"sizes": len(sw[algos[0]]), "differs_at": diffs}
    return out


def other_configs(vc, dev, peaks):
    """The other four workload configurations, timed (parity for them is in
    tests/test_gpu_configs.py).  Device-side seeded torch inputs: the values
    do not change the time of a copy or a sum."""
    import torch

    gen = torch.Generator(device=dev)
    gen.manual_seed(3)
    stream = torch.cuda.current_stream(dev)
    res = {}

    def entry(coll, algo, N, count, dtype, fn, bytes_moved_per_rank, factor, root=0):
        ms = time_calls(fn, stream, min_ms=50.0)
        hbm, steps = plan_shape(vc, coll, algo, N, count, dtype, root)
        if algo.startswith("pipe_"):
            steps = (steps, "chunks from the cost model")
        return {"ms": ms, "busbw": bytes_moved_per_rank * factor / (ms * 1e-3) / 1e9,
                "hbm_gbs": hbm / (ms * 1e-3) / 1e9, "frac_of_measured": hbm / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                "frac_of_nominal_8TBs": hbm / (ms * 1e-3) / 1e9 / NOMINAL_HBM_GBS, "steps": steps,
                "algorithmic_bytes": hbm}

    # 1. Ring AllReduce, N=4, 4096 fp32 (latency-bound)
    x = [torch.rand(4096, device=dev, generator=gen) * 2 - 1 for _ in range(4)]
    y = [torch.empty_like(t) for t in x]
    r = {}
    for a in ("ring", "rhd", "dbt", "fused"):
        fn = lambda a=a: vc.vc_allreduce(x, y, algo=a)
        r[a] = {"us": time_graph(fn, stream) * 1e3, "us_eager": time_calls(fn, stream, min_ms=5.0) * 1e3}
    res["ring_allreduce_n4_4096_f32"] = r
    del x, y
    # 3. bf16 gradient bucket, N=8, 64M elements: AllReduce, ReduceScatter, AllGather
    N, cnt = 8, 64 << 20
    xb = [(torch.randn(cnt, device=dev, generator=gen) * 1e-3).to(torch.bfloat16) for _ in range(N)]
    yb = [torch.empty_like(t) for t in xb]
    r = {}
    for a in ("ring", "fused", "rhd", "dbt"):
        r["allreduce_" + a] = entry("allreduce", a, N, cnt, "bf16", lambda a=a: vc.vc_allreduce(xb, yb, algo=a),
                                    cnt * 2, 2 * (N - 1) / N)
    rs_out = [t[: cnt // N] for t in yb]
    for a in ("ring", "fused"):
        r["reduce_scatter_" + a] = entry("reduce_scatter", a, N, cnt // N, "bf16",
                                         lambda a=a: vc.vc_reduce_scatter(xb, rs_out, algo=a), cnt * 2, (N - 1) / N)
    ag_in = [t[: cnt // N] for t in xb]
    for a in ("ring", "fused"):
        r["allgather_" + a] = entry("allgather", a, N, cnt // N, "bf16",
                                    lambda a=a: vc.vc_allgather(ag_in, yb, algo=a), cnt * 2, (N - 1) / N)
    res["bf16_bucket_n8_64M"] = r
    del xb, yb, rs_out, ag_in
    torch.cuda.empty_cache()
    # 4. MoE AllToAll, N=8, 8192 x 4096 bf16 per rank in 8 blocks
    cnt = 8192 * 4096
    xa = [torch.randn(cnt, device=dev, generator=gen).to(torch.bfloat16) for _ in range(N)]
    ya = [torch.empty_like(t) for t in xa]
    r = {}
    for a in ("pairwise", "bruck", "fused"):
        r[a] = entry("alltoall", a, N, cnt // N, "bf16", lambda a=a: vc.vc_alltoall(xa, ya, algo=a),
                     cnt * 2, (N - 1) / N)
    res["moe_alltoall_n8_8192x4096_bf16"] = r
    del xa, ya
    torch.cuda.empty_cache()
    # 5. Broadcast and Scatter, root 0, int32, 1 GiB total, N = 8 and 16
    cnt = (1 << 30) // 4
    src = torch.randint(-2**31, 2**31 - 1, (cnt,), dtype=torch.int32, device=dev, generator=gen)
    r = {}
    for N in (8, 16):
        outs = [torch.empty_like(src) for _ in range(N)]
        for a in ("binomial", "scatter_allgather", "fused", "pipe_chain", "pipe_tree"):
            r[f"broadcast_n{N}_{a}"] = entry("broadcast", a, N, cnt, "i32",
                                             lambda a=a: vc.vc_broadcast(src, outs, root=0, algo=a), cnt * 4, 1.0)
        del outs
        sc = [torch.empty(cnt // N, dtype=torch.int32, device=dev) for _ in range(N)]
        for a in ("binomial", "fused"):
            r[f"scatter_n{N}_{a}"] = entry("scatter", a, N, cnt // N, "i32",
                                           lambda a=a: vc.vc_scatter(src, sc, root=0, algo=a), cnt * 4, (N - 1) / N)
        del sc
        torch.cuda.empty_cache()
    res["bcast_scatter_int32_1GiB"] = r
    res["pipelined_broadcast_chunks_n8_1GiB"] = chunk_sweep(vc, src, stream)
    return res


def chunk_sweep(vc, src, stream, N: int = 8):
    """The pipelined Broadcasts' chunk count k measured: every k from 1 to 256
    (powers of 2) next to the k the cost model picks, k* = sqrt(h M / (alpha
    beta)) with h = N-2 (chain) or ceil(log2 N)-1 (tree) -- the
    Bcast/Scatter page's eqs. pipe-chain-bcast and pipe-tree-bcast optimised
    in k (the page prints N-1 for the chain; the derivative gives N-2)."""
    import math
    import torch

    M = src.numel() * 4
    alpha, beta = vc.vc_get_cost_model()[1:]
    outs = [torch.empty_like(src) for _ in range(N)]
    res = {"bytes": M, "cost_model": {"alpha_s": alpha, "beta_bytes_per_s": beta}}
    for algo, h in (("pipe_chain", N - 2), ("pipe_tree", math.ceil(math.log2(N)) - 1)):
        ks = [1 << i for i in range(9)]
        ms = [time_calls(lambda k=k: vc.vc_broadcast_pipelined(src, outs, root=0, algo=algo, nchunks=k), stream,
                         min_ms=30.0) for k in ks]
        model_k = min(256, max(1, round(math.sqrt(h * M / (alpha * beta)))))
        model_ms = time_calls(lambda: vc.vc_broadcast_pipelined(src, outs, root=0, algo=algo, nchunks=0), stream,
                              min_ms=30.0)
        best = min(range(len(ks)), key=lambda i: ms[i])
        res[algo] = {"k": ks, "ms": ms, "measured_best_k": ks[best], "measured_best_ms": ms[best],
                     "model_k": model_k, "model_ms": model_ms}
    del outs
    return res


def e2e(vc, host, send, recv, stream, args, world, dev, M):
    """End to end through host memory: every step uploads the N inputs from
    pinned host buffers, runs the four AllReduces and reads every output back
    into pinned host buffers.  Two device buffer sets alternate so that a
    step's uploads overlap the previous step's read-backs (the copy engines
    run both directions at once); events keep each set from being refilled
    before its previous step has finished with it."""
    import torch

    N = len(send)
    pin_in = [torch.from_numpy(h).pin_memory() for h in host]
    pin_out = {a: [torch.empty(M // 4, dtype=torch.float32).pin_memory() for _ in range(N)] for a in ALGOS}
    dsend = [send, [torch.empty_like(x) for x in send]]
    drecv = [recv, {a: [torch.empty_like(x) for x in recv[a]] for a in ALGOS}]
    up, comp, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    uploaded = [torch.cuda.Event(), torch.cuda.Event()]
    computed = [torch.cuda.Event(), torch.cuda.Event()]
    downloaded = [torch.cuda.Event(), torch.cuda.Event()]
    used = [False, False]

    def step(i):
        b = i % 2
        with torch.cuda.stream(up):
            if used[b]:
                up.wait_event(computed[b])  # set b's inputs were read by step i-2
            for r in range(N):
                dsend[b][r].copy_(pin_in[r], non_blocking=True)
            uploaded[b].record(up)
        with torch.cuda.stream(comp):
            comp.wait_event(uploaded[b])
            if used[b]:
                comp.wait_event(downloaded[b])  # set b's outputs were read back by step i-2
            for a in ALGOS:
                vc.vc_allreduce(dsend[b], drecv[b][a], algo=a, stream=comp)
            computed[b].record(comp)
        with torch.cuda.stream(down):
            down.wait_event(computed[b])
            for a in ALGOS:
                for r in range(N):
                    pin_out[a][r].copy_(drecv[b][a][r], non_blocking=True)
            downloaded[b].record(down)
        used[b] = True

    def join():
        for st in (up, comp, down):
            stream.wait_stream(st)

    steps = max(1, min(args.steps, args.e2e_steps))
    for i in range(2):
        step(i)
    join()
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for st in (up, comp, down):
        st.wait_event(e0)
    for i in range(2, 2 + steps):
        step(i)
    join()
    e1.record(stream)
    torch.cuda.synchronize()
    # the last step's outputs are on the host: spot-check them against the device copy
    for a in ALGOS:
        assert torch.equal(pin_out[a][N - 1][:4096], drecv[(1 + steps) % 2][a][N - 1][:4096].cpu())
    ms = reduce_max(e0.elapsed_time(e1), world, dev) / steps
    return {"value": step_bus_bytes(M) * world / (ms * 1e-3) / 1e9, "unit": "GB/s",
            "h2d_bytes_per_step": N * M, "d2h_bytes_per_step": len(ALGOS) * N * M,
            "ms_per_step": ms, "steps": steps,
            "pipeline": "two buffer sets; uploads overlap the previous step's read-backs"}


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--algos", default="ring,rhd,dbt,fused",
                    help="AllReduce algorithms in one step (profiling a single kernel uses one)")
    ap.add_argument("--mib-per-rank", type=float, default=BYTES_PER_RANK / (1 << 20),
                    help="message per rank (the workload is 256; smaller only for profiling captures)")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-per-algo", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip timing the other workload configurations")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--slice-limit", type=int, default=None,
                    help="bytes per rank up to which calls take the sliced form (default: the library's)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--e2e-steps", type=int, default=8)
    ap.add_argument("--details-out", default=None, help="also write every section as one JSON file here")
    ap.add_argument("--ref-mib", type=float, default=None,
                    help="reference arm: MiB per rank (default: the workload's 256)")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
