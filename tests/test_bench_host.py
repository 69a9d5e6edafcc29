"""bench.py's host logic on the CPU: the reference arm's JSON line, the
replica timing reductions over two gloo ranks (world size 2), the final
line's size, the alpha-beta fit and the collectives sweep's slices and busbw
(with the library calls and the timing stubbed)."""
import io
import json
import os
import socket
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

import bench


def test_reference_arm_prints_one_json_line():
    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0", "--ref-mib", "1"])
    assert rc == 0
    lines = [l for l in buf.getvalue().splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "impl"):
        assert key in d, key
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["config"]["workload"] == bench.WORKLOAD
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["cpu_baseline"]["kind"] == "oracle"


def test_step_bus_bytes():
    assert bench.step_bus_bytes(256 << 20) == 4 * (256 << 20) * 1.75


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import torch.distributed as dist

    r, w, _ = bench.dist_env()
    bench.dist_init(w, "gloo")
    bench.barrier(w)
    mx = bench.reduce_max(10.0 + r, w)
    sm = bench.reduce_sum(1.0 + r, w)
    out.put((r, mx, sm))
    dist.destroy_process_group()


def test_replica_timing_reductions_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, mx, sm in res:
        assert mx == 11.0 and sm == 3.0


def _stub_result():
    """A GPU-arm result as run_ours builds it, with full-size detail sections."""
    algos = ["ring", "rhd", "dbt", "fused"]
    pt = {"bytes_per_rank": 1 << 20, "us": 30.123456, "us_eager": 36.1, "busbw": 61.2345678, "busbw_eager": 50.1,
          "steps": 14, "algorithmic_bytes": 36700160, "l2_resident": True}
    return {
        "metric": bench.METRIC, "value": 417.123456789, "unit": "GB/s", "n_gpus": 1, "steps": 200, "warmup": 5,
        "ms_per_step": 4.50412345, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic", "config": bench.config_block(256 << 20),
        "roofline": {"bound": "hbm", "kernel": "step_kernel<sum_f32>", "achieved": 6624.123456, "peak": 6659.6,
                     "unit": "GB/s", "frac": 0.99465, "peak_source": "measured", "traffic": 1.34e9,
                     "algorithmic_bytes_per_launch": 1.3997e9, "launches": 2800, "avg_launch_ms": 0.2113,
                     "frac_of_nominal_8TBs": 0.82, "kernels": {f"k{i}": {"launches": 1, "share": 0.1, "gbs": 1.0}
                                                               for i in range(12)},
                     "measured": "x" * 300, "ms_per_step_traced": 4.68},
        "gpu_launches": 12345,
        "clocks": {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 120},
        "per_algo": {a: {"ms": 1.3, "algbw": 200.1, "busbw": 352.123, "hbm_gbs": 7031.2, "algorithmic_bytes": 1 << 33,
                         "frac_of_measured": 1.0561, "frac_of_nominal_8TBs": 0.879} for a in algos},
        "sweep": {a: [dict(pt) for _ in range(19)] for a in algos},
        "alpha_beta": {"alpha_us": 1.48, "crossovers": {f"{a}/{b}": {"measured_bytes_per_rank": 1 << 25}
                                                        for a in algos for b in algos}},
        "configs": {f"cfg{i}": {"ms": 1.0, "busbw": 2.0, "steps": 3, "note": "y" * 200} for i in range(40)},
        "e2e": {"value": 27.33, "unit": "GB/s", "h2d_bytes_per_step": 2147483648,
                "d2h_bytes_per_step": 8589934592, "ms_per_step": 68.7, "steps": 8, "pipeline": "z" * 100},
        "cpu_baseline": {"value": 0.4776, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": "s" * 400},
    }


def test_final_line_is_short_and_last(tmp_path):
    out = _stub_result()
    buf = io.StringIO()
    with redirect_stdout(buf):
        s = bench.emit(out, str(tmp_path / "d.json"))
    lines = [l for l in buf.getvalue().splitlines() if l.strip()]
    assert lines[-1] == s
    assert len(s.encode()) <= bench.FINAL_LINE_MAX
    d = json.loads(s)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "clocks",
                "gpu_launches"):
        assert key in d, key
    assert d["value"] > 0 and d["config"]["workload"] == bench.WORKLOAD
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in d["roofline"], key
    assert d["e2e"]["h2d_bytes_per_step"] == 2147483648 and d["e2e"]["d2h_bytes_per_step"] == 8589934592
    # every detail section is on an earlier line, whole
    sections = {json.loads(l)["detail"] for l in lines[:-1]}
    assert {"per_algo", "sweep", "alpha_beta", "configs", "roofline"} <= sections
    with open(tmp_path / "d.json") as f:
        assert json.load(f)["sweep"] == out["sweep"]


def test_alpha_beta_fit_predicts_every_pair():
    """A sweep that follows T = steps * alpha + bytes / beta exactly, with the
    latency-formula page's NVLink constants (alpha 5 us, beta 450 GB/s): the fit
    recovers them, the page formula puts the Ring/DBT crossover at 14.4 MB
    (eq. model-algo-ring-dbt-crossover), and every pair gets a prediction from
    both models (a size, or which algorithm is faster at every size)."""
    alpha, beta = 5e-6, 450e9
    shape = {"ring": (14, 35), "rhd": (6, 35), "dbt": (6, 29), "fused": (1, 16)}
    sw = {a: [] for a in shape}
    for lg in range(10, 29):
        M = 1 << lg
        for a, (s, k) in shape.items():
            t = s * alpha + k * M / beta
            sw[a].append({"bytes_per_rank": M, "us": t * 1e6, "steps": s, "algorithmic_bytes": k * M})
    r = bench.alpha_beta_fit(sw, auto=lambda M: "fused")
    assert abs(r["alpha_us"] - 5.0) < 1e-6 and abs(r["beta_gbs"] - 450.0) < 1e-6
    assert len(r["crossovers"]) == 6
    for pair, c in r["crossovers"].items():
        for key in ("predicted_hbm_model", "predicted_page_formula", "measured"):
            v = c[key]
            assert v["bytes_per_rank"] is not None or v.get("never"), (pair, key, v)
    page = r["crossovers"]["ring/dbt"]["predicted_page_formula"]
    assert abs(page["bytes_per_rank"] - 1.44e7) / 1.44e7 < 1e-9 and page["below"] == "dbt"
    # in the HBM model DBT moves fewer bytes in fewer steps than Ring: no crossover
    assert r["crossovers"]["ring/dbt"]["predicted_hbm_model"]["never"] == "dbt faster at every size"
    # measured on this exact sweep: the same as the HBM model
    assert r["crossovers"]["ring/dbt"]["measured"]["never"] == "dbt faster at every swept size"
    assert r["auto_vs_measured"]["differs_at"] == []
    assert "schedule_model_vs_measured" not in r


class _FakeVC:
    """Records the library calls the collectives sweep makes (no GPU)."""

    def __init__(self):
        self.calls = []

    def _rec(self, name, *args, **kw):
        self.calls.append((name, args, kw))

    def vc_reduce_scatter(self, ins, outs, algo):
        self._rec("reduce_scatter", len(ins[0]), len(outs[0]), algo=algo)

    def vc_allgather(self, ins, outs, algo):
        self._rec("allgather", len(ins[0]), len(outs[0]), algo=algo)

    def vc_broadcast(self, src, outs, root, algo):
        self._rec("broadcast", len(src), len(outs[0]), algo=algo)

    def vc_broadcast_pipelined(self, src, outs, root, algo):
        self._rec("broadcast", len(src), len(outs[0]), algo=algo)

    def vc_alltoall(self, ins, outs, algo):
        self._rec("alltoall", len(ins[0]), len(outs[0]), algo=algo)

    def vc_scatter(self, src, outs, root, algo):
        self._rec("scatter", len(src), len(outs[0]), algo=algo)

    def vc_gather(self, ins, out, root, algo):
        self._rec("gather", len(ins[0]), len(out), algo=algo)

    def vc_reduce(self, ins, out, root, algo):
        self._rec("reduce", len(ins[0]), len(out), algo=algo)

    def vc_plan_describe(self, coll, algo, N, count, dtype, root=0):
        return [], 0, 1


def test_sweep_collectives_sizes_and_busbw(monkeypatch):
    """Every collective and algorithm at every size, with the buffer slices
    the pages' busbw convention implies and busbw = M x factor / time."""
    N = 8
    import torch

    import collective_communication_algorithms_virtual_gb300 as vc_lib

    send = [torch.empty((1 << 20) // 4) for _ in range(N)]  # 1 MiB per rank, host tensors
    recv = {bench.ALGOS[0]: [torch.empty((1 << 20) // 4) for _ in range(N)]}
    vc = _FakeVC()
    monkeypatch.setattr(bench, "time_graph", lambda fn, stream: (fn(), 0.01)[1])  # 10 us a call
    sizes = (4 << 10, 1 << 20, 4 << 20)  # the last exceeds the buffers and is skipped
    res = bench.sweep_collectives(vc, send, recv, None, sizes)
    assert set(res) == {f"{c}_{a}" for c, algos in bench.COLL_SWEEP.items() for a in algos}
    for key, rows in res.items():
        assert [r["bytes_per_rank"] for r in rows] == [4 << 10, 1 << 20], key
        coll = next(c for c in bench.COLL_SWEEP if key.startswith(c + "_"))
        f = vc_lib.vc_busbw_factor(coll, N)  # the library's table
        assert bench.coll_busbw_factor(coll, N) == f, coll
        for r in rows:
            assert r["busbw"] == pytest.approx(r["bytes_per_rank"] * f / 10e-6 / 1e9), key
    # the slices: RS and Scatter input M / output M/N, AG and Gather input M/N /
    # output M, Bcast, Reduce and A2A M
    for name, args, kw in vc.calls:
        n_in, n_out = args
        if name in ("reduce_scatter", "scatter"):
            assert n_in == N * n_out, name
        elif name in ("allgather", "gather"):
            assert n_out == N * n_in, name
        else:
            assert n_in == n_out, name
