"""bench.py's host logic on the CPU: the reference arm's JSON line and the
replica timing reductions over two gloo ranks (world size 2)."""
import io
import json
import os
import socket
import sys
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
