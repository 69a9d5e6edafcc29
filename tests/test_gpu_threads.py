"""Concurrent calls from several host threads, each on its own CUDA stream.

The library's host state (plan cache, support cache, one-launch plan
descriptions and their first upload, scratch pool) is shared by all threads.
Four threads issue interleaved calls; some shapes are the same in every
thread, so first uses race.  Every result must equal the oracle bit for bit.
"""
import threading

import numpy as np
import pytest
import torch

import collective_communication_algorithms_virtual_gb300 as vc
from oracle import cxx
from synthetic_inputs import rank_buffers

from .gpu_util import same_bits, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from collective_communication_algorithms_virtual_gb300 import build

    build.build()
    vc.lib()
    yield


# (algo, N, count, dtype): shared shapes first (every thread uses them), then per-thread ones
SHARED = [("ring", 8, 4096 + 5, "f32"), ("rhd", 5, 3001, "bf16"), ("dbt", 8, 65536, "f32"), ("fused", 16, 777, "bf16")]


def _worker(tid, errors):
    try:
        stream = torch.cuda.Stream()
        rng = np.random.default_rng(100 + tid)
        shapes = SHARED + [("ring", int(rng.integers(2, 12)), int(rng.integers(1, 20000)), "f32") for _ in range(4)]
        with torch.cuda.stream(stream):
            for rep in range(3):
                for j, (algo, N, count, dtype) in enumerate(shapes):
                    kind = "uniform_f32" if dtype == "f32" else "normal_bf16"
                    xs = rank_buffers(kind, 1000 * tid + 10 * rep + j, N, count)
                    sends = [to_dev(x) for x in xs]
                    recvs = [torch.empty_like(s) for s in sends]
                    vc.vc_allreduce(sends, recvs, algo=algo, stream=stream)
                    stream.synchronize()
                    want = cxx.allreduce(xs, algo, dtype).outputs
                    for r in range(N):
                        if not same_bits(to_host(recvs[r]), want[r]):
                            errors.append((tid, rep, algo, N, count, dtype, r))
                            return
    except Exception as e:  # reported by the main thread
        errors.append((tid, repr(e)))


def test_concurrent_threads_on_separate_streams():
    errors = []
    threads = [threading.Thread(target=_worker, args=(t, errors)) for t in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=600)
    assert not any(t.is_alive() for t in threads)
    assert not errors, errors
