"""vc_reduce_scatter_noalloc: the Ring ReduceScatter for callers that cannot
allocate device memory (code running inside an allocator or an out-of-memory
handler, loops that forbid cudaMalloc or pool growth, fixed memory budgets).

It keeps its partial sums in a fixed array the library reserves on every GPU
instead of in the library's memory pool.  Checked through the C ABI on two
calls in a row (the array keeps the previous call's contents): bit for bit
against the oracle's ring ReduceScatter and against the allocating
vc_reduce_scatter(..., ring).  The size limit is checked at its exact boundary
(each rank's pair of partial slots is rounded up to 256 bytes), and MAX / MIN
are rejected.  This file is collected last so that a failure here cannot hide
another test's result.
"""
import ctypes

import numpy as np
import pytest
import torch

import collective_communication_algorithms_virtual_gb300 as vc
from oracle import cxx
from synthetic_inputs import normal_f32, rank_buffers

from .gpu_util import first_diff, same_bits, to_dev, to_host

pytestmark = pytest.mark.gpu

LIMIT = 16 << 20  # VC_NOALLOC_SCRATCH_BYTES
CODE = {"f32": 0, "bf16": 1, "i32": 2, "f16": 3}
TDT = {"f32": torch.float32, "bf16": torch.bfloat16, "i32": torch.int32, "f16": torch.float16}


def scratch_bytes(N, rc):
    """Two 4-byte partial slots of rc elements per rank, each rank's pair
    rounded up to 256 bytes."""
    return N * (-(-(2 * rc * 4) // 256) * 256)


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from collective_communication_algorithms_virtual_gb300 import build

    build.build()
    lib = vc.lib()
    PP = ctypes.POINTER(ctypes.c_void_p)
    lib.vc_reduce_scatter_noalloc.argtypes = [PP, PP, ctypes.c_int, ctypes.c_size_t, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_void_p]
    lib.vc_reduce_scatter_noalloc.restype = ctypes.c_int
    return lib


def _ptrs(ts):
    return (ctypes.c_void_p * len(ts))(*[ctypes.c_void_p(t.data_ptr()) for t in ts])


def _inputs(dtype, seed, N, n):
    if dtype == "f16":
        return [normal_f32(seed, r, n).astype(np.float16) for r in range(N)]
    kind = {"f32": "uniform_f32", "bf16": "normal_bf16", "i32": "int32_bits"}[dtype]
    return rank_buffers(kind, seed, N, n)


def _check_two_calls(L, dtype, N, rc, seed0):
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):  # two calls in a row, different data
        xs = _inputs(dtype, seed0 + call, N, N * rc)
        want = cxx.reduce_scatter(xs, "ring", dtype).outputs
        send = [to_dev(x) for x in xs]
        alloc = [torch.empty(rc, dtype=TDT[dtype], device="cuda") for _ in range(N)]
        got = [torch.full((rc,), -7, dtype=TDT[dtype], device="cuda") for _ in range(N)]
        vc.vc_reduce_scatter(send, alloc, algo="ring")
        status = L.vc_reduce_scatter_noalloc(_ptrs(send), _ptrs(got), N, rc, CODE[dtype], 0, stream)
        assert status == 0, L.vc_last_error().decode()
        torch.cuda.synchronize()
        for r in range(N):
            g = to_host(got[r])
            assert same_bits(g, want[r]), (dtype, N, call, r, first_diff(g, want[r]))
            assert torch.equal(got[r], alloc[r]), (dtype, N, call, r)


@pytest.mark.parametrize("dtype,N,rc", [("f32", 8, 100_003), ("bf16", 8, 100_003), ("i32", 8, 100_003),
                                        ("f16", 8, 50_001), ("f32", 3, 77_777), ("bf16", 5, 65_537),
                                        ("f16", 5, 1_001)])
def test_noalloc_matches_oracle_and_allocating_call(L, dtype, N, rc):
    assert scratch_bytes(N, rc) <= LIMIT
    _check_two_calls(L, dtype, N, rc, 40 + N)


def test_noalloc_size_limit_boundary_n3(L):
    N = 3
    rc_max = 699_040  # the largest recvcount whose scratch fits at N = 3
    assert scratch_bytes(N, rc_max) <= LIMIT < scratch_bytes(N, rc_max + 1)
    _check_two_calls(L, "f32", N, rc_max, 90)
    rc = rc_max + 1
    send = [torch.zeros(N * rc, device="cuda") for _ in range(N)]
    out = [torch.full((rc,), 3.0, device="cuda") for _ in range(N)]
    status = L.vc_reduce_scatter_noalloc(_ptrs(send), _ptrs(out), N, rc, 0, 0,
                                         torch.cuda.current_stream().cuda_stream)
    assert status == 1  # VC_ERR_INVALID_ARG
    assert "scratch" in L.vc_last_error().decode()
    torch.cuda.synchronize()
    assert all(bool((o == 3.0).all()) for o in out)


def test_noalloc_rejects_sizes_beyond_the_array(L):
    N = 8
    rc = LIMIT // (2 * N * 4) + 1
    assert scratch_bytes(N, rc) > LIMIT
    send = [torch.zeros(N * rc, device="cuda") for _ in range(N)]
    out = [torch.full((rc,), 3.0, device="cuda") for _ in range(N)]
    status = L.vc_reduce_scatter_noalloc(_ptrs(send), _ptrs(out), N, rc, 0, 0,
                                         torch.cuda.current_stream().cuda_stream)
    assert status == 1  # VC_ERR_INVALID_ARG
    assert "scratch" in L.vc_last_error().decode()
    torch.cuda.synchronize()
    assert all(bool((o == 3.0).all()) for o in out)


@pytest.mark.parametrize("op", [1, 2])  # VC_MAX, VC_MIN
def test_noalloc_rejects_max_and_min(L, op):
    N, rc = 4, 1000
    send = [torch.ones(N * rc, device="cuda") for _ in range(N)]
    out = [torch.full((rc,), 3.0, device="cuda") for _ in range(N)]
    status = L.vc_reduce_scatter_noalloc(_ptrs(send), _ptrs(out), N, rc, 0, op,
                                         torch.cuda.current_stream().cuda_stream)
    assert status == 2  # VC_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert all(bool((o == 3.0).all()) for o in out)
