"""vc_reduce_scatter_noalloc: the Ring ReduceScatter for callers that cannot
allocate device memory (code running inside an allocator or an out-of-memory
handler, loops that forbid cudaMalloc or pool growth, fixed memory budgets).

It keeps its partial sums in a fixed array the library reserves on every GPU
instead of in the library's memory pool, and must give exactly what the
allocating vc_reduce_scatter(..., ring) gives.  Checked through the C ABI on
two calls in a row (the array keeps the previous call's contents), with a
size above the array's limit rejected without enqueuing anything.  This file
is collected last so that a failure here cannot hide another test's result.
"""
import ctypes

import numpy as np
import pytest
import torch

import collective_communication_algorithms_virtual_gb300 as vc
from synthetic_inputs import rank_buffers

pytestmark = pytest.mark.gpu

LIMIT = 16 << 20  # VC_NOALLOC_SCRATCH_BYTES


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


def _to_dev(x):
    if x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(x).cuda()


@pytest.mark.parametrize("dtype,kind,code", [("f32", "uniform_f32", 0), ("bf16", "normal_bf16", 1),
                                              ("i32", "int32_bits", 2)])
def test_noalloc_matches_allocating_ring_reduce_scatter(L, dtype, kind, code):
    N, rc = 8, 100_003
    assert 2 * N * rc * 4 <= LIMIT
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):  # two calls in a row, different data
        xs = rank_buffers(kind, 40 + call, N, N * rc)
        send = [_to_dev(x) for x in xs]
        want = [torch.empty(rc, dtype=send[0].dtype, device="cuda") for _ in range(N)]
        got = [torch.full((rc,), -7, dtype=send[0].dtype, device="cuda") for _ in range(N)]
        vc.vc_reduce_scatter(send, want, algo="ring")
        rc_ = L.vc_reduce_scatter_noalloc(_ptrs(send), _ptrs(got), N, rc, code, 0, stream)
        assert rc_ == 0, L.vc_last_error().decode()
        torch.cuda.synchronize()
        for r in range(N):
            assert torch.equal(got[r], want[r]), (dtype, call, r)


def test_noalloc_rejects_sizes_beyond_the_array(L):
    N = 8
    rc = LIMIT // (2 * N * 4) + 1
    send = [torch.zeros(N * rc, device="cuda") for _ in range(N)]
    out = [torch.full((rc,), 3.0, device="cuda") for _ in range(N)]
    status = L.vc_reduce_scatter_noalloc(_ptrs(send), _ptrs(out), N, rc, 0, 0,
                                         torch.cuda.current_stream().cuda_stream)
    assert status == 1  # VC_ERR_INVALID_ARG
    assert "scratch" in L.vc_last_error().decode()
    torch.cuda.synchronize()
    assert all(bool((o == 3.0).all()) for o in out)
