"""Thin ctypes binding over the C ABI of include/vc.h.

Argument marshalling only: tensors become device pointers, counts and enum
codes; every step of every collective runs in libvcoll.so.  The functions
keep the C names.  There is no fallback: if the library is not built, or a
call fails, an exception is raised.

The C ABI takes bare pointers and counts and cannot see a buffer's size, so
before each call every tensor is checked to hold at least the elements the
call reads or writes there, contiguous, of the call's dtype, on one CUDA
device; anything else raises VCError(VC_ERR_INVALID_ARG) before the library
is called.  The checks cost about 5 us of host time for 16 tensors;
VC_CHECK_TENSORS=0 in the environment skips them.
"""
from __future__ import annotations

import ctypes
import os
from typing import Sequence

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libvcoll.so")

VC_SUCCESS, VC_ERR_INVALID_ARG, VC_ERR_UNSUPPORTED, VC_ERR_CUDA, VC_ERR_NOMEM, VC_ERR_TIMEOUT = range(6)
DTYPES = {"f32": 0, "bf16": 1, "i32": 2, "f16": 3}
OPS = {"sum": 0, "max": 1, "min": 2}
ALGOS = {"fused": 0, "ring": 1, "rhd": 2, "dbt": 3, "binomial": 4, "scatter_allgather": 5,
         "pairwise": 6, "bruck": 7, "auto": 8, "pipe_chain": 9, "pipe_tree": 10, "mesh": 11, "ring_hop": 12}
ALGO_NAMES = {v: k for k, v in ALGOS.items()}
COST_POLICIES = {"hbm": 0, "link": 1}
COLLS = {"allreduce": 0, "reduce_scatter": 1, "allgather": 2, "broadcast": 3, "scatter": 4,
         "alltoall": 5, "gather": 6, "reduce": 7}


class VCError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


class TraceRecord(ctypes.Structure):
    _fields_ = [("coll", ctypes.c_int32), ("algo", ctypes.c_int32), ("step", ctypes.c_int32),
                ("kernel", ctypes.c_int32), ("bytes", ctypes.c_int64), ("nops", ctypes.c_int32),
                ("ms", ctypes.c_float)]


KERNEL_MODES = {0: "copy", 1: "f32", 2: "i32", 3: "bf16", 4: "bf16_pure", 5: "f16", 6: "f16_pure"}
KERNEL_OPS = {0: "sum", 1: "max", 2: "min"}


def kernel_name(code: int) -> str:
    mode = KERNEL_MODES[code & 7]
    name = mode if mode == "copy" else f"{KERNEL_OPS[(code >> 3) & 3]}_{mode}"
    if code & 256:  # one launch over the whole GPU, each thread carrying its group through every step
        return name + "_sliced"
    if code & 128:  # one cluster launch for the whole plan
        return name + "_single_launch"
    extra = ("_tma" if mode == "copy" else "_batched") if code & 64 else ""
    return name + ("_large" if code & 32 else "") + extra


class PlanEntry(ctypes.Structure):
    _fields_ = [("step", ctypes.c_int32), ("op", ctypes.c_int32), ("role", ctypes.c_int32),
                ("pos", ctypes.c_int32), ("buf", ctypes.c_int32), ("owner", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("reduce", ctypes.c_int32), ("byte_off", ctypes.c_int64),
                ("n", ctypes.c_int64), ("nb", ctypes.c_int64), ("stride_bytes", ctypes.c_int64),
                ("elem0", ctypes.c_int64)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (loaded once); raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, I, Z, V = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p
        PP = ctypes.POINTER(ctypes.c_void_p)
        for name, args in {
            "vc_allreduce": [PP, PP, I, Z, I, I, I, V],
            "vc_reduce_scatter": [PP, PP, I, Z, I, I, I, V],
            "vc_allgather": [PP, PP, I, Z, I, I, V],
            "vc_broadcast": [P, PP, I, Z, I, I, I, V],
            "vc_scatter": [P, PP, I, Z, I, I, I, V],
            "vc_alltoall": [PP, PP, I, Z, I, I, V],
            "vc_broadcast_pipelined": [P, PP, I, Z, I, I, I, I, V],
            "vc_gather": [PP, P, I, Z, I, I, I, V],
            "vc_reduce": [PP, P, I, Z, I, I, I, I, V],
        }.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = I
        L.vc_status_string.argtypes = [I]
        L.vc_status_string.restype = ctypes.c_char_p
        L.vc_last_error.argtypes = []
        L.vc_last_error.restype = ctypes.c_char_p
        L.vc_busbw_factor.argtypes = [I, I]
        L.vc_busbw_factor.restype = ctypes.c_double
        L.vc_plan_describe.argtypes = [I, I, I, Z, I, I, I, I, I, ctypes.POINTER(PlanEntry), Z,
                                       ctypes.POINTER(Z), ctypes.POINTER(Z), ctypes.POINTER(I)]
        L.vc_plan_describe.restype = I
        U32P, U8P = ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(ctypes.c_uint8)
        L.vc_plan_exec_order.argtypes = [I, I, I, Z, I, I, I, I, I, U32P, U8P, Z, U8P, Z, ctypes.POINTER(Z),
                                         ctypes.POINTER(I)]
        L.vc_plan_exec_order.restype = I
        L.vc_plan_form.argtypes = [I, I, I, Z, I, I, I, I, I, ctypes.POINTER(I), ctypes.POINTER(I),
                                   ctypes.POINTER(I)]
        L.vc_plan_form.restype = I
        L.vc_trace_enable.argtypes = [I]
        L.vc_trace_enable.restype = I
        L.vc_trace_read.argtypes = [ctypes.POINTER(TraceRecord), Z, ctypes.POINTER(Z)]
        L.vc_trace_read.restype = I
        L.vc_set_cost_model.argtypes = [I, ctypes.c_double, ctypes.c_double]
        L.vc_set_cost_model.restype = I
        L.vc_get_cost_model.argtypes = [ctypes.POINTER(I), ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)]
        L.vc_get_cost_model.restype = I
        L.vc_select_algo.argtypes = [I, I, Z, I, I, ctypes.POINTER(I), ctypes.POINTER(ctypes.c_double)]
        L.vc_select_algo.restype = I
        L.vc_device_errors.argtypes = [V, ctypes.POINTER(ctypes.c_uint32)]
        L.vc_device_errors.restype = I
        L.vc_copy_selftest.argtypes = [V, ctypes.POINTER(ctypes.c_uint32)]
        L.vc_copy_selftest.restype = I
        L.vc_set_single_launch.argtypes = [Z]
        L.vc_set_single_launch.restype = I
        L.vc_get_single_launch.argtypes = [ctypes.POINTER(Z)]
        L.vc_get_single_launch.restype = I
        L.vc_set_merge_steps.argtypes = [I]
        L.vc_set_merge_steps.restype = I
        L.vc_get_merge_steps.argtypes = [ctypes.POINTER(I)]
        L.vc_get_merge_steps.restype = I
        L.vc_set_slice_limit.argtypes = [Z]
        L.vc_set_slice_limit.restype = I
        L.vc_get_slice_limit.argtypes = [ctypes.POINTER(Z)]
        L.vc_get_slice_limit.restype = I
        L.vc_set_reuse_order.argtypes = [Z]
        L.vc_set_reuse_order.restype = I
        L.vc_get_reuse_order.argtypes = [ctypes.POINTER(Z)]
        L.vc_get_reuse_order.restype = I
        L.vc_set_copy_pipeline.argtypes = [Z]
        L.vc_set_copy_pipeline.restype = I
        L.vc_get_copy_pipeline.argtypes = [ctypes.POINTER(Z)]
        L.vc_get_copy_pipeline.restype = I
        L.vc_version.argtypes = []
        L.vc_version.restype = I
        _lib = L
    return _lib


def check(status: int) -> None:
    if status != VC_SUCCESS:
        L = lib()
        raise VCError(status, f"{L.vc_status_string(status).decode()}: {L.vc_last_error().decode()}")


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------

_ARRAY_TYPES: dict = {}


def _ptr_array(ptrs: Sequence[int]):
    n = len(ptrs)
    typ = _ARRAY_TYPES.get(n)
    if typ is None:
        typ = _ARRAY_TYPES[n] = ctypes.c_void_p * n
    return typ(*ptrs)


_TORCH_DTYPES: dict = {}


def _dtype_code(t) -> int:
    if not _TORCH_DTYPES:
        import torch

        _TORCH_DTYPES.update({torch.float32: 0, torch.bfloat16: 1, torch.int32: 2, torch.float16: 3})
    code = _TORCH_DTYPES.get(t.dtype)
    if code is None:
        raise VCError(VC_ERR_INVALID_ARG, f"unsupported dtype {t.dtype}")
    return code


_raw_stream = None


def _stream_handle(stream, like) -> int:
    """The cudaStream_t to enqueue on: `stream` (a torch stream or a raw
    handle), else the current stream of `like`'s device."""
    global _raw_stream
    if stream is None:
        if _raw_stream is None:
            import torch

            # the raw handle without building a Stream object (measured ~3 us per call)
            _raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None) or \
                (lambda dev: torch.cuda.current_stream(dev).cuda_stream)
        return int(_raw_stream(like.get_device()))
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


CHECK_TENSORS = os.environ.get("VC_CHECK_TENSORS", "1") != "0"


def _checked(ts, need: int, like) -> list[int]:
    """Pointers of `ts`, each tensor checked to hold at least `need`
    contiguous elements of `like`'s dtype on `like`'s CUDA device."""
    if not CHECK_TENSORS:
        return [t.data_ptr() for t in ts]
    dt, dev = like.dtype, like.get_device()
    if dev < 0:
        raise VCError(VC_ERR_INVALID_ARG, f"tensors must be on a CUDA device, not {like.device}")
    out = []
    for t in ts:
        if t.numel() < need or t.dtype is not dt or t.get_device() != dev or not t.is_contiguous():
            raise VCError(VC_ERR_INVALID_ARG,
                          f"each tensor must be contiguous {dt} on cuda:{dev} with at least {need} elements, "
                          f"not {tuple(t.shape)} {t.dtype} on {t.device}"
                          + ("" if t.is_contiguous() else " (not contiguous)"))
        out.append(t.data_ptr())
    return out


def _ranks(ts, N: int, what: str):
    if len(ts) != N:
        raise VCError(VC_ERR_INVALID_ARG, f"{what}: {len(ts)} tensors for {N} ranks")
    return ts


def _code(table: dict, key) -> int:
    return table[key] if isinstance(key, str) else int(key)


# ---------------------------------------------------------------------------
# collectives (tensor arguments; one tensor per virtual rank)
# ---------------------------------------------------------------------------

def vc_allreduce(send, recv, algo="fused", op="sum", stream=None) -> None:
    """recv[r] = sum over ranks of send[q]; ``send[r] is recv[r]`` allowed."""
    N = len(send)
    n = send[0].numel()
    sp, rp = _checked(send, n, send[0]), _checked(_ranks(recv, N, "recv"), n, send[0])
    check(lib().vc_allreduce(_ptr_array(sp), _ptr_array(rp), N, n, _dtype_code(send[0]), _code(OPS, op),
                             _code(ALGOS, algo), _stream_handle(stream, send[0])))


def vc_reduce_scatter(send, recv, algo="fused", op="sum", stream=None) -> None:
    """recv[r] = block r of the sum; send[q] holds N blocks of recv[r].numel()."""
    N = len(send)
    rc = recv[0].numel()
    sp, rp = _checked(send, N * rc, send[0]), _checked(_ranks(recv, N, "recv"), rc, send[0])
    check(lib().vc_reduce_scatter(_ptr_array(sp), _ptr_array(rp), N, rc, _dtype_code(send[0]), _code(OPS, op),
                                  _code(ALGOS, algo), _stream_handle(stream, send[0])))


def vc_allgather(send, recv, algo="fused", stream=None) -> None:
    """recv[r] = concatenation of send[0..N-1]."""
    N = len(send)
    sc = send[0].numel()
    sp, rp = _checked(send, sc, send[0]), _checked(_ranks(recv, N, "recv"), N * sc, send[0])
    check(lib().vc_allgather(_ptr_array(sp), _ptr_array(rp), N, sc, _dtype_code(send[0]), _code(ALGOS, algo),
                             _stream_handle(stream, send[0])))


def vc_broadcast(send_root, recv, root=0, algo="fused", stream=None) -> None:
    """recv[r] = send_root for every rank; ``send_root is recv[root]`` allowed."""
    N = len(recv)
    n = recv[0].numel()
    (sp,), rp = _checked([send_root], n, send_root), _checked(recv, n, send_root)
    check(lib().vc_broadcast(ctypes.c_void_p(sp), _ptr_array(rp), N, n, _dtype_code(send_root), int(root),
                             _code(ALGOS, algo), _stream_handle(stream, send_root)))


def vc_scatter(send_root, recv, root=0, algo="fused", stream=None) -> None:
    """recv[r] = block r of send_root."""
    N = len(recv)
    rc = recv[0].numel()
    (sp,), rp = _checked([send_root], N * rc, send_root), _checked(recv, rc, send_root)
    check(lib().vc_scatter(ctypes.c_void_p(sp), _ptr_array(rp), N, rc, _dtype_code(send_root), int(root),
                           _code(ALGOS, algo), _stream_handle(stream, send_root)))


def vc_alltoall(send, recv, algo="fused", stream=None) -> None:
    """recv[j] block i = send[i] block j; every buffer holds N blocks."""
    N = len(send)
    blk = send[0].numel() // N
    sp, rp = _checked(send, N * blk, send[0]), _checked(_ranks(recv, N, "recv"), N * blk, send[0])
    check(lib().vc_alltoall(_ptr_array(sp), _ptr_array(rp), N, blk, _dtype_code(send[0]), _code(ALGOS, algo),
                            _stream_handle(stream, send[0])))


def vc_broadcast_pipelined(send_root, recv, root=0, algo="pipe_tree", nchunks=0, stream=None) -> None:
    """Chunked Broadcast; nchunks=0 takes the cost model's optimum."""
    N = len(recv)
    n = recv[0].numel()
    (sp,), rp = _checked([send_root], n, send_root), _checked(recv, n, send_root)
    check(lib().vc_broadcast_pipelined(ctypes.c_void_p(sp), _ptr_array(rp), N, n, _dtype_code(send_root),
                                       int(root), _code(ALGOS, algo), int(nchunks),
                                       _stream_handle(stream, send_root)))


def vc_gather(send, recv_root, root=0, algo="fused", stream=None) -> None:
    """recv_root = concatenation of send[0..N-1] (on the root only)."""
    N = len(send)
    sc = send[0].numel()
    sp, (rp,) = _checked(send, sc, send[0]), _checked([recv_root], N * sc, send[0])
    check(lib().vc_gather(_ptr_array(sp), ctypes.c_void_p(rp), N, sc, _dtype_code(send[0]), int(root),
                          _code(ALGOS, algo), _stream_handle(stream, send[0])))


def vc_reduce(send, recv_root, root=0, algo="fused", op="sum", stream=None) -> None:
    """recv_root = sum over ranks of send[q]; ``recv_root is send[root]`` allowed."""
    N = len(send)
    n = send[0].numel()
    sp, (rp,) = _checked(send, n, send[0]), _checked([recv_root], n, send[0])
    check(lib().vc_reduce(_ptr_array(sp), ctypes.c_void_p(rp), N, n, _dtype_code(send[0]), _code(OPS, op),
                          int(root), _code(ALGOS, algo), _stream_handle(stream, send[0])))


def vc_busbw_factor(coll, nranks: int) -> float:
    return lib().vc_busbw_factor(_code(COLLS, coll), int(nranks))


def vc_status_string(status: int) -> str:
    return lib().vc_status_string(int(status)).decode()


def vc_last_error() -> str:
    return lib().vc_last_error().decode()


def vc_version() -> int:
    return lib().vc_version()


def vc_set_cost_model(policy="hbm", alpha_s: float = 0.0, beta_bytes_per_s: float = 0.0) -> None:
    """Cost model behind algo="auto" (0 keeps the policy's default constant)."""
    check(lib().vc_set_cost_model(_code(COST_POLICIES, policy), float(alpha_s), float(beta_bytes_per_s)))


def vc_get_cost_model():
    p, a, b = ctypes.c_int(0), ctypes.c_double(0), ctypes.c_double(0)
    check(lib().vc_get_cost_model(ctypes.byref(p), ctypes.byref(a), ctypes.byref(b)))
    return {0: "hbm", 1: "link"}[p.value], a.value, b.value


def vc_select_algo(coll, nranks: int, count: int, dtype="f32", root: int = 0):
    """(algorithm name, predicted seconds) that algo="auto" would use."""
    a, t = ctypes.c_int(0), ctypes.c_double(0)
    check(lib().vc_select_algo(_code(COLLS, coll), int(nranks), int(count), _code(DTYPES, dtype), int(root),
                               ctypes.byref(a), ctypes.byref(t)))
    return ALGO_NAMES[a.value], t.value


def vc_set_single_launch(max_step_bytes: int) -> None:
    """Run schedules whose steps each move at most this many bytes in one
    launch (0: never; SINGLE_LAUNCH_ALWAYS: whenever eligible)."""
    check(lib().vc_set_single_launch(int(max_step_bytes)))


def vc_get_single_launch() -> int:
    v = ctypes.c_size_t(0)
    check(lib().vc_get_single_launch(ctypes.byref(v)))
    return v.value


SINGLE_LAUNCH_ALWAYS = (1 << 64) - 1
VC_SINGLE_LAUNCH_DEFAULT = 768 << 10  # VC_SINGLE_LAUNCH_DEFAULT


def vc_set_slice_limit(max_bytes_per_rank: int) -> None:
    """Run eligible schedules (fp32 / int32 AllReduce and the like) whose
    message per rank is at most this many bytes in the sliced form (0: never;
    SLICE_ALWAYS: whenever eligible)."""
    check(lib().vc_set_slice_limit(int(max_bytes_per_rank)))


def vc_get_slice_limit() -> int:
    v = ctypes.c_size_t(0)
    check(lib().vc_get_slice_limit(ctypes.byref(v)))
    return v.value


def vc_set_merge_steps(on: bool) -> None:
    """Run consecutive steps that depend on nothing among themselves as one
    launch (default on).  Clears the plan cache."""
    check(lib().vc_set_merge_steps(int(bool(on))))


def vc_get_merge_steps() -> bool:
    v = ctypes.c_int(0)
    check(lib().vc_get_merge_steps(ctypes.byref(v)))
    return bool(v.value)


SLICE_ALWAYS = (1 << 64) - 1
VC_SLICE_DEFAULT = 16 << 20  # VC_SLICE_LIMIT_DEFAULT


def vc_set_reuse_order(min_step_bytes: int) -> None:
    """Steps after one writing at least this many bytes are ordered for L2 reuse
    (0: every step; REUSE_ORDER_NEVER: none).  Clears the plan cache."""
    check(lib().vc_set_reuse_order(int(min_step_bytes)))


def vc_get_reuse_order() -> int:
    v = ctypes.c_size_t(0)
    check(lib().vc_get_reuse_order(ctypes.byref(v)))
    return v.value


REUSE_ORDER_NEVER = (1 << 64) - 1


def vc_set_copy_pipeline(min_bytes: int) -> None:
    """Copy launches of whole 16-byte groups that write at least this many
    bytes take the bulk-copy pipeline (0: every one; COPY_PIPELINE_NEVER: none)."""
    check(lib().vc_set_copy_pipeline(int(min_bytes)))


def vc_get_copy_pipeline() -> int:
    v = ctypes.c_size_t(0)
    check(lib().vc_get_copy_pipeline(ctypes.byref(v)))
    return v.value


COPY_PIPELINE_NEVER = (1 << 64) - 1


def vc_device_errors(stream=None) -> int:
    """Waits for the stream, then reads and clears the device error word."""
    v = ctypes.c_uint32(0)
    s = None if stream is None else (stream if isinstance(stream, int) else int(stream.cuda_stream))
    check(lib().vc_device_errors(s, ctypes.byref(v)))
    return v.value


def vc_copy_selftest(stream=None) -> int:
    """Error word left by a bulk-copy launch whose first wait is made to run out."""
    v = ctypes.c_uint32(0)
    s = None if stream is None else (stream if isinstance(stream, int) else int(stream.cuda_stream))
    check(lib().vc_copy_selftest(s, ctypes.byref(v)))
    return v.value


def vc_trace_enable(on: bool = True) -> None:
    """Start (clearing old records) or stop the launch trace."""
    check(lib().vc_trace_enable(int(bool(on))))


def vc_trace_read(capacity: int = 1 << 20) -> list:
    """Wait for the traced launches and return their records (dicts)."""
    buf = (TraceRecord * capacity)()
    n = ctypes.c_size_t(0)
    check(lib().vc_trace_read(buf, capacity, ctypes.byref(n)))
    out = []
    for r in buf[:n.value]:
        out.append({"coll": r.coll, "algo": r.algo, "step": r.step, "kernel": kernel_name(r.kernel),
                    "bytes": r.bytes, "nops": r.nops, "ms": r.ms})
    return out


def vc_plan_describe(coll, algo, nranks: int, count: int, dtype="f32", root: int = 0, inplace: bool = False,
                     nchunks: int = 0, op="sum"):
    """The step plan the library would run, as (entries, scratch_bytes, n_steps);
    host only, needs no GPU."""
    L = lib()
    need, scratch = ctypes.c_size_t(0), ctypes.c_size_t(0)
    steps = ctypes.c_int(0)
    args = (_code(COLLS, coll), _code(ALGOS, algo), int(nranks), int(count), _code(DTYPES, dtype),
            _code(OPS, op), int(root), int(bool(inplace)), int(nchunks))
    check(L.vc_plan_describe(*args, None, 0, ctypes.byref(need), ctypes.byref(scratch), ctypes.byref(steps)))
    buf = (PlanEntry * max(1, need.value))()
    check(L.vc_plan_describe(*args, buf, need.value, ctypes.byref(need), ctypes.byref(scratch),
                             ctypes.byref(steps)))
    return list(buf[:need.value]), scratch.value, steps.value


FORMS = {0: "steps", 1: "cluster", 2: "sliced"}


def vc_plan_form(coll, algo, nranks: int, count: int, dtype="f32", root: int = 0, inplace: bool = False,
                 nchunks: int = 0, op="sum"):
    """The execution form a call takes under the current settings, on aligned
    buffers: ("sliced" | "cluster" | "steps", launches, host_ranges); host
    only, needs no GPU."""
    L = lib()
    form, launches, hr = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    check(L.vc_plan_form(_code(COLLS, coll), _code(ALGOS, algo), int(nranks), int(count), _code(DTYPES, dtype),
                         _code(OPS, op), int(root), int(bool(inplace)), int(nchunks), ctypes.byref(form),
                         ctypes.byref(launches), ctypes.byref(hr)))
    return FORMS[form.value], launches.value, bool(hr.value)


def vc_plan_exec_order(coll, algo, nranks: int, count: int, dtype="f32", root: int = 0, inplace: bool = False,
                       nchunks: int = 0, op="sum"):
    """The order the library executes the plan in (the L2 reuse order): per
    step, the operations' indices as vc_plan_describe numbers them, their keep
    flags, and whether the step walks its tiles backwards.  Returns
    (order, keep, reverse) with order and keep lists of lists per step; host
    only, needs no GPU."""
    L = lib()
    nops, steps = ctypes.c_size_t(0), ctypes.c_int(0)
    args = (_code(COLLS, coll), _code(ALGOS, algo), int(nranks), int(count), _code(DTYPES, dtype),
            _code(OPS, op), int(root), int(bool(inplace)), int(nchunks))
    check(L.vc_plan_exec_order(*args, None, None, 0, None, 0, ctypes.byref(nops), ctypes.byref(steps)))
    order = (ctypes.c_uint32 * max(1, nops.value))()
    keep = (ctypes.c_uint8 * max(1, nops.value))()
    rev = (ctypes.c_uint8 * max(1, steps.value))()
    check(L.vc_plan_exec_order(*args, order, keep, nops.value, rev, steps.value, ctypes.byref(nops),
                               ctypes.byref(steps)))
    entries, _, _ = vc_plan_describe(coll, algo, nranks, count, dtype, root, inplace, nchunks, op)
    per_step = [0] * steps.value
    for e in entries:
        per_step[e.step] = max(per_step[e.step], e.op + 1)
    out_order, out_keep, k = [], [], 0
    for n in per_step:
        out_order.append(list(order[k:k + n]))
        out_keep.append(list(keep[k:k + n]))
        k += n
    return out_order, out_keep, list(rev[:steps.value])
