"""ctypes wrapper of the C++ oracle (``oracle/sim.cpp``) -- TEST INFRASTRUCTURE ONLY.

The C++ oracle is a plain, single-threaded simulation of N ranks running the
pages' schedules step by step (see the header of ``sim.cpp``).  This module
builds it (``g++ -O2``) into ``oracle/libvcoracle.so`` and exposes it with the
same functions and results as the numpy oracle in ``oracle.schedules``
(``allreduce``, ``reduce_scatter``, ``allgather``, ``broadcast``,
``broadcast_pipelined``, ``scatter``, ``gather``, ``reduce``, ``alltoall``),
plus the closed-form association trees (``allreduce_at``,
``reduce_scatter_at``) and the element conversions.

Only ``tests/``, ``__graft_entry__`` (build and smoke) and the benchmark's
CPU-baseline and reference legs may load it.  The CUDA library never links or
calls it.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import shutil
import subprocess
from dataclasses import dataclass

import numpy as np

from .translog import Transfer, TransferLog

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "sim.cpp")
HDR = os.path.join(HERE, "sim.h")
LIB_PATH = os.path.join(HERE, "libvcoracle.so")

DTYPE_CODE = {"f32": 0, "bf16": 1, "i32": 2, "f16": 3}
OP_CODE = {"sum": 0, "max": 1, "min": 2}
STORAGE = {"f32": np.float32, "bf16": np.uint16, "i32": np.int32, "f16": np.float16}

ALGOS = {
    "allreduce": ("fused", "ring", "rhd", "dbt", "mesh", "ring_hop"),
    "reduce_scatter": ("fused", "ring"),
    "allgather": ("fused", "ring"),
    "broadcast": ("fused", "binomial", "scatter_allgather"),
    "scatter": ("fused", "binomial"),
    "alltoall": ("fused", "pairwise", "bruck", "ring"),
}
ALGOS_EXTRA = {
    "broadcast": ("pipe_chain", "pipe_tree"),
    "gather": ("fused", "binomial"),
    "reduce": ("fused", "binomial"),
}


class Unsupported(ValueError):
    """The schedule is not defined for these arguments."""


def build(force: bool = False) -> str:
    """Compile the oracle if its source is newer than the library."""
    if (not force and os.path.exists(LIB_PATH)
            and os.path.getmtime(LIB_PATH) >= max(os.path.getmtime(SRC), os.path.getmtime(HDR))):
        return LIB_PATH
    cxx = os.environ.get("CXX") or shutil.which("g++") or "c++"
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [cxx, "-std=c++17", "-O2", "-Wall", "-fPIC", "-shared", SRC, "-o", tmp]
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"oracle build failed ({' '.join(cmd)}):\n{r.stdout}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


_LIB = None


def lib():
    global _LIB
    if _LIB is None:
        build()
        L = ctypes.CDLL(LIB_PATH)
        P, I, I64, C = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_char_p
        L.vo_run.argtypes = [C, C, I, ctypes.POINTER(P), I64, I, I, I, I, I, ctypes.POINTER(P), C, I]
        L.vo_run.restype = I
        for name, args, res in [
            ("vo_noutputs", [P], I), ("vo_output_elems", [P, I], I64), ("vo_output_copy", [P, I, P], None),
            ("vo_hbm_bytes", [P], I64), ("vo_local_steps", [P], I), ("vo_nrecords", [P], I64),
            ("vo_records", [P, P], None), ("vo_nchunks_total", [P], I64), ("vo_record_chunks", [P, P], None),
            ("vo_record_phase", [P, I64], C), ("vo_free", [P], None), ("vo_set_fault", [I, I], None),
            ("vo_bf16_from_f32", [P, P, I64], None), ("vo_f32_from_bf16", [P, P, I64], None),
            ("vo_f16_from_f32", [P, P, I64], None), ("vo_f32_from_f16", [P, P, I64], None),
        ]:
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        for name in ("vo_allreduce_at", "vo_reduce_scatter_at"):
            f = getattr(L, name)
            f.argtypes = [ctypes.POINTER(P), I, C, I64, I, P, I64, I, P, C, I]
            f.restype = I
        _LIB = L
    return _LIB


@dataclass
class Result:
    outputs: list
    log: TransferLog
    hbm_bytes: int
    local_steps: int = 0

    @property
    def nsteps(self) -> int:
        """Steps that carry messages: the coefficient of alpha."""
        return len(self.log.steps())

    @property
    def launch_steps(self) -> int:
        """Steps that move any data on one device (messages or local copies)."""
        if self.nsteps == 0:
            return 1 if self.hbm_bytes > 0 else 0
        return self.nsteps + self.local_steps


def _ptrs(arrs):
    return (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])


def _as_storage(x, dtype):
    x = np.ascontiguousarray(x)
    want = STORAGE[dtype]
    assert x.dtype == want and x.ndim == 1, (x.dtype, want, x.shape)
    return x


def _run(coll, algo, arrays, n_in, N, dtype, op="sum", root=0, inplace=False, nchunks=0, want_log=True,
         want_outputs=True, keep=None):
    """Run one collective.  ``keep`` lists the outputs to copy back (None: all;
    the others are returned as None), for full-size checks that need one."""
    L = lib()
    arrays = [_as_storage(a, dtype) for a in arrays]
    for a in arrays:
        assert len(a) == n_in, (len(a), n_in)
    res = ctypes.c_void_p()
    err = ctypes.create_string_buffer(512)
    rc = L.vo_run(coll.encode(), algo.encode(), N, _ptrs(arrays), n_in, DTYPE_CODE[dtype], OP_CODE[op], root,
                  int(bool(inplace)), int(nchunks), ctypes.byref(res), err, len(err))
    if rc == 1:
        raise Unsupported(err.value.decode())
    if rc != 0:
        raise ValueError(err.value.decode())
    try:
        outs = []
        if want_outputs:
            es = np.dtype(STORAGE[dtype]).itemsize
            for i in range(L.vo_noutputs(res)):
                if keep is not None and i not in keep:
                    outs.append(None)
                    continue
                nbytes = L.vo_output_elems(res, i)
                o = np.empty(nbytes // es, dtype=STORAGE[dtype])
                L.vo_output_copy(res, i, o.ctypes.data)
                outs.append(o)
        log = TransferLog()
        if want_log:
            n = L.vo_nrecords(res)
            f = np.empty((n, 9), dtype=np.int64)
            if n:
                L.vo_records(res, f.ctypes.data)
            ch = np.empty(L.vo_nchunks_total(res), dtype=np.int64)
            if len(ch):
                L.vo_record_chunks(res, ch.ctypes.data)
            at = 0
            for i in range(n):
                step, src, dst, cnt, red, esz, so, do, nch = (int(v) for v in f[i])
                chunks = tuple(int(c) for c in ch[at:at + nch])
                at += nch
                phase = L.vo_record_phase(res, i).decode()
                if coll == "alltoall" and algo == "ring":
                    chunks = tuple(divmod(c, N) for c in chunks)  # (source, destination) of each block
                log.records.append(Transfer(step=step, phase=phase, src=src, dst=dst, n=cnt, reduce=bool(red),
                                            esize=esz, src_off=None if so < 0 else so,
                                            dst_off=None if do < 0 else do, chunks=chunks))
        return Result(outs, log, int(L.vo_hbm_bytes(res)), int(L.vo_local_steps(res)))
    finally:
        L.vo_free(res)


def _check_same(inputs, dtype):
    assert len(inputs) >= 1
    n = len(inputs[0])
    for x in inputs:
        assert len(x) == n
    return len(inputs), n


def allreduce(inputs, algo: str, dtype: str, inplace: bool = False, op: str = "sum", **kw) -> Result:
    N, n = _check_same(inputs, dtype)
    return _run("allreduce", algo, inputs, n, N, dtype, op=op, inplace=inplace, **kw)


def reduce_scatter(inputs, algo: str, dtype: str, op: str = "sum", **kw) -> Result:
    N, n = _check_same(inputs, dtype)
    return _run("reduce_scatter", algo, inputs, n, N, dtype, op=op, **kw)


def allgather(inputs, algo: str, dtype: str, **kw) -> Result:
    N, n = _check_same(inputs, dtype)
    return _run("allgather", algo, inputs, n, N, dtype, **kw)


def broadcast(root_input, N: int, root: int, algo: str, dtype: str, inplace: bool = False, **kw) -> Result:
    return _run("broadcast", algo, [root_input], len(root_input), N, dtype, root=root, inplace=inplace, **kw)


def broadcast_pipelined(root_input, N: int, root: int, algo: str, dtype: str, k: int, inplace: bool = False,
                        **kw) -> Result:
    if algo not in ALGOS_EXTRA["broadcast"]:
        raise Unsupported(f"broadcast/{algo}")
    return _run("broadcast", algo, [root_input], len(root_input), N, dtype, root=root, inplace=inplace,
                nchunks=k, **kw)


def scatter(root_input, N: int, root: int, algo: str, dtype: str, **kw) -> Result:
    return _run("scatter", algo, [root_input], len(root_input), N, dtype, root=root, **kw)


def gather(inputs, root: int, algo: str, dtype: str, **kw) -> Result:
    N, n = _check_same(inputs, dtype)
    return _run("gather", algo, inputs, n, N, dtype, root=root, **kw)


def reduce(inputs, root: int, algo: str, dtype: str, inplace: bool = False, op: str = "sum", **kw) -> Result:
    N, n = _check_same(inputs, dtype)
    return _run("reduce", algo, inputs, n, N, dtype, op=op, root=root, inplace=inplace, **kw)


def alltoall(inputs, algo: str, dtype: str, **kw) -> Result:
    N, n = _check_same(inputs, dtype)
    return _run("alltoall", algo, inputs, n, N, dtype, **kw)


@contextlib.contextmanager
def fault(kind: str, step: int):
    """Test-only: lose ("drop_step") or duplicate ("dup_step") every message of one step."""
    lib().vo_set_fault({"drop_step": 1, "dup_step": 2}[kind], step)
    try:
        yield
    finally:
        lib().vo_set_fault(0, -1)


def _at(fn, values_at, algo, size, dtype, idx, op):
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    vals = [_as_storage(np.asarray(v), dtype) for v in values_at]
    for v in vals:
        assert len(v) == len(idx)
    out = np.empty(len(idx), dtype=STORAGE[dtype])
    err = ctypes.create_string_buffer(512)
    rc = fn(_ptrs(vals), len(vals), algo.encode(), size, DTYPE_CODE[dtype], idx.ctypes.data, len(idx),
            OP_CODE[op], out.ctypes.data, err, len(err))
    if rc == 1:
        raise Unsupported(err.value.decode())
    if rc != 0:
        raise ValueError(err.value.decode())
    return out


def allreduce_at(values_at, algo: str, count: int, dtype: str, idx, op: str = "sum") -> np.ndarray:
    """Expected AllReduce output at element indices ``idx`` from the closed-form
    association tree; ``values_at[r]`` holds rank r's stored inputs there."""
    return _at(lib().vo_allreduce_at, values_at, algo, count, dtype, idx, op)


def reduce_scatter_at(values_at, algo: str, rc: int, dtype: str, idx, op: str = "sum") -> np.ndarray:
    """Expected ReduceScatter result for input-space element indices ``idx``
    (element e lands on rank e // rc at offset e % rc)."""
    return _at(lib().vo_reduce_scatter_at, values_at, algo, rc, dtype, idx, op)


def _conv(name, x, in_dt, out_dt):
    x = np.ascontiguousarray(x, dtype=in_dt)
    out = np.empty(len(x), dtype=out_dt)
    getattr(lib(), name)(x.ctypes.data, out.ctypes.data, len(x))
    return out


def f32_to_bf16(x):
    return _conv("vo_bf16_from_f32", x, np.float32, np.uint16)


def bf16_to_f32(b):
    return _conv("vo_f32_from_bf16", b, np.uint16, np.float32)


def f32_to_f16_bits(x):
    return _conv("vo_f16_from_f32", x, np.float32, np.uint16)


def f16_bits_to_f32(h):
    return _conv("vo_f32_from_f16", h, np.uint16, np.float32)
