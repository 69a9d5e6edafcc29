"""CPU replay of the library's step plans (test infrastructure).

``vc_plan_describe`` exports, without a GPU, the steps and operations the
library would launch.  This module executes them with numpy on byte buffers
standing in for device memory, checks that no operation of a step writes
bytes that another operation of the same step reads or writes (the plans'
race-freedom contract), and derives the rank-to-rank transfers each step
implies.  It shares nothing with the oracle: tests compare the two.
"""
from __future__ import annotations

from collections import Counter, defaultdict

import numpy as np
import torch

from collective_communication_algorithms_virtual_gb300 import vc_plan_describe

SEND, RECV, SCRATCH = 0, 1, 2
NPT = {0: np.float32, 1: np.uint16, 2: np.int32, 3: np.float16}
ESZ = {0: 4, 1: 2, 2: 4, 3: 2}
DT = {"f32": 0, "bf16": 1, "i32": 2, "f16": 3}


def get_plan(coll, algo, N, count, dtype, root=0, inplace=False, nchunks=0, op="sum"):
    entries, scratch, nsteps = vc_plan_describe(coll, algo, N, count, dtype, root, inplace, nchunks, op)
    steps = [dict() for _ in range(nsteps)]
    for e in entries:
        op = steps[e.step].setdefault(e.op, {"reduce": bool(e.reduce), "red": e.reduce, "n": e.n,
                                             "nb": e.nb, "src": [], "dst": []})
        (op["src"] if e.role == 0 else op["dst"]).append(
            (e.pos, e.buf, e.owner, e.dtype, e.byte_off, e.stride_bytes))
    out = []
    for st in steps:
        ops = []
        for k in sorted(st):
            op = st[k]
            op["src"] = [x[1:] for x in sorted(op["src"])]
            op["dst"] = [x[1:] for x in sorted(op["dst"])]
            ops.append(op)
        out.append(ops)
    return out, scratch


class Memory:
    """Byte buffers of every rank plus the scratch block."""

    def __init__(self, send, recv, scratch_bytes, inplace_ranks=()):
        self.send = [None if s is None else np.frombuffer(bytearray(s.tobytes()), np.uint8) for s in send]
        self.recv = [np.zeros(r, np.uint8) for r in recv]
        for r in inplace_ranks:
            self.recv[r] = self.send[r]
        self.scratch = np.full(max(1, scratch_bytes), 0xA5, np.uint8)
        self.inplace = set(inplace_ranks)

    def buf(self, kind, owner):
        if kind == SEND:
            return self.send[owner]
        if kind == RECV:
            return self.recv[owner]
        return self.scratch

    def ident(self, kind, owner):
        if kind == SCRATCH:
            return ("X", 0)
        if kind == SEND and owner in self.inplace:
            return ("R", owner)
        return ("S" if kind == SEND else "R", owner)

    def view(self, kind, owner, dt, off, n):
        b = self.buf(kind, owner)
        nbytes = n * ESZ[dt]
        assert off >= 0 and off + nbytes <= len(b), (kind, owner, off, nbytes, len(b))
        return b[off:off + nbytes]


def _widen(raw, dt):
    if dt == 0:
        return raw.view(np.float32).copy()
    if dt == 3:
        return raw.view(np.float16).astype(np.float32)
    if dt == 1:
        return (raw.view(np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)
    return raw.view(np.int32).view(np.uint32).copy()


def _narrow(acc, dt):
    if dt == 0:
        return acc.astype(np.float32).view(np.uint8)
    if dt == 3:
        with np.errstate(over="ignore"):
            return acc.astype(np.float32).astype(np.float16).view(np.uint8)
    if dt == 1:
        t = torch.from_numpy(acc.astype(np.float32)).to(torch.bfloat16)
        return t.view(torch.int16).numpy().view(np.uint8)
    return acc.astype(np.uint32).view(np.uint8)


def _combine(a, b, red):
    """1 sum, 2 max, 3 min (max/min: take b if it is larger/smaller or a is NaN)."""
    with np.errstate(over="ignore", invalid="ignore"):
        if red == 1:
            return a + b
        if a.dtype == np.uint32:
            ai, bi = a.view(np.int32), b.view(np.int32)
            return np.where(bi > ai if red == 2 else bi < ai, b, a)
        return np.where(((b > a) if red == 2 else (b < a)) | (a != a), b, a)


def run_plan(plan, mem: Memory) -> None:
    for ops in plan:
        for op in ops:
            n = op["n"]
            for b in range(op["nb"]):
                srcs = [mem.view(k, o, dt, off + b * stride, n) for (k, o, dt, off, stride) in op["src"]]
                if op["reduce"]:
                    acc = _widen(srcs[0], op["src"][0][2])
                    for s, (k, o, dt, off, stride) in zip(srcs[1:], op["src"][1:]):
                        acc = _combine(acc, _widen(s, dt), op["red"])
                for (k, o, dt, off, stride) in op["dst"]:
                    dstv = mem.view(k, o, dt, off + b * stride, n)
                    dstv[:] = _narrow(acc, dt) if op["reduce"] else srcs[0]


def hazards(plan, mem: Memory) -> list:
    """Pairs of operations of one step where one writes bytes the other touches."""
    found = []
    for si, ops in enumerate(plan):
        reads, writes = [], []
        for oi, op in enumerate(ops):
            for role, lst in (("r", op["src"]), ("w", op["dst"])):
                for (k, o, dt, off, stride) in lst:
                    for b in range(op["nb"]):
                        lo = off + b * stride
                        iv = (mem.ident(k, o), lo, lo + op["n"] * ESZ[dt], oi)
                        (reads if role == "r" else writes).append(iv)
        by_buf = defaultdict(list)
        for iv in writes:
            by_buf[iv[0]].append(("w",) + iv)
        for iv in reads:
            by_buf[iv[0]].append(("r",) + iv)
        for key, ivs in by_buf.items():
            ivs.sort(key=lambda x: x[2])
            for i in range(len(ivs)):
                for j in range(i + 1, len(ivs)):
                    a, c = ivs[i], ivs[j]
                    if c[2] >= a[3]:
                        break
                    if a[4] == c[4] or (a[0] == "r" and c[0] == "r"):
                        continue
                    found.append((si, a, c))
    return found


def transfers(plan) -> Counter:
    """(step, src rank, dst rank, reduce) -> elements, for every read of another rank's buffer."""
    tot = Counter()
    for si, ops in enumerate(plan):
        for op in ops:
            for (kd, od, dtd, offd, sd) in op["dst"]:
                for (ks, os_, dts, offs, ss) in op["src"]:
                    if os_ != od:
                        tot[(si, os_, od, op["reduce"])] += op["n"] * op["nb"]
    return tot


def oracle_transfers(log) -> Counter:
    tot = Counter()
    for t in log.records:
        if t.n:
            tot[(t.step, t.src, t.dst, t.reduce)] += t.n
    return tot
