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
                                             "nb": e.nb, "elem0": e.elem0, "src": [], "dst": []})
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


def _apply(op, mem: Memory, b: int, i0: int, i1: int) -> None:
    """Elements [i0, i1) of run b of one operation."""
    n = i1 - i0
    srcs = [mem.view(k, o, dt, off + b * stride + i0 * ESZ[dt], n) for (k, o, dt, off, stride) in op["src"]]
    if op["reduce"]:
        acc = _widen(srcs[0], op["src"][0][2])
        for s, (k, o, dt, off, stride) in zip(srcs[1:], op["src"][1:]):
            acc = _combine(acc, _widen(s, dt), op["red"])
    for (k, o, dt, off, stride) in op["dst"]:
        dstv = mem.view(k, o, dt, off + b * stride + i0 * ESZ[dt], n)
        dstv[:] = _narrow(acc, dt) if op["reduce"] else srcs[0]


def run_plan(plan, mem: Memory) -> None:
    for ops in plan:
        for op in ops:
            for b in range(op["nb"]):
                _apply(op, mem, b, 0, op["n"])


def position_places(plan, mem: Memory, group: int) -> list:
    """The sliced form's precondition, checked on the described plan: every
    operation names its first element position (elem0), a multiple of
    `group`, covers one run, and every operand holds position elem0 + i at a
    fixed place of its buffer -- byte off - elem0 * size + position * size,
    with one origin (off - elem0 * size) for all operands whose bytes overlap.
    Returns the violations (empty: each byte belongs to one position, so a
    thread that owns a group of positions owns every byte of them)."""
    bad = []
    spans = defaultdict(list)  # buffer -> (lo, hi, origin, size)
    for si, ops in enumerate(plan):
        for oi, op in enumerate(ops):
            e0 = op["elem0"]
            if e0 < 0 or e0 % group or op["nb"] != 1:
                bad.append((si, oi, "elem0", e0, op["nb"]))
                continue
            for (k, o, dt, off, stride) in op["src"] + op["dst"]:
                z = ESZ[dt]
                spans[mem.ident(k, o)].append((off, off + op["n"] * z, off - e0 * z, z, si, oi))
    for key, lst in spans.items():
        lst.sort()
        reach, place = None, None
        for (lo, hi, origin, z, si, oi) in lst:
            if reach is not None and lo < reach and (origin, z) != place:
                bad.append((si, oi, key, lo, origin, place))
            if reach is None or lo >= reach:
                place = (origin, z)
            reach = hi if reach is None else max(reach, hi)
    return bad


def origins(plan, es: int) -> list:
    """Every operand's (origin, alignment it needs): origin = byte offset -
    elem0 x its element size; 16 bytes, or 32 for the fp32 partial sums of
    16-bit data in scratch (accessed 32 bytes at a time)."""
    out = []
    for ops in plan:
        for op in ops:
            for (k, o, dt, off, stride) in op["src"] + op["dst"]:
                z = ESZ[dt]
                need = 32 if (k == SCRATCH and es == 2 and z == 4) else 16
                out.append((off - op["elem0"] * z, need))
    return out


def reads_before_writes(plan, mem: Memory) -> list:
    """Reads of a receive buffer or of scratch whose bytes no earlier step
    wrote (the sliced form reads those through L1 and needs none: what it
    reads there, the reading thread stored earlier in the launch).  Send
    buffers are inputs and may be read at any step; nothing may write them.
    Returns the violations."""
    bad = []
    written = defaultdict(list)  # buffer -> [(lo, hi)] written by earlier steps
    for si, ops in enumerate(plan):
        for oi, op in enumerate(ops):
            for (k, o, dt, off, stride) in op["dst"]:
                if k == SEND:
                    bad.append((si, oi, "writes a send buffer", o))
            for (k, o, dt, off, stride) in op["src"]:
                if k == SEND:
                    continue
                lo, hi = off, off + op["n"] * ESZ[dt]
                key = ("X", 0) if k == SCRATCH else ("R", o)
                cov = lo
                for (a, b) in sorted(written[key]):
                    if a <= cov < b:
                        cov = b
                if cov < hi:
                    bad.append((si, oi, key, lo, hi, cov))
        for op in ops:
            for (k, o, dt, off, stride) in op["dst"]:
                key = ("X", 0) if k == SCRATCH else ("R", o)
                written[key].append((off, off + op["n"] * ESZ[dt]))
    return bad


def run_plan_sliced(plan, mem: Memory, count: int, group: int, schedule) -> None:
    """The sliced form's execution with its owners interleaved as given: each
    group of `group` element positions walks the steps in order, applying the
    part of each operation that covers it; every entry of `schedule` (group
    indices, each len(plan) times) advances that group by one step.  Equal to
    run_plan for any schedule when the plan meets position_places."""
    ranges = [[(op["elem0"], op["elem0"] + op["n"]) for op in ops] for ops in plan]
    at = defaultdict(int)  # group -> next step
    for g in schedule:
        s = at[g]
        at[g] = s + 1
        a, z = g * group, min(count, (g + 1) * group)
        for op, (lo, hi) in zip(plan[s], ranges[s]):
            x, y = max(a, lo), min(z, hi)
            if x < y:
                _apply(op, mem, 0, x - lo, y - lo)


def one_after_another(groups: int, steps: int, reverse: bool = True) -> list:
    """Every group to the end before the next (last group first)."""
    order = range(groups - 1, -1, -1) if reverse else range(groups)
    return [g for g in order for _ in range(steps)]


def shuffled(groups: int, steps: int, rng) -> list:
    """A random interleaving of the groups' steps."""
    sched = np.repeat(np.arange(groups), steps)
    rng.shuffle(sched)
    return sched.tolist()


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


def slice_bytes(coll, N, count, es):
    """What a sliced call carries per rank, against the size limit: AllReduce
    and Reduce 4 bytes per element (fp32 / int32 data, or fp32 partials of
    16-bit data), ReduceScatter likewise per input element, AllGather, Gather
    and Scatter their N x count message, Broadcast its message; None for the
    AllToAlls."""
    return {"allreduce": count * 4, "reduce": count * 4, "reduce_scatter": count * N * 4,
            "allgather": count * N * es, "gather": count * N * es, "scatter": count * N * es,
            "broadcast": count * es}.get(coll)


def predict_sliced(coll, algo, N, count, dtype, root=0, inplace=False, nchunks=0, op="sum", limit=16 << 20):
    """The sliced form predicted from the described plan alone, with the checks
    above: two or more steps, every operation keeping positions (one run; a
    copy from one source), each byte at one position, origins aligned,
    write-before-read, within the size limit and not in place (AllReduce
    excepted).  Returns (sliced, host_ranges): the kernel derives operation
    ranges itself only where every origin is 0 and the data is 4 bytes wide.
    Left out: the library also needs the plan's description to fit a block's
    shared memory, which holds at the rank counts the tests use (16 or
    fewer; the ring AllReduce's is the first to outgrow it, at 19)."""
    plan, scratch = get_plan(coll, algo, N, count, dtype, root=root, inplace=inplace, nchunks=nchunks, op=op)
    es = ESZ[DT[dtype]]
    mem = Memory([None] * N, [0] * N, scratch)
    sb = slice_bytes(coll, N, count, es)
    ok = len(plan) >= 2 and sb is not None and sb <= limit and count < (1 << 29)
    ok = ok and not (inplace and coll != "allreduce")
    ok = ok and all(o["elem0"] >= 0 and o["nb"] == 1 and (o["reduce"] or len(o["src"]) == 1)
                    for ops in plan for o in ops)
    ok = ok and not position_places(plan, mem, 16 // es) and not reads_before_writes(plan, mem)
    orig = origins(plan, es) if ok else []
    ok = ok and all(o % need == 0 for o, need in orig)
    return ok, ok and (es == 2 or any(o != 0 for o, _ in orig))


def step_kind(ops):
    """A step's kernel kind as the plan description gives it: 0 for a copy
    step, 1 + op for a reduction step (one data type per plan).  None for a
    step without operations."""
    return ops[0]["red"] if ops else None


def launch_groups(plan, ident) -> list:
    """Runs of consecutive steps of one kind in which no step reads bytes an
    earlier step of the run wrote, or writes bytes an earlier one read or
    wrote: each (first, end) range may run as one launch.  `ident(kind,
    owner)` names the buffer an operand lies in, so that buffers that are one
    (an in-place call's send and receive buffers of a rank) compare equal.  An
    operand's bytes are the hull of its nb runs."""

    def spans(ops, role):
        out = []
        for op in ops:
            for (k, o, dt, off, stride) in op[role]:
                last = off + (op["nb"] - 1) * stride
                out.append((ident(k, o), min(off, last), max(off, last) + op["n"] * ESZ[dt]))
        return out

    def hit(a, b):
        return any(x[0] == y[0] and x[1] < y[2] and y[1] < x[2] for x in a for y in b)

    groups, s = [], 0
    while s < len(plan):
        reads, writes = spans(plan[s], "src"), spans(plan[s], "dst")
        e = s + 1
        while e < len(plan) and step_kind(plan[e]) == step_kind(plan[s]):
            r, w = spans(plan[e], "src"), spans(plan[e], "dst")
            if hit(writes, r) or hit(writes, w) or hit(reads, w):
                break
            reads, writes, e = reads + r, writes + w, e + 1
        groups.append((s, e))
        s = e
    return groups


def launches_of(ops) -> int:
    """Launches one (merged) step takes: all remaining operations at once if
    they fit the small kernel parameter block (16 operations, 64 operand
    pointers), else the largest prefix that fits the large one (128, 512)."""
    n, i = 0, 0
    ptrs = [len(op["src"]) + len(op["dst"]) for op in ops]
    while i < len(ops):
        j, p = i, 0
        while j < len(ops) and j - i < 16 and p + ptrs[j] <= 64:
            p, j = p + ptrs[j], j + 1
        if j < len(ops):
            j, p = i, 0
            while j < len(ops) and j - i < 128 and p + ptrs[j] <= 512:
                p, j = p + ptrs[j], j + 1
            assert j > i, "an operation with more operand pointers than the large block holds"
        n, i = n + 1, j
    return n
