"""Transfer log written by every simulated schedule.

One record per message: at step ``step`` rank ``src`` sends ``n`` elements to
rank ``dst``; ``reduce`` says whether the receiver adds them to its own data
(ReduceScatter / Reduce phases) or stores them (AllGather / Broadcast phases).
``src_off`` / ``dst_off`` are element offsets in the sender's and receiver's
logical buffers (None where a message carries several chunks; then ``chunks``
lists the chunk indices it carries).  ``esize`` is bytes per element on the
wire.
"""
from __future__ import annotations

from collections import Counter, defaultdict
from dataclasses import dataclass, field


@dataclass(frozen=True)
class Transfer:
    step: int
    phase: str
    src: int
    dst: int
    n: int
    reduce: bool
    esize: int
    src_off: int | None = None
    dst_off: int | None = None
    chunks: tuple = ()

    @property
    def nbytes(self) -> int:
        return self.n * self.esize


@dataclass
class TransferLog:
    records: list = field(default_factory=list)

    def add(self, **kw) -> None:
        self.records.append(Transfer(**kw))

    def steps(self) -> list[int]:
        """Distinct step indices that carry data (a message of at least one
        element), in order."""
        return sorted({t.step for t in self.records if t.n > 0})

    def bytes_sent_by(self, rank: int) -> int:
        return sum(t.nbytes for t in self.records if t.src == rank)

    def bytes_received_by(self, rank: int) -> int:
        return sum(t.nbytes for t in self.records if t.dst == rank)

    def max_message_bytes_per_step(self) -> dict[int, int]:
        """Largest single message of each step: what one link carries per step
        in the alpha-beta model, where a step's messages travel in parallel."""
        out: dict[int, int] = defaultdict(int)
        for t in self.records:
            out[t.step] = max(out[t.step], t.nbytes)
        return dict(out)

    def bandwidth_bytes(self) -> int:
        """Sum over steps of the step's largest message (the M/beta factor)."""
        return sum(self.max_message_bytes_per_step().values())

    def pattern(self) -> Counter:
        """Multiset of (step, src, dst, reduce, n): the comparison key."""
        return Counter((t.step, t.src, t.dst, t.reduce, t.n) for t in self.records)

    def table(self) -> list[tuple[int, int, int]]:
        """(step, src, dst) triples sorted: the shape printed in the pages' tables."""
        return sorted((t.step, t.src, t.dst) for t in self.records)
