"""How a rank buffer is cut into N chunks.

[hccl article], section "Ring算法：环形流水线传输": ``chunk_size = count / size``
in C integer division, which silently drops ``count mod size`` elements.  The
[Latency-formula page], section "Ring AllReduce：带宽最优", splits the data into
N equal chunks of M/N.  Neither says what happens to a remainder.

Reading taken: chunk c of a buffer of ``count`` elements is
``[min(c*ce, count), min((c+1)*ce, count))`` with
``ce = ceil(count / N)`` rounded up to a multiple of ``16 / esize`` elements, so
every chunk starts 16 bytes from the previous one's start.  All elements are
covered exactly once; the last chunks may be short or empty.  When N divides
count into 16-byte multiples this is exactly the pages' equal split.
"""
from __future__ import annotations


def chunk_elems(count: int, nparts: int, esize: int) -> int:
    """ce: the (aligned) elements per chunk."""
    if count <= 0:
        return 0
    align = 16 // esize
    ce = -(-count // nparts)
    return -(-ce // align) * align


def chunk_range(c: int, count: int, nparts: int, esize: int) -> tuple[int, int]:
    """[lo, hi) element range of chunk c."""
    ce = chunk_elems(count, nparts, esize)
    return min(c * ce, count), min((c + 1) * ce, count)


def chunk_of(e: int, count: int, nparts: int, esize: int) -> int:
    """Index of the chunk holding element e."""
    ce = chunk_elems(count, nparts, esize)
    return e // ce
