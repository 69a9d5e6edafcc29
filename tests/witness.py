"""Expansion of the order-witness fixtures into inputs and expected outputs.

A row of ``order_witness_n8_foldin.txt`` names the rank count N, the ranks a, b
and u that hold +2^24, -2^24 and +1 (every other rank holds 0) and the expected
fp32 result per part: one value (fused, rhd), one per tree half (dbt: the first
4N elements, then the rest), or one per chunk of 8 elements (ring, rs_ring).
Every rank holds 8N elements.
"""
import numpy as np

BIG = float(2 ** 24)


def inputs(N: int, a: int, b: int, u: int, n: int):
    vals = [0.0] * N
    vals[a], vals[b], vals[u] = BIG, -BIG, 1.0
    return [np.full(n, v, dtype=np.float32) for v in vals]


def rows(read_golden):
    out = []
    for row in read_golden("order_witness_n8_foldin.txt"):
        wid, N, a, b, u, algo = row[0], int(row[1]), int(row[2]), int(row[3]), int(row[4]), row[5]
        exp = [float(v) for v in row[6:]]
        count = 8 * N
        if len(exp) == 1:
            want = np.full(count, exp[0], dtype=np.float32)
        elif len(exp) == 2:
            want = np.repeat(np.array(exp, dtype=np.float32), 4 * N)
        else:
            assert len(exp) == N, row
            want = np.repeat(np.array(exp, dtype=np.float32), 8)
        out.append((wid, N, algo, inputs(N, a, b, u, count), want))
    return out
