"""The Python binding's tensor checks, on the CPU with fake tensors.

The C ABI takes bare pointers and counts, so the binding checks every tensor
before a call: at least the elements the call reads or writes there,
contiguous, the call's dtype, one CUDA device, one tensor per rank.  Here the
library is replaced by a recorder: each collective with tensors of the right
sizes (or larger outputs) must reach it with the count the C ABI expects, and
every mismatch must raise VCError(VC_ERR_INVALID_ARG) without reaching it.
"""
import pytest
import torch

from collective_communication_algorithms_virtual_gb300 import binding as b


class FakeTensor:
    """What the binding reads of a tensor, with each property settable."""

    def __init__(self, n, dtype=torch.float32, dev=0, contiguous=True, ptr=0x10000):
        self._n, self.dtype, self._dev, self._contig, self._ptr = n, dtype, dev, contiguous, ptr
        self.shape = (n,)
        self.device = f"cuda:{dev}" if dev >= 0 else "cpu"

    def numel(self):
        return self._n

    def get_device(self):
        return self._dev

    def is_contiguous(self):
        return self._contig

    def data_ptr(self):
        return self._ptr


class Recorder:
    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def call(*args):
            self.calls.append((name, args))
            return 0
        return call


@pytest.fixture
def rec(monkeypatch):
    r = Recorder()
    monkeypatch.setattr(b, "lib", lambda: r)
    monkeypatch.setattr(b, "CHECK_TENSORS", True)
    return r


N = 4


def ts(n, k=N, **kw):
    return [FakeTensor(n, ptr=0x10000 * (i + 1), **kw) for i in range(k)]


def calls(rc):
    """Each collective with correct sizes, its C function and the count it must pass."""
    return [
        (lambda: b.vc_allreduce(ts(100), ts(100), stream=1), "vc_allreduce", 100),
        (lambda: b.vc_reduce_scatter(ts(N * rc), ts(rc), stream=1), "vc_reduce_scatter", rc),
        (lambda: b.vc_allgather(ts(rc), ts(N * rc), stream=1), "vc_allgather", rc),
        (lambda: b.vc_broadcast(FakeTensor(100), ts(100), stream=1), "vc_broadcast", 100),
        (lambda: b.vc_broadcast_pipelined(FakeTensor(100), ts(100), stream=1), "vc_broadcast_pipelined", 100),
        (lambda: b.vc_scatter(FakeTensor(N * rc), ts(rc), stream=1), "vc_scatter", rc),
        (lambda: b.vc_gather(ts(rc), FakeTensor(N * rc), stream=1), "vc_gather", rc),
        (lambda: b.vc_reduce(ts(100), FakeTensor(100), stream=1), "vc_reduce", 100),
        (lambda: b.vc_alltoall(ts(N * rc), ts(N * rc), stream=1), "vc_alltoall", rc),
    ]


def test_correct_tensors_reach_the_library_with_their_counts(rec):
    for fn, name, count in calls(7):
        fn()
        got, args = rec.calls[-1]
        assert got == name and args[2] == N and args[3] == count, (name, args[2:4])


def test_larger_outputs_are_accepted(rec):
    b.vc_allreduce(ts(100), ts(128), stream=1)
    b.vc_allgather(ts(5), ts(N * 5 + 3), stream=1)
    b.vc_gather(ts(5), FakeTensor(N * 5 + 1), stream=1)
    assert [c[0] for c in rec.calls] == ["vc_allreduce", "vc_allgather", "vc_gather"]


@pytest.mark.parametrize("bad", [
    lambda: b.vc_allreduce(ts(100), ts(99), stream=1),                           # an output too small
    lambda: b.vc_reduce_scatter(ts(N * 7 - 1), ts(7), stream=1),                 # inputs short of N blocks
    lambda: b.vc_allgather(ts(7), ts(N * 7 - 1), stream=1),                      # outputs short of N blocks
    lambda: b.vc_scatter(FakeTensor(N * 7 - 1), ts(7), stream=1),                # the root's message short
    lambda: b.vc_gather(ts(7), FakeTensor(N * 7 - 1), stream=1),                 # the root's output short
    lambda: b.vc_reduce(ts(100), FakeTensor(50), stream=1),
    lambda: b.vc_broadcast(FakeTensor(99), ts(100), stream=1),
    lambda: b.vc_allreduce(ts(100), ts(100, dtype=torch.bfloat16), stream=1),    # another dtype
    lambda: b.vc_allreduce(ts(100), ts(100, dev=1), stream=1),                   # another device
    lambda: b.vc_allreduce(ts(100, dev=-1), ts(100, dev=-1), stream=1),          # host tensors
    lambda: b.vc_alltoall(ts(N * 7), ts(N * 7, contiguous=False), stream=1),     # a strided view
    lambda: b.vc_allreduce(ts(100), ts(100, k=N - 1), stream=1),                 # a rank short
])
def test_mismatched_tensors_never_reach_the_library(rec, bad):
    with pytest.raises(b.VCError) as e:
        bad()
    assert e.value.status == b.VC_ERR_INVALID_ARG
    assert rec.calls == []


def test_checks_can_be_switched_off(rec, monkeypatch):
    monkeypatch.setattr(b, "CHECK_TENSORS", False)
    b.vc_allreduce(ts(100), ts(99), stream=1)
    assert rec.calls[-1][0] == "vc_allreduce"


def test_real_host_tensors_are_refused(rec):
    """torch's own host tensors (get_device() == -1): refused before the
    library, which would otherwise hand host pointers to a kernel."""
    xs = [torch.ones(16) for _ in range(N)]
    for fn in (lambda: b.vc_allreduce(xs, xs), lambda: b.vc_broadcast(xs[0], xs), lambda: b.vc_alltoall(xs, xs)):
        with pytest.raises(b.VCError) as e:
            fn()
        assert e.value.status == b.VC_ERR_INVALID_ARG and "CUDA" in str(e.value)
    assert rec.calls == []
