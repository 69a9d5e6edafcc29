"""The execution form vc_plan_form reports, against the launches a call makes.

vc_plan_form answers on the host which form a call takes (sliced, one
cluster, or per step) and how many launches it makes.  Here calls of every
collective run on the GPU under the launch trace, with the default settings,
at sizes on both sides of the limits: one-rank in place (nothing to do),
unaligned chunk origins, in-place Broadcast, merged AllToAll rounds, and
steps that outgrow the kernel parameter block and split.  The trace must
show what vc_plan_form reported: the same number of launches, one sliced
launch for the sliced form, one cluster launch for the cluster form and
neither for per-step execution.  (Results are compared with the oracle in the
other GPU tests.)
"""
import pytest
import torch

import collective_communication_algorithms_virtual_gb300 as vc

pytestmark = pytest.mark.gpu

TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16, "i32": torch.int32}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from collective_communication_algorithms_virtual_gb300 import build

    build.build()
    vc.lib()
    old = (vc.vc_get_slice_limit(), vc.vc_get_single_launch(), vc.vc_get_merge_steps())
    vc.vc_set_slice_limit(vc.VC_SLICE_DEFAULT)
    vc.vc_set_single_launch(vc.VC_SINGLE_LAUNCH_DEFAULT)
    vc.vc_set_merge_steps(True)
    yield
    vc.vc_set_slice_limit(old[0])
    vc.vc_set_single_launch(old[1])
    vc.vc_set_merge_steps(old[2])
    assert vc.vc_device_errors() == 0


def _call(coll, algo, N, count, dtype, root=0, k=0, inplace=False):
    """The call, on zero-filled device buffers (the form does not depend on
    the data)."""
    dt = TORCH_DT[dtype]

    def z(n):
        return torch.zeros(n, dtype=dt, device="cuda")

    if coll == "allreduce":
        xs = [z(count) for _ in range(N)]
        ys = xs if inplace else [z(count) for _ in range(N)]
        return lambda: vc.vc_allreduce(xs, ys, algo=algo)
    if coll == "reduce_scatter":
        xs, ys = [z(N * count) for _ in range(N)], [z(count) for _ in range(N)]
        return lambda: vc.vc_reduce_scatter(xs, ys, algo=algo)
    if coll == "allgather":
        xs, ys = [z(count) for _ in range(N)], [z(N * count) for _ in range(N)]
        return lambda: vc.vc_allgather(xs, ys, algo=algo)
    if coll == "broadcast":
        ys = [z(count) for _ in range(N)]
        x = ys[root] if inplace else z(count)
        if algo.startswith("pipe_"):
            return lambda: vc.vc_broadcast_pipelined(x, ys, root=root, algo=algo, nchunks=k)
        return lambda: vc.vc_broadcast(x, ys, root=root, algo=algo)
    if coll == "scatter":
        x, ys = z(N * count), [z(count) for _ in range(N)]
        return lambda: vc.vc_scatter(x, ys, root=root, algo=algo)
    if coll == "gather":
        xs, y = [z(count) for _ in range(N)], z(N * count)
        return lambda: vc.vc_gather(xs, y, root=root, algo=algo)
    if coll == "reduce":
        xs = [z(count) for _ in range(N)]
        y = xs[root] if inplace else z(count)
        return lambda: vc.vc_reduce(xs, y, root=root, algo=algo)
    xs, ys = [z(N * count) for _ in range(N)], [z(N * count) for _ in range(N)]
    return lambda: vc.vc_alltoall(xs, ys, algo=algo)


# (coll, algo, N, count, dtype, root, nchunks, inplace)
CASES = [
    ("allreduce", "ring", 8, 1 << 18, "f32", 0, 0, False),  # 1 MiB per rank
    ("allreduce", "ring", 8, 1 << 18, "bf16", 0, 0, False),
    ("allreduce", "ring", 8, 5 << 20, "f32", 0, 0, False),  # 20 MiB per rank: above the slice limit
    ("allreduce", "rhd", 6, 1000, "f32", 0, 0, False),
    ("allreduce", "dbt", 16, 4096, "i32", 0, 0, False),
    ("allreduce", "mesh", 16, 5 << 20, "f32", 0, 0, False),
    ("allreduce", "ring_hop", 8, 4096, "f16", 0, 0, False),
    ("allreduce", "fused", 8, 4096, "f32", 0, 0, False),
    ("allreduce", "ring", 8, 4096, "f32", 0, 0, True),
    ("allreduce", "ring", 1, 4096, "f32", 0, 0, True),  # one rank in place: no launch
    ("reduce_scatter", "ring", 8, 4096, "f32", 0, 0, False),
    ("reduce_scatter", "ring", 8, 5, "f32", 0, 0, False),  # chunk origins not 16-byte aligned
    ("allgather", "ring", 8, 1024, "bf16", 0, 0, False),
    ("allgather", "ring", 8, 5, "f32", 0, 0, False),
    ("broadcast", "binomial", 8, 1000, "f32", 3, 0, False),
    ("broadcast", "binomial", 8, 1000, "f32", 3, 0, True),  # in place
    ("broadcast", "scatter_allgather", 5, 23, "f32", 4, 0, False),
    ("broadcast", "pipe_tree", 8, 4096, "bf16", 0, 4, False),
    ("broadcast", "pipe_chain", 8, 4096, "i32", 2, 0, False),
    ("scatter", "binomial", 8, 1024, "f32", 2, 0, False),
    ("gather", "binomial", 8, 1024, "f32", 5, 0, False),
    ("reduce", "binomial", 8, 1000, "f32", 7, 0, False),
    ("reduce", "binomial", 8, 1000, "bf16", 0, 0, True),
    ("alltoall", "pairwise", 8, 1024, "f32", 0, 0, False),  # rounds merged: one launch
    ("alltoall", "pairwise", 16, 1024, "f32", 0, 0, False),  # 256 operations: split in two
    ("alltoall", "bruck", 8, 128, "f32", 0, 0, False),
    ("alltoall", "ring", 8, 128, "bf16", 0, 0, False),
    ("alltoall", "bruck", 64, 16, "f32", 0, 0, False),  # steps beyond the parameter block
]


def test_reported_form_is_the_launches_made():
    seen = set()
    split = False
    for coll, algo, N, count, dtype, root, k, inplace in CASES:
        form, launches, _ = vc.vc_plan_form(coll, algo, N, count, dtype, root, inplace, k)
        fn = _call(coll, algo, N, count, dtype, root, k, inplace)
        fn()  # first call of the shape: the plan description becomes resident
        torch.cuda.synchronize()
        vc.vc_trace_enable(True)
        try:
            fn()
            torch.cuda.synchronize()
            recs = vc.vc_trace_read()
        finally:
            vc.vc_trace_enable(False)
        what = (coll, algo, N, count, dtype, root, k, inplace, form, launches, [r["kernel"] for r in recs[:4]])
        assert len(recs) == launches, what
        kinds = [r["kernel"] for r in recs]
        if form == "sliced":
            assert kinds[0].endswith("_sliced"), what
        elif form == "cluster":
            assert kinds[0].endswith("_single_launch"), what
        else:
            assert not any(x.endswith(("_sliced", "_single_launch")) for x in kinds), what
            split = split or launches > vc.vc_plan_describe(coll, algo, N, count, dtype, root, inplace, k)[2]
        seen.add(form)
    assert seen == {"sliced", "cluster", "steps"}
    assert split, "no case split a step over several launches"
