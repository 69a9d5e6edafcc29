"""Virtual-rank collectives on one GB300.

N logical ranks are N buffers in one GPU's HBM.  The collectives and schedules
(Ring / Recursive Halving-Doubling / Double Binary Tree AllReduce, Ring
ReduceScatter and AllGather, binomial Broadcast and Scatter, Pairwise and
Bruck AllToAll, and a fused one-pass form of each) run in hand-written sm_103a
CUDA kernels behind the C ABI of ``include/vc.h``; this package is the thin
Python binding over it.
"""
from .binding import (  # noqa: F401
    ALGOS,
    COLLS,
    DTYPES,
    LIB_PATH,
    VCError,
    lib,
    vc_allgather,
    vc_allreduce,
    vc_alltoall,
    vc_broadcast,
    vc_broadcast_pipelined,
    vc_gather,
    vc_reduce,
    vc_busbw_factor,
    vc_last_error,
    vc_plan_describe,
    vc_plan_exec_order,
    vc_plan_form,
    vc_reduce_scatter,
    vc_scatter,
    vc_select_algo,
    vc_set_cost_model,
    vc_set_single_launch,
    vc_get_single_launch,
    vc_device_errors,
    vc_copy_selftest,
    SINGLE_LAUNCH_ALWAYS,
    VC_SINGLE_LAUNCH_DEFAULT,
    vc_set_slice_limit,
    vc_set_merge_steps,
    vc_get_merge_steps,
    vc_get_slice_limit,
    SLICE_ALWAYS,
    VC_SLICE_DEFAULT,
    vc_set_reuse_order,
    vc_get_reuse_order,
    REUSE_ORDER_NEVER,
    vc_set_copy_pipeline,
    vc_get_copy_pipeline,
    COPY_PIPELINE_NEVER,
    vc_get_cost_model,
    vc_status_string,
    vc_trace_enable,
    vc_trace_read,
    vc_version,
)
