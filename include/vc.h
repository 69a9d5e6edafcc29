/*
 * vc.h -- virtual-rank collectives on one GPU.
 *
 * N logical ranks are N buffers in one GPU's memory.  Each call reduces or
 * redistributes those buffers with one of the schedules analysed on three
 * pages: the Broadcast/Scatter page "一对多通信：Broadcast 与 Scatter"
 * (one-to-many communication), the CSDN article on CANN hccl's AllReduce
 * algorithms, and the latency-formula page "集合通信算法延迟公式" (alpha-beta
 * latency formulas of collective algorithms).  The call shape follows the
 * article's hccl_allreduce(sendbuf, recvbuf, count, dataType, op, comm,
 * stream) (section "hccl_allreduce接口详解"); the communicator becomes an
 * explicit rank count and one pointer per rank.
 *
 * Common rules for every collective below:
 *
 *  - Counts are in ELEMENTS, not bytes.
 *  - `send` / `recv` are HOST arrays of `nranks` DEVICE pointers, one per
 *    virtual rank, all on the current CUDA device.  The arrays are read
 *    during the call only; the buffers belong to the caller and must stay
 *    alive until the work enqueued on `stream` has finished.
 *  - Every call only enqueues work on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream) and returns without waiting for it.  Scratch
 *    memory, where a schedule needs it, comes from a memory pool owned by the
 *    library, is allocated and freed in stream order, and stays cached in the
 *    pool for later calls.
 *  - Output buffers must not overlap each other or any input, except where a
 *    function allows in-place operation.  Inputs may overlap each other.
 *  - Any alignment is accepted.  When every pointer a step touches is 16-byte
 *    aligned the vector path runs; otherwise a slower element-wise path.
 *  - Errors are returned, never raised: VC_ERR_INVALID_ARG (null pointer,
 *    nranks outside [1, VC_MAX_RANKS], root outside [0, nranks), overlapping
 *    buffers, a count above INT64_MAX / (16 nranks^2), beyond which some
 *    schedule's sizes would overflow), VC_ERR_UNSUPPORTED (an algorithm
 *    that is not defined for the collective or the rank count),
 *    VC_ERR_NOMEM (scratch allocation failed), VC_ERR_CUDA (a CUDA call or
 *    launch failed; vc_last_error() has the text).  On any error nothing has
 *    been enqueued, except for VC_ERR_CUDA from a launch after earlier steps.
 *  - A count of 0 returns VC_SUCCESS without enqueuing anything.
 *
 * Reductions (VC_SUM, VC_MAX, VC_MIN) on VC_FLOAT32 (in fp32), VC_BFLOAT16
 * and VC_FLOAT16 (inputs widened exactly to fp32, combined in fp32, rounded
 * once to the 16-bit type, round to nearest even) and VC_INT32 (sums wrap
 * around).  Every algorithm fixes the association per element, so results
 * are reproducible bit for bit run to run; different algorithms may differ
 * in the last bits of a sum.
 */
#ifndef VC_H_
#define VC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so that the header needs no CUDA headers. */
typedef struct CUstream_st* vc_stream_t;

#define VC_MAX_RANKS 64

typedef enum {
  VC_SUCCESS = 0,
  VC_ERR_INVALID_ARG = 1,
  VC_ERR_UNSUPPORTED = 2,
  VC_ERR_CUDA = 3,
  VC_ERR_NOMEM = 4,
  VC_ERR_TIMEOUT = 5
} vc_status_t;

typedef enum { VC_FLOAT32 = 0, VC_BFLOAT16 = 1, VC_INT32 = 2, VC_FLOAT16 = 3 } vc_dtype_t;

/*
 * Reduction ops, as the hccl article lists them (SUM / MAX / MIN).  MAX and
 * MIN keep the first operand unless the second is larger (smaller) or the
 * first is NaN: a NaN is passed over while a number is present, and of +0
 * and -0 the one met first in the algorithm's fixed association is kept.
 * int32 compares signed.  16-bit floats are compared after exact widening.
 */
typedef enum { VC_SUM = 0, VC_MAX = 1, VC_MIN = 2 } vc_op_t;

typedef enum {
  VC_ALGO_FUSED = 0,             /* one pass over all ranks: every collective          */
  VC_ALGO_RING = 1,              /* AllReduce, ReduceScatter, AllGather, AllToAll      */
  VC_ALGO_RHD = 2,               /* AllReduce; fold-in when nranks is not 2^k          */
  VC_ALGO_DBT = 3,               /* AllReduce                                          */
  VC_ALGO_BINOMIAL = 4,          /* Broadcast, Scatter, Gather, Reduce                 */
  VC_ALGO_SCATTER_ALLGATHER = 5, /* Broadcast                                          */
  VC_ALGO_PAIRWISE = 6,          /* AllToAll                                           */
  VC_ALGO_BRUCK = 7,             /* AllToAll                                           */
  VC_ALGO_AUTO = 8,              /* any collective: cheapest under the cost model      */
  VC_ALGO_PIPE_CHAIN = 9,        /* Broadcast, message cut into chunks along a chain   */
  VC_ALGO_PIPE_TREE = 10,        /* Broadcast, chunks down the binomial tree           */
  VC_ALGO_MESH = 11,             /* AllReduce: root 0 folds every rank, then sends     */
  VC_ALGO_RING_HOP = 12          /* AllReduce: ring, partials rounded on every hop     */
} vc_algo_t;

typedef enum {
  VC_COLL_ALLREDUCE = 0,
  VC_COLL_REDUCE_SCATTER = 1,
  VC_COLL_ALLGATHER = 2,
  VC_COLL_BROADCAST = 3,
  VC_COLL_SCATTER = 4,
  VC_COLL_ALLTOALL = 5,
  VC_COLL_GATHER = 6,
  VC_COLL_REDUCE = 7
} vc_coll_t;

/*
 * AllReduce: recv[r][i] = sum over q of send[q][i], for every rank r and
 * element i < count.  Latency-formula page, sections "Ring AllReduce",
 * "Recursive Halving-Doubling" and "Double Binary Tree" (eqs.
 * model-algo-ring-ar, model-algo-rhd-ar, model-algo-dbt-ar); hccl article,
 * sections "Ring算法", "Tree算法".
 *   send[r], recv[r]: `count` elements each.  send[r] == recv[r] (in place)
 *   is allowed, as hccl_allreduce allows sendbuf == recvbuf.
 *   algo: FUSED (rank-order sum in one pass), RING (ReduceScatter + AllGather
 *   in 2(N-1) steps; 16-bit data keeps fp32 partial sums in library scratch),
 *   RING_HOP (the same ring with the partial sums kept in the data type and
 *   rounded on every hop; equals RING for fp32 and int32), RHD (2 log2 N
 *   rounds for N a power of 2; otherwise the first 2(N-P) ranks, P the
 *   largest power of 2 below N, fold in pairwise before and get the result
 *   back after), DBT (two mirrored heap trees, 2 floor(log2 N) levels),
 *   MESH (hccl article, section "Mesh算法：全连接广播": rank 0 folds the other
 *   ranks in rank order, one per step, then sends the result to each, one
 *   per step; 2(N-1) steps).
 */
vc_status_t vc_allreduce(const void* const* send, void* const* recv, int nranks, size_t count,
                         vc_dtype_t dtype, vc_op_t op, vc_algo_t algo, vc_stream_t stream);

/*
 * ReduceScatter: recv[r][j] = sum over q of send[q][r*recvcount + j].
 * Latency-formula page, section "Ring ReduceScatter" (eq.
 * model-algo-ring-reducescatter).
 *   send[q]: nranks*recvcount elements; recv[r]: recvcount elements.  No in-place.
 *   algo: FUSED or RING (N-1 steps; rank r's chain ends on rank r).
 */
vc_status_t vc_reduce_scatter(const void* const* send, void* const* recv, int nranks,
                              size_t recvcount, vc_dtype_t dtype, vc_op_t op, vc_algo_t algo,
                              vc_stream_t stream);

/*
 * AllGather: recv[r][q*sendcount + j] = send[q][j].  Latency-formula page,
 * section "Ring AllGather" (eq. model-algo-ring-allgather).
 *   send[q]: sendcount elements; recv[r]: nranks*sendcount elements.  No in-place.
 *   algo: FUSED or RING (a local copy, then N-1 ring steps).
 */
vc_status_t vc_allgather(const void* const* send, void* const* recv, int nranks, size_t sendcount,
                         vc_dtype_t dtype, vc_algo_t algo, vc_stream_t stream);

/*
 * Broadcast: recv[r][i] = send_root[i] for every rank r.  Broadcast/Scatter
 * page, section "Broadcast" (eq. onetoall-bcast-semantic) and its algorithm
 * sections.
 *   send_root, recv[r]: `count` elements.  send_root == recv[root] is allowed.
 *   algo: FUSED (one read, N writes), BINOMIAL (ceil(log2 N) steps),
 *   SCATTER_ALLGATHER (binomial Scatter of N chunks, then a Ring AllGather),
 *   PIPE_CHAIN or PIPE_TREE (as vc_broadcast_pipelined with nchunks = 0).
 */
vc_status_t vc_broadcast(const void* send_root, void* const* recv, int nranks, size_t count,
                         vc_dtype_t dtype, int root, vc_algo_t algo, vc_stream_t stream);

/*
 * Scatter: recv[r][j] = send_root[r*recvcount + j].  Broadcast/Scatter page,
 * section "Scatter" (eq. onetoall-scatter-semantic) and "二叉树 Scatter".
 *   send_root: nranks*recvcount elements; recv[r]: recvcount elements.  No in-place.
 *   algo: FUSED or BINOMIAL (ceil(log2 N) steps, halving sizes).
 */
vc_status_t vc_scatter(const void* send_root, void* const* recv, int nranks, size_t recvcount,
                       vc_dtype_t dtype, int root, vc_algo_t algo, vc_stream_t stream);

/*
 * AllToAll: recv[j][i*blockcount + e] = send[i][j*blockcount + e].
 * Latency-formula page, section "AllToAll 算法怎么选" (eqs.
 * model-algo-a2a-pairwise, model-algo-a2a-bruck).
 *   send[i], recv[j]: nranks*blockcount elements.  No in-place.
 *   algo: FUSED (one pass), PAIRWISE (N-1 exchange rounds plus the local
 *   block), BRUCK (ceil(log2 N) rounds through two library scratch buffers),
 *   RING (eq. model-algo-a2a-ring: N-1 rounds of store and forward to the
 *   right-hand neighbour, through two library forwarding buffers).
 */
vc_status_t vc_alltoall(const void* const* send, void* const* recv, int nranks, size_t blockcount,
                        vc_dtype_t dtype, vc_algo_t algo, vc_stream_t stream);

/*
 * Cost model behind VC_ALGO_AUTO (process-wide, thread-safe).  The model is
 * the latency-formula page's alpha-beta (Hockney) model, T = alpha terms +
 * data terms.
 *
 *   VC_COST_HBM (default): the model on one GPU, where every virtual rank
 *     lives in the same HBM: T = (steps that launch work) * alpha +
 *     (algorithmic bytes the call reads and writes) / beta, both taken from
 *     the call's plan.  Candidates: every algorithm of the collective, the
 *     fused one included.  Defaults: alpha = 1.9e-6 s (one dependent step on
 *     a GB300 with programmatic dependent launch, fitted to the message-size
 *     sweep), beta = 6.6e12 B/s (measured HBM copy rate).
 *   VC_COST_LINK: the pages' own formulas with M the per-rank message and
 *     beta a link bandwidth (eqs. model-algo-ring-ar, -rhd-ar, -dbt-ar,
 *     -ring-reducescatter, -ring-allgather, -a2a-pairwise, -a2a-bruck,
 *     -a2a-ring, -reduce-tree; Broadcast/Scatter page eqs. binomial-bcast,
 *     binomial-scatter, onetoall-gather-scatter-duality, pipe-chain-bcast,
 *     pipe-tree-bcast).
 *     Candidates: the pages' algorithms only (no fused).  Defaults: alpha =
 *     5e-6 s, beta = 450e9 B/s, the page's NVLink example.
 *
 * alpha <= 0 or beta <= 0 selects the policy's default; a NaN or infinite
 * alpha or beta returns VC_ERR_INVALID_ARG and leaves the model unchanged.
 * Ties go to the first candidate in enum order.
 */
typedef enum { VC_COST_HBM = 0, VC_COST_LINK = 1 } vc_cost_policy_t;

vc_status_t vc_set_cost_model(vc_cost_policy_t policy, double alpha_s, double beta_bytes_per_s);
vc_status_t vc_get_cost_model(vc_cost_policy_t* policy, double* alpha_s, double* beta_bytes_per_s);

/*
 * The algorithm VC_ALGO_AUTO would run for these arguments and the time the
 * model predicts for it (host only, no CUDA call).  `count` follows the
 * collective's convention; `root` is used by the rooted collectives
 * (Broadcast, Scatter, Gather, Reduce).
 */
vc_status_t vc_select_algo(vc_coll_t coll, int nranks, size_t count, vc_dtype_t dtype, int root,
                           vc_algo_t* algo, double* predicted_s);

/*
 * Broadcast with the message cut into `nchunks` chunks that travel one
 * behind another (Broadcast/Scatter page, sections "分块链式流水线", eq.
 * pipe-chain-bcast: N+k-2 steps, and "分块二叉树流水线", eq. pipe-tree-bcast:
 * ceil(log2 N)+k-1 steps).  Chunk j follows the chain (PIPE_CHAIN) or the
 * binomial tree (PIPE_TREE) delayed by j steps.  nchunks = 0 takes the
 * optimum of the page's formula under the current cost model,
 * k* = sqrt(h M / (alpha beta)) with h = N-2 (chain) or ceil(log2 N)-1
 * (tree), within [1, 256] and at most one chunk per 16 bytes; otherwise
 * nchunks must be in [1, 1024].  vc_broadcast with a PIPE algorithm uses
 * nchunks = 0.  Other algorithms ignore nchunks.  Buffers as vc_broadcast.
 */
vc_status_t vc_broadcast_pipelined(const void* send_root, void* const* recv, int nranks, size_t count,
                                   vc_dtype_t dtype, int root, vc_algo_t algo, int nchunks,
                                   vc_stream_t stream);

/*
 * Gather: recv_root[q*sendcount + j] = send[q][j] -- Scatter's dual
 * (Broadcast/Scatter page, section "对偶性：Scatter 与 Gather", eq.
 * onetoall-gather-scatter-duality: its data flow reversed, same cost).
 *   send[q]: sendcount elements; recv_root (a single device pointer, the
 *   root's buffer): nranks*sendcount elements.  No in-place.
 *   algo: FUSED or BINOMIAL (distances 1, 2, 4, ...: each subtree hands
 *   everything it holds to its parent).
 */
vc_status_t vc_gather(const void* const* send, void* recv_root, int nranks, size_t sendcount,
                      vc_dtype_t dtype, int root, vc_algo_t algo, vc_stream_t stream);

/*
 * Reduce: recv_root[i] = sum over q of send[q][i] (latency-formula page,
 * section "Broadcast / Reduce 怎么用 Tree 算法", eq. model-algo-reduce-tree).
 *   send[q], recv_root: `count` elements.  recv_root == send[root] is allowed.
 *   algo: FUSED (rank-order sum) or BINOMIAL (the binomial Broadcast run
 *   backwards with adds: distances 1, 2, 4, ...; the sum is the balanced
 *   tree over adjacent ranks counted from the root).
 */
vc_status_t vc_reduce(const void* const* send, void* recv_root, int nranks, size_t count, vc_dtype_t dtype,
                      vc_op_t op, int root, vc_algo_t algo, vc_stream_t stream);

/* Name of a status code (static string). */
const char* vc_status_string(vc_status_t status);

/* Text of the last error on the calling thread ("" if none). */
const char* vc_last_error(void);

/*
 * busbw = algbw * factor: AllReduce 2(N-1)/N; AllGather, ReduceScatter,
 * AllToAll (N-1)/N; Broadcast, Reduce 1 (latency-formula page, table
 * tbl-model-algo-busbw-coef).  Scatter and Gather are not in that table and
 * get (N-1)/N.
 * Returns 0 for an unknown collective or nranks < 1.
 */
double vc_busbw_factor(vc_coll_t coll, int nranks);

/*
 * Schedule introspection (host only; no CUDA call, usable without a GPU).
 *
 * Builds the step plan a call with these arguments would execute (nchunks:
 * as vc_broadcast_pipelined, ignored by other algorithms; inplace: 1 for an
 * AllReduce with send[r] == recv[r], a Broadcast with send_root ==
 * recv[root] or a Reduce with recv_root == send[root], and
 * VC_ERR_INVALID_ARG for the other collectives, which do not run in place)
 * and writes
 * one entry per operand of every operation.  An operation reads its sources
 * in the listed order (`pos`), combines them left to right with the step's
 * op (reduction steps) or copies its single source (copy steps), and writes
 * the result to each of its
 * destinations; it covers `nb` runs of `n` elements, run b starting
 * b*stride_bytes after run 0.  All operations of one step are independent;
 * steps run in order (vc_plan_form reports how they are launched).
 *   buf: 0 send, 1 recv, 2 library scratch; owner: the rank that holds it;
 *   byte_off: from the start of that rank's buffer (scratch: of the scratch
 *   block); dtype: storage type of the operand; elem0: the element position
 *   of the operation's first element, where the schedule keeps positions --
 *   its element i is position elem0 + i, held in order by each operand's
 *   region.  Positions are the elements of the message: AllReduce's and the
 *   tree Reduce's buffer, ring ReduceScatter's input, ring AllGather's
 *   output, the Broadcasts' message, the binomial Scatter's input and
 *   Gather's output at the root.  Else -1.
 * Returns VC_ERR_INVALID_ARG if `capacity` is too small (with *n_entries set
 * to the size needed).  *scratch_bytes receives the scratch the call needs,
 * *n_steps the number of steps.
 */
typedef struct {
  int32_t step;
  int32_t op;     /* operation index within the step */
  int32_t role;   /* 0 source, 1 destination */
  int32_t pos;    /* position within the sources or destinations */
  int32_t buf;    /* 0 send, 1 recv, 2 scratch */
  int32_t owner;  /* rank */
  int32_t dtype;  /* vc_dtype_t of the operand */
  int32_t reduce; /* 0 copy; reduction: 1 sum, 2 max, 3 min */
  int64_t byte_off;
  int64_t n;
  int64_t nb;
  int64_t stride_bytes;
  int64_t elem0;  /* element position of the first element, or -1 (above) */
} vc_plan_entry_t;

vc_status_t vc_plan_describe(vc_coll_t coll, vc_algo_t algo, int nranks, size_t count,
                             vc_dtype_t dtype, vc_op_t op, int root, int inplace, int nchunks,
                             vc_plan_entry_t* entries,
                             size_t capacity, size_t* n_entries, size_t* scratch_bytes,
                             int* n_steps);

/*
 * Host-only: the execution form a call with these arguments takes under the
 * current settings (vc_set_slice_limit, vc_set_single_launch,
 * vc_set_merge_steps), on 16-byte aligned buffers with a resident plan
 * description (a call whose buffers are not aligned, or whose shape is first
 * seen while its stream is captured, runs per step).
 *   *form: VC_FORM_SLICED (one launch over the GPU, each thread carrying its
 *     group of positions through every step), VC_FORM_CLUSTER (one launch of
 *     one thread-block cluster with a barrier between steps) or VC_FORM_STEPS
 *     (one launch per step, or per run of independent steps, and more than
 *     one for a step whose operations outgrow the kernel parameter block);
 *   *launches: the launches the call makes (1 for the one-launch forms; 0 for
 *     a call with nothing to do);
 *   *host_ranges: for the sliced form, 1 if its kernel reads the operation
 *     ranges the host lists (16-bit data, or a region not at origin 0), 0 if
 *     it derives them from each operation's first operand.
 * VC_ERR_INVALID_ARG for a null output; other errors as vc_plan_describe.
 * Needs no GPU.
 */
typedef enum { VC_FORM_STEPS = 0, VC_FORM_CLUSTER = 1, VC_FORM_SLICED = 2 } vc_form_t;
vc_status_t vc_plan_form(vc_coll_t coll, vc_algo_t algo, int nranks, size_t count, vc_dtype_t dtype, vc_op_t op,
                         int root, int inplace, int nchunks, int* form, int* launches, int* host_ranges);

/*
 * Host-only introspection of the L2 reuse order (vc_set_reuse_order, read at
 * the call): the plan vc_plan_describe returns, in the order the library
 * executes it (no counterpart on the source pages).  For the k-th operation
 * executed (steps in order, a step's operations consecutive):
 *   order[k]: its index within its step as vc_plan_describe numbers it;
 *   keep[k]: 1 if its results are stored with the default L2 policy (the
 *            next step reads them), else 0 (streaming);
 * reverse[s]: 1 if step s walks its tiles last to first.
 * This is the order of per-step launches; a one-launch plan (vc_set_single_
 * launch) runs the same operation order with every step walked forward and
 * plain stores, and launches of multi-destination (fused) operations walk
 * forward with streaming stores.
 * *n_ops and *n_steps receive the sizes; null arrays with both capacities 0
 * ask for the sizes only.  VC_ERR_INVALID_ARG if a capacity is too small.
 * Needs no GPU.
 */
vc_status_t vc_plan_exec_order(vc_coll_t coll, vc_algo_t algo, int nranks, size_t count, vc_dtype_t dtype,
                               vc_op_t op, int root, int inplace, int nchunks, uint32_t* order, uint8_t* keep,
                               size_t op_capacity, uint8_t* reverse, size_t step_capacity, size_t* n_ops,
                               int* n_steps);

/*
 * Launch trace (off by default; host bookkeeping plus two CUDA events per
 * launch while on).  While enabled, every kernel launch the library makes is
 * bracketed by CUDA events recorded on the caller's stream, and a record
 * keeps the collective, algorithm, step, kernel variant and the launch's
 * algorithmic bytes (every operand of every operation read or written once,
 * at its storage size); at most 2^20 records are kept between reads (later
 * launches run untraced).  vc_trace_enable(1) clears old records;
 * vc_trace_read waits for the recorded events, writes up to `capacity`
 * records with their event-timed durations and clears them.
 *   kernel: bits 0-2 the mode (0 copy, 1 fp32, 2 int32, 3 bf16 with fp32
 *   partials among the sources, 4 bf16 only, 5 fp16 with fp32 partials, 6
 *   fp16 only), bits 3-4 the op (0 sum, 1 max, 2 min), bit 5 set when the
 *   launch used the large parameter block (more than 16 operations or 64
 *   operand pointers), bit 6 set when an fp32 / int32 launch too small to
 *   fill the GPU took the kernel that loads four sources at a time or a copy
 *   launch took the bulk-copy (TMA) pipeline, bit 7
 *   set for a single-launch plan (vc_set_single_launch: one record for the
 *   whole call, step -1, bytes and nops of all steps; bits 0-2 then give the
 *   mode of the plan's reduction steps), bit 8 set as well when that launch
 *   ran the sliced form (vc_set_slice_limit).
 */
typedef struct {
  int32_t coll;   /* vc_coll_t */
  int32_t algo;   /* vc_algo_t */
  int32_t step;
  int32_t kernel;
  int64_t bytes;
  int32_t nops;
  float ms;
} vc_trace_record_t;

vc_status_t vc_trace_enable(int on);
vc_status_t vc_trace_read(vc_trace_record_t* records, size_t capacity, size_t* n_records);

/*
 * Single-launch execution.
 *
 * By default every step of a schedule is one kernel launch and stream order
 * is the barrier between steps.  A call whose schedule has two or more steps,
 * each moving at most `max_step_bytes` (algorithmic bytes: every operand of
 * every operation read or written once), instead runs ALL its steps in one
 * launch: a single thread-block cluster (16 blocks where the device allows,
 * else 8) executes the steps in order with a cluster-wide barrier between
 * consecutive steps.  The operations, their order and every element's
 * association are unchanged, so results are identical bit for bit; what goes
 * away is one launch and one grid drain per step, which dominate small
 * messages.  It applies when, in addition,
 *   - the schedule's reduction steps share one data type and op (true of
 *     every schedule of this library),
 *   - its description fits the kernel's shared memory (96 KB; e.g. the ring
 *     AllReduce up to 21 ranks),
 *   - every buffer pointer of the call is 16-byte aligned,
 *   - it is not an AllToAll (their steps of many small block copies measured
 *     faster as one launch a step; a Pairwise AllToAll's independent rounds
 *     share one launch under vc_set_merge_steps), and
 *   - the description is resident on the device.  It is uploaded once per
 *     call shape (collective, algorithm, ranks, count, type, op, root, in
 *     place), at the first call that is not being captured into a CUDA graph
 *     (a capture of a shape not seen before takes the per-step path), into
 *     at most 64 MB of device memory per device that is kept until the
 *     process exits; shapes beyond that take the per-step path.
 *  max_step_bytes: 0 disables single-launch execution, SIZE_MAX applies it
 *  to every eligible call.  Default VC_SINGLE_LAUNCH_DEFAULT, the measured
 *  crossover on a GB300 (8 ranks, fp32): at steps of 768 KB or less one
 *  cluster beats a launch per step over the whole GPU, above it the full
 *  GPU's bandwidth wins.  Process-wide.
 */
#define VC_SINGLE_LAUNCH_DEFAULT ((size_t)768 << 10)
vc_status_t vc_set_single_launch(size_t max_step_bytes);
vc_status_t vc_get_single_launch(size_t* max_step_bytes);

/*
 * Sliced execution (a form of single-launch execution, tried before the
 * cluster form).
 *
 * In the AllReduce schedules (Ring, RHD, DBT, Mesh, RING_HOP), the ring
 * ReduceScatter and AllGather, the Broadcasts (binomial, Scatter+AllGather,
 * pipelined), the binomial Scatter and Gather and the tree Reduce, every
 * operation maps element position e of each source to position e of each
 * destination, where positions are the elements of the message (AllReduce's
 * and Reduce's buffer, ReduceScatter's input, AllGather's output, the
 * Broadcast message, Scatter's input and Gather's output at the root), and
 * each buffer region holds its positions in order at
 * one place: the send and receive buffers and the partial sums the schedule
 * keeps in scratch (fp32 for bf16 / fp16 data).  A call of such a schedule
 * runs all its steps in one launch over the whole GPU when, per rank, it
 * carries at most `max_bytes_per_rank`: AllReduce 4 bytes per element (the
 * fp32 / int32 data, or the fp32 partials of 16-bit data), ReduceScatter 4
 * bytes per input element likewise, AllGather its output, Broadcast its
 * message (Reduce, Scatter and Gather likewise).  Each thread owns one group
 * of positions (16 bytes of the data
 * type) of every buffer and carries it through every step of the plan in
 * order, applying each operation that covers it.  What a step reads at a
 * position was written there by an earlier step, by the same thread, so the
 * thread's program order is the step barrier and no thread reads what
 * another wrote.  The steps, operations, operands and every element's
 * association (16-bit data: widened, combined in fp32, rounded once) are
 * unchanged, so results are identical bit for bit; different positions
 * merely run out of step with each other, as when a ring is pipelined in
 * slices.  The 16-bit AllReduce Ring and the ReduceScatter ring keep one
 * partial per element while the partials take at most 16 MiB per rank;
 * above that they alternate two chunk-sized slots per rank, which several
 * positions share, and do not run sliced at 5 ranks or more.  In-place
 * calls other than AllReduce, and the AllToAlls, take the other forms.  The
 * conditions of single-launch execution on alignment and the resident
 * description apply as well, and the description with each operation's
 * element range and each operand's address must fit the kernel's 96 KB of
 * shared memory (the ring AllReduce up to 18 ranks, the ring ReduceScatter
 * and AllGather up to 25 and 26, the tree schedules up to 64).  max_bytes_per_rank: 0 disables it, SIZE_MAX
 * applies it to every eligible call.  Default VC_SLICE_LIMIT_DEFAULT: up to
 * 16 MiB per rank the form measured faster than the cluster form and than
 * per-step launches (8 ranks, fp32 and bf16, GB300; above, the whole GPU's
 * bandwidth per step wins for AllReduce).  Process-wide.
 */
#define VC_SLICE_LIMIT_DEFAULT ((size_t)16 << 20)
vc_status_t vc_set_slice_limit(size_t max_bytes_per_rank);
vc_status_t vc_get_slice_limit(size_t* max_bytes_per_rank);

/*
 * Independent steps in one launch.
 *
 * With one launch per step, stream order is the barrier between steps; a
 * barrier is needed only where a step reads what an earlier one wrote, or
 * writes what an earlier one read or wrote.  When `on` (the default), a run of
 * consecutive steps of one kind in which no step does either with respect to
 * the earlier steps of the run runs as one launch, the steps' operations in
 * step order (each block takes them in that order), without a barrier
 * between them.  Such runs: Pairwise AllToAll's rounds, each reading only the
 * send buffers and writing its own output blocks; the Ring AllToAll's local
 * copy with its first round; the Mesh AllReduce's copies of the result to
 * each rank; binomial steps (Broadcast, Scatter, Gather, the pipelined
 * tree) at rank counts that are not powers of 2, where a rank reached in one
 * step forwards nothing in the next.  Every operation, operand and byte is
 * unchanged; vc_plan_describe still reports the schedule's steps, and
 * vc_plan_form the launches.  Process-wide; applies to plans built after the
 * call (the plan cache is cleared).
 */
vc_status_t vc_set_merge_steps(int on);
vc_status_t vc_get_merge_steps(int* on);

/*
 * Bulk-copy pipeline for large copy steps (no counterpart on the source
 * pages: an execution choice that leaves every result unchanged, bit for
 * bit).  A per-step copy launch whose operations move whole 16-byte groups
 * and that writes at least min_bytes in total, in a call with no bf16 / fp16
 * reduction step, runs as a pipeline of bulk (TMA) loads into shared memory,
 * three 32 KB stages per SM, each landed tile written to every destination
 * with bulk stores; other copy launches load and store through registers.
 * The pipeline holds most of an SM's shared memory while the reduction
 * kernels run best with a large L1 (the 16-bit ones most), so each switch
 * between the two reconfigures the SMs; the default, VC_COPY_PIPELINE_DEFAULT,
 * is where the pipeline's higher copy bandwidth pays for that on a GB300
 * (8 ranks: AllGather 4-6% faster from 128 MiB per step, fp32 ring and
 * halving-doubling AllReduce 2-4% at 256 MiB per rank; slower below).  0
 * takes it for every eligible copy launch, SIZE_MAX for none.  Process-wide.
 */
#define VC_COPY_PIPELINE_DEFAULT ((size_t)128 << 20)
vc_status_t vc_set_copy_pipeline(size_t min_bytes);
vc_status_t vc_get_copy_pipeline(size_t* min_bytes);

/*
 * L2 reuse order (no counterpart on the source pages: an execution choice
 * that leaves every result unchanged, bit for bit).  A step that follows one
 * writing at least min_step_bytes walks its tiles in the direction opposite
 * to that step, with its (independent) operations listed so that the one
 * whose inputs were written last comes first; results the next step reads
 * are stored with the default L2 policy instead of streaming.  The step then
 * starts on lines still in L2.  Below the default, VC_REUSE_ORDER_DEFAULT,
 * the data stay in L2 anyway and the reordering measured slower on a GB300.
 * 0 orders every step, SIZE_MAX none.  Process-wide; applies to plans built
 * after the call (the plan cache is cleared).
 */
#define VC_REUSE_ORDER_DEFAULT ((size_t)16 << 20)
vc_status_t vc_set_reuse_order(size_t min_step_bytes);
vc_status_t vc_get_reuse_order(size_t* min_step_bytes);

/*
 * Device error word.  Waits for `stream` (after the work enqueued so far),
 * then reads and clears the word: bit 1 set when a bulk-copy pipeline's wait
 * for a tile's load gave up (the launch then stopped issuing copies and
 * returned; its outputs are incomplete).  Never set in correct operation;
 * the waits are bounded so that a fault elsewhere cannot hang a launch.
 */
vc_status_t vc_device_errors(vc_stream_t stream, uint32_t* flags);

/* Exercises that bounded wait (no counterpart on the source pages): runs the
 * bulk-copy pipeline on a 64 KB copy whose first tile's load is announced but
 * never issued, so the wait for it gives up (within about a second) and
 * the launch returns.  *flags receives the error word that launch left
 * (bit 1 set); the word is cleared before and after.  Allocates and frees
 * 128 KB of device memory and waits for `stream`. */
vc_status_t vc_copy_selftest(vc_stream_t stream, uint32_t* flags);

/*
 * Ring ReduceScatter that allocates no device memory.
 *
 * The source pages have no counterpart to this call: it exists for callers
 * that cannot allocate device memory while they run -- code inside a custom
 * allocator or an out-of-memory handler, real-time loops that forbid
 * cudaMalloc and pool growth, or hosts whose memory budget is fixed ahead of
 * time.  It computes exactly what vc_reduce_scatter(..., VC_ALGO_RING, ...)
 * computes (same schedule and execution order, same results bit for bit),
 * but its partial sums live in one fixed array that the library places in
 * each GPU's memory when its device code is loaded there, instead of in the
 * library's pool, in two block slots per rank (the allocating call keeps one
 * slot per block while they take at most 16 MiB per rank).
 *
 *   op: VC_SUM only; VC_MAX and VC_MIN return VC_ERR_UNSUPPORTED.
 *   dtype: VC_FLOAT32, VC_BFLOAT16, VC_FLOAT16 or VC_INT32.
 *   send[q]: nranks*recvcount elements; recv[r]: recvcount elements; no in-place.
 *   Scratch needed: nranks * roundup(2 * recvcount * 4, 256) bytes (two
 *   4-byte partial slots per rank -- 16-bit partials are kept in fp32 --
 *   each rank's pair rounded up to 256 bytes), at most
 *   VC_NOALLOC_SCRATCH_BYTES (16 MiB); larger calls return VC_ERR_INVALID_ARG
 *   and enqueue nothing.
 *   The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current.  With CUDA's lazy module
 *   loading that lookup (or the first launch of any of this library's
 *   kernels) is also when the device code, and with it the array, is loaded
 *   onto the device, which takes device memory.  So make the first call of
 *   this entry point on each device outside the code that must not allocate,
 *   and before any stream capture; later calls allocate nothing.
 *   Every call shares the one array and leaves its last contents behind (no
 *   part of it needs to start at zero: every partial sum is written before
 *   it is read).  Calls whose work overlaps on the GPU -- on two streams, or
 *   from two threads -- race on the array: serialise them.
 */
#define VC_NOALLOC_SCRATCH_BYTES (16u << 20)
vc_status_t vc_reduce_scatter_noalloc(const void* const* send, void* const* recv, int nranks,
                                      size_t recvcount, vc_dtype_t dtype, vc_op_t op,
                                      vc_stream_t stream);

/* Library version, major*10000 + minor*100 + patch. */
int vc_version(void);

#ifdef __cplusplus
}
#endif

#endif /* VC_H_ */
