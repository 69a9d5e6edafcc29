// Launcher and C ABI of the virtual-rank collectives (host side).
//
// A call becomes a plan (plan.h, cached per call shape).  Its steps run one
// launch each on the caller's stream (kernels.cuh step_kernel), with the
// parameter block filled here from the plan and the call's pointers; or, for
// a small plan, all in one cluster launch of the plan kernel, whose
// description is uploaded to device memory once per call shape.  Also here:
// argument checks, the scratch pool, the cost-model selection of
// VC_ALGO_AUTO, the launch trace, and the C entry points of vc.h.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstddef>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <tuple>
#include <map>
#include <memory>
#include <unordered_map>
#include <mutex>
#include <string>
#include <vector>

#include "kernels.cuh"
#include "slice.cuh"
#include "plan.h"
#include "vc.h"

#define VC_EXPORT extern "C" __attribute__((visibility("default")))

namespace vc {

// ---------------------------------------------------------------------------
// errors
// ---------------------------------------------------------------------------
namespace {
thread_local std::string g_last_error;

vc_status_t fail(vc_status_t s, const std::string& msg) {
  g_last_error = msg;
  return s;
}
vc_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(VC_ERR_CUDA, std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")");
}
// VC_PDL=0 launches every step in plain stream order (for comparison).
bool pdl_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("VC_PDL");
    return !(v && std::strcmp(v, "0") == 0);
  }();
  return on;
}
// Copy launches writing at least this many bytes take the bulk-copy pipeline
// (vc_set_copy_pipeline).
std::atomic<size_t> g_copy_pipeline{VC_COPY_PIPELINE_DEFAULT};
// Steps after one that writes at least this many bytes are ordered for L2
// reuse (vc_set_reuse_order); read when a plan is built.
std::atomic<size_t> g_reuse_min{VC_REUSE_ORDER_DEFAULT};
bool log_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("VC_LOG");
    return v && v[0] && std::strcmp(v, "0") != 0;
  }();
  return on;
}
}  // namespace



// ---------------------------------------------------------------------------
// per-device state: SM count, occupancy, scratch pool
// ---------------------------------------------------------------------------
namespace {

// Blocks of one kernel resident per SM.
struct Residency {
  int blocks = 1;
};
struct DeviceState {
  bool init = false;
  int nsm = 0;
  cudaMemPool_t pool = nullptr;
  std::map<const void*, Residency> occupancy;
};
std::mutex g_mu;
DeviceState g_dev[64];

vc_status_t device_state(DeviceState** out, int* dev_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(VC_ERR_CUDA, "device index out of range");
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.init) {
    e = cudaDeviceGetAttribute(&st.nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    st.init = true;
  }
  *out = &st;
  *dev_out = dev;
  return VC_SUCCESS;
}

vc_status_t scratch_pool(DeviceState* st, int dev, cudaMemPool_t* pool) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!st->pool) {
    cudaMemPoolProps props;
    std::memset(&props, 0, sizeof(props));
    props.allocType = cudaMemAllocationTypePinned;
    props.handleTypes = cudaMemHandleTypeNone;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaError_t e = cudaMemPoolCreate(&st->pool, &props);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemPoolCreate");
    uint64_t keep = UINT64_MAX;  // keep freed scratch cached for the next call
    e = cudaMemPoolSetAttribute(st->pool, cudaMemPoolAttrReleaseThreshold, &keep);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemPoolSetAttribute");
  }
  *pool = st->pool;
  return VC_SUCCESS;
}

// Resident blocks per SM of a kernel (its occupancy limit), queried once.
template <class K>
Residency residency(DeviceState* st, K kernel) {
  std::lock_guard<std::mutex> lk(g_mu);
  const void* key = reinterpret_cast<const void*>(kernel);
  auto it = st->occupancy.find(key);
  if (it != st->occupancy.end()) return it->second;
  Residency r;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, dev::kThreads, 0) != cudaSuccess || n < 1) n = 1;
  r.blocks = n;
  st->occupancy[key] = r;
  return r;
}

// ---------------------------------------------------------------------------
// launch trace
// ---------------------------------------------------------------------------
// What a step launch knows of its call: collective, algorithm and step (for
// the trace), and whether its copies may take the bulk-copy pipeline.
struct LaunchCtx {
  int coll = 0, algo = 0, step = 0;
  bool pipeline = true;
};
struct Pending {
  vc_trace_record_t rec;
  cudaEvent_t start, stop;
};
std::mutex g_trace_mu;
bool g_trace_on = false;
size_t g_trace_dropped = 0;
constexpr size_t kTraceMax = 1u << 20;  // records kept until vc_trace_read

std::vector<Pending> g_trace;
// With g_trace_mu held: whether this launch is traced (tracing on and room
// left; launches past the cap are counted, not recorded).
bool trace_slot() {
  if (!g_trace_on) return false;
  if (g_trace.size() < kTraceMax) return true;
  ++g_trace_dropped;
  return false;
}
std::vector<cudaEvent_t> g_event_pool;

cudaError_t take_event(cudaEvent_t* ev) {
  if (!g_event_pool.empty()) {
    *ev = g_event_pool.back();
    g_event_pool.pop_back();
    return cudaSuccess;
  }
  return cudaEventCreate(ev);
}

int64_t launch_bytes(const Step& st, size_t i, size_t j) {
  int64_t b = 0;
  for (size_t k = i; k < j; ++k) {
    const Op& op = st.ops[k];
    int64_t per = 0;
    for (const Operand& o : op.src) per += esize(o.dt);
    for (const Operand& o : op.dst) per += esize(o.dt);
    b += per * op.n * op.nb;
  }
  return b;
}

// ---------------------------------------------------------------------------
// launching one step
// ---------------------------------------------------------------------------
struct Bases {
  const void* const* send;  // per rank (broadcast/scatter: only the root's entry is used)
  void* const* recv;
  char* scratch;
};

const char* base_ptr(const Bases& b, const Operand& o) {
  switch (o.buf) {
    case Buf::Send: return static_cast<const char*>(b.send[o.owner]) + o.byte_off;
    case Buf::Recv: return static_cast<const char*>(b.recv[o.owner]) + o.byte_off;
    default: return b.scratch + o.byte_off;
  }
}

// Elements in one vector group of a step's kernel (must match the device's
// group_elems): 16 bytes of the copied type; 4 fp32 / int32 values; 8 values
// of a 16-bit type (fp32 partial sums among them move 32 bytes).
int64_t group_elements(Mode mode, int esz) {
  switch (mode) {
    case Mode::Copy: return 16 / esz;
    case Mode::F32:
    case Mode::I32: return 4;
    case Mode::BF16:
    case Mode::F16: return 8;
  }
  return 0;
}

// Descriptor of one operation, except its tiling and pointer index.
// `ptrs_aligned`: every operand address is 16-byte aligned.
void describe_op(dev::OpDesc& d, const Op& op, Mode mode, bool ptrs_aligned) {
  d.n = op.n;
  d.nb = op.nb;
  d.sstride = op.sstride;
  d.dstride = op.dstride;
  d.ns = static_cast<uint8_t>(op.src.size());
  d.nd = static_cast<uint8_t>(op.dst.size());
  d.esz = static_cast<uint8_t>(esize(op.src[0].dt));
  d.smask = d.dmask = 0;
  for (size_t s = 0; s < op.src.size(); ++s)
    if (op.src[s].dt == DT::F32) d.smask |= 1ull << s;
  for (size_t s = 0; s < op.dst.size(); ++s)
    if (op.dst[s].dt == DT::F32) d.dmask |= 1ull << s;
  const int64_t gelems = group_elements(mode, d.esz);
  bool aligned = ptrs_aligned;
  if (op.nb > 1) aligned &= (op.n % gelems) == 0 && (op.sstride % 16) == 0 && (op.dstride % 16) == 0;
  d.vec = aligned ? 1 : 0;
  d.groups = aligned ? op.n / gelems : 0;
  d.keep = op.keep ? 1 : 0;
}

// Tiles operations d[0, n): the largest number of groups per thread (4, 2 or
// 1) that still gives `cap` tiles (one per resident block), so a small step
// is spread over many blocks instead of a few doing all of it.  Returns the
// tile count, or -1 if it does not fit the 32-bit tile numbers.
int64_t assign_tiles(dev::OpDesc* d, size_t n, int64_t cap, int max_upt = dev::kUnroll) {
  auto tiles_per_run = [](const dev::OpDesc& o, int upt) {
    const int64_t per = o.vec ? int64_t(upt) * dev::kThreads : dev::kTileElems;
    const int64_t units = o.vec ? o.groups : o.n;
    return std::max<int64_t>(1, (units + per - 1) / per);
  };
  auto count_tiles = [&](int upt) {
    int64_t total = 0;
    for (size_t k = 0; k < n; ++k) total += tiles_per_run(d[k], upt) * d[k].nb;
    return total;
  };
  int upt = max_upt;
  while (upt > 1 && count_tiles(upt) < cap) upt /= 2;
  int64_t tiles = 0;
  for (size_t k = 0; k < n; ++k) {
    d[k].upt = static_cast<uint8_t>(upt);
    const int64_t tpr = tiles_per_run(d[k], upt);
    d[k].tpr = static_cast<uint32_t>(tpr);
    d[k].tile0 = static_cast<uint32_t>(tiles);
    tiles += tpr * d[k].nb;
    if (tiles > 0xFFFFFFFFll || tpr > 0xFFFFFFFFll) return -1;
  }
  return tiles;
}

// Fills the parameter block of operations [i, j) of a step.
template <class P>
bool fill_params(P& p, const Step& st, size_t i, size_t j, const Bases& b, int64_t cap, int64_t* tiles_out,
                 int max_upt = dev::kUnroll) {
  std::memset(&p, 0, sizeof(P));
  int np = 0;
  for (size_t k = i; k < j; ++k) {
    const Op& op = st.ops[k];
    bool aligned = true;
    const int p0 = np;
    for (const Operand& o : op.src) {
      const char* ptr = base_ptr(b, o);
      p.ptr[np++] = ptr;
      aligned &= (reinterpret_cast<uintptr_t>(ptr) & 15) == 0;
    }
    for (const Operand& o : op.dst) {
      const char* ptr = base_ptr(b, o);
      p.ptr[np++] = ptr;
      aligned &= (reinterpret_cast<uintptr_t>(ptr) & 15) == 0;
    }
    describe_op(p.op[k - i], op, st.mode, aligned);
    p.op[k - i].p0 = static_cast<uint16_t>(p0);
  }
  const int64_t tiles = assign_tiles(p.op, j - i, cap, max_upt);
  if (tiles < 0) return false;
  p.nops = static_cast<uint32_t>(j - i);
  p.rev = st.reverse ? 1 : 0;
  p.late = 0;
  p.ntiles = static_cast<uint32_t>(tiles);
  *tiles_out = tiles;
  return true;
}

template <int MODE, int OP, class P>
vc_status_t launch_typed(DeviceState* st, const Step& s, size_t i, size_t j, const Bases& b, cudaStream_t stream,
                         const LaunchCtx& tc) {
  static thread_local P p;  // large: keep off the stack
  // tiles are sized against the vector-only kernel's residency
  auto kernel = dev::step_kernel<MODE, OP, P, 1, false, false>;
  Residency res = residency(st, kernel);
  int64_t cap = int64_t(st->nsm) * res.blocks;
  int64_t tiles = 0;
  if (!fill_params(p, s, i, j, b, cap, &tiles)) return fail(VC_ERR_INVALID_ARG, "operation too large for one launch");
  if (tiles == 0) return VC_SUCCESS;
  bool elem = false, fan = false;
  int maxns = 0;
  for (uint32_t k = 0; k < p.nops; ++k) {
    const dev::OpDesc& d = p.op[k];
    elem |= !d.vec || d.groups * group_elements(s.mode, d.esz) < d.n;
    // multi-destination operations: bulk-store kernels for copies and fp32 / int32 sums
    fan |= (MODE == dev::kCopy || MODE == dev::kF32 || MODE == dev::kI32) && d.nd > 1;
    maxns = std::max<int>(maxns, d.ns);
  }
  // fp32 / int32: a launch that does not fill the GPU (tiles were shrunk)
  // with a many-source operation loads four sources at a time
  bool batched = false;
  if constexpr (MODE == dev::kF32 || MODE == dev::kI32) {
    batched = p.op[0].upt < dev::kUnroll && maxns > 2;
    if (batched)
      kernel = elem ? dev::step_kernel<MODE, OP, P, 4, true, false> : dev::step_kernel<MODE, OP, P, 4, false, false>;
  }
  if constexpr (MODE == dev::kCopy || MODE == dev::kF32 || MODE == dev::kI32) {
    if (fan && !batched)
      kernel = elem ? dev::step_kernel<MODE, OP, P, 1, true, true> : dev::step_kernel<MODE, OP, P, 1, false, true>;
  }
  if (!batched && !fan && elem) kernel = dev::step_kernel<MODE, OP, P, 1, true, false>;
  if (batched || elem || fan) {
    res = residency(st, kernel);
    cap = int64_t(st->nsm) * res.blocks;
  }
  // copies of aligned whole groups: the bulk-copy pipeline, one block per SM, tiles of up to 32 KB
  unsigned block = dev::kThreads;
  size_t dyn_smem = 0;
  bool tma = false;
  if constexpr (MODE == dev::kCopy) {
    // Only for launches that write at least the set minimum (128 MiB by
    // default) in calls without 16-bit reductions: the pipeline wants most of
    // an SM's shared memory while the other step kernels run with a large L1,
    // so the SMs are reconfigured at each switch, and a reduction kernel that
    // starts early behind the pipeline runs in its configuration; smaller
    // copies, and the 16-bit reductions (the most sensitive to L1), lose more
    // there than the pipeline gains.
    int64_t groups = 0;  // 16-byte groups the launch writes
    for (uint32_t k = 0; k < p.nops; ++k) groups += p.op[k].groups * p.op[k].nb * p.op[k].nd;
    const size_t min_bytes = g_copy_pipeline.load(std::memory_order_relaxed);
    if (!elem && tc.pipeline && min_bytes != SIZE_MAX && static_cast<size_t>(groups) * 16 >= min_bytes) {
      cap = st->nsm;
      if (!fill_params(p, s, i, j, b, cap, &tiles, dev::kCopyTileBytes / (dev::kThreads * 16)))
        return fail(VC_ERR_INVALID_ARG, "operation too large for one launch");
      kernel = dev::tma_copy_kernel<P>;
      block = dev::kCopyThreads;
      dyn_smem = dev::kCopyStages * dev::kCopyTileBytes + dev::kCopyStages * sizeof(uint64_t);
      tma = true;
      static std::once_flag once[64];  // per device
      cudaError_t ea = cudaSuccess;
      std::call_once(once[st - g_dev], [&] {
        ea = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(dyn_smem));
      });
      if (ea != cudaSuccess) return cuda_fail(ea, "cudaFuncSetAttribute");
    }
  }
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(tiles, cap));
  p.late = tiles < cap ? 1 : 0;  // the grid leaves room: the next grid only after this one's wait
  std::unique_lock<std::mutex> lk(g_trace_mu);
  const bool trace = trace_slot();
  if (!trace) lk.unlock();
  Pending pend{};
  if (trace) {
    cudaError_t e = take_event(&pend.start);
    if (e == cudaSuccess) e = take_event(&pend.stop);
    if (e == cudaSuccess) e = cudaEventRecord(pend.start, stream);
    if (e != cudaSuccess) return cuda_fail(e, "trace event");
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = dyn_smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  if (trace) {
    e = cudaEventRecord(pend.stop, stream);
    if (e != cudaSuccess) return cuda_fail(e, "trace event");
    pend.rec.coll = tc.coll;
    pend.rec.algo = tc.algo;
    pend.rec.step = tc.step;
    pend.rec.kernel = MODE | (OP << 3) | (sizeof(P) == sizeof(dev::LargeParams) ? 32 : 0) | (batched || tma ? 64 : 0);
    pend.rec.bytes = launch_bytes(s, i, j);
    pend.rec.nops = static_cast<int32_t>(j - i);
    g_trace.push_back(pend);
  }
  return VC_SUCCESS;
}

template <int MODE, class P>
vc_status_t launch_op(DeviceState* st, const Step& s, size_t i, size_t j, const Bases& b, cudaStream_t stream,
                      const LaunchCtx& tc) {
  switch (s.red) {
    case RedOp::Max: return launch_typed<MODE, dev::kMax, P>(st, s, i, j, b, stream, tc);
    case RedOp::Min: return launch_typed<MODE, dev::kMin, P>(st, s, i, j, b, stream, tc);
    default: return launch_typed<MODE, dev::kSum, P>(st, s, i, j, b, stream, tc);
  }
}

template <class P>
vc_status_t launch_mode(DeviceState* st, const Step& s, size_t i, size_t j, const Bases& b, cudaStream_t stream,
                        const LaunchCtx& tc) {
  // 16-bit steps whose sources are all of the data type take the batched kernel
  auto pure = [&](DT want) {
    for (size_t k = i; k < j; ++k)
      for (const Operand& o : s.ops[k].src)
        if (o.dt != want) return false;
    return true;
  };
  switch (s.mode) {
    case Mode::Copy: return launch_typed<dev::kCopy, dev::kSum, P>(st, s, i, j, b, stream, tc);
    case Mode::F32: return launch_op<dev::kF32, P>(st, s, i, j, b, stream, tc);
    case Mode::I32: return launch_op<dev::kI32, P>(st, s, i, j, b, stream, tc);
    case Mode::BF16:
      return pure(DT::BF16) ? launch_op<dev::kBF16P, P>(st, s, i, j, b, stream, tc)
                            : launch_op<dev::kBF16, P>(st, s, i, j, b, stream, tc);
    default:
      return pure(DT::F16) ? launch_op<dev::kF16P, P>(st, s, i, j, b, stream, tc)
                           : launch_op<dev::kF16, P>(st, s, i, j, b, stream, tc);
  }
}

int op_ptrs(const Op& op) { return static_cast<int>(op.src.size() + op.dst.size()); }

// The launch of step `s` that starts at operation i: all the remaining
// operations if they fit the small parameter block (16 operations, 64
// operand pointers), else the largest prefix that fits the large one (128,
// 512; *large set).  Returns the end of its operations; i itself when one
// operation alone has too many operands.
size_t launch_span(const Step& s, size_t i, bool* large) {
  size_t j = i;
  int ptrs = 0;
  while (j < s.ops.size() && j - i < 16 && ptrs + op_ptrs(s.ops[j]) <= 64) ptrs += op_ptrs(s.ops[j++]);
  *large = j != s.ops.size();
  if (!*large) return j;
  j = i;
  ptrs = 0;
  while (j < s.ops.size() && j - i < 128 && ptrs + op_ptrs(s.ops[j]) <= 512) ptrs += op_ptrs(s.ops[j++]);
  return j;
}

vc_status_t launch_step(DeviceState* st, const Step& s, const Bases& b, cudaStream_t stream, int* launches,
                        const LaunchCtx& tc) {
  for (size_t i = 0; i < s.ops.size();) {
    bool large = false;
    const size_t j = launch_span(s, i, &large);
    if (j == i) return fail(VC_ERR_INVALID_ARG, "operation has too many operands");
    const vc_status_t rc = large ? launch_mode<dev::LargeParams>(st, s, i, j, b, stream, tc)
                                 : launch_mode<dev::SmallParams>(st, s, i, j, b, stream, tc);
    if (rc != VC_SUCCESS) return rc;
    ++*launches;
    i = j;
  }
  return VC_SUCCESS;
}

// Per-step execution of a plan: f(first step, step) for each step, where a
// run of independent steps (Plan::launch_end) is one step holding their
// operations in step order.  Stops at the first status other than success.
template <class F>
vc_status_t for_each_launch_group(const Plan& plan, F&& f) {
  for (size_t si = 0; si < plan.steps.size();) {
    const size_t se = plan.launch_end.empty() ? si + 1 : plan.launch_end[si];
    vc_status_t rc;
    if (se == si + 1) {
      rc = f(si, plan.steps[si]);
    } else {
      Step merged = plan.steps[si];
      for (size_t k = si + 1; k < se; ++k)
        merged.ops.insert(merged.ops.end(), plan.steps[k].ops.begin(), plan.steps[k].ops.end());
      rc = f(si, static_cast<const Step&>(merged));
    }
    if (rc != VC_SUCCESS) return rc;
    si = se;
  }
  return VC_SUCCESS;
}

// ---------------------------------------------------------------------------
// argument checks shared by the entry points
// ---------------------------------------------------------------------------
const char* coll_name(Coll c) {
  static const char* n[] = {"allreduce", "reduce_scatter", "allgather", "broadcast", "scatter", "alltoall",
                            "gather", "reduce"};
  return n[static_cast<int>(c)];
}
const char* algo_name(Algo a) {
  static const char* n[] = {"fused", "ring", "rhd", "dbt", "binomial", "scatter_allgather", "pairwise", "bruck",
                            "auto", "pipe_chain", "pipe_tree", "mesh", "ring_hop"};
  return n[static_cast<int>(a)];
}

struct Call {
  Coll coll;
  Algo algo;
  bool autoalgo = false;  // VC_ALGO_AUTO: pick algo from the cost model
  int nranks;
  int64_t count;
  DT dt;
  int root = 0;
  const void* const* send = nullptr;  // per-rank inputs (AllReduce, ReduceScatter, AllGather, AllToAll)
  const void* send_root = nullptr;    // Broadcast, Scatter
  void* const* recv = nullptr;
  void* recv_root = nullptr;          // Gather, Reduce
  int nchunks = 0;                    // pipelined Broadcast (0: from the cost model)
  RedOp red = RedOp::Sum;
  cudaStream_t stream = nullptr;
};

bool overlap(const void* a, int64_t na, const void* b, int64_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + static_cast<uintptr_t>(nb) && y < x + static_cast<uintptr_t>(na);
}

vc_status_t plan_status(PlanStatus ps, const std::string& why) {
  if (ps == PlanStatus::Invalid) return fail(VC_ERR_INVALID_ARG, why);
  if (ps == PlanStatus::Unsupported) return fail(VC_ERR_UNSUPPORTED, why);
  return VC_SUCCESS;
}

vc_status_t to_op(vc_op_t op, RedOp* out) {
  switch (op) {
    case VC_SUM: *out = RedOp::Sum; return VC_SUCCESS;
    case VC_MAX: *out = RedOp::Max; return VC_SUCCESS;
    case VC_MIN: *out = RedOp::Min; return VC_SUCCESS;
  }
  return fail(VC_ERR_INVALID_ARG, "unknown reduction op");
}

vc_status_t to_dt(vc_dtype_t d, DT* out) {
  switch (d) {
    case VC_FLOAT32: *out = DT::F32; return VC_SUCCESS;
    case VC_BFLOAT16: *out = DT::BF16; return VC_SUCCESS;
    case VC_INT32: *out = DT::I32; return VC_SUCCESS;
    case VC_FLOAT16: *out = DT::F16; return VC_SUCCESS;
  }
  return fail(VC_ERR_INVALID_ARG, "unknown dtype");
}

// Cost model of VC_ALGO_AUTO.
std::mutex g_cost_mu;
CostModel g_cost{CostPolicy::Hbm, 1.9e-6, 6.6e12};

CostModel default_cost(CostPolicy p) {
  return p == CostPolicy::Hbm ? CostModel{p, 1.9e-6, 6.6e12} : CostModel{p, 5e-6, 450e9};
}
CostModel current_cost() {
  std::lock_guard<std::mutex> lk(g_cost_mu);
  return g_cost;
}

// VC_ALGO_AUTO is returned as Algo::Fused with *is_auto set; the caller resolves it.
vc_status_t to_algo(vc_algo_t a, Algo* out, bool* is_auto = nullptr) {
  const int v = static_cast<int>(a);
  if (v == VC_ALGO_AUTO && is_auto) {
    *is_auto = true;
    *out = Algo::Fused;
    return VC_SUCCESS;
  }
  if (v < 0 || v > 12 || v == VC_ALGO_AUTO) return fail(VC_ERR_INVALID_ARG, "unknown algorithm");
  if (is_auto) *is_auto = false;
  *out = static_cast<Algo>(v);
  return VC_SUCCESS;
}

vc_status_t resolve_auto(PlanArgs* pa) {
  Algo chosen;
  std::string why;
  const PlanStatus ps = select_algo(*pa, current_cost(), &chosen, nullptr, &why);
  if (ps != PlanStatus::Ok) return plan_status(ps, why);
  pa->algo = chosen;
  return VC_SUCCESS;
}

// Plans are pure functions of the call's shape, so they are built once and
// kept (a bounded cache, cleared when full).
struct PlanKey {
  int coll, algo, nranks, dt, root, inplace, nchunks, op;
  int64_t count;
  int compact;
  bool operator==(const PlanKey& o) const {
    return coll == o.coll && algo == o.algo && nranks == o.nranks && dt == o.dt && root == o.root &&
           inplace == o.inplace && nchunks == o.nchunks && op == o.op && count == o.count && compact == o.compact;
  }
};
struct PlanKeyHash {
  size_t operator()(const PlanKey& k) const {
    uint64_t h = 1469598103934665603ull;
    for (int64_t v : {int64_t(k.coll), int64_t(k.algo), int64_t(k.nranks), int64_t(k.dt), int64_t(k.root),
                      int64_t(k.inplace), int64_t(k.nchunks), int64_t(k.op), k.count, int64_t(k.compact)})
      h = (h ^ static_cast<uint64_t>(v)) * 1099511628211ull;
    return static_cast<size_t>(h);
  }
};
std::mutex g_plan_mu;
std::unordered_map<PlanKey, std::shared_ptr<const Plan>, PlanKeyHash> g_plans;

PlanKey plan_key(const PlanArgs& pa) {
  return PlanKey{static_cast<int>(pa.coll), static_cast<int>(pa.algo), pa.nranks, static_cast<int>(pa.dt),
                 pa.root, pa.inplace ? 1 : 0, pa.nchunks, static_cast<int>(pa.op), pa.count,
                 pa.compact_partials ? 1 : 0};
}

// Orders each step for reuse of what the previous step wrote while it is
// still in L2.  A step walks its tiles in the direction opposite to the step
// before it (one flag per launch), and its operations are listed so that,
// walked that way, the one whose sources the previous step wrote last comes
// first: every step starts on the most recent lines.  Operations whose results
// the next step reads are marked keep and stored with the default L2 policy
// instead of streaming.  Only where a step writes at least the set minimum:
// below that everything stays in L2 anyway, and the reordered walks and plain
// stores measured 3-7% slower (ring, 8 ranks, 1-8 MiB per rank), while from
// 16 MiB per step on they win.  Operations of a step are independent, and
// neither their order, a tile's order nor a cache policy changes any
// element's association.
int64_t step_written_bytes(const Step& s) {
  int64_t b = 0;
  for (const Op& op : s.ops)
    for (const Operand& d : op.dst) b += op.n * op.nb * esize(d.dt);
  return b;
}
void order_for_reuse(Plan* plan) {
  for (Step& s : plan->steps)
    for (size_t i = 0; i < s.ops.size(); ++i) s.ops[i].built = static_cast<uint32_t>(i);
  const size_t min_bytes = g_reuse_min.load(std::memory_order_relaxed);
  if (min_bytes == SIZE_MAX) return;
  auto small = [&](const Step& s) { return static_cast<size_t>(step_written_bytes(s)) < min_bytes; };
  struct Span {
    Buf buf;
    int owner;
    int64_t lo, hi;
  };
  auto span = [](const Operand& o, const Op& op, int64_t stride) {
    const int64_t last = o.byte_off + (op.nb - 1) * stride;
    return Span{o.buf, o.buf == Buf::Scratch ? -1 : o.owner, std::min(o.byte_off, last),
                std::max(o.byte_off, last) + op.n * esize(o.dt)};
  };
  auto overlap = [](const Span& a, const Span& b) {
    return a.buf == b.buf && a.owner == b.owner && a.lo < b.hi && b.lo < a.hi;
  };
  for (size_t s = 0; s + 1 < plan->steps.size(); ++s) {
    if (small(plan->steps[s])) continue;
    std::vector<Span> reads;
    for (const Op& op : plan->steps[s + 1].ops)
      for (const Operand& src : op.src) reads.push_back(span(src, op, op.sstride));
    for (Op& op : plan->steps[s].ops)
      for (const Operand& d : op.dst) {
        const Span w = span(d, op, op.dstride);
        for (const Span& r : reads) op.keep = op.keep || overlap(r, w);
      }
  }
  for (size_t s = 1; s < plan->steps.size(); ++s) {
    const Step& prev = plan->steps[s - 1];
    if (small(prev)) continue;
    Step& cur = plan->steps[s];
    // when each of the previous step's operations ran: its place in the list,
    // counted from the end if that step walked backwards
    const int np = static_cast<int>(prev.ops.size());
    std::vector<std::pair<Span, int>> writes;
    for (int j = 0; j < np; ++j)
      for (const Operand& d : prev.ops[j].dst)
        writes.push_back({span(d, prev.ops[j], prev.ops[j].dstride), prev.reverse ? np - 1 - j : j});
    const size_t n = cur.ops.size();
    std::vector<int> when(n, -1);
    for (size_t i = 0; i < n; ++i)
      for (const Operand& src : cur.ops[i].src) {
        const Span sp = span(src, cur.ops[i], cur.ops[i].sstride);
        for (const auto& w : writes)
          if (overlap(w.first, sp)) when[i] = std::max(when[i], w.second);
      }
    std::vector<size_t> idx(n);
    for (size_t i = 0; i < n; ++i) idx[i] = i;
    std::stable_sort(idx.begin(), idx.end(), [&](size_t a, size_t b) { return when[a] > when[b]; });
    cur.reverse = !prev.reverse;
    if (cur.reverse) std::reverse(idx.begin(), idx.end());  // walked from the end of the list
    std::vector<Op> ops;
    ops.reserve(n);
    for (size_t i : idx) ops.push_back(cur.ops[i]);
    cur.ops = std::move(ops);
  }
}

// Steps that share a launch.  The stream order between launches is the step
// barrier, and a barrier is needed only where a step reads what an earlier
// one wrote or writes what an earlier one read or wrote.  A run of
// consecutive steps of one kernel mode in which no step does either with
// respect to the earlier steps of the run runs as one launch: its steps'
// operations in step order, so each block still takes the steps in order,
// without a barrier between them.  Every operation's operands and bytes are
// unchanged.  Such runs: Pairwise AllToAll's rounds (each reads only the send
// buffers and writes its own output blocks), the Ring AllToAll's local copy
// with its first round, the Mesh AllReduce's copies of the result to each
// rank, and binomial steps at rank counts that are not powers of 2, where a
// rank reached in one step forwards nothing in the next.
std::atomic<int> g_merge_steps{1};
void mark_independent_steps(Plan* plan) {
  plan->launch_end.clear();
  if (!g_merge_steps.load(std::memory_order_relaxed)) return;
  struct Span {
    Buf buf;
    int owner;
    int64_t lo, hi;
  };
  auto span = [](const Operand& o, const Op& op, int64_t stride) {
    const int64_t last = o.byte_off + (op.nb - 1) * stride;
    return Span{o.buf, o.buf == Buf::Scratch ? -1 : o.owner, std::min(o.byte_off, last),
                std::max(o.byte_off, last) + op.n * esize(o.dt)};
  };
  auto hit = [](const std::vector<Span>& a, const Span& b) {
    for (const Span& x : a)
      if (x.buf == b.buf && x.owner == b.owner && x.lo < b.hi && b.lo < x.hi) return true;
    return false;
  };
  const size_t n = plan->steps.size();
  std::vector<uint32_t> end(n, 0);
  bool any = false;
  for (size_t s = 0; s < n;) {
    std::vector<Span> reads, writes;
    auto add = [&](const Step& st) {
      for (const Op& op : st.ops) {
        for (const Operand& o : op.src) reads.push_back(span(o, op, op.sstride));
        for (const Operand& o : op.dst) writes.push_back(span(o, op, op.dstride));
      }
    };
    add(plan->steps[s]);
    size_t e = s + 1;
    for (; e < n; ++e) {
      const Step& st = plan->steps[e];
      if (st.mode != plan->steps[s].mode || st.red != plan->steps[s].red) break;
      bool dep = false;
      for (const Op& op : st.ops) {
        for (const Operand& o : op.src) dep = dep || hit(writes, span(o, op, op.sstride));
        for (const Operand& o : op.dst) {
          const Span w = span(o, op, op.dstride);
          dep = dep || hit(writes, w) || hit(reads, w);
        }
      }
      if (dep) break;
      add(st);
    }
    any = any || e > s + 1;
    for (size_t k = s; k < e; ++k) end[k] = static_cast<uint32_t>(e);
    s = e;
  }
  if (any) plan->launch_end = std::move(end);
}

PlanStatus cached_plan(const PlanArgs& pa, std::shared_ptr<const Plan>* out, std::string* why) {
  const PlanKey key = plan_key(pa);
  {
    std::lock_guard<std::mutex> lk(g_plan_mu);
    auto it = g_plans.find(key);
    if (it != g_plans.end()) {
      *out = it->second;
      return PlanStatus::Ok;
    }
  }
  auto plan = std::make_shared<Plan>();
  const PlanStatus ps = build_plan(pa, plan.get(), why);
  if (ps != PlanStatus::Ok) return ps;
  order_for_reuse(plan.get());
  mark_independent_steps(plan.get());
  std::lock_guard<std::mutex> lk(g_plan_mu);
  if (g_plans.size() >= 256) g_plans.clear();
  g_plans.emplace(key, plan);
  *out = plan;
  return PlanStatus::Ok;
}

// ---------------------------------------------------------------------------
// one-launch plans (host side)
// ---------------------------------------------------------------------------
std::mutex g_sl_mu;
size_t g_sl_limit = VC_SINGLE_LAUNCH_DEFAULT;
size_t g_slice_limit = VC_SLICE_LIMIT_DEFAULT;
constexpr int kPlanSmemMax = 96 << 10;            // description + bases in shared memory
constexpr size_t kPlanArenaChunk = 4u << 20;      // device memory for descriptions, per allocation
constexpr size_t kPlanArenaMax = 64u << 20;       // and in total, per device

size_t single_launch_limit() {
  std::lock_guard<std::mutex> lk(g_sl_mu);
  return g_sl_limit;
}
size_t slice_limit() {
  std::lock_guard<std::mutex> lk(g_sl_mu);
  return g_slice_limit;
}

struct DevPlan {
  bool eligible = false;
  const char* why = "";          // when not eligible
  const uint4* dptr = nullptr;   // description in device memory
  uint32_t words = 0;
  int rmode = dev::kCopy;        // kernel mode of the reduction steps
  RedOp red = RedOp::Sum;
  int64_t max_step_bytes = 0;
  int64_t bytes = 0;
  int nops = 0;
  bool sliced = false;           // every operation keeps element positions: the sliced form applies
  uint32_t nrefs = 0;
  uint32_t slice_words = 0;      // the description with the operations' element ranges
  int slice_es = 0;              // sliced form: bytes of the data type
  bool slice_host_ranges = false;  // the kernel takes the ranges the host lists (else derives them)
  int64_t slice_positions = 0;   // element positions the sliced plan covers
};
struct PlanStore {
  std::unordered_map<PlanKey, DevPlan, PlanKeyHash> plans;
  std::vector<void*> chunks;
  size_t chunk_used = kPlanArenaChunk;  // forces the first allocation
  size_t total = 0;
  cudaStream_t upload = nullptr;
  int cluster = 0;  // blocks per cluster (0: not yet chosen)
};
PlanStore g_store[64];

int kernel_mode(Mode m) {
  switch (m) {
    case Mode::Copy: return dev::kCopy;
    case Mode::F32: return dev::kF32;
    case Mode::I32: return dev::kI32;
    case Mode::BF16: return dev::kBF16;
    case Mode::F16: return dev::kF16;
  }
  return dev::kCopy;
}

using PlanKernel = void (*)(dev::PlanParams);
template <int RMODE>
PlanKernel plan_kernel_op(RedOp r) {
  switch (r) {
    case RedOp::Max: return dev::plan_kernel<RMODE, dev::kMax>;
    case RedOp::Min: return dev::plan_kernel<RMODE, dev::kMin>;
    default: return dev::plan_kernel<RMODE, dev::kSum>;
  }
}
PlanKernel plan_kernel_for(int rmode, RedOp r) {
  switch (rmode) {
    case dev::kF32: return plan_kernel_op<dev::kF32>(r);
    case dev::kI32: return plan_kernel_op<dev::kI32>(r);
    case dev::kBF16: return plan_kernel_op<dev::kBF16>(r);
    case dev::kF16: return plan_kernel_op<dev::kF16>(r);
    default: return dev::plan_kernel<dev::kCopy, dev::kSum>;
  }
}

// Blocks per cluster: 16 (non-portable size) where the device can place such
// a cluster with the largest description, else 8.
int plan_cluster(PlanStore& ps) {
  if (ps.cluster) return ps.cluster;
  PlanKernel k = dev::plan_kernel<dev::kF32, dev::kSum>;
  int best = 8;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kPlanSmemMax) == cudaSuccess &&
      cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(16);
    cfg.blockDim = dim3(dev::kPlanThreads);
    cfg.dynamicSmemBytes = kPlanSmemMax;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 16;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) == cudaSuccess && n >= 1) best = 16;
  }
  cudaGetLastError();
  ps.cluster = best;
  return best;
}

// Byte ranges of one buffer written so far (start -> end, disjoint).
struct Written {
  std::map<int64_t, int64_t> runs;
  void add(int64_t lo, int64_t hi) {
    auto it = runs.upper_bound(lo);
    if (it != runs.begin() && std::prev(it)->second >= lo) {
      --it;
      lo = it->first;
      hi = std::max(hi, it->second);
      it = runs.erase(it);
    }
    while (it != runs.end() && it->first <= hi) {
      hi = std::max(hi, it->second);
      it = runs.erase(it);
    }
    runs.emplace(lo, hi);
  }
  bool covers(int64_t lo, int64_t hi) const {
    auto it = runs.upper_bound(lo);
    return it != runs.begin() && std::prev(it)->second >= hi;
  }
};

// The sliced form (slice_kernel, slice16_kernel) applies to a plan whose
// every operation keeps element positions: operation element i is position
// pos0 + i, one run, a copy from one source.  Each operand holds the
// positions of its region of a buffer in order: position e at byte
// origin + e * size, where origin = offset - pos0 * size.  Regions of one
// buffer whose bytes overlap share one origin and size, so each byte any
// operation touches belongs to one position; with groups and origins on
// 16-byte boundaries (32 for the fp32 partial sums of 16-bit data, accessed
// 32 bytes at a time) a thread that owns a group of positions owns every byte
// of them.  Send and receive buffers hold the data type; scratch holds it too,
// or fp32 partial sums of 16-bit reductions.  Send buffers are only read, and
// every byte of a receive buffer or of scratch that a step reads was written
// by an earlier step -- by the thread that owns it, which therefore reads it
// through L1.  Positions stay below 2^29, so the kernels' 32-bit element
// offsets hold.  Where every region, scratch included, has origin 0 (the
// 4-byte AllReduce schedules, the Broadcasts), a 4-byte kernel derives each
// operation's range from its first operand's offset; otherwise it takes the
// ranges the host lists (a Reduce's first operand can be a partial sum in
// scratch, whose origin is its slot).
struct SliceShape {
  int es = 0;              // bytes of the data type
  bool absolute = true;    // every region has origin 0 (an operation's range follows from any operand)
  int64_t positions = 0;   // positions the plan covers
};
bool sliceable(const Plan& plan, int rmode, SliceShape* sh) {
  int es = 0;
  if (rmode == dev::kF32 || rmode == dev::kI32) es = 4;
  else if (rmode == dev::kBF16 || rmode == dev::kF16) es = 2;
  else if (rmode == dev::kCopy)  // copies only: the data type of any operand (a step may have none)
    for (const Step& st : plan.steps)
      if (!st.ops.empty()) {
        es = esize(st.ops[0].src[0].dt);
        break;
      }
  if (es != 2 && es != 4) return false;
  const int64_t gelems = 16 / es;
  struct Region {
    int64_t lo, hi, origin;
    int size;
  };
  std::map<std::pair<int, int>, std::vector<Region>> regions;  // (buffer kind, owner) -> regions
  auto key = [](const Operand& o) {
    return std::make_pair(static_cast<int>(o.buf), o.buf == Buf::Scratch ? 0 : o.owner);
  };
  bool absolute = true;
  int64_t positions = 0;
  for (const Step& st : plan.steps)
    for (const Op& op : st.ops) {
      if (op.pos0 < 0 || op.nb != 1 || op.pos0 % gelems != 0 || op.pos0 + op.n > (int64_t(1) << 29)) return false;
      if (st.mode == Mode::Copy && op.src.size() != 1) return false;
      positions = std::max(positions, op.pos0 + op.n);
      auto fits = [&](const Operand& o) {
        const int z = esize(o.dt);
        const bool partial = es == 2 && o.dt == DT::F32 && o.buf == Buf::Scratch && st.mode != Mode::Copy;
        if (z != es && !partial) return false;
        const int64_t origin = o.byte_off - op.pos0 * z;
        if (origin % (partial ? 32 : 16) != 0) return false;
        absolute = absolute && origin == 0;
        regions[key(o)].push_back({o.byte_off, o.byte_off + op.n * z, origin, z});
        return true;
      };
      for (const Operand& o : op.src)
        if (!fits(o)) return false;
      for (const Operand& o : op.dst)
        if (o.buf == Buf::Send || !fits(o)) return false;
    }
  // receive buffers and scratch: written before read, step by step
  std::map<std::pair<int, int>, Written> written;
  for (const Step& st : plan.steps) {
    for (const Op& op : st.ops)
      for (const Operand& o : op.src) {
        if (o.buf == Buf::Send) continue;
        const auto it = written.find(key(o));
        if (it == written.end() || !it->second.covers(o.byte_off, o.byte_off + op.n * esize(o.dt))) return false;
      }
    for (const Op& op : st.ops)
      for (const Operand& o : op.dst) written[key(o)].add(o.byte_off, o.byte_off + op.n * esize(o.dt));
  }
  for (auto& kv : regions) {
    std::vector<Region>& rs = kv.second;
    std::sort(rs.begin(), rs.end(), [](const Region& x, const Region& y) { return x.lo < y.lo; });
    int64_t reach = INT64_MIN, origin = 0;  // furthest byte of the regions so far, and their origin and size
    int size = 0;
    for (const Region& g : rs) {
      if (g.lo < reach && (g.origin != origin || g.size != size)) return false;
      if (g.lo >= reach) {
        origin = g.origin;
        size = g.size;
      }
      reach = std::max(reach, g.hi);
    }
  }
  sh->es = es;
  sh->absolute = absolute;
  sh->positions = positions;
  return true;
}

// Builds the description of `plan` for N ranks tiled for `workers` tile
// walkers (sub-blocks of the cluster), assuming every buffer base is 16-byte
// aligned (checked at each call).
void build_image(const Plan& plan, int N, int workers, std::vector<uint4>* img, DevPlan* dp) {
  dp->eligible = false;
  const size_t S = plan.steps.size();
  if (S < 2) { dp->why = "single step"; return; }
  bool have_red = false;
  size_t nops = 0, nrefs = 0;
  for (const Step& s : plan.steps) {
    nops += s.ops.size();
    for (const Op& op : s.ops) nrefs += op.src.size() + op.dst.size();
    if (s.mode == Mode::Copy) continue;
    if (have_red && (kernel_mode(s.mode) != dp->rmode || s.red != dp->red)) { dp->why = "mixed reductions"; return; }
    have_red = true;
    dp->rmode = kernel_mode(s.mode);
    dp->red = s.red;
  }
  if (nrefs > 0xFFFF) { dp->why = "too many operands"; return; }
  const size_t words = 1 + S + nops * (sizeof(dev::OpDesc) / 16) + nrefs;
  if (words * 16 + (2 * N + 1) * sizeof(void*) > static_cast<size_t>(kPlanSmemMax)) { dp->why = "too large"; return; }
  img->assign(words, make_uint4(0, 0, 0, 0));
  auto* hdr = reinterpret_cast<dev::PlanHeader*>(img->data());
  auto* steps = reinterpret_cast<dev::PlanStep*>(img->data() + 1);
  auto* ops = reinterpret_cast<dev::OpDesc*>(img->data() + 1 + S);
  auto* refs = reinterpret_cast<dev::OperandRef*>(ops + nops);
  hdr->nsteps = static_cast<uint32_t>(S);
  hdr->nops = static_cast<uint32_t>(nops);
  hdr->nrefs = static_cast<uint32_t>(nrefs);
  auto ref_of = [&](const Operand& o) {
    dev::OperandRef r{};
    r.base = o.buf == Buf::Send ? o.owner : o.buf == Buf::Recv ? N + o.owner : 2 * N;
    r.off = o.byte_off;
    return r;
  };
  size_t oi = 0, ri = 0;
  std::vector<const Op*> order;  // the operations as listed
  order.reserve(nops);
  for (size_t si = 0; si < S; ++si) {
    const Step& s = plan.steps[si];
    steps[si].op0 = static_cast<uint32_t>(oi);
    steps[si].nops = static_cast<uint32_t>(s.ops.size());
    steps[si].mode = static_cast<uint32_t>(s.mode == Mode::Copy ? dev::kCopy : dp->rmode);
    int64_t step_bytes = 0;
    // A step's operations are independent: they are listed here by their
    // first element position (else the byte offset of their first
    // destination), so that a sliced thread can stop looking once an
    // operation starts past its groups.
    std::vector<size_t> by_pos(s.ops.size());
    for (size_t k = 0; k < by_pos.size(); ++k) by_pos[k] = k;
    auto position = [&](const Op& op) {
      return op.pos0 >= 0 ? op.pos0 : op.dst.empty() ? 0 : op.dst[0].byte_off;
    };
    std::stable_sort(by_pos.begin(), by_pos.end(),
                     [&](size_t x, size_t y) { return position(s.ops[x]) < position(s.ops[y]); });
    for (size_t k : by_pos) {
      order.push_back(&s.ops[k]);
      const Op& op = s.ops[k];
      bool aligned = true;
      dev::OpDesc& d = ops[oi++];
      d.p0 = static_cast<uint16_t>(ri);
      for (const Operand& o : op.src) {
        refs[ri++] = ref_of(o);
        aligned &= (o.byte_off & 15) == 0;
        step_bytes += esize(o.dt) * op.n * op.nb;
      }
      for (const Operand& o : op.dst) {
        refs[ri++] = ref_of(o);
        aligned &= (o.byte_off & 15) == 0;
        step_bytes += esize(o.dt) * op.n * op.nb;
      }
      describe_op(d, op, s.mode, aligned);
    }
    const int64_t tiles = assign_tiles(ops + steps[si].op0, s.ops.size(), workers);
    if (tiles < 0) { dp->why = "too many tiles"; return; }
    steps[si].ntiles = static_cast<uint32_t>(tiles);
    dp->max_step_bytes = std::max(dp->max_step_bytes, step_bytes);
    dp->bytes += step_bytes;
  }
  dp->words = static_cast<uint32_t>(words);
  dp->nops = static_cast<int>(nops);
  dp->nrefs = static_cast<uint32_t>(nrefs);
  dp->eligible = true;
  SliceShape sh;
  dp->sliced = sliceable(plan, dp->rmode, &sh) &&
               dev::slice_smem_bytes(dp->words, 2 * N + 1, static_cast<uint32_t>(nops + 1), static_cast<uint32_t>(nrefs)) <=
                   static_cast<size_t>(kPlanSmemMax);
  dp->slice_es = sh.es;
  dp->slice_host_ranges = sh.es == 2 || !sh.absolute;
  dp->slice_positions = sh.positions;
  if (dp->sliced) {  // after the description: the operations' element ranges [e0, e1), in listed order
    dp->slice_words = dp->words + static_cast<uint32_t>((nops + 1) / 2);
    img->resize(dp->slice_words, make_uint4(0, 0, 0, 0));
    auto* rng = reinterpret_cast<int2*>(img->data() + dp->words);
    for (size_t k = 0; k < nops; ++k)
      rng[k] = make_int2(static_cast<int>(order[k]->pos0), static_cast<int>(order[k]->pos0 + order[k]->n));
  }
}

// The resident description of a plan shape, uploading it at the first call
// that may (not while `stream` is being captured).  nullptr: not available
// for this call.
const DevPlan* resident_plan(int dev, const PlanKey& key, const Plan& plan, int N, cudaStream_t stream) {
  std::lock_guard<std::mutex> lk(g_sl_mu);
  PlanStore& ps = g_store[dev];
  auto it = ps.plans.find(key);
  if (it != ps.plans.end()) return &it->second;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
    cudaGetLastError();
    return nullptr;
  }
  DevPlan dp;
  std::vector<uint4> img;
  build_image(plan, N, plan_cluster(ps) * dev::kPlanSubs, &img, &dp);
  if (dp.eligible) {
    const size_t bytes = (img.size() * 16 + 255) / 256 * 256;
    // another thread's capture in global mode must not see these calls
    cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
    cudaThreadExchangeStreamCaptureMode(&mode);
    cudaError_t e = cudaSuccess;
    if (ps.chunk_used + bytes > kPlanArenaChunk) {
      if (ps.total + kPlanArenaChunk > kPlanArenaMax) {
        e = cudaErrorMemoryAllocation;
      } else {
        void* chunk = nullptr;
        e = cudaMalloc(&chunk, kPlanArenaChunk);
        if (e == cudaSuccess) {
          ps.chunks.push_back(chunk);
          ps.total += kPlanArenaChunk;
          ps.chunk_used = 0;
        }
      }
    }
    if (e == cudaSuccess && !ps.upload) e = cudaStreamCreateWithFlags(&ps.upload, cudaStreamNonBlocking);
    char* dst = nullptr;
    if (e == cudaSuccess) {
      dst = static_cast<char*>(ps.chunks.back()) + ps.chunk_used;
      e = cudaMemcpyAsync(dst, img.data(), img.size() * 16, cudaMemcpyHostToDevice, ps.upload);
      if (e == cudaSuccess) e = cudaStreamSynchronize(ps.upload);
    }
    cudaThreadExchangeStreamCaptureMode(&mode);
    if (e == cudaSuccess) {
      ps.chunk_used += bytes;
      dp.dptr = reinterpret_cast<const uint4*>(dst);
    } else {
      cudaGetLastError();
      dp.eligible = false;
      dp.why = "no device memory for the description";
    }
  }
  return &ps.plans.emplace(key, dp).first->second;
}

using SliceKernel = void (*)(dev::PlanParams);
template <int RMODE, int U, int BT, bool HR>
SliceKernel slice_kernel_op(RedOp r) {
  switch (r) {
    case RedOp::Max: return dev::slice_kernel<RMODE, dev::kMax, U, BT, HR>;
    case RedOp::Min: return dev::slice_kernel<RMODE, dev::kMin, U, BT, HR>;
    default: return dev::slice_kernel<RMODE, dev::kSum, U, BT, HR>;
  }
}
template <bool F16, int U, int BT>
SliceKernel slice16_kernel_op(RedOp r) {
  switch (r) {
    case RedOp::Max: return dev::slice16_kernel<F16, dev::kMax, U, BT>;
    case RedOp::Min: return dev::slice16_kernel<F16, dev::kMin, U, BT>;
    default: return dev::slice16_kernel<F16, dev::kSum, U, BT>;
  }
}
// The kernel for a sliced plan: 16-bit data (reductions, or copies alone) the
// 16-bit kernel; 4-byte data the 4-byte one, taking the host's ranges where
// positions are not absolute.  Copy-only plans never combine, so any
// reduction variant serves.
template <int U, int BT>
SliceKernel slice_kernel_for(const DevPlan& dp) {
  if (dp.slice_es == 2) {
    if constexpr (U <= 4) return dp.rmode == dev::kF16 ? slice16_kernel_op<true, U, BT>(dp.red)
                                                      : slice16_kernel_op<false, U, BT>(dp.red);
    return nullptr;
  }
  if (dp.rmode == dev::kI32)
    return dp.slice_host_ranges ? slice_kernel_op<dev::kI32, U, BT, true>(dp.red)
                                : slice_kernel_op<dev::kI32, U, BT, false>(dp.red);
  return dp.slice_host_ranges ? slice_kernel_op<dev::kF32, U, BT, true>(dp.red)
                              : slice_kernel_op<dev::kF32, U, BT, false>(dp.red);
}
// The sliced form's launch shape, measured on 8 ranks (ring / DBT / RHD, 256 KiB
// to 8 MiB per rank): 256-thread blocks; one group a thread while that takes
// at most 256 blocks, else the fewest groups a thread (2, 4 or 8, whose loads
// of a step a thread issues together) that take at most two blocks per SM.
// One group a thread up to 256 blocks against up to 64: 512 KiB - 1 MiB per
// rank 0.3-1 us faster, fp32 and bf16.  (Before a grid let the next one in
// only after its wait, grids of more than 64 blocks of one group a thread
// measured up to twice as slow.)  512- or 1024-thread blocks were slower at
// small sizes.  16-bit plans stop at 4 groups a thread (8 elements each,
// fp32 sums: 128 registers for bf16, two blocks per SM, 144 for fp16; 8
// groups take 240).
constexpr int kSliceBlock = 256;
constexpr int kSliceSmallGrid = 256;

// A sliced plan (slice_kernel): one launch over the whole GPU, each thread
// carrying its 16-byte group of every buffer through every step.
vc_status_t launch_sliced(const DevPlan& dp, DeviceState* st, const dev::PlanParams& prm, cudaStream_t stream,
                          const LaunchCtx& tc) {
  const int64_t g = prm.groups, per_block = kSliceBlock;
  const int umax = dp.slice_es == 2 ? 4 : 8;
  int U = 1;
  if (g > int64_t(kSliceSmallGrid) * per_block) {
    U = 2;
    while (U < umax && g > int64_t(2) * st->nsm * per_block * U) U *= 2;
  }
  const SliceKernel kernel = U == 1 ? slice_kernel_for<1, kSliceBlock>(dp)
                           : U == 2 ? slice_kernel_for<2, kSliceBlock>(dp)
                           : U == 4 ? slice_kernel_for<4, kSliceBlock>(dp)
                                    : slice_kernel_for<8, kSliceBlock>(dp);
  if (!kernel) return fail(VC_ERR_UNSUPPORTED, "no sliced kernel for this launch shape");
  // (16-bit: the ranges within the description, up to 8 bytes more than the table)
  const size_t smem = dev::slice_smem_bytes(dp.words, prm.nbases, dp.nops + 1, dp.nrefs);
  int per_sm = 0;
  {
    static std::mutex mu;
    static std::map<std::tuple<const void*, size_t, DeviceState*>, int> occ;
    std::lock_guard<std::mutex> lk(mu);
    auto key = std::make_tuple(reinterpret_cast<const void*>(kernel), smem, st);
    auto it = occ.find(key);
    if (it == occ.end()) {
      cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPlanSmemMax);
      if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kSliceBlock, smem);
      if (e != cudaSuccess) return cuda_fail(e, "sliced plan occupancy");
      it = occ.emplace(key, std::max(1, per_sm)).first;
    }
    per_sm = it->second;
  }
  const int64_t slices = (prm.groups + int64_t(U) * kSliceBlock - 1) / (int64_t(U) * kSliceBlock);
  const unsigned grid = static_cast<unsigned>(std::max<int64_t>(1, std::min<int64_t>(slices, int64_t(st->nsm) * per_sm)));
  std::unique_lock<std::mutex> lk(g_trace_mu);
  const bool trace = trace_slot();
  if (!trace) lk.unlock();
  Pending pend{};
  if (trace) {
    cudaError_t e = take_event(&pend.start);
    if (e == cudaSuccess) e = take_event(&pend.stop);
    if (e == cudaSuccess) e = cudaEventRecord(pend.start, stream);
    if (e != cudaSuccess) return cuda_fail(e, "trace event");
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kSliceBlock);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, prm);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  if (trace) {
    e = cudaEventRecord(pend.stop, stream);
    if (e != cudaSuccess) return cuda_fail(e, "trace event");
    pend.rec.coll = tc.coll;
    pend.rec.algo = tc.algo;
    pend.rec.step = -1;
    pend.rec.kernel = dp.rmode | (static_cast<int>(dp.red) << 3) | 128 | 256;
    pend.rec.bytes = dp.bytes;
    pend.rec.nops = dp.nops;
    g_trace.push_back(pend);
  }
  return VC_SUCCESS;
}

// slice_groups > 0: run the plan in the sliced form over that many 16-byte
// groups per buffer; otherwise as one cluster with a barrier between steps.
vc_status_t launch_plan(const DevPlan& dp, int dev, int N, const std::vector<const void*>& sends,
                        const std::vector<void*>& recvs, char* scratch, cudaStream_t stream, const LaunchCtx& tc,
                        DeviceState* st = nullptr, int64_t slice_groups = 0) {
  dev::PlanParams prm{};
  prm.plan = dp.dptr;
  prm.words = dp.words;
  prm.nbases = static_cast<uint32_t>(2 * N + 1);
  prm.groups = slice_groups;
  if (slice_groups > 0 && dp.slice_host_ranges) prm.words = dp.slice_words;
  for (int r = 0; r < N; ++r) {
    prm.base[r] = sends[r];
    prm.base[N + r] = recvs[r];
  }
  prm.base[2 * N] = scratch;
  if (slice_groups > 0) return launch_sliced(dp, st, prm, stream, tc);
  const PlanKernel kernel = plan_kernel_for(dp.rmode, dp.red);
  int cluster;
  {
    std::lock_guard<std::mutex> lk(g_sl_mu);
    cluster = g_store[dev].cluster;
  }
  static std::mutex attr_mu;
  static std::map<std::pair<int, const void*>, bool> attr_done;
  {
    std::lock_guard<std::mutex> lk(attr_mu);
    auto key = std::make_pair(dev, reinterpret_cast<const void*>(kernel));
    if (!attr_done[key]) {
      cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPlanSmemMax);
      if (e == cudaSuccess && cluster > 8) e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
      attr_done[key] = true;
    }
  }
  std::unique_lock<std::mutex> lk(g_trace_mu);
  const bool trace = trace_slot();
  if (!trace) lk.unlock();
  Pending pend{};
  if (trace) {
    cudaError_t e = take_event(&pend.start);
    if (e == cudaSuccess) e = take_event(&pend.stop);
    if (e == cudaSuccess) e = cudaEventRecord(pend.start, stream);
    if (e != cudaSuccess) return cuda_fail(e, "trace event");
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster);
  cfg.blockDim = dim3(dev::kPlanThreads);
  cfg.dynamicSmemBytes = dp.words * 16 + prm.nbases * sizeof(void*);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, prm);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  if (trace) {
    e = cudaEventRecord(pend.stop, stream);
    if (e != cudaSuccess) return cuda_fail(e, "trace event");
    pend.rec.coll = tc.coll;
    pend.rec.algo = tc.algo;
    pend.rec.step = -1;
    pend.rec.kernel = dp.rmode | (static_cast<int>(dp.red) << 3) | 128;
    pend.rec.bytes = dp.bytes;
    pend.rec.nops = dp.nops;
    g_trace.push_back(pend);
  }
  return VC_SUCCESS;
}

std::mutex g_support_mu;
std::unordered_map<PlanKey, std::pair<PlanStatus, std::string>, PlanKeyHash> g_support;

PlanStatus supported(const PlanArgs& zero, std::string* why) {
  const PlanKey key = plan_key(zero);
  {
    std::lock_guard<std::mutex> lk(g_support_mu);
    auto it = g_support.find(key);
    if (it != g_support.end()) {
      *why = it->second.second;
      return it->second.first;
    }
  }
  Plan probe;
  const PlanStatus ps = build_plan(zero, &probe, why);
  std::lock_guard<std::mutex> lk(g_support_mu);
  if (g_support.size() >= 4096) g_support.clear();
  g_support.emplace(key, std::make_pair(ps, *why));
  return ps;
}

// Which one-launch forms a call may take, before its device description
// says whether the plan qualifies.  `aligned`: every buffer pointer and the
// scratch block 16-byte aligned; `scratch32`: the scratch block 32-byte
// aligned (16-bit sliced plans access their fp32 partials 32 bytes at a time).
struct FormGate {
  bool sliced = false;   // try the sliced form
  bool cluster = false;  // else try one cluster
  size_t cluster_limit = 0;
};
FormGate form_gate(const PlanArgs& pa, const Plan& plan, int64_t es, bool aligned, bool scratch32) {
  FormGate g;
  const int64_t N = pa.nranks, count = pa.count;
  if (!aligned || plan.steps.size() < 2) return g;
  // the sliced form's size per rank: AllReduce and Reduce the 4 bytes a
  // thread carries through the steps per element (fp32 / int32 data, or the
  // fp32 partial sums of 16-bit data), ReduceScatter its input likewise,
  // AllGather and Gather their output, Broadcast and Scatter their message.
  // Not for in-place calls of the other collectives, whose send and receive
  // buffers would hold positions at two places.
  int64_t slice_bytes = -1;
  switch (pa.coll) {
    case Coll::AllReduce:
    case Coll::Reduce: slice_bytes = count * 4; break;
    case Coll::ReduceScatter: slice_bytes = count * N * 4; break;
    case Coll::AllGather:
    case Coll::Gather:
    case Coll::Scatter: slice_bytes = count * N * es; break;
    case Coll::Broadcast: slice_bytes = count * es; break;
    default: break;
  }
  if (pa.inplace && pa.coll != Coll::AllReduce) slice_bytes = -1;
  const size_t slim = slice_limit();
  g.sliced = slim > 0 && slice_bytes >= 0 && (es == 4 || scratch32) && count < (int64_t(1) << 29) &&
             static_cast<uint64_t>(slice_bytes) <= std::min<uint64_t>(slim, INT64_MAX);
  // a plan whose steps all share one launch (step merging: Pairwise
  // AllToAll's rounds) runs that launch, not a cluster with a barrier per step
  // (8 ranks, 64 KiB per rank: 10.4 us as a cluster, 2-3 us as one launch).
  // AllToAll plans run per step: their steps are many small block copies, and
  // one launch a step measured faster than one cluster (8 ranks, 1-16 KiB per
  // rank: Bruck 7.3-7.5 against 10.1-10.6 us, Ring 12.0-12.3 against
  // 14.2-14.9).
  const bool one_launch = !plan.launch_end.empty() && plan.launch_end[0] == plan.steps.size();
  g.cluster_limit = single_launch_limit();
  g.cluster = !one_launch && pa.coll != Coll::AllToAll && g.cluster_limit > 0 &&
              plan_bytes(plan) / static_cast<int64_t>(plan.steps.size()) <=
                  static_cast<int64_t>(std::min<size_t>(g.cluster_limit, INT64_MAX));
  return g;
}

vc_status_t run(const Call& c) {
  const int N = c.nranks;
  if (N < 1 || N > VC_MAX_RANKS) return fail(VC_ERR_INVALID_ARG, "nranks must be in [1, 64]");
  const bool root_send = c.coll == Coll::Broadcast || c.coll == Coll::Scatter;  // one input: the root's
  const bool root_recv = c.coll == Coll::Gather || c.coll == Coll::Reduce;      // one output: the root's
  const bool rooted = root_send || root_recv;
  if (!root_recv && !c.recv) return fail(VC_ERR_INVALID_ARG, "null recv array");
  if (rooted && (c.root < 0 || c.root >= N)) return fail(VC_ERR_INVALID_ARG, "root outside [0, nranks)");
  if (!root_send && !c.send) return fail(VC_ERR_INVALID_ARG, "null send array");
  if (c.count < 0) return fail(VC_ERR_INVALID_ARG, "count too large");
  // algorithm / rank-count support is decided before looking at sizes
  PlanArgs pa{c.coll, c.algo, N, c.count, c.dt, c.root, false};
  pa.op = c.red;
  if (c.autoalgo) {
    const vc_status_t rs = resolve_auto(&pa);
    if (rs != VC_SUCCESS) return rs;
  }
  pa.nchunks = 1;
  if (pa.algo == Algo::PipeChain || pa.algo == Algo::PipeTree)
    pa.nchunks = c.nchunks > 0 ? c.nchunks : default_chunks(pa.algo, N, c.count, c.dt, current_cost());
  {
    // support of the algorithm for this collective and rank count, decided
    // on a zero-size plan (cached: it does not depend on the size)
    PlanArgs zero = pa;
    zero.count = 0;
    std::string why;
    const PlanStatus ps = supported(zero, &why);
    if (ps != PlanStatus::Ok) return plan_status(ps, why);
  }
  if (c.count == 0) return VC_SUCCESS;

  // element counts of each send / recv buffer
  const int64_t es = esize(c.dt);
  int64_t send_elems = c.count, recv_elems = c.count;
  if (c.coll == Coll::ReduceScatter || c.coll == Coll::Scatter) send_elems = c.count * N;
  if (c.coll == Coll::AllGather || c.coll == Coll::Gather) recv_elems = c.count * N;
  if (c.coll == Coll::AllToAll) send_elems = recv_elems = c.count * N;
  if (c.count > count_limit(N)) return fail(VC_ERR_INVALID_ARG, "count too large");
  const int64_t sbytes = send_elems * es, rbytes = recv_elems * es;

  std::vector<const void*> sends;
  if (root_send) {
    if (!c.send_root) return fail(VC_ERR_INVALID_ARG, "null root send buffer");
    sends.assign(N, nullptr);
    sends[c.root] = c.send_root;
  } else {
    for (int r = 0; r < N; ++r) {
      if (!c.send[r]) return fail(VC_ERR_INVALID_ARG, "null send buffer");
      sends.push_back(c.send[r]);
    }
  }
  std::vector<void*> recvs(N, nullptr);
  if (root_recv) {
    if (!c.recv_root) return fail(VC_ERR_INVALID_ARG, "null root recv buffer");
    recvs[c.root] = c.recv_root;
  } else {
    for (int r = 0; r < N; ++r) {
      if (!c.recv[r]) return fail(VC_ERR_INVALID_ARG, "null recv buffer");
      recvs[r] = c.recv[r];
    }
  }

  // outputs must not overlap each other or any input, except in place
  bool inplace = false;
  for (int i = 0; i < N; ++i) {
    if (!recvs[i]) continue;
    for (int j = i + 1; j < N; ++j)
      if (recvs[j] && overlap(recvs[i], rbytes, recvs[j], rbytes)) return fail(VC_ERR_INVALID_ARG, "receive buffers overlap");
    for (int q = 0; q < N; ++q) {
      if (!sends[q] || !overlap(recvs[i], rbytes, sends[q], sbytes)) continue;
      const bool same = sends[q] == recvs[i] && q == i && sbytes == rbytes;
      const bool allowed = same && (c.coll == Coll::AllReduce ||
                                    ((c.coll == Coll::Broadcast || c.coll == Coll::Reduce) && i == c.root));
      if (!allowed) return fail(VC_ERR_INVALID_ARG, "a receive buffer overlaps a send buffer");
      inplace = true;
    }
  }
  pa.inplace = c.coll == Coll::AllReduce ? (N == 1 && inplace) : inplace;

  std::shared_ptr<const Plan> plan_ptr;
  std::string why;
  const PlanStatus ps = cached_plan(pa, &plan_ptr, &why);
  if (ps != PlanStatus::Ok) return plan_status(ps, why);
  const Plan& plan = *plan_ptr;

  DeviceState* st = nullptr;
  int dev = 0;
  vc_status_t rc = device_state(&st, &dev);
  if (rc != VC_SUCCESS) return rc;

  char* scratch = nullptr;
  if (plan.scratch_bytes > 0) {
    cudaMemPool_t pool;
    rc = scratch_pool(st, dev, &pool);
    if (rc != VC_SUCCESS) return rc;
    cudaError_t e = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&scratch), plan.scratch_bytes, pool, c.stream);
    if (e == cudaErrorMemoryAllocation) {
      cudaGetLastError();
      return fail(VC_ERR_NOMEM, "scratch allocation of " + std::to_string(plan.scratch_bytes) + " bytes failed");
    }
    if (e != cudaSuccess) return cuda_fail(e, "cudaMallocFromPoolAsync");
  }
  const Bases b{sends.data(), recvs.data(), scratch};
  int launches = 0;
  LaunchCtx tc;
  tc.coll = static_cast<int>(c.coll);
  tc.algo = static_cast<int>(pa.algo);
  for (const Step& s : plan.steps) tc.pipeline &= s.mode != Mode::BF16 && s.mode != Mode::F16;
  // one launch for the whole plan when it is small enough and eligible: the
  // sliced form where every operation keeps element positions, else one
  // cluster with a barrier between steps
  const DevPlan* dp = nullptr;
  int64_t slice_groups = 0;
  bool aligned = (reinterpret_cast<uintptr_t>(scratch) & 15) == 0;
  for (int r = 0; r < N; ++r)
    aligned &= (!sends[r] || (reinterpret_cast<uintptr_t>(sends[r]) & 15) == 0) &&
               (!recvs[r] || (reinterpret_cast<uintptr_t>(recvs[r]) & 15) == 0);
  const FormGate gate = form_gate(pa, plan, es, aligned, (reinterpret_cast<uintptr_t>(scratch) & 31) == 0);
  if (gate.sliced) {
    dp = resident_plan(dev, plan_key(pa), plan, N, c.stream);
    if (dp && dp->eligible && dp->sliced) slice_groups = (dp->slice_positions * es + 15) / 16;
    else dp = nullptr;
  }
  if (!dp && gate.cluster) {
    dp = resident_plan(dev, plan_key(pa), plan, N, c.stream);
    if (dp && (!dp->eligible || static_cast<uint64_t>(dp->max_step_bytes) > gate.cluster_limit)) dp = nullptr;
  }
  if (dp) {
    tc.step = -1;
    rc = launch_plan(*dp, dev, N, sends, recvs, scratch, c.stream, tc, st, slice_groups);
    if (rc == VC_SUCCESS) launches = 1;
  } else {
    rc = for_each_launch_group(plan, [&](size_t si, const Step& s) {
      tc.step = static_cast<int>(si);
      return launch_step(st, s, b, c.stream, &launches, tc);
    });
  }
  if (scratch) {
    cudaError_t e = cudaFreeAsync(scratch, c.stream);
    if (e != cudaSuccess && rc == VC_SUCCESS) rc = cuda_fail(e, "cudaFreeAsync");
  }
  if (log_enabled()) {
    size_t ops = 0;
    for (const Step& s : plan.steps) ops += s.ops.size();
    std::fprintf(stderr, "[vc] %s algo=%s nranks=%d count=%lld dtype=%d root=%d steps=%zu ops=%zu launches=%d%s scratch=%lld\n",
                 coll_name(c.coll), algo_name(pa.algo), N, static_cast<long long>(c.count), static_cast<int>(c.dt),
                 c.root, plan.steps.size(), ops, launches, dp ? " (single launch)" : "",
                 static_cast<long long>(plan.scratch_bytes));
  }
  return rc;
}

template <class F>
vc_status_t entry(F&& f) {
  g_last_error.clear();
  try {
    return f();
  } catch (const std::bad_alloc&) {
    return fail(VC_ERR_NOMEM, "host allocation failed");
  } catch (...) {
    return fail(VC_ERR_INVALID_ARG, "internal error");
  }
}

}  // namespace
}  // namespace vc

using namespace vc;

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------
VC_EXPORT vc_status_t vc_allreduce(const void* const* send, void* const* recv, int nranks, size_t count,
                                   vc_dtype_t dtype, vc_op_t op, vc_algo_t algo, vc_stream_t stream) {
  return entry([&] {
    Call c;
    c.coll = Coll::AllReduce;
    vc_status_t rc = to_algo(algo, &c.algo, &c.autoalgo);
    if (rc == VC_SUCCESS) rc = to_dt(dtype, &c.dt);
    if (rc != VC_SUCCESS) return rc;
    rc = to_op(op, &c.red);
    if (rc != VC_SUCCESS) return rc;
    c.nranks = nranks;
    c.count = static_cast<int64_t>(count);
    c.send = send;
    c.recv = recv;
    c.stream = reinterpret_cast<cudaStream_t>(stream);
    return run(c);
  });
}

VC_EXPORT vc_status_t vc_reduce_scatter(const void* const* send, void* const* recv, int nranks, size_t recvcount,
                                        vc_dtype_t dtype, vc_op_t op, vc_algo_t algo, vc_stream_t stream) {
  return entry([&] {
    Call c;
    c.coll = Coll::ReduceScatter;
    vc_status_t rc = to_algo(algo, &c.algo, &c.autoalgo);
    if (rc == VC_SUCCESS) rc = to_dt(dtype, &c.dt);
    if (rc != VC_SUCCESS) return rc;
    rc = to_op(op, &c.red);
    if (rc != VC_SUCCESS) return rc;
    c.nranks = nranks;
    c.count = static_cast<int64_t>(recvcount);
    c.send = send;
    c.recv = recv;
    c.stream = reinterpret_cast<cudaStream_t>(stream);
    return run(c);
  });
}

VC_EXPORT vc_status_t vc_allgather(const void* const* send, void* const* recv, int nranks, size_t sendcount,
                                   vc_dtype_t dtype, vc_algo_t algo, vc_stream_t stream) {
  return entry([&] {
    Call c;
    c.coll = Coll::AllGather;
    vc_status_t rc = to_algo(algo, &c.algo, &c.autoalgo);
    if (rc == VC_SUCCESS) rc = to_dt(dtype, &c.dt);
    if (rc != VC_SUCCESS) return rc;
    c.nranks = nranks;
    c.count = static_cast<int64_t>(sendcount);
    c.send = send;
    c.recv = recv;
    c.stream = reinterpret_cast<cudaStream_t>(stream);
    return run(c);
  });
}

VC_EXPORT vc_status_t vc_broadcast(const void* send_root, void* const* recv, int nranks, size_t count,
                                   vc_dtype_t dtype, int root, vc_algo_t algo, vc_stream_t stream) {
  return entry([&] {
    Call c;
    c.coll = Coll::Broadcast;
    vc_status_t rc = to_algo(algo, &c.algo, &c.autoalgo);
    if (rc == VC_SUCCESS) rc = to_dt(dtype, &c.dt);
    if (rc != VC_SUCCESS) return rc;
    c.nranks = nranks;
    c.count = static_cast<int64_t>(count);
    c.root = root;
    c.send_root = send_root;
    c.recv = recv;
    c.stream = reinterpret_cast<cudaStream_t>(stream);
    return run(c);
  });
}

VC_EXPORT vc_status_t vc_scatter(const void* send_root, void* const* recv, int nranks, size_t recvcount,
                                 vc_dtype_t dtype, int root, vc_algo_t algo, vc_stream_t stream) {
  return entry([&] {
    Call c;
    c.coll = Coll::Scatter;
    vc_status_t rc = to_algo(algo, &c.algo, &c.autoalgo);
    if (rc == VC_SUCCESS) rc = to_dt(dtype, &c.dt);
    if (rc != VC_SUCCESS) return rc;
    c.nranks = nranks;
    c.count = static_cast<int64_t>(recvcount);
    c.root = root;
    c.send_root = send_root;
    c.recv = recv;
    c.stream = reinterpret_cast<cudaStream_t>(stream);
    return run(c);
  });
}

VC_EXPORT vc_status_t vc_alltoall(const void* const* send, void* const* recv, int nranks, size_t blockcount,
                                  vc_dtype_t dtype, vc_algo_t algo, vc_stream_t stream) {
  return entry([&] {
    Call c;
    c.coll = Coll::AllToAll;
    vc_status_t rc = to_algo(algo, &c.algo, &c.autoalgo);
    if (rc == VC_SUCCESS) rc = to_dt(dtype, &c.dt);
    if (rc != VC_SUCCESS) return rc;
    c.nranks = nranks;
    c.count = static_cast<int64_t>(blockcount);
    c.send = send;
    c.recv = recv;
    c.stream = reinterpret_cast<cudaStream_t>(stream);
    return run(c);
  });
}

VC_EXPORT vc_status_t vc_broadcast_pipelined(const void* send_root, void* const* recv, int nranks, size_t count,
                                             vc_dtype_t dtype, int root, vc_algo_t algo, int nchunks,
                                             vc_stream_t stream) {
  return entry([&] {
    Call c;
    c.coll = Coll::Broadcast;
    vc_status_t rc = to_algo(algo, &c.algo, &c.autoalgo);
    if (rc == VC_SUCCESS) rc = to_dt(dtype, &c.dt);
    if (rc != VC_SUCCESS) return rc;
    if (nchunks < 0 || nchunks > 1024) return fail(VC_ERR_INVALID_ARG, "nchunks must be in [0, 1024]");
    c.nranks = nranks;
    c.count = static_cast<int64_t>(count);
    c.root = root;
    c.send_root = send_root;
    c.recv = recv;
    c.nchunks = nchunks;
    c.stream = reinterpret_cast<cudaStream_t>(stream);
    return run(c);
  });
}

VC_EXPORT vc_status_t vc_gather(const void* const* send, void* recv_root, int nranks, size_t sendcount,
                                vc_dtype_t dtype, int root, vc_algo_t algo, vc_stream_t stream) {
  return entry([&] {
    Call c;
    c.coll = Coll::Gather;
    vc_status_t rc = to_algo(algo, &c.algo, &c.autoalgo);
    if (rc == VC_SUCCESS) rc = to_dt(dtype, &c.dt);
    if (rc != VC_SUCCESS) return rc;
    c.nranks = nranks;
    c.count = static_cast<int64_t>(sendcount);
    c.root = root;
    c.send = send;
    c.recv_root = recv_root;
    c.stream = reinterpret_cast<cudaStream_t>(stream);
    return run(c);
  });
}

VC_EXPORT vc_status_t vc_reduce(const void* const* send, void* recv_root, int nranks, size_t count,
                                vc_dtype_t dtype, vc_op_t op, int root, vc_algo_t algo, vc_stream_t stream) {
  return entry([&] {
    Call c;
    c.coll = Coll::Reduce;
    vc_status_t rc = to_algo(algo, &c.algo, &c.autoalgo);
    if (rc == VC_SUCCESS) rc = to_dt(dtype, &c.dt);
    if (rc != VC_SUCCESS) return rc;
    rc = to_op(op, &c.red);
    if (rc != VC_SUCCESS) return rc;
    c.nranks = nranks;
    c.count = static_cast<int64_t>(count);
    c.root = root;
    c.send = send;
    c.recv_root = recv_root;
    c.stream = reinterpret_cast<cudaStream_t>(stream);
    return run(c);
  });
}

VC_EXPORT const char* vc_status_string(vc_status_t s) {
  switch (s) {
    case VC_SUCCESS: return "VC_SUCCESS";
    case VC_ERR_INVALID_ARG: return "VC_ERR_INVALID_ARG";
    case VC_ERR_UNSUPPORTED: return "VC_ERR_UNSUPPORTED";
    case VC_ERR_CUDA: return "VC_ERR_CUDA";
    case VC_ERR_NOMEM: return "VC_ERR_NOMEM";
    case VC_ERR_TIMEOUT: return "VC_ERR_TIMEOUT";
  }
  return "VC_ERR_UNKNOWN";
}

VC_EXPORT const char* vc_last_error(void) { return g_last_error.c_str(); }

VC_EXPORT vc_status_t vc_set_cost_model(vc_cost_policy_t policy, double alpha_s, double beta_bytes_per_s) {
  return entry([&]() -> vc_status_t {
    if (policy != VC_COST_HBM && policy != VC_COST_LINK) return fail(VC_ERR_INVALID_ARG, "unknown cost policy");
    if (!std::isfinite(alpha_s) || !std::isfinite(beta_bytes_per_s))
      return fail(VC_ERR_INVALID_ARG, "alpha and beta must be finite");
    CostModel m = default_cost(static_cast<CostPolicy>(static_cast<int>(policy)));
    if (alpha_s > 0) m.alpha = alpha_s;
    if (beta_bytes_per_s > 0) m.beta = beta_bytes_per_s;
    std::lock_guard<std::mutex> lk(g_cost_mu);
    g_cost = m;
    return VC_SUCCESS;
  });
}

VC_EXPORT vc_status_t vc_get_cost_model(vc_cost_policy_t* policy, double* alpha_s, double* beta_bytes_per_s) {
  return entry([&]() -> vc_status_t {
    const CostModel m = current_cost();
    if (policy) *policy = static_cast<vc_cost_policy_t>(static_cast<int>(m.policy));
    if (alpha_s) *alpha_s = m.alpha;
    if (beta_bytes_per_s) *beta_bytes_per_s = m.beta;
    return VC_SUCCESS;
  });
}

VC_EXPORT vc_status_t vc_select_algo(vc_coll_t coll, int nranks, size_t count, vc_dtype_t dtype, int root,
                                     vc_algo_t* algo, double* predicted_s) {
  return entry([&]() -> vc_status_t {
    if (static_cast<int>(coll) < 0 || static_cast<int>(coll) > 7) return fail(VC_ERR_INVALID_ARG, "unknown collective");
    if (!algo) return fail(VC_ERR_INVALID_ARG, "null algo");
    PlanArgs pa;
    pa.coll = static_cast<Coll>(static_cast<int>(coll));
    vc_status_t rc = to_dt(dtype, &pa.dt);
    if (rc != VC_SUCCESS) return rc;
    pa.nranks = nranks;
    pa.count = static_cast<int64_t>(count);
    pa.root = root;
    Algo chosen;
    std::string why;
    const PlanStatus ps = select_algo(pa, current_cost(), &chosen, predicted_s, &why);
    if (ps != PlanStatus::Ok) return plan_status(ps, why);
    *algo = static_cast<vc_algo_t>(static_cast<int>(chosen));
    return VC_SUCCESS;
  });
}

VC_EXPORT double vc_busbw_factor(vc_coll_t coll, int nranks) {
  if (nranks < 1) return 0.0;
  const double N = nranks;
  switch (coll) {
    case VC_COLL_ALLREDUCE: return 2.0 * (N - 1) / N;
    case VC_COLL_REDUCE_SCATTER:
    case VC_COLL_ALLGATHER:
    case VC_COLL_ALLTOALL:
    case VC_COLL_SCATTER:
    case VC_COLL_GATHER: return (N - 1) / N;
    case VC_COLL_BROADCAST:
    case VC_COLL_REDUCE: return 1.0;
  }
  return 0.0;
}

// The plan of a host-only description call (vc_plan_describe, vc_plan_exec_order).
vc_status_t describe_plan(vc_coll_t coll, vc_algo_t algo, int nranks, size_t count, vc_dtype_t dtype, vc_op_t op,
                          int root, int inplace, int nchunks, Plan* plan, PlanArgs* args = nullptr) {
  if (static_cast<int>(coll) < 0 || static_cast<int>(coll) > 7) return fail(VC_ERR_INVALID_ARG, "unknown collective");
  PlanArgs pa;
  pa.coll = static_cast<Coll>(static_cast<int>(coll));
  bool is_auto = false;
  vc_status_t rc = to_algo(algo, &pa.algo, &is_auto);
  if (rc == VC_SUCCESS) rc = to_dt(dtype, &pa.dt);
  if (rc == VC_SUCCESS) rc = to_op(op, &pa.op);
  if (rc != VC_SUCCESS) return rc;
  pa.nranks = nranks;
  pa.count = static_cast<int64_t>(count);
  pa.root = root;
  pa.inplace = inplace != 0;
  // as the calls allow it: AllReduce, and a Broadcast or Reduce at its root
  if (pa.inplace && pa.coll != Coll::AllReduce && pa.coll != Coll::Broadcast && pa.coll != Coll::Reduce)
    return fail(VC_ERR_INVALID_ARG, "in place only for AllReduce, Broadcast and Reduce");
  if (is_auto) {
    rc = resolve_auto(&pa);
    if (rc != VC_SUCCESS) return rc;
  }
  if (pa.algo == Algo::PipeChain || pa.algo == Algo::PipeTree) {
    // as vc_broadcast_pipelined takes it
    if (nchunks < 0 || nchunks > 1024) return fail(VC_ERR_INVALID_ARG, "nchunks must be in [0, 1024]");
    pa.nchunks = nchunks > 0 ? nchunks : default_chunks(pa.algo, nranks, pa.count, pa.dt, current_cost());
  }
  std::string why;
  const PlanStatus ps = build_plan(pa, plan, &why);
  if (ps != PlanStatus::Ok) return plan_status(ps, why);
  if (args) *args = pa;
  return VC_SUCCESS;
}

VC_EXPORT vc_status_t vc_plan_describe(vc_coll_t coll, vc_algo_t algo, int nranks, size_t count,
                                       vc_dtype_t dtype, vc_op_t op, int root, int inplace, int nchunks,
                                       vc_plan_entry_t* entries,
                                       size_t capacity, size_t* n_entries, size_t* scratch_bytes, int* n_steps) {
  return entry([&]() -> vc_status_t {
    Plan plan;
    const vc_status_t rc = describe_plan(coll, algo, nranks, count, dtype, op, root, inplace, nchunks, &plan);
    if (rc != VC_SUCCESS) return rc;
    size_t need = 0;
    for (const Step& s : plan.steps)
      for (const Op& op : s.ops) need += op.src.size() + op.dst.size();
    if (n_entries) *n_entries = need;
    if (scratch_bytes) *scratch_bytes = static_cast<size_t>(plan.scratch_bytes);
    if (n_steps) *n_steps = static_cast<int>(plan.steps.size());
    if (!entries) return capacity == 0 ? VC_SUCCESS : fail(VC_ERR_INVALID_ARG, "null entries");
    if (capacity < need) return fail(VC_ERR_INVALID_ARG, "capacity too small");
    size_t k = 0;
    for (size_t si = 0; si < plan.steps.size(); ++si) {
      const Step& s = plan.steps[si];
      for (size_t oi = 0; oi < s.ops.size(); ++oi) {
        const Op& op = s.ops[oi];
        for (int role = 0; role < 2; ++role) {
          const auto& list = role == 0 ? op.src : op.dst;
          for (size_t pos = 0; pos < list.size(); ++pos) {
            vc_plan_entry_t& e = entries[k++];
            e.step = static_cast<int32_t>(si);
            e.op = static_cast<int32_t>(oi);
            e.role = role;
            e.pos = static_cast<int32_t>(pos);
            e.buf = static_cast<int32_t>(list[pos].buf);
            e.owner = list[pos].owner;
            e.dtype = static_cast<int32_t>(list[pos].dt);
            e.reduce = s.mode == Mode::Copy ? 0 : 1 + static_cast<int32_t>(s.red);
            e.byte_off = list[pos].byte_off;
            e.n = op.n;
            e.nb = op.nb;
            e.stride_bytes = role == 0 ? op.sstride : op.dstride;
            e.elem0 = op.pos0;
          }
        }
      }
    }
    return VC_SUCCESS;
  });
}

VC_EXPORT vc_status_t vc_plan_exec_order(vc_coll_t coll, vc_algo_t algo, int nranks, size_t count, vc_dtype_t dtype,
                                         vc_op_t op, int root, int inplace, int nchunks, uint32_t* order,
                                         uint8_t* keep, size_t op_capacity, uint8_t* reverse, size_t step_capacity,
                                         size_t* n_ops, int* n_steps) {
  return entry([&]() -> vc_status_t {
    Plan plan;
    const vc_status_t rc = describe_plan(coll, algo, nranks, count, dtype, op, root, inplace, nchunks, &plan);
    if (rc != VC_SUCCESS) return rc;
    order_for_reuse(&plan);
    size_t nops = 0;
    for (const Step& s : plan.steps) nops += s.ops.size();
    if (n_ops) *n_ops = nops;
    if (n_steps) *n_steps = static_cast<int>(plan.steps.size());
    if (!order && !keep && !reverse && op_capacity == 0 && step_capacity == 0) return VC_SUCCESS;
    if (!order || !keep || !reverse) return fail(VC_ERR_INVALID_ARG, "null output array");
    if (op_capacity < nops || step_capacity < plan.steps.size()) return fail(VC_ERR_INVALID_ARG, "capacity too small");
    size_t k = 0;
    for (size_t si = 0; si < plan.steps.size(); ++si) {
      reverse[si] = plan.steps[si].reverse ? 1 : 0;
      for (const Op& o : plan.steps[si].ops) {
        order[k] = o.built;
        keep[k] = o.keep ? 1 : 0;
        ++k;
      }
    }
    return VC_SUCCESS;
  });
}

VC_EXPORT vc_status_t vc_plan_form(vc_coll_t coll, vc_algo_t algo, int nranks, size_t count, vc_dtype_t dtype,
                                   vc_op_t op, int root, int inplace, int nchunks, int* form, int* launches,
                                   int* host_ranges) {
  return entry([&]() -> vc_status_t {
    if (!form || !launches || !host_ranges) return fail(VC_ERR_INVALID_ARG, "null output");
    if (nranks < 1 || nranks > VC_MAX_RANKS) return fail(VC_ERR_INVALID_ARG, "nranks must be in [1, 64]");
    Plan plan;
    PlanArgs pa;
    const vc_status_t rc = describe_plan(coll, algo, nranks, count, dtype, op, root, inplace, nchunks, &plan, &pa);
    if (rc != VC_SUCCESS) return rc;
    // as a call builds it (cached_plan), and an AllReduce in place as a call runs it
    order_for_reuse(&plan);
    mark_independent_steps(&plan);
    if (pa.coll == Coll::AllReduce) pa.inplace = nranks == 1 && pa.inplace;
    const FormGate gate = form_gate(pa, plan, esize(pa.dt), true, true);
    DevPlan dp;
    std::vector<uint4> img;
    if (gate.sliced || gate.cluster) build_image(plan, nranks, 16 * dev::kPlanSubs, &img, &dp);
    *host_ranges = 0;
    if (gate.sliced && dp.eligible && dp.sliced) {
      *form = VC_FORM_SLICED;
      *launches = 1;
      *host_ranges = dp.slice_host_ranges ? 1 : 0;
    } else if (gate.cluster && dp.eligible && static_cast<uint64_t>(dp.max_step_bytes) <= gate.cluster_limit) {
      *form = VC_FORM_CLUSTER;
      *launches = 1;
    } else {  // as run() launches it: empty steps launch nothing, large ones split
      *form = VC_FORM_STEPS;
      int n = 0;
      const vc_status_t rs = for_each_launch_group(plan, [&](size_t, const Step& s) -> vc_status_t {
        for (size_t i = 0; i < s.ops.size(); ++n) {
          bool large = false;
          const size_t j = launch_span(s, i, &large);
          if (j == i) return fail(VC_ERR_INVALID_ARG, "operation has too many operands");
          i = j;
        }
        return VC_SUCCESS;
      });
      if (rs != VC_SUCCESS) return rs;
      *launches = n;
    }
    return VC_SUCCESS;
  });
}

VC_EXPORT vc_status_t vc_trace_enable(int on) {
  return entry([&]() -> vc_status_t {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    for (Pending& p : g_trace) {
      g_event_pool.push_back(p.start);
      g_event_pool.push_back(p.stop);
    }
    g_trace.clear();
    g_trace_dropped = 0;
    g_trace_on = on != 0;
    return VC_SUCCESS;
  });
}

VC_EXPORT vc_status_t vc_trace_read(vc_trace_record_t* records, size_t capacity, size_t* n_records) {
  return entry([&]() -> vc_status_t {
    std::lock_guard<std::mutex> lk(g_trace_mu);
    size_t n = 0;
    vc_status_t rc = VC_SUCCESS;
    for (Pending& p : g_trace) {
      if (records && n < capacity && rc == VC_SUCCESS) {
        cudaError_t e = cudaEventSynchronize(p.stop);
        float ms = 0.f;
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, p.start, p.stop);
        if (e != cudaSuccess) {
          rc = cuda_fail(e, "trace event");
        } else {
          records[n] = p.rec;
          records[n].ms = ms;
          ++n;
        }
      }
      g_event_pool.push_back(p.start);
      g_event_pool.push_back(p.stop);
    }
    g_trace.clear();
    if (n_records) *n_records = n;
    return rc;
  });
}

// ---------------------------------------------------------------------------
// Ring ReduceScatter without device allocation
// ---------------------------------------------------------------------------
// For callers that cannot allocate device memory during the call (see vc.h).
// The partial sums use this fixed array instead of the library's pool.  Host
// code may not use the array's name as a device address: it is looked up once
// per device with cudaGetSymbolAddress while that device is current.
static __device__ __align__(256) unsigned char g_noalloc_scratch[VC_NOALLOC_SCRATCH_BYTES];

namespace vc {
namespace {
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {};

vc_status_t noalloc_scratch(int dev, char** out) {
  if (dev < 0 || dev >= static_cast<int>(sizeof(g_noalloc_ptr) / sizeof(g_noalloc_ptr[0])))
    return fail(VC_ERR_CUDA, "device index out of range for the fixed scratch table");
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress");
    g_noalloc_ptr[dev] = p;
  }
  *out = static_cast<char*>(g_noalloc_ptr[dev]);
  return VC_SUCCESS;
}

vc_status_t run_reduce_scatter_noalloc(const void* const* send, void* const* recv, int N, int64_t rc, DT dt,
                                       cudaStream_t stream) {
  if (N < 1 || N > VC_MAX_RANKS) return fail(VC_ERR_INVALID_ARG, "nranks must be in [1, 64]");
  if (!send || !recv) return fail(VC_ERR_INVALID_ARG, "null send or recv array");
  if (rc < 0) return fail(VC_ERR_INVALID_ARG, "count too large");
  if (rc == 0) return VC_SUCCESS;
  if (rc > (INT64_MAX / 8) / N) return fail(VC_ERR_INVALID_ARG, "count too large");
  const int64_t es = esize(dt);
  const int64_t sbytes = rc * N * es, rbytes = rc * es;
  for (int r = 0; r < N; ++r)
    if (!send[r] || !recv[r]) return fail(VC_ERR_INVALID_ARG, "null send or recv buffer");
  for (int i = 0; i < N; ++i) {
    for (int j = i + 1; j < N; ++j)
      if (overlap(recv[i], rbytes, recv[j], rbytes)) return fail(VC_ERR_INVALID_ARG, "receive buffers overlap");
    for (int q = 0; q < N; ++q)
      if (overlap(recv[i], rbytes, send[q], sbytes))
        return fail(VC_ERR_INVALID_ARG, "a receive buffer overlaps a send buffer");
  }
  // the allocating call's steps, operations and execution order, with the
  // partial sums in two block slots per rank (the allocating call keeps one
  // slot per block while they take at most 16 MiB per rank)
  PlanArgs pa{Coll::ReduceScatter, Algo::Ring, N, rc, dt, 0, false};
  pa.compact_partials = true;
  std::shared_ptr<const Plan> plan_ptr;
  std::string why;
  const PlanStatus ps = cached_plan(pa, &plan_ptr, &why);
  if (ps != PlanStatus::Ok) return plan_status(ps, why);
  const Plan& plan = *plan_ptr;
  if (plan.scratch_bytes > static_cast<int64_t>(VC_NOALLOC_SCRATCH_BYTES))
    return fail(VC_ERR_INVALID_ARG, "vc_reduce_scatter_noalloc needs " + std::to_string(plan.scratch_bytes) +
                                        " bytes of scratch; the fixed array holds " +
                                        std::to_string(VC_NOALLOC_SCRATCH_BYTES) +
                                        " (nranks * roundup(2 * recvcount * 4, 256) must not exceed it)");
  DeviceState* st = nullptr;
  int dev = 0;
  vc_status_t rc_ = device_state(&st, &dev);
  if (rc_ != VC_SUCCESS) return rc_;
  char* scratch = nullptr;
  rc_ = noalloc_scratch(dev, &scratch);
  if (rc_ != VC_SUCCESS) return rc_;
  const Bases b{send, recv, scratch};
  int launches = 0;
  LaunchCtx tc;
  tc.coll = static_cast<int>(Coll::ReduceScatter);
  tc.algo = static_cast<int>(Algo::Ring);
  for (const Step& s : plan.steps) tc.pipeline &= s.mode != Mode::BF16 && s.mode != Mode::F16;
  for (size_t si = 0; si < plan.steps.size(); ++si) {
    tc.step = static_cast<int>(si);
    rc_ = launch_step(st, plan.steps[si], b, stream, &launches, tc);
    if (rc_ != VC_SUCCESS) return rc_;
  }
  return VC_SUCCESS;
}
}  // namespace
}  // namespace vc

VC_EXPORT vc_status_t vc_reduce_scatter_noalloc(const void* const* send, void* const* recv, int nranks,
                                                size_t recvcount, vc_dtype_t dtype, vc_op_t op,
                                                vc_stream_t stream) {
  return entry([&]() -> vc_status_t {
    DT dt;
    vc_status_t rc = to_dt(dtype, &dt);
    if (rc != VC_SUCCESS) return rc;
    if (op != VC_SUM) return fail(op == VC_MAX || op == VC_MIN ? VC_ERR_UNSUPPORTED : VC_ERR_INVALID_ARG, "only VC_SUM is implemented");
    return run_reduce_scatter_noalloc(send, recv, nranks, static_cast<int64_t>(recvcount), dt,
                                      reinterpret_cast<cudaStream_t>(stream));
  });
}

VC_EXPORT vc_status_t vc_device_errors(vc_stream_t stream, uint32_t* flags) {
  return entry([&]() -> vc_status_t {
    if (!flags) return fail(VC_ERR_INVALID_ARG, "null output pointer");
    *flags = 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint32_t zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(flags, dev::g_device_error, sizeof(uint32_t), 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemcpyToSymbolAsync(dev::g_device_error, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
    return VC_SUCCESS;
  });
}

VC_EXPORT vc_status_t vc_copy_selftest(vc_stream_t stream, uint32_t* flags) {
  return entry([&]() -> vc_status_t {
    if (!flags) return fail(VC_ERR_INVALID_ARG, "null output pointer");
    DeviceState* st = nullptr;
    int dev = 0;
    vc_status_t rc = device_state(&st, &dev);
    if (rc != VC_SUCCESS) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // one copy of 64 KB (two 32 KB tiles) from a zeroed buffer to another
    char* mem = nullptr;
    cudaError_t e = cudaMalloc(&mem, 2 << 16);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc");
    Step step;
    step.mode = Mode::Copy;
    Op op;
    op.src.push_back(Operand{Buf::Send, 0, 0, DT::I32});
    op.dst.push_back(Operand{Buf::Recv, 0, 0, DT::I32});
    op.n = (1 << 16) / 4;
    step.ops.push_back(op);
    const void* send[1] = {mem};
    void* recv[1] = {mem + (1 << 16)};
    const Bases b{send, recv, nullptr};
    static thread_local dev::SmallParams p;
    int64_t tiles = 0;
    fill_params(p, step, 0, 1, b, 1, &tiles, dev::kCopyTileBytes / (dev::kThreads * 16));
    auto kernel = dev::tma_copy_kernel<dev::SmallParams, true>;
    const size_t smem = dev::kCopyStages * dev::kCopyTileBytes + dev::kCopyStages * sizeof(uint64_t);
    const uint32_t zero = 0;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e == cudaSuccess) e = cudaMemsetAsync(mem, 0, 2 << 16, s);
    if (e == cudaSuccess)
      e = cudaMemcpyToSymbolAsync(dev::g_device_error, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(1);
      cfg.blockDim = dim3(dev::kCopyThreads);
      cfg.dynamicSmemBytes = smem;
      cfg.stream = s;
      e = cudaLaunchKernelEx(&cfg, kernel, p);
    }
    if (e == cudaSuccess)
      e = cudaMemcpyFromSymbolAsync(flags, dev::g_device_error, sizeof(uint32_t), 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
      e = cudaMemcpyToSymbolAsync(dev::g_device_error, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    cudaFree(mem);
    if (e != cudaSuccess) return cuda_fail(e, "copy self-test");
    return VC_SUCCESS;
  });
}

VC_EXPORT vc_status_t vc_set_single_launch(size_t max_step_bytes) {
  std::lock_guard<std::mutex> lk(g_sl_mu);
  g_sl_limit = max_step_bytes;
  return VC_SUCCESS;
}

VC_EXPORT vc_status_t vc_get_single_launch(size_t* max_step_bytes) {
  if (!max_step_bytes) return fail(VC_ERR_INVALID_ARG, "null output pointer");
  std::lock_guard<std::mutex> lk(g_sl_mu);
  *max_step_bytes = g_sl_limit;
  return VC_SUCCESS;
}

VC_EXPORT vc_status_t vc_set_merge_steps(int on) {
  g_merge_steps.store(on ? 1 : 0, std::memory_order_relaxed);
  std::lock_guard<std::mutex> lk(g_plan_mu);  // cached plans carry the grouping they were built with
  g_plans.clear();
  return VC_SUCCESS;
}

VC_EXPORT vc_status_t vc_get_merge_steps(int* on) {
  if (!on) return fail(VC_ERR_INVALID_ARG, "null output pointer");
  *on = g_merge_steps.load(std::memory_order_relaxed);
  return VC_SUCCESS;
}

VC_EXPORT vc_status_t vc_set_slice_limit(size_t max_bytes_per_rank) {
  std::lock_guard<std::mutex> lk(g_sl_mu);
  g_slice_limit = max_bytes_per_rank;
  return VC_SUCCESS;
}

VC_EXPORT vc_status_t vc_get_slice_limit(size_t* max_bytes_per_rank) {
  if (!max_bytes_per_rank) return fail(VC_ERR_INVALID_ARG, "null output pointer");
  std::lock_guard<std::mutex> lk(g_sl_mu);
  *max_bytes_per_rank = g_slice_limit;
  return VC_SUCCESS;
}

VC_EXPORT vc_status_t vc_set_reuse_order(size_t min_step_bytes) {
  g_reuse_min.store(min_step_bytes, std::memory_order_relaxed);
  std::lock_guard<std::mutex> lk(g_plan_mu);  // cached plans carry the order they were built with
  g_plans.clear();
  return VC_SUCCESS;
}

VC_EXPORT vc_status_t vc_get_reuse_order(size_t* min_step_bytes) {
  if (!min_step_bytes) return fail(VC_ERR_INVALID_ARG, "null output pointer");
  *min_step_bytes = g_reuse_min.load(std::memory_order_relaxed);
  return VC_SUCCESS;
}

VC_EXPORT vc_status_t vc_set_copy_pipeline(size_t min_bytes) {
  g_copy_pipeline.store(min_bytes, std::memory_order_relaxed);
  return VC_SUCCESS;
}

VC_EXPORT vc_status_t vc_get_copy_pipeline(size_t* min_bytes) {
  if (!min_bytes) return fail(VC_ERR_INVALID_ARG, "null output pointer");
  *min_bytes = g_copy_pipeline.load(std::memory_order_relaxed);
  return VC_SUCCESS;
}

VC_EXPORT int vc_version(void) { return 100; }
