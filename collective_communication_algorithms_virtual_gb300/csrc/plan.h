// Step plans of the virtual-rank collectives (host C++, no CUDA).
//
// A plan is a list of steps; a step is a list of independent operations; an
// operation reads its sources, adds them left to right (or copies its single
// source) and writes every destination.  Steps run in order, one kernel
// launch each; the operations of a step never write what another operation of
// the same step reads or writes, so they run in any order or all at once.
#pragma once

#include <cstdint>
#include <string>
#include <vector>

namespace vc {

enum class Buf : uint8_t { Send = 0, Recv = 1, Scratch = 2 };
enum class DT : uint8_t { F32 = 0, BF16 = 1, I32 = 2, F16 = 3 };
enum class Mode : uint8_t { Copy = 0, F32 = 1, I32 = 2, BF16 = 3, F16 = 4 };
enum class RedOp : uint8_t { Sum = 0, Max = 1, Min = 2 };

enum class Coll : int {
  AllReduce = 0, ReduceScatter = 1, AllGather = 2, Broadcast = 3, Scatter = 4, AllToAll = 5, Gather = 6, Reduce = 7
};
enum class Algo : int {
  Fused = 0, Ring = 1, RHD = 2, DBT = 3, Binomial = 4, ScatterAllGather = 5, Pairwise = 6, Bruck = 7,
  PipeChain = 9, PipeTree = 10, Mesh = 11, RingHop = 12
};

inline int esize(DT t) { return (t == DT::BF16 || t == DT::F16) ? 2 : 4; }

struct Operand {
  Buf buf;
  int owner;         // rank holding the buffer (scratch: the rank it belongs to)
  int64_t byte_off;  // from the rank's buffer start (scratch: from the scratch block start)
  DT dt;             // storage type
};

struct Op {
  std::vector<Operand> src;
  std::vector<Operand> dst;
  int64_t n = 0;        // elements per run
  int64_t nb = 1;       // runs
  int64_t sstride = 0;  // bytes between runs, every source
  int64_t dstride = 0;  // bytes between runs, every destination
  bool keep = false;    // execution only: the next step reads the results (keep them in L2)
  uint32_t built = 0;   // introspection: the operation's index in its step as built
  // Element position of the operation's first element: element i of the
  // operation is position pos0 + i, and each operand holds the positions of
  // its region of a buffer in order.  Positions are the elements of the
  // message: AllReduce's and the tree Reduce's buffer, ring ReduceScatter's
  // input, ring AllGather's output, the Broadcasts' message (binomial,
  // Scatter+AllGather, pipelined), the binomial Scatter's input and Gather's
  // output at the root.  -1: the operation does not keep positions.
  int64_t pos0 = -1;
};

struct Step {
  Mode mode;
  std::vector<Op> ops;
  RedOp red = RedOp::Sum;  // how a reduction step combines its sources
  bool reverse = false;    // execution order only: walk the step's tiles from the last one
};

struct Plan {
  std::vector<Step> steps;
  int64_t scratch_bytes = 0;
  // Execution only (set by the library, not by build_plan): launch_end[s] >
  // s + 1 when steps s .. launch_end[s]-1 depend on nothing among themselves
  // and share one launch; empty when every step is its own launch.
  std::vector<uint32_t> launch_end;
};

struct PlanArgs {
  Coll coll;
  Algo algo;
  int nranks;
  int64_t count;  // per the collective's convention (see vc.h)
  DT dt;
  int root = 0;
  bool inplace = false;
  int nchunks = 1;  // pipelined Broadcasts: chunks of the message (>= 1)
  RedOp op = RedOp::Sum;
  // ring ReduceScatter: partial sums in two block slots per rank even where
  // one slot per block would fit (the entry point without allocation)
  bool compact_partials = false;
};

enum class PlanStatus { Ok, Invalid, Unsupported };

// The largest count a plan for `nranks` ranks takes: every byte offset and
// size in it then fits int64 (an AllToAll's working buffers, the largest,
// hold 2 N x N x count elements of 4 bytes).
int64_t count_limit(int nranks);

// Builds the plan; on failure `why` says what is wrong (counts above
// count_limit are Invalid).
PlanStatus build_plan(const PlanArgs& a, Plan* out, std::string* why);

// Algorithmic bytes of a plan (every operand read or written once) and the
// number of steps that launch work.
int64_t plan_bytes(const Plan& p);
int plan_launch_steps(const Plan& p);

// Cost models for choosing an algorithm (see vc.h, vc_set_cost_model).
enum class CostPolicy : int { Hbm = 0, Link = 1 };
struct CostModel {
  CostPolicy policy = CostPolicy::Hbm;
  double alpha = 0;  // seconds per step
  double beta = 0;   // bytes per second
};

// Chunks of a pipelined Broadcast when the caller does not choose: the
// optimum of the page's pipelined formula, k* = sqrt(h M / (alpha beta)) with
// h = N-2 (chain) or ceil(log2 N)-1 (tree), rounded, within [1, 256] and at
// most one chunk per 16 bytes.
int default_chunks(Algo a, int nranks, int64_t count, DT dt, const CostModel& cm);

// Picks the cheapest algorithm for a.coll under the model (a.algo is ignored).
PlanStatus select_algo(const PlanArgs& a, const CostModel& cm, Algo* out, double* predicted_s, std::string* why);

}  // namespace vc
