// Step plans of the virtual-rank collectives.
//
// Each builder below turns one schedule of the source pages into steps of
// independent operations over the N rank buffers.  A "send" of the pages is a
// read of the sender's buffer by the receiver's operation; a "recv" is the
// write of that operation.  Chunk indices, step order and the order in which
// each operation adds its sources follow the pages' schedules exactly:
//
//  * Ring AllReduce / ReduceScatter / AllGather: CSDN hccl article, section
//    "Ring算法：环形流水线传输"; latency-formula page "集合通信算法延迟公式",
//    eqs. model-algo-ring-rs / -ag / -ar, -allgather, -reducescatter.
//  * Recursive Halving-Doubling: latency-formula page, eqs. model-algo-rhd-*.
//  * Double Binary Tree: latency-formula page, eq. model-algo-dbt-ar, with the
//    heap tree of the hccl article, section "Tree算法：层次化规约".
//  * Binomial Broadcast / Scatter and Scatter+AllGather Broadcast:
//    Broadcast/Scatter page "一对多通信：Broadcast 与 Scatter", sections
//    "二叉树（Binomial Tree）", "二叉树 Scatter", "Broadcast 与 Scatter 的关系".
//  * Pairwise / Bruck AllToAll: latency-formula page, eqs.
//    model-algo-a2a-pairwise / -bruck.
//
// Readings where the pages leave a step open (chunk remainders, the ring
// AllGather indices, ReduceScatter block ownership, how the two DBT trees are
// built, Bruck's direction) are stated next to the code that takes them.
#include "plan.h"

#include <algorithm>
#include <cmath>
#include <functional>

namespace vc {
namespace {

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int ceil_log2(int n) {
  int l = 0;
  while ((1 << l) < n) ++l;
  return l;
}
int heap_depth(int i) {
  int d = 0;
  for (int v = i + 1; v > 1; v >>= 1) ++d;
  return d;
}
int lowbit(int v) { return v & -v; }

// Ring AllReduce of 16-bit data and ring ReduceScatter: while their partial
// sums take at most this many bytes per rank, they keep one place per element
// (see allreduce_ring, reduce_scatter).
constexpr int64_t kFlatPartialBytes = int64_t(16) << 20;
int md(int a, int n) { return ((a % n) + n) % n; }
bool is_pow2(int n) { return n >= 1 && (n & (n - 1)) == 0; }

// Chunk c of a buffer of `count` elements cut into `parts`: ce = ceil(count /
// parts) rounded up to a whole number of 16-byte groups, chunk c = [c*ce,
// (c+1)*ce) clipped to count.  The hccl article's ring divides count by the
// rank count and drops the remainder; the pages never say where it goes.
// With this rule every chunk starts on a 16-byte boundary of the buffer and
// the last chunks may be short or empty.
struct Chunks {
  int64_t count = 0, ce = 0;
  Chunks(int64_t count_, int parts, int es) : count(count_) {
    if (count <= 0) return;
    const int64_t align = 16 / es;
    ce = ceil_div(ceil_div(count, parts), align) * align;
  }
  int64_t lo(int64_t c) const { return std::min(c * ce, count); }
  int64_t hi(int64_t c) const { return std::min((c + 1) * ce, count); }
  int64_t len(int64_t c) const { return hi(c) - lo(c); }
};

class Builder {
 public:
  explicit Builder(const PlanArgs& a) : a_(a), N_(a.nranks), es_(esize(a.dt)) {}

  Plan take() { return std::move(plan_); }

  void build() {
    switch (a_.coll) {
      case Coll::AllReduce: allreduce(); break;
      case Coll::ReduceScatter: reduce_scatter(); break;
      case Coll::AllGather: allgather(); break;
      case Coll::Broadcast: broadcast(); break;
      case Coll::Scatter: scatter(); break;
      case Coll::AllToAll: alltoall(); break;
      case Coll::Gather: gather(); break;
      case Coll::Reduce: reduce(); break;
    }
  }

 private:
  const PlanArgs& a_;
  const int N_;
  const int es_;
  Plan plan_;

  // ---- operands and steps -------------------------------------------------
  Operand S(int r, int64_t elem) const { return {Buf::Send, r, elem * es_, a_.dt}; }
  Operand R(int r, int64_t elem) const { return {Buf::Recv, r, elem * es_, a_.dt}; }
  static Operand Sc(int owner, int64_t byte_off, DT dt) { return {Buf::Scratch, owner, byte_off, dt}; }

  int64_t alloc(int64_t bytes) {
    const int64_t off = plan_.scratch_bytes;
    plan_.scratch_bytes += ceil_div(std::max<int64_t>(bytes, 0), 256) * 256;
    return off;
  }

  Mode reduce_mode() const {
    switch (a_.dt) {
      case DT::F32: return Mode::F32;
      case DT::I32: return Mode::I32;
      case DT::BF16: return Mode::BF16;
      default: return Mode::F16;
    }
  }
  // Partial results are stored as fp32 when the data is 16-bit, else in the data type.
  DT acc_dt() const { return bf16() ? DT::F32 : a_.dt; }
  // 16-bit floating point data (bf16 or fp16): partials go to fp32 scratch.
  bool bf16() const { return a_.dt == DT::BF16 || a_.dt == DT::F16; }

  size_t new_step(Mode m) {
    Step st{m, {}};
    if (m != Mode::Copy) st.red = a_.op;
    plan_.steps.push_back(std::move(st));
    return plan_.steps.size() - 1;
  }
  // pos0: the operation's first element position (AllReduce schedules), or -1.
  void add(size_t st, std::vector<Operand> src, std::vector<Operand> dst, int64_t n, int64_t pos0 = -1) {
    if (n <= 0) return;
    Op op;
    op.src = std::move(src);
    op.dst = std::move(dst);
    op.n = n;
    op.pos0 = pos0;
    plan_.steps[st].ops.push_back(std::move(op));
  }
  void copy(size_t st, Operand src, Operand dst, int64_t n, int64_t pos0 = -1) { add(st, {src}, {dst}, n, pos0); }

  // ---- AllReduce ------------------------------------------------------------
  void allreduce() {
    if (a_.count == 0) return;
    if (N_ == 1) {
      if (!a_.inplace) copy(new_step(Mode::Copy), S(0, 0), R(0, 0), a_.count, 0);
      return;
    }
    switch (a_.algo) {
      case Algo::Fused: allreduce_fused(); break;
      case Algo::Ring:
      case Algo::RingHop: allreduce_ring(); break;
      case Algo::RHD: allreduce_rhd(); break;
      case Algo::DBT: allreduce_dbt(); break;
      case Algo::Mesh: allreduce_mesh(); break;
      default: break;
    }
  }

  // Mesh AllReduce (hccl article, section "Mesh算法：全连接广播"), step for
  // step from its code: the root folds every other rank's buffer into its own
  // in rank order, one rank per step, then sends the result to every other
  // rank in rank order, one per step.  The article's call takes a root; an
  // AllReduce here has none and rank 0 is the root.  The root's running
  // result lives in its receive buffer (fp32 scratch for 16-bit data).
  void allreduce_mesh() {
    const int root = 0;
    const int64_t count = a_.count;
    const int64_t part = bf16() ? alloc(count * 4) : -1;
    auto acc = [&]() { return part >= 0 ? Sc(root, part, DT::F32) : R(root, 0); };
    int t = 0;
    for (int i = 0; i < N_; ++i) {
      if (i == root) continue;
      const bool last = t == N_ - 2;
      add(new_step(reduce_mode()), {t == 0 ? S(root, 0) : acc(), S(i, 0)}, {last ? R(root, 0) : acc()}, count, 0);
      ++t;
    }
    for (int i = 0; i < N_; ++i)
      if (i != root) copy(new_step(Mode::Copy), R(root, 0), R(i, 0), count, 0);
  }

  // One pass: every output element is ((x0 + x1) + x2) + ... in rank order,
  // the fold of the hccl article's Mesh root (section "Mesh算法").
  void allreduce_fused() {
    const size_t st = new_step(reduce_mode());
    std::vector<Operand> src, dst;
    for (int q = 0; q < N_; ++q) src.push_back(S(q, 0));
    for (int r = 0; r < N_; ++r) dst.push_back(R(r, 0));
    add(st, src, dst, a_.count, 0);
  }

  // ReduceScatter step s: rank r adds chunk (r-s-1) mod N, sent by rank r-1,
  // to its own copy.  AllGather step s: rank r stores chunk (r-s) mod N from
  // rank r-1, i.e. every rank forwards the chunk it obtained the step before.
  // (The article prints the AllGather indices as r+s+1 / r+s; those agree with
  // the forwarding only at s = 0 and would leave chunk r-1 undelivered.)
  // Partial sums live in the receive buffers, or for bf16 in fp32 scratch:
  // up to kFlatPartialBytes of partials per rank one fp32 buffer per rank,
  // element e of chunk c at position e (every scratch byte then belongs to
  // one element of the buffers, which the sliced form needs); above that, two
  // fp32 chunk slots per rank used alternately (step s writes slot s%2 while
  // rank r+1 reads rank r's slot (s-1)%2), a quarter of the memory at 8
  // ranks.  The last ReduceScatter step writes the final (rounded) chunk into
  // the receive buffer.
  // RingHop: the same schedule with the partial sums kept in the data type,
  // rounded on every hop (no scratch); for fp32 / int32 it is the ring.
  void allreduce_ring() {
    const Chunks ch(a_.count, N_, es_);
    const bool wide = bf16() && a_.algo != Algo::RingHop;  // fp32 partials in scratch
    const bool flat = wide && a_.count * 4 <= kFlatPartialBytes;
    std::vector<int64_t> slot0(N_, 0);
    if (wide)
      for (int r = 0; r < N_; ++r) slot0[r] = alloc(flat ? a_.count * 4 : 2 * ch.ce * 4);
    auto part = [&](int r, int s, int64_t lo) {
      return Sc(r, flat ? slot0[r] + lo * 4 : slot0[r] + (s & 1) * ch.ce * 4, DT::F32);
    };
    for (int s = 0; s < N_ - 1; ++s) {
      const size_t st = new_step(reduce_mode());
      for (int r = 0; r < N_; ++r) {
        const int c = md(r - s - 1, N_), left = md(r - 1, N_);
        const int64_t lo = ch.lo(c);
        const Operand own = S(r, lo);
        const Operand in = s == 0 ? S(left, lo) : (wide ? part(left, s - 1, lo) : R(left, lo));
        const Operand out = s == N_ - 2 ? R(r, lo) : (wide ? part(r, s, lo) : R(r, lo));
        add(st, {own, in}, {out}, ch.len(c), lo);
      }
    }
    for (int s = 0; s < N_ - 1; ++s) {
      const size_t st = new_step(Mode::Copy);
      for (int r = 0; r < N_; ++r) {
        const int c = md(r - s, N_);
        copy(st, R(md(r - 1, N_), ch.lo(c)), R(r, ch.lo(c)), ch.len(c), ch.lo(c));
      }
    }
  }

  // Halving round k: rank r and r^2^k hold the same run of chunks; the rank
  // with bit k clear keeps the lower half, the other the upper half, and each
  // adds the partner's copy of the half it keeps.  Doubling round j: partners
  // at distance 2^(L-1-j) copy each other's segment.  Partial sums stay at
  // their own offsets (receive buffers, or one fp32 scratch buffer per rank
  // for bf16); a rank writes only the half it keeps while its partner reads
  // the other half, so no round overwrites what another op of it reads.
  void allreduce_rhd() {
    // N not a power of 2 (the pages require one; Rabenseifner's fold-in is the
    // reading taken): with P the largest power of 2 below N and r = N - P,
    // rank 2i+1 first hands its buffer to rank 2i (i < r), RHD runs on the P
    // virtual ranks v (real rank 2v for v < r, v + r after), and rank 2i
    // finally copies the result to 2i+1.
    int P = 1;
    while (P * 2 <= N_) P *= 2;
    const int rr = N_ - P;
    std::vector<int> real(P);
    for (int v = 0; v < P; ++v) real[v] = v < rr ? 2 * v : v + rr;
    const Chunks ch(a_.count, P, es_);
    const int L = ceil_log2(P);
    std::vector<int64_t> base(N_, 0);
    if (bf16())
      for (int v = 0; v < P; ++v) base[real[v]] = alloc(a_.count * 4);
    auto X = [&](int r, int64_t lo) { return bf16() ? Sc(r, base[r] + lo * 4, DT::F32) : R(r, lo); };
    std::vector<bool> folded(N_, false);
    if (rr > 0) {
      const size_t st = new_step(reduce_mode());
      for (int i = 0; i < rr; ++i) {
        add(st, {S(2 * i, 0), S(2 * i + 1, 0)}, {X(2 * i, 0)}, a_.count, 0);
        folded[2 * i] = true;
      }
    }
    std::vector<std::pair<int, int>> seg(P, {0, P});
    for (int k = 0; k < L; ++k) {
      const size_t st = new_step(reduce_mode());
      auto next = seg;
      for (int v = 0; v < P; ++v) {
        const int w = v ^ (1 << k);
        const int c0 = seg[v].first, c1 = seg[v].second, h = (c1 - c0) / 2;
        const std::pair<int, int> keep = ((v >> k) & 1) ? std::make_pair(c0 + h, c1) : std::make_pair(c0, c0 + h);
        next[v] = keep;
        const int64_t lo = ch.lo(keep.first), hi = ch.hi(keep.second - 1);
        const int rv = real[v], rw = real[w];
        const Operand own = (k == 0 && !folded[rv]) ? S(rv, lo) : X(rv, lo);
        const Operand partner = (k == 0 && !folded[rw]) ? S(rw, lo) : X(rw, lo);
        const Operand out = k == L - 1 ? R(rv, lo) : X(rv, lo);
        add(st, {own, partner}, {out}, hi - lo, lo);
      }
      seg = next;
    }
    for (int j = 0; j < L; ++j) {
      const int d = 1 << (L - 1 - j);
      const size_t st = new_step(Mode::Copy);
      auto next = seg;
      for (int v = 0; v < P; ++v) {
        const int w = v ^ d;
        const int64_t lo = ch.lo(seg[w].first), hi = ch.hi(seg[w].second - 1);
        copy(st, R(real[w], lo), R(real[v], lo), hi - lo, lo);
        next[v] = {std::min(seg[v].first, seg[w].first), std::max(seg[v].second, seg[w].second)};
      }
      seg = next;
    }
    if (rr > 0) {
      const size_t st = new_step(Mode::Copy);
      for (int i = 0; i < rr; ++i) copy(st, R(2 * i, 0), R(2 * i + 1, 0), a_.count, 0);
    }
  }

  // Two heap trees run their levels in the same steps.  Tree A: heap index i
  // on rank i (parent (i-1)/2, children 2i+1, 2i+2, as in the hccl article's
  // Tree); tree B: heap index i on rank N-1-i, so that each rank is interior
  // in at most one tree -- the pages ask for two trees with different
  // parent/child relations without saying how they are built.  Tree A takes
  // chunk 0 of a two-way split of the buffer, tree B chunk 1.  Reduce: the
  // deepest level first; a node adds its left child's subtree sum, then its
  // right child's, to its own value.  Broadcast: the root's sum goes down one
  // level per step.  The root writes the final (rounded) value into its
  // receive buffer; partial sums of other interior nodes live in their
  // receive buffers, or for bf16 in fp32 scratch.
  void allreduce_dbt() {
    const Chunks halves(a_.count, 2, es_);
    const int D = heap_depth(N_ - 1);
    std::vector<int64_t> base(N_, 0);
    if (bf16()) {
      const int64_t hmax = std::max(halves.len(0), halves.len(1));
      for (int r = 0; r < N_; ++r) base[r] = alloc(hmax * 4);
    }
    auto rank_of = [&](int tree, int i) { return tree == 0 ? i : N_ - 1 - i; };
    auto X = [&](int v, int64_t lo) { return bf16() ? Sc(v, base[v], DT::F32) : R(v, lo); };
    for (int t = 0; t < D; ++t) {
      const int depth = D - 1 - t;
      const size_t st = new_step(reduce_mode());
      for (int tree = 0; tree < 2; ++tree) {
        const int64_t lo = halves.lo(tree), n = halves.len(tree);
        for (int i = 0; i < N_; ++i) {
          if (heap_depth(i) != depth || 2 * i + 1 >= N_) continue;
          const int v = rank_of(tree, i);
          std::vector<Operand> src{S(v, lo)};
          for (int c = 2 * i + 1; c <= 2 * i + 2 && c < N_; ++c) {
            const bool leaf = 2 * c + 1 >= N_;
            src.push_back(leaf ? S(rank_of(tree, c), lo) : X(rank_of(tree, c), lo));
          }
          add(st, src, {i == 0 ? R(v, lo) : X(v, lo)}, n, lo);
        }
      }
    }
    for (int t = 0; t < D; ++t) {
      const int depth = t + 1;
      const size_t st = new_step(Mode::Copy);
      for (int tree = 0; tree < 2; ++tree) {
        const int64_t lo = halves.lo(tree), n = halves.len(tree);
        for (int i = 0; i < N_; ++i)
          if (heap_depth(i) == depth) copy(st, R(rank_of(tree, (i - 1) / 2), lo), R(rank_of(tree, i), lo), n, lo);
      }
    }
  }

  // ---- ReduceScatter / AllGather --------------------------------------------
  void reduce_scatter() {
    const int64_t rc = a_.count;
    if (rc == 0) return;
    if (N_ == 1) {
      copy(new_step(Mode::Copy), S(0, 0), R(0, 0), rc);
      return;
    }
    if (a_.algo == Algo::Fused) {
      const size_t st = new_step(reduce_mode());
      for (int r = 0; r < N_; ++r) {
        std::vector<Operand> src;
        for (int q = 0; q < N_; ++q) src.push_back(S(q, r * rc));
        add(st, src, {R(r, 0)}, rc);
      }
      return;
    }
    // Ring: the AllReduce ReduceScatter shifted by one block so that rank r
    // ends with block r (block ownership is left open by the pages): at step s
    // rank r adds block (r-s-2) mod N from rank r-1.  Partials travel through
    // scratch: while they take at most kFlatPartialBytes per rank, one buffer
    // of N blocks per rank, block c at its own place (every scratch byte then
    // belongs to one element of the input, which the sliced form needs);
    // above that two block slots per rank (step s writes slot s%2).
    std::vector<int64_t> slot0(N_);
    const DT adt = acc_dt();
    const bool flat = !a_.compact_partials && int64_t(N_) * rc * esize(adt) <= kFlatPartialBytes;
    for (int r = 0; r < N_; ++r) slot0[r] = alloc((flat ? N_ : 2) * rc * esize(adt));
    auto part = [&](int r, int s, int c) {
      return Sc(r, slot0[r] + (flat ? c : (s & 1)) * rc * esize(adt), adt);
    };
    for (int s = 0; s < N_ - 1; ++s) {
      const size_t st = new_step(reduce_mode());
      for (int r = 0; r < N_; ++r) {
        const int c = md(r - s - 2, N_), left = md(r - 1, N_);
        const Operand in = s == 0 ? S(left, c * rc) : part(left, s - 1, c);
        const Operand out = s == N_ - 2 ? R(r, 0) : part(r, s, c);
        add(st, {S(r, c * rc), in}, {out}, rc, c * rc);  // positions: the input's elements
      }
    }
  }

  void allgather() {
    const int64_t sc = a_.count;
    if (sc == 0) return;
    if (a_.algo == Algo::Fused || N_ == 1) {
      const size_t st = new_step(Mode::Copy);
      for (int q = 0; q < N_; ++q) {
        std::vector<Operand> dst;
        for (int r = 0; r < N_; ++r) dst.push_back(R(r, q * sc));
        add(st, {S(q, 0)}, dst, sc);
      }
      return;
    }
    // Ring: step 0 also places every rank's own block; at step s rank r stores
    // block (r-s-1) mod N from rank r-1 (read from rank r-1's input at step 0,
    // since its receive copy is being written in that same step).
    for (int s = 0; s < N_ - 1; ++s) {
      const size_t st = new_step(Mode::Copy);
      if (s == 0)
        for (int r = 0; r < N_; ++r) copy(st, S(r, 0), R(r, r * sc), sc, r * sc);
      for (int r = 0; r < N_; ++r) {
        const int c = md(r - s - 1, N_), left = md(r - 1, N_);
        copy(st, s == 0 ? S(left, 0) : R(left, c * sc), R(r, c * sc), sc, c * sc);  // positions: the output's elements
      }
    }
  }

  // ---- Broadcast / Scatter ----------------------------------------------------
  int absr(int v) const { return (v + a_.root) % N_; }

  void broadcast() {
    const int64_t count = a_.count;
    if (count == 0) return;
    const int root = a_.root;
    if (a_.algo == Algo::Fused || N_ == 1) {
      std::vector<Operand> dst;
      for (int r = 0; r < N_; ++r)
        if (r != root || !a_.inplace) dst.push_back(R(r, 0));
      if (!dst.empty()) add(new_step(Mode::Copy), {S(root, 0)}, dst, count);
      return;
    }
    if (a_.algo == Algo::PipeChain || a_.algo == Algo::PipeTree) {
      broadcast_pipelined();
      return;
    }
    if (a_.algo == Algo::Binomial) {
      // At distance d = 2^(L-1-s), every relative rank v with v mod 2d == 0
      // and v + d < N sends the whole message to v + d.
      const int L = ceil_log2(N_);
      for (int s = 0; s < L; ++s) {
        const int d = 1 << (L - 1 - s);
        const size_t st = new_step(Mode::Copy);
        if (s == 0 && !a_.inplace) copy(st, S(root, 0), R(root, 0), count, 0);
        for (int v = 0; v + d < N_; v += 2 * d)
          copy(st, v == 0 ? S(root, 0) : R(absr(v), 0), R(absr(v + d), 0), count, 0);
      }
      return;
    }
    // Scatter + AllGather: the message is cut into N chunks; rank r receives
    // chunk r straight into its place in its receive buffer; then a ring
    // AllGather in the receive buffers (step s: rank r stores chunk (r-s-1)
    // from rank r-1).
    const Chunks ch(count, N_, es_);
    auto clo = [&](int c) { return ch.lo(c); };
    auto clen = [&](int c) { return ch.len(c); };
    size_t first = plan_.steps.size();
    binomial_scatter(clo, clen, ch.ce, [&](int r) { return R(r, ch.lo(r)); });
    if (!a_.inplace) copy(first, S(root, ch.lo(root)), R(root, ch.lo(root)), ch.len(root), ch.lo(root));
    for (int s = 0; s < N_ - 1; ++s) {
      const size_t st = new_step(Mode::Copy);
      for (int r = 0; r < N_; ++r) {
        const int c = md(r - s - 1, N_);
        copy(st, R(md(r - 1, N_), ch.lo(c)), R(r, ch.lo(c)), ch.len(c), ch.lo(c));
      }
    }
  }

  // Chunked Broadcasts (Broadcast/Scatter page, sections "分块链式流水线" and
  // "分块二叉树流水线"): the message is cut into k chunks and chunk j follows
  // the unpipelined route delayed by j steps -- along the chain, relative rank
  // v forwards chunk j to v+1 at step v+j (N+k-2 steps); down the binomial
  // tree, chunk j takes binomial step s at step j+s (ceil(log2 N)+k-1 steps).
  // The pages give the step counts and chunk sizes; following the unpipelined
  // route with a delay per chunk is the reading taken.  In any one step a rank
  // receives one chunk and forwards other, earlier chunks.
  void broadcast_pipelined() {
    const int k = std::max(1, a_.nchunks);
    const Chunks ch(a_.count, k, es_);
    const int root = a_.root;
    const bool chain = a_.algo == Algo::PipeChain;
    const int L = ceil_log2(N_);
    const int nsteps = chain ? N_ + k - 2 : L + k - 1;
    for (int t = 0; t < nsteps; ++t) {
      const size_t st = new_step(Mode::Copy);
      if (t == 0 && !a_.inplace) copy(st, S(root, 0), R(root, 0), count_all(), 0);
      for (int j = 0; j < k; ++j) {
        const int s = t - j;
        if (chain) {
          if (s < 0 || s >= N_ - 1) continue;
          const int v = s;
          copy(st, v == 0 ? S(root, ch.lo(j)) : R(absr(v), ch.lo(j)), R(absr(v + 1), ch.lo(j)), ch.len(j), ch.lo(j));
        } else {
          if (s < 0 || s >= L) continue;
          const int d = 1 << (L - 1 - s);
          for (int v = 0; v + d < N_; v += 2 * d)
            copy(st, v == 0 ? S(root, ch.lo(j)) : R(absr(v), ch.lo(j)), R(absr(v + d), ch.lo(j)), ch.len(j),
                 ch.lo(j));
        }
      }
    }
  }
  int64_t count_all() const { return a_.count; }

  // Gather: the Scatter run backwards (Broadcast/Scatter page, section
  // "对偶性：Scatter 与 Gather").  Distances 1, 2, 4, ...: relative rank v with
  // v mod 2d == d hands the chunks of relative ranks [v, min(v+d, N)) -- its
  // own input and what its subtree gave it, kept in its staging scratch -- to
  // v - d; the root places them straight into its receive buffer.
  void gather() {
    const int64_t rc = a_.count;
    if (rc == 0) return;
    const int root = a_.root;
    if (a_.algo == Algo::Fused || N_ == 1) {
      const size_t st = new_step(Mode::Copy);
      for (int q = 0; q < N_; ++q) copy(st, S(q, 0), R(root, q * rc), rc);
      return;
    }
    const int L = ceil_log2(N_);
    std::vector<int64_t> stage(N_, 0);
    for (int v = 1; v < N_; ++v) {
      const int cap = std::min(lowbit(v), N_ - v) - 1;
      if (cap > 0) stage[v] = alloc(cap * rc * es_);
    }
    auto stage_op = [&](int v, int q) { return Sc(absr(v), stage[v] + (q - v - 1) * rc * es_, a_.dt); };
    for (int s = 0; s < L; ++s) {
      const int d = 1 << s;
      const size_t st = new_step(Mode::Copy);
      if (s == 0) copy(st, S(root, 0), R(root, root * rc), rc, root * rc);  // positions: the root's output
      for (int u = 0; u + d < N_; u += 2 * d) {
        const int v = u + d, end = std::min(v + d, N_);
        auto dst = [&](int q) { return u == 0 ? R(root, absr(q) * rc) : stage_op(u, q); };
        copy(st, S(absr(v), 0), dst(v), rc, absr(v) * rc);
        int q = v + 1;
        while (q < end) {  // runs contiguous at both ends (the root's buffer wraps past rank N-1)
          int q2 = q + 1;
          while (q2 < end && !(u == 0 && absr(q2) == 0)) ++q2;
          copy(st, stage_op(v, q), dst(q), int64_t(q2 - q) * rc, absr(q) * rc);
          q = q2;
        }
      }
    }
  }

  // Reduce to the root: the binomial Broadcast run backwards with adds
  // (latency-formula page, section "Broadcast / Reduce 怎么用 Tree 算法").
  // Distances 1, 2, 4, ...: relative rank u with u mod 2d == 0 adds the value
  // of u + d (its partial sum, or its input if it has none yet) to its own.
  // Partial sums live in scratch (fp32 for bf16); the root's last step writes
  // the (rounded) result into its receive buffer, which may be its input.
  void reduce() {
    const int64_t count = a_.count;
    if (count == 0) return;
    const int root = a_.root;
    if (N_ == 1) {
      if (!a_.inplace) copy(new_step(Mode::Copy), S(0, 0), R(0, 0), count);
      return;
    }
    if (a_.algo == Algo::Fused) {
      std::vector<Operand> src;
      for (int q = 0; q < N_; ++q) src.push_back(S(q, 0));
      add(new_step(reduce_mode()), src, {R(root, 0)}, count);
      return;
    }
    const int L = ceil_log2(N_);
    const DT adt = acc_dt();
    std::vector<int64_t> base(N_, -1);
    for (int u = 0; u + 1 < N_; u += 2)
      if (u != 0 || bf16()) base[u] = alloc(count * esize(adt));
    auto P = [&](int u) { return base[u] >= 0 ? Sc(absr(u), base[u], adt) : R(root, 0); };
    std::vector<bool> partial(N_, false);
    for (int s = 0; s < L; ++s) {
      const int d = 1 << s;
      const size_t st = new_step(reduce_mode());
      for (int u = 0; u + d < N_; u += 2 * d) {
        const int v = u + d;
        const Operand own = partial[u] ? P(u) : S(absr(u), 0);
        const Operand other = partial[v] ? P(v) : S(absr(v), 0);
        const bool last = u == 0 && s == L - 1;
        add(st, {own, other}, {last ? R(root, 0) : P(u)}, count, 0);
        partial[u] = true;
      }
    }
  }

  void scatter() {
    const int64_t rc = a_.count;
    if (rc == 0) return;
    const int root = a_.root;
    if (a_.algo == Algo::Fused || N_ == 1) {
      const size_t st = new_step(Mode::Copy);
      for (int r = 0; r < N_; ++r) copy(st, S(root, r * rc), R(r, 0), rc);
      return;
    }
    size_t first = plan_.steps.size();
    binomial_scatter([&](int c) { return c * rc; }, [&](int) { return rc; }, rc, [&](int r) { return R(r, 0); });
    copy(first, S(root, root * rc), R(root, 0), rc, root * rc);
  }

  // Binomial Scatter over absolute chunks [clo(c), clo(c)+clen(c)) of the
  // root's buffer.  At distance d, relative rank v hands the chunks of
  // relative ranks [v+d, min(v+2d, N)) to rank v+d: the receiver's own chunk
  // goes to own_dst(receiver), the rest to its staging scratch, which holds
  // relative chunks v+1 .. v+cap(v) in slots of `slot` elements.
  void binomial_scatter(const std::function<int64_t(int)>& clo, const std::function<int64_t(int)>& clen,
                        int64_t slot, const std::function<Operand(int)>& own_dst) {
    const int L = ceil_log2(N_);
    std::vector<int64_t> stage(N_, 0);
    for (int v = 1; v < N_; ++v) {
      const int cap = std::min(lowbit(v), N_ - v) - 1;
      if (cap > 0) stage[v] = alloc(cap * slot * es_);
    }
    auto stage_op = [&](int v, int q) { return Sc(absr(v), stage[v] + (q - v - 1) * slot * es_, a_.dt); };
    // Operand holding relative chunk q at sender v.
    auto held = [&](int v, int q) { return v == 0 ? S(a_.root, clo(absr(q))) : stage_op(v, q); };
    for (int s = 0; s < L; ++s) {
      const int d = 1 << (L - 1 - s);
      const size_t st = new_step(Mode::Copy);
      for (int v = 0; v + d < N_; v += 2 * d) {
        const int w = v + d, end = std::min(v + 2 * d, N_);
        copy(st, held(v, w), own_dst(absr(w)), clen(absr(w)), clo(absr(w)));  // positions: the root's buffer
        // the rest, in runs that stay contiguous in the root's buffer (split
        // where absolute chunk numbers wrap past N-1)
        int q = w + 1;
        while (q < end) {
          int q2 = q + 1;
          while (q2 < end && absr(q2) != 0) ++q2;
          int64_t n = 0;
          for (int k = q; k < q2; ++k) n += clen(absr(k));
          copy(st, held(v, q), stage_op(w, q), n, clo(absr(q)));
          q = q2;
        }
      }
    }
  }

  // ---- AllToAll -------------------------------------------------------------
  struct BlockCopy {
    Operand src, dst;
  };
  static bool same_bufs(const BlockCopy& x, const BlockCopy& y) {
    return x.src.buf == y.src.buf && x.src.owner == y.src.owner && x.dst.buf == y.dst.buf &&
           x.dst.owner == y.dst.owner;
  }
  // Emits block copies as runs with constant source and destination strides.
  void emit_runs(size_t st, const std::vector<BlockCopy>& v, int64_t B) {
    size_t i = 0;
    while (i < v.size()) {
      size_t j = i + 1;
      int64_t ss = 0, ds = 0;
      if (j < v.size() && same_bufs(v[i], v[j])) {
        ss = v[j].src.byte_off - v[i].src.byte_off;
        ds = v[j].dst.byte_off - v[i].dst.byte_off;
        ++j;
        while (j < v.size() && same_bufs(v[i], v[j]) && v[j].src.byte_off - v[j - 1].src.byte_off == ss &&
               v[j].dst.byte_off - v[j - 1].dst.byte_off == ds)
          ++j;
      }
      Op op;
      op.src = {v[i].src};
      op.dst = {v[i].dst};
      op.n = B;
      op.nb = static_cast<int64_t>(j - i);
      op.sstride = ss;
      op.dstride = ds;
      if (op.nb > 1 && ss == B * es_ && ds == B * es_) {  // one contiguous run
        op.n = B * op.nb;
        op.nb = 1;
        op.sstride = op.dstride = 0;
      }
      if (op.nb == 1) op.sstride = op.dstride = 0;
      plan_.steps[st].ops.push_back(std::move(op));
      i = j;
    }
  }

  // Ring AllToAll (latency-formula page, eq. model-algo-a2a-ring), store and
  // forward: in round k rank i receives from rank i-1 the blocks that left
  // rank s = i-k k rounds ago and are addressed to ranks i, i+1, ..., s-1;
  // it keeps the one for itself (block s of its output) and stages the rest,
  // indexed by destination, in one of two forwarding buffers (round k writes
  // buffer k%2 while rank i+1 reads rank i's buffer (k-1)%2).  Round 0 is the
  // local block.
  void alltoall_ring(int64_t B) {
    const int64_t fbytes = int64_t(N_) * B * es_;
    int64_t F[2] = {0, 0};
    if (N_ > 2) {
      F[0] = alloc(int64_t(N_) * fbytes);
      F[1] = alloc(int64_t(N_) * fbytes);
    }
    auto fwd = [&](int which, int rank, int d) { return Sc(rank, F[which] + rank * fbytes + d * B * es_, a_.dt); };
    {
      const size_t st = new_step(Mode::Copy);
      for (int i = 0; i < N_; ++i) copy(st, S(i, i * B), R(i, i * B), B);
    }
    for (int k = 1; k < N_; ++k) {
      const size_t st = new_step(Mode::Copy);
      for (int i = 0; i < N_; ++i) {
        const int from = md(i - 1, N_), src = md(i - k, N_);
        auto held = [&](int d) { return k == 1 ? S(from, int64_t(d) * B) : fwd((k - 1) & 1, from, d); };
        copy(st, held(i), R(i, int64_t(src) * B), B);
        std::vector<BlockCopy> rest;
        for (int h = 1; h < N_ - k; ++h) {  // destinations i+1 .. s-1, in ring order
          const int d = (i + h) % N_;
          rest.push_back({held(d), fwd(k & 1, i, d)});
        }
        emit_runs(st, rest, B);
      }
    }
  }

  void alltoall() {
    const int64_t B = a_.count;
    if (B == 0) return;
    if (a_.algo == Algo::Fused || N_ == 1) {
      const size_t st = new_step(Mode::Copy);
      for (int j = 0; j < N_; ++j)
        for (int i = 0; i < N_; ++i) copy(st, S(i, j * B), R(j, i * B), B);
      return;
    }
    if (a_.algo == Algo::Pairwise) {
      // Round 0 is the local block; in round k rank i writes its block for
      // rank (i+k) mod N into block i of that rank's output.
      for (int k = 0; k < N_; ++k) {
        const size_t st = new_step(Mode::Copy);
        for (int i = 0; i < N_; ++i) {
          const int j = (i + k) % N_;
          copy(st, S(i, j * B), R(j, i * B), B);
        }
      }
      return;
    }
    if (a_.algo == Algo::Ring) {
      alltoall_ring(B);
      return;
    }
    // Bruck (Bruck et al. 1997, cited by the latency-formula page): position p
    // of rank i's working buffer holds its block for rank (i+p) mod N.  Round
    // k rewrites every working buffer: positions with bit k set come from rank
    // i - 2^k (the packed send to distance 2^k), the others stay.  The first
    // round reads the inputs through the rotation, the last writes the outputs
    // through the inverse rotation (out_i[block (i-p) mod N] = position p), and
    // rounds in between use two scratch working buffers alternately.
    const int L = ceil_log2(N_);
    const int64_t wbytes = N_ * B * es_;
    int64_t W[2] = {0, 0};
    if (L >= 2) W[0] = alloc(int64_t(N_) * wbytes);
    if (L >= 3) W[1] = alloc(int64_t(N_) * wbytes);
    auto work = [&](int which, int rank, int p) { return Sc(rank, W[which] + rank * wbytes + p * B * es_, a_.dt); };
    for (int k = 0; k < L; ++k) {
      const size_t st = new_step(Mode::Copy);
      for (int i = 0; i < N_; ++i) {
        std::vector<BlockCopy> moving, staying;
        for (int p = 0; p < N_; ++p) {
          const bool mv = (p >> k) & 1;
          const int from = mv ? md(i - (1 << k), N_) : i;
          const Operand src = k == 0 ? S(from, int64_t((from + p) % N_) * B) : work((k - 1) & 1, from, p);
          const Operand dst = k == L - 1 ? R(i, int64_t(md(i - p, N_)) * B) : work(k & 1, i, p);
          (mv ? moving : staying).push_back({src, dst});
        }
        emit_runs(st, moving, B);
        emit_runs(st, staying, B);
      }
    }
  }
};

}  // namespace

int64_t count_limit(int nranks) { return INT64_MAX / 16 / (int64_t(nranks) * nranks); }

PlanStatus build_plan(const PlanArgs& a, Plan* out, std::string* why) {
  auto bad = [&](PlanStatus s, const char* msg) {
    if (why) *why = msg;
    return s;
  };
  if (a.nranks < 1 || a.nranks > 64) return bad(PlanStatus::Invalid, "nranks must be in [1, 64]");
  if (a.count < 0) return bad(PlanStatus::Invalid, "negative count");
  const bool rooted = a.coll == Coll::Broadcast || a.coll == Coll::Scatter || a.coll == Coll::Gather ||
                      a.coll == Coll::Reduce;
  if (rooted && (a.root < 0 || a.root >= a.nranks)) return bad(PlanStatus::Invalid, "root outside [0, nranks)");
  if (a.nchunks < 1 || a.nchunks > 1024) return bad(PlanStatus::Invalid, "nchunks must be in [1, 1024]");
  bool ok = false;
  switch (a.coll) {
    case Coll::AllReduce:
      ok = a.algo == Algo::Fused || a.algo == Algo::Ring || a.algo == Algo::RHD || a.algo == Algo::DBT ||
           a.algo == Algo::Mesh || a.algo == Algo::RingHop;
      break;
    case Coll::ReduceScatter:
    case Coll::AllGather: ok = a.algo == Algo::Fused || a.algo == Algo::Ring; break;
    case Coll::Broadcast:
      ok = a.algo == Algo::Fused || a.algo == Algo::Binomial || a.algo == Algo::ScatterAllGather;
      break;
    case Coll::Scatter: ok = a.algo == Algo::Fused || a.algo == Algo::Binomial; break;
    case Coll::AllToAll:
      ok = a.algo == Algo::Fused || a.algo == Algo::Pairwise || a.algo == Algo::Bruck || a.algo == Algo::Ring;
      break;
    case Coll::Gather:
    case Coll::Reduce: ok = a.algo == Algo::Fused || a.algo == Algo::Binomial; break;
  }
  if (a.coll == Coll::Broadcast && (a.algo == Algo::PipeChain || a.algo == Algo::PipeTree)) ok = true;
  if (!ok) return bad(PlanStatus::Unsupported, "algorithm not defined for this collective");
  if (a.count > count_limit(a.nranks)) return bad(PlanStatus::Invalid, "count too large");
  Builder b(a);
  b.build();
  *out = b.take();
  return PlanStatus::Ok;
}

int64_t plan_bytes(const Plan& p) {
  int64_t b = 0;
  for (const Step& s : p.steps)
    for (const Op& op : s.ops) {
      int64_t per = 0;
      for (const Operand& o : op.src) per += esize(o.dt);
      for (const Operand& o : op.dst) per += esize(o.dt);
      b += per * op.n * op.nb;
    }
  return b;
}

int plan_launch_steps(const Plan& p) {
  int n = 0;
  for (const Step& s : p.steps) n += s.ops.empty() ? 0 : 1;
  return n;
}

namespace {

// The pages' alpha-beta formulas with M the per-rank message in bytes
// (latency-formula page: eqs. model-algo-ring-ar, -rhd-ar, -dbt-ar,
// -ring-reducescatter, -ring-allgather, -a2a-pairwise, -a2a-bruck, -a2a-ring,
// -reduce-tree; Broadcast/Scatter page: eqs. binomial-bcast, binomial-scatter,
// onetoall-gather-scatter-duality, pipe-chain-bcast, pipe-tree-bcast).
double link_time(Coll c, Algo a, int N, double M, double al, double be, double k) {
  const double n = N, lg = std::log2(n), cl = ceil_log2(N);
  switch (c) {
    case Coll::AllReduce:
      if (a == Algo::Ring) return 2 * (n - 1) * al + 2 * (n - 1) / n * M / be;
      if (a == Algo::RHD) return 2 * lg * al + 2 * (n - 1) / n * M / be;
      return 2 * lg * al + lg * M / be;  // DBT
    case Coll::ReduceScatter:
    case Coll::AllGather: return (n - 1) * al + (n - 1) / n * M / be;
    case Coll::Broadcast:
      if (a == Algo::Binomial) return cl * (al + M / be);
      if (a == Algo::PipeChain) return (n + k - 2) * (al + M / (k * be));
      if (a == Algo::PipeTree) return (cl + k - 1) * (al + M / (k * be));
      return cl * al + (n - 1) * M / (n * be) + (n - 1) * al + (n - 1) / n * M / be;  // scatter + ring AG
    case Coll::Scatter:
    case Coll::Gather: return cl * al + (n - 1) * M / (n * be);
    case Coll::Reduce: return lg * (al + M / be);
    case Coll::AllToAll:
      if (a == Algo::Pairwise) return (n - 1) * (al + M / (n * be));
      if (a == Algo::Ring) return (n - 1) * al + (n - 1) / n * M / be;  // as printed (see the oracle)
      return cl * al + (n - 1) / n * M / be;  // Bruck
  }
  return 0;
}

}  // namespace

int default_chunks(Algo a, int nranks, int64_t count, DT dt, const CostModel& cm) {
  const double h = a == Algo::PipeChain ? nranks - 2 : ceil_log2(nranks) - 1;
  const double M = double(count) * esize(dt);
  int64_t k = 1;
  if (h > 0 && M > 0 && cm.alpha > 0 && cm.beta > 0) k = static_cast<int64_t>(std::floor(std::sqrt(h * M / (cm.alpha * cm.beta)) + 0.5));
  const int64_t groups = std::max<int64_t>(1, count * esize(dt) / 16);
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>({k, 256, groups})));
}

PlanStatus select_algo(const PlanArgs& a, const CostModel& cm, Algo* out, double* predicted_s, std::string* why) {
  std::vector<Algo> cand;
  const bool link = cm.policy == CostPolicy::Link;
  switch (a.coll) {
    case Coll::AllReduce:
      cand = link ? std::vector<Algo>{Algo::Ring, Algo::RHD, Algo::DBT}
                  : std::vector<Algo>{Algo::Fused, Algo::Ring, Algo::RHD, Algo::DBT, Algo::Mesh, Algo::RingHop};
      if (link && !is_pow2(a.nranks)) cand.erase(cand.begin() + 1);  // the page's RHD formula needs 2^k
      break;
    case Coll::ReduceScatter:
    case Coll::AllGather:
      cand = link ? std::vector<Algo>{Algo::Ring} : std::vector<Algo>{Algo::Fused, Algo::Ring};
      break;
    case Coll::Broadcast:
      cand = link ? std::vector<Algo>{Algo::Binomial, Algo::ScatterAllGather}
                  : std::vector<Algo>{Algo::Fused, Algo::Binomial, Algo::ScatterAllGather};
      break;
    case Coll::Scatter:
      cand = link ? std::vector<Algo>{Algo::Binomial} : std::vector<Algo>{Algo::Fused, Algo::Binomial};
      break;
    case Coll::AllToAll:
      cand = link ? std::vector<Algo>{Algo::Pairwise, Algo::Bruck, Algo::Ring}
                  : std::vector<Algo>{Algo::Fused, Algo::Pairwise, Algo::Bruck, Algo::Ring};
      break;
    case Coll::Gather:
    case Coll::Reduce:
      cand = link ? std::vector<Algo>{Algo::Binomial} : std::vector<Algo>{Algo::Fused, Algo::Binomial};
      break;
  }
  if (a.coll == Coll::Broadcast) {
    cand.push_back(Algo::PipeChain);
    cand.push_back(Algo::PipeTree);
  }
  const int64_t es = esize(a.dt);
  const bool per_rank = a.coll == Coll::AllReduce || a.coll == Coll::Broadcast || a.coll == Coll::Reduce;
  const double M = per_rank ? double(a.count * es) : double(a.count * es * a.nranks);
  bool found = false;
  double best = 0;
  PlanStatus last = PlanStatus::Unsupported;
  for (Algo al : cand) {
    PlanArgs pa = a;
    pa.algo = al;
    pa.nchunks = (al == Algo::PipeChain || al == Algo::PipeTree) ? default_chunks(al, a.nranks, a.count, a.dt, cm) : 1;
    Plan p;
    std::string w;
    last = build_plan(pa, &p, &w);
    if (last == PlanStatus::Invalid) {
      if (why) *why = w;
      return last;
    }
    if (last != PlanStatus::Ok) continue;
    const double t = link ? link_time(a.coll, al, a.nranks, M, cm.alpha, cm.beta, pa.nchunks)
                          : plan_launch_steps(p) * cm.alpha + double(plan_bytes(p)) / cm.beta;
    if (!found || t < best) {
      found = true;
      best = t;
      *out = al;
    }
  }
  if (!found) {
    if (why) *why = "no algorithm is defined for these arguments";
    return PlanStatus::Unsupported;
  }
  if (predicted_s) *predicted_s = best;
  return PlanStatus::Ok;
}

}  // namespace vc
