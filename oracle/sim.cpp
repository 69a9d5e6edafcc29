// The oracle for the virtual-rank collectives -- TEST INFRASTRUCTURE ONLY.
//
// A plain, single-threaded C++17 simulation of N ranks exchanging messages
// step by step, written from three source pages:
//   [Bcast/Scatter page]    "一对多通信：Broadcast 与 Scatter" (one-to-many
//                           communication: Broadcast and Scatter);
//   [hccl article]          the CSDN article on CANN hccl's AllReduce
//                           algorithms, sections "Ring算法：环形流水线传输",
//                           "Mesh算法：全连接广播", "Tree算法：层次化规约";
//   [Latency-formula page]  "集合通信算法延迟公式" (alpha-beta latency formulas
//                           of collective algorithms), cited by equation label.
//
// Model (the alpha-beta model of the latency-formula page): every rank holds
// its own buffers; a step is a list of messages; every payload is copied from
// its sender before any message of the step is delivered, so the messages of
// one step travel at the same time.  A receiver either stores a payload or
// combines it into its own data, in the order the messages are listed.  Each
// schedule records a transfer log (step, sender, receiver, elements, reduce or
// store, bytes per element on the wire, offsets or chunk indices) and its
// algorithmic HBM bytes: every operand a step reads and every result it writes
// once, at its storage size, when the N ranks are N buffers of one memory.
//
// Arithmetic.  fp32: one IEEE binary32 add (round to nearest even) per
// combine, in the schedule's own association.  int32: addition modulo 2^32.
// bf16 and fp16: widened exactly to fp32, accumulated in fp32 -- partial sums
// travel and are stored as fp32 -- and rounded once, to nearest even, when the
// result is stored (the ring_hop schedule instead rounds after every hop).
// MAX / MIN: max(a, b) = b when b > a or a is NaN, else a (min likewise); the
// pages list the ops without NaN or signed-zero rules, and this is the reading
// taken.  int32 compares signed.
//
// Where the pages are silent the readings are stated at the schedule.  This
// file shares no code with the CUDA library, and nothing in it is used by the
// library.

#include "sim.h"

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <stdexcept>
#include <string>
#include <vector>

namespace {

enum DType { F32 = 0, BF16 = 1, I32 = 2, F16 = 3 };
enum Op { SUM = 0, MAX = 1, MIN = 2 };

struct Unsupported : std::runtime_error {
  using std::runtime_error::runtime_error;
};
struct BadArg : std::runtime_error {
  using std::runtime_error::runtime_error;
};

int esize_of(int dt) { return (dt == F32 || dt == I32) ? 4 : 2; }

// ---------------------------------------------------------------------------
// element conversions, from the IEEE 754 binary32 / binary16 layouts and the
// bf16 layout (the upper half of a binary32)
// ---------------------------------------------------------------------------
uint32_t bits_of(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return u;
}
float float_of(uint32_t u) {
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

uint32_t widen_bf16(uint16_t b) { return static_cast<uint32_t>(b) << 16; }

// Round to nearest, ties to even: with the kept part k = u >> 16 and the
// dropped part d = u & 0xFFFF, u + 0x7FFF + (k & 1) carries into k exactly
// when d > 0x8000, or d == 0x8000 and k is odd.  A carry out of the mantissa
// moves into the exponent, so the largest finite values round to infinity.
// NaN keeps its sign and top payload bits and gets the quiet bit.
uint16_t narrow_bf16(uint32_t u) {
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return static_cast<uint16_t>((u >> 16) | 0x0040u);
  const uint64_t k_odd = (u >> 16) & 1u;
  return static_cast<uint16_t>((static_cast<uint64_t>(u) + 0x7FFFu + k_odd) >> 16);
}

// binary16: sign, 5 exponent bits (bias 15), 10 mantissa bits.  Exact.
uint32_t widen_f16(uint16_t h) {
  const uint32_t sign = static_cast<uint32_t>(h & 0x8000u) << 16;
  const uint32_t ex = (h >> 10) & 0x1Fu;
  const uint32_t man = h & 0x3FFu;
  if (ex == 0) {
    // zero or subnormal: man * 2^-24, exact in binary32
    const float v = std::ldexp(static_cast<float>(man), -24);
    return sign | bits_of(v);
  }
  if (ex == 31) return sign | 0x7F800000u | (man << 13);
  return sign | ((ex - 15 + 127) << 23) | (man << 13);
}

// binary32 -> binary16, round to nearest, ties to even.  Above the largest
// finite half plus half an ulp (65520) the result is infinity.  NaN keeps its
// sign and top payload bits and gets the quiet bit.
uint16_t narrow_f16(uint32_t u) {
  const uint16_t sign = static_cast<uint16_t>((u >> 16) & 0x8000u);
  const uint32_t a = u & 0x7FFFFFFFu;
  if (a > 0x7F800000u) return static_cast<uint16_t>(sign | 0x7E00u | ((a >> 13) & 0x3FFu));
  if (a >= 0x477FF000u) return static_cast<uint16_t>(sign | 0x7C00u);  // |x| >= 65520 (or inf)
  if (a >= 0x38800000u) {                                               // |x| >= 2^-14: normal half
    const uint32_t ex = (a >> 23) - 127 + 15;
    const uint32_t m = a & 0x7FFFFFu;
    uint32_t h = (ex << 10) | (m >> 13);
    const uint32_t rem = m & 0x1FFFu;
    if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) ++h;
    return static_cast<uint16_t>(sign | h);
  }
  if (a <= 0x33000000u) return sign;  // |x| <= 2^-25: the tie at 2^-25 goes to the even 0
  // subnormal half: |x| = m * 2^(E-23) with the implicit bit in m; in units
  // of 2^-24 that is m * 2^(E+1), E in [-25, -15]
  const int E = static_cast<int>(a >> 23) - 127;
  const uint32_t m = (a & 0x7FFFFFu) | 0x800000u;
  const int shift = -(E + 1);  // 14 .. 24
  uint32_t q = m >> shift;
  const uint32_t r = m & ((1u << shift) - 1u);
  const uint32_t half = 1u << (shift - 1);
  if (r > half || (r == half && (q & 1u))) ++q;
  return static_cast<uint16_t>(sign | q);
}

// ---------------------------------------------------------------------------
// lanes: every reduction runs on 32-bit lanes (fp32 bits, or uint32 for int32)
// ---------------------------------------------------------------------------
using Lane = uint32_t;

bool lanes_are_float(int dt) { return dt != I32; }

Lane widen_elem(const uint8_t* p, int dt) {
  switch (dt) {
    case F32:
    case I32: {
      uint32_t v;
      std::memcpy(&v, p, 4);
      return v;
    }
    case BF16: {
      uint16_t v;
      std::memcpy(&v, p, 2);
      return widen_bf16(v);
    }
    default: {
      uint16_t v;
      std::memcpy(&v, p, 2);
      return widen_f16(v);
    }
  }
}

void narrow_elem(Lane v, int dt, uint8_t* p) {
  switch (dt) {
    case F32:
    case I32:
      std::memcpy(p, &v, 4);
      break;
    case BF16: {
      const uint16_t b = narrow_bf16(v);
      std::memcpy(p, &b, 2);
      break;
    }
    default: {
      const uint16_t h = narrow_f16(v);
      std::memcpy(p, &h, 2);
      break;
    }
  }
}

Lane combine1(Lane a, Lane b, int op, bool fl) {
  if (op == SUM) return fl ? bits_of(float_of(a) + float_of(b)) : a + b;
  if (fl) {
    const float x = float_of(a), y = float_of(b);
    const bool take_b = (op == MAX ? y > x : y < x) || std::isnan(x);
    return take_b ? b : a;
  }
  const int32_t x = static_cast<int32_t>(a), y = static_cast<int32_t>(b);
  return (op == MAX ? y > x : y < x) ? b : a;
}

// dst[i] = dst[i] (op) src[i]
void combine_into(Lane* dst, const Lane* src, int64_t n, int op, bool fl) {
  if (op == SUM && fl) {
    for (int64_t i = 0; i < n; ++i) dst[i] = bits_of(float_of(dst[i]) + float_of(src[i]));
  } else if (op == SUM) {
    for (int64_t i = 0; i < n; ++i) dst[i] = dst[i] + src[i];
  } else {
    for (int64_t i = 0; i < n; ++i) dst[i] = combine1(dst[i], src[i], op, fl);
  }
}

std::vector<Lane> widen_buf(const uint8_t* p, int64_t n, int dt) {
  std::vector<Lane> v(static_cast<size_t>(n));
  const int es = esize_of(dt);
  for (int64_t i = 0; i < n; ++i) v[i] = widen_elem(p + i * es, dt);
  return v;
}

std::vector<uint8_t> narrow_buf(const Lane* v, int64_t n, int dt) {
  const int es = esize_of(dt);
  std::vector<uint8_t> out(static_cast<size_t>(n * es));
  for (int64_t i = 0; i < n; ++i) narrow_elem(v[i], dt, out.data() + i * es);
  return out;
}

// ---------------------------------------------------------------------------
// how a buffer is cut into parts ([hccl article] "Ring算法": chunk_size =
// count / size drops the remainder; reading taken: ce = ceil(count / parts)
// rounded up to a 16-byte multiple, chunk c = [min(c ce, count),
// min((c+1) ce, count)), so the last chunks may be short or empty)
// ---------------------------------------------------------------------------
int64_t part_elems(int64_t count, int64_t parts, int es) {
  if (count <= 0) return 0;
  const int64_t align = 16 / es;
  const int64_t ce = (count + parts - 1) / parts;
  return (ce + align - 1) / align * align;
}
std::pair<int64_t, int64_t> part_range(int64_t c, int64_t count, int64_t parts, int es) {
  const int64_t ce = part_elems(count, parts, es);
  return {std::min(c * ce, count), std::min((c + 1) * ce, count)};
}

int ceil_log2(int n) {
  int L = 0;
  while ((1 << L) < n) ++L;
  return L;
}
int mod(int a, int n) { return ((a % n) + n) % n; }

// ---------------------------------------------------------------------------
// the simulation: buffers, messages, steps
// ---------------------------------------------------------------------------
// A buffer is either lanes (a rank's data during a reduction) or stored
// elements (data movement).  A message is a list of pieces, each copying n
// elements from a sender's buffer to a receiver's.
struct Buf {
  bool lanes = false;
  int es = 4;
  std::vector<Lane> l;
  std::vector<uint8_t> b;
};

struct Piece {
  Buf* src;
  int64_t soff;
  Buf* dst;
  int64_t doff;
  int64_t n;
};

struct Record {
  int64_t step, src, dst, n, reduce, esize, src_off, dst_off;
  std::string phase;
  std::vector<int64_t> chunks;
};

struct Msg {
  Record rec;
  std::vector<Piece> pieces;
  bool round_after = false;  // ring_hop: round the combined values to the data type
};

int g_fault_kind = 0, g_fault_step = -1;

struct Sim {
  int dt, op;
  int e_in, e_out, e_acc;
  int64_t hbm = 0;
  int local_steps = 0;
  std::vector<Record> log;

  Sim(int dtype, int op_) : dt(dtype), op(op_) {
    e_in = e_out = esize_of(dtype);
    e_acc = 4;
  }

  // algorithmic bytes: n elements, each read or written once at these sizes
  void rw(int64_t n, std::initializer_list<int> sizes) {
    int64_t s = 0;
    for (int x : sizes) s += x;
    hbm += n * s;
  }
  void rw(int64_t n, const std::vector<int>& sizes) {
    int64_t s = 0;
    for (int x : sizes) s += x;
    hbm += n * s;
  }

  Msg msg(int src, int dst, int64_t n, bool reduce, int wire, const char* phase, int64_t src_off = -1,
          int64_t dst_off = -1, std::vector<int64_t> chunks = {}) {
    Msg m;
    m.rec = Record{0, src, dst, n, reduce ? 1 : 0, wire, src_off, dst_off, phase, std::move(chunks)};
    return m;
  }

  void deliver(const Msg& m, const std::vector<std::vector<uint8_t>>& sent_bytes,
               const std::vector<std::vector<Lane>>& sent_lanes, size_t mi) {
    int64_t at = 0;
    for (const Piece& p : m.pieces) {
      if (p.dst->lanes) {
        Lane* d = p.dst->l.data() + p.doff;
        const Lane* s = sent_lanes[mi].data() + at;
        if (m.rec.reduce)
          combine_into(d, s, p.n, op, lanes_are_float(dt));
        else
          std::memcpy(d, s, static_cast<size_t>(p.n) * 4);
        if (m.round_after)
          for (int64_t i = 0; i < p.n; ++i) {
            uint8_t tmp[4];
            narrow_elem(d[i], dt, tmp);
            d[i] = widen_elem(tmp, dt);
          }
      } else {
        std::memcpy(p.dst->b.data() + p.doff * p.dst->es, sent_bytes[mi].data() + at * p.dst->es,
                    static_cast<size_t>(p.n * p.dst->es));
      }
      at += p.n;
    }
  }

  // payload snapshots, kept from step to step so that their memory is reused
  std::vector<std::vector<uint8_t>> pb;
  std::vector<std::vector<Lane>> pl;

  // All payloads are read from their senders first, then delivered in order.
  void run_step(int step, std::vector<Msg>& msgs) {
    if (g_fault_kind == 1 && g_fault_step == step) return;
    if (pb.size() < msgs.size()) {
      pb.resize(msgs.size());
      pl.resize(msgs.size());
    }
    for (size_t i = 0; i < msgs.size(); ++i) {
      pb[i].clear();
      pl[i].clear();
      for (const Piece& p : msgs[i].pieces) {
        if (p.src->lanes)
          pl[i].insert(pl[i].end(), p.src->l.begin() + p.soff, p.src->l.begin() + p.soff + p.n);
        else
          pb[i].insert(pb[i].end(), p.src->b.begin() + p.soff * p.src->es,
                       p.src->b.begin() + (p.soff + p.n) * p.src->es);
      }
    }
    for (size_t i = 0; i < msgs.size(); ++i) {
      msgs[i].rec.step = step;
      log.push_back(msgs[i].rec);
      deliver(msgs[i], pb, pl, i);
      if (g_fault_kind == 2 && g_fault_step == step) deliver(msgs[i], pb, pl, i);
    }
  }
};

Buf lane_buf(const uint8_t* p, int64_t n, int dt) {
  Buf b;
  b.lanes = true;
  b.l = widen_buf(p, n, dt);
  return b;
}
Buf byte_buf(int64_t n, int es) {
  Buf b;
  b.es = es;
  b.b.assign(static_cast<size_t>(n * es), 0);
  return b;
}
Buf byte_copy(const uint8_t* p, int64_t n, int es) {
  Buf b;
  b.es = es;
  b.b.assign(p, p + n * es);
  return b;
}

struct Out {
  std::vector<std::vector<uint8_t>> outputs;
};

using In = std::vector<const uint8_t*>;

// one rank, nothing to exchange: every output is a copy of the input
void self_copy(Sim& sm, const In& in, int64_t count, Out& o) {
  sm.rw(count, {sm.e_in, sm.e_out});
  for (const uint8_t* p : in) o.outputs.emplace_back(p, p + count * sm.e_in);
}

void narrow_all(Sim& sm, std::vector<Buf>& acc, int64_t count, Out& o) {
  for (Buf& b : acc) o.outputs.push_back(narrow_buf(b.l.data(), count, sm.dt));
}

// ---------------------------------------------------------------------------
// AllReduce: out_r = the elementwise reduction of every rank's input, on every
// rank ([Latency-formula page] section "Ring AllReduce"; [hccl article]
// section "集合通信vs点对点")
// ---------------------------------------------------------------------------

// Fused: every rank's element is read once and folded in rank order,
// ((x0 + x1) + x2) + ..., the order in which the [hccl article]'s Mesh root
// folds ranks 0..N-1 into its buffer; the result is written to all N outputs.
void allreduce_fused(Sim& sm, const In& in, int64_t count, Out& o) {
  const int N = static_cast<int>(in.size());
  std::vector<Lane> acc = widen_buf(in[0], count, sm.dt);
  for (int q = 1; q < N; ++q) {
    const std::vector<Lane> x = widen_buf(in[q], count, sm.dt);
    combine_into(acc.data(), x.data(), count, sm.op, lanes_are_float(sm.dt));
  }
  if (N > 1)
    for (int q = 0; q < N; ++q)
      for (int r = 0; r < N; ++r)
        if (q != r) sm.log.push_back(Record{0, q, r, count, 1, sm.e_in, 0, 0, "fused", {}});
  std::vector<int> sizes(N, sm.e_in);
  sizes.insert(sizes.end(), N, sm.e_out);
  sm.rw(count, sizes);
  const std::vector<uint8_t> res = narrow_buf(acc.data(), count, sm.dt);
  for (int r = 0; r < N; ++r) o.outputs.push_back(res);
}

// Mesh ([hccl article] "Mesh算法：全连接广播"), from its code: the root
// receives every other rank's buffer in rank order and folds each into its
// own (N-1 steps of one message), then sends the result to every other rank
// in rank order (N-1 steps).  An AllReduce call has no root: root 0.
void allreduce_mesh(Sim& sm, const In& in, int64_t count, Out& o) {
  const int N = static_cast<int>(in.size());
  if (N == 1) return self_copy(sm, in, count, o);
  std::vector<Buf> acc;
  for (int r = 0; r < N; ++r) acc.push_back(lane_buf(in[r], count, sm.dt));
  int step = 0;
  for (int i = 1, t = 0; i < N; ++i, ++t) {
    std::vector<Msg> ms;
    Msg m = sm.msg(i, 0, count, true, sm.e_in, "mesh_reduce", 0, 0);
    m.pieces.push_back({&acc[i], 0, &acc[0], 0, count});
    ms.push_back(std::move(m));
    sm.rw(count, {t == 0 ? sm.e_in : sm.e_acc, sm.e_in, t == N - 2 ? sm.e_out : sm.e_acc});
    sm.run_step(step++, ms);
  }
  for (int i = 1; i < N; ++i) {
    std::vector<Msg> ms;
    Msg m = sm.msg(0, i, count, false, sm.e_out, "mesh_bcast", 0, 0);
    m.pieces.push_back({&acc[0], 0, &acc[i], 0, count});
    ms.push_back(std::move(m));
    sm.rw(count, {sm.e_out, sm.e_out});
    sm.run_step(step++, ms);
  }
  narrow_all(sm, acc, count, o);
}

// Ring AllReduce = Ring ReduceScatter then Ring AllGather, N-1 steps each
// ([hccl article] "Ring算法"; [Latency-formula page] eqs. model-algo-ring-rs,
// -ag, -ar).  ReduceScatter step s: rank r sends chunk (r - s) mod N to r + 1,
// which adds it to its own copy; chunk c ends on rank c - 1 summed as
// x_c + x_{c+1} + ... + x_{c+N-1}.  AllGather step s: rank r forwards the
// chunk it completed or received last, (r + 1 - s) mod N, which r + 1 stores
// (reading taken of the article's garbled AllGather indices: forwarding, as
// its prose and the formula page describe).  16-bit data: fp32 partials, one
// rounding on the last ReduceScatter step; round_each_hop (ring_hop) rounds to
// the data type after every hop instead.
void allreduce_ring(Sim& sm, const In& in, int64_t count, Out& o, bool round_each_hop) {
  const int N = static_cast<int>(in.size());
  if (N == 1) return self_copy(sm, in, count, o);
  const int es = esize_of(sm.dt);
  std::vector<Buf> acc;
  for (int r = 0; r < N; ++r) acc.push_back(lane_buf(in[r], count, sm.dt));
  const int e_part = round_each_hop ? sm.e_in : sm.e_acc;
  int step = 0;
  for (int s = 0; s < N - 1; ++s) {
    std::vector<Msg> ms;
    for (int r = 0; r < N; ++r) {
      const int c = mod(r - s, N);
      const auto [lo, hi] = part_range(c, count, N, es);
      const int dst = (r + 1) % N;
      const int wire = s == 0 ? sm.e_in : e_part;
      Msg m = sm.msg(r, dst, hi - lo, true, wire, "rs", lo, lo, {c});
      m.pieces.push_back({&acc[r], lo, &acc[dst], lo, hi - lo});
      m.round_after = round_each_hop;
      ms.push_back(std::move(m));
      sm.rw(hi - lo, {sm.e_in, wire, s == N - 2 ? sm.e_out : e_part});
    }
    sm.run_step(step++, ms);
  }
  for (int s = 0; s < N - 1; ++s) {
    std::vector<Msg> ms;
    for (int r = 0; r < N; ++r) {
      const int c = mod(r + 1 - s, N);
      const auto [lo, hi] = part_range(c, count, N, es);
      const int dst = (r + 1) % N;
      Msg m = sm.msg(r, dst, hi - lo, false, sm.e_out, "ag", lo, lo, {c});
      m.pieces.push_back({&acc[r], lo, &acc[dst], lo, hi - lo});
      ms.push_back(std::move(m));
      sm.rw(hi - lo, {sm.e_out, sm.e_out});
    }
    sm.run_step(step++, ms);
  }
  narrow_all(sm, acc, count, o);
}

// Recursive Halving-Doubling (Rabenseifner) ([Latency-formula page] section
// "Recursive Halving-Doubling", eqs. model-algo-rhd-rs, -ag, -ar, for N a
// power of 2).  Halving round k pairs virtual rank v with v XOR 2^k; both
// hold the same run of chunks; the one with bit k clear keeps the lower half
// (reading: the page does not say which), each sends the half it gives up
// and adds the half it keeps.  Doubling (the reverse process) pairs v with
// v XOR 2^(L-1-j) in round j; each sends its whole run and stores the
// partner's.  N not a power of 2 (reading: Rabenseifner's own fold-in): with
// P the largest power of 2 not above N and r = N - P, odd rank 2i+1 (i < r)
// first hands its buffer to 2i, which adds it; the halving and doubling run
// on virtual ranks v = 0..P-1 living on real rank 2v (v < r) or v + r; rank
// 2i finally hands the result back to 2i+1.
void allreduce_rhd(Sim& sm, const In& in, int64_t count, Out& o) {
  const int N = static_cast<int>(in.size());
  if (N == 1) return self_copy(sm, in, count, o);
  const int es = esize_of(sm.dt);
  int P = 1;
  while (P * 2 <= N) P *= 2;
  const int rr = N - P;
  int L = 0;
  while ((1 << L) < P) ++L;
  std::vector<int> real(P);
  for (int v = 0; v < P; ++v) real[v] = v < rr ? 2 * v : v + rr;
  std::vector<Buf> acc;
  for (int r = 0; r < N; ++r) acc.push_back(lane_buf(in[r], count, sm.dt));
  std::vector<bool> folded(N, false);
  int step = 0;
  if (rr) {
    std::vector<Msg> ms;
    for (int i = 0; i < rr; ++i) {
      Msg m = sm.msg(2 * i + 1, 2 * i, count, true, sm.e_in, "fold", 0, 0);
      m.pieces.push_back({&acc[2 * i + 1], 0, &acc[2 * i], 0, count});
      ms.push_back(std::move(m));
      sm.rw(count, {sm.e_in, sm.e_in, sm.e_acc});
      folded[2 * i] = true;
    }
    sm.run_step(step++, ms);
  }
  std::vector<std::pair<int, int>> seg(P, {0, P});  // chunk run [c0, c1) of each virtual rank
  auto elems = [&](int c0, int c1) {
    return std::make_pair(part_range(c0, count, P, es).first, part_range(c1 - 1, count, P, es).second);
  };
  auto chunk_list = [](int c0, int c1) {
    std::vector<int64_t> v;
    for (int c = c0; c < c1; ++c) v.push_back(c);
    return v;
  };
  for (int k = 0; k < L; ++k) {
    std::vector<Msg> ms;
    std::vector<std::pair<int, int>> nseg = seg;
    for (int v = 0; v < P; ++v) {
      const int w = v ^ (1 << k);
      const auto [c0, c1] = seg[v];
      const int h = (c1 - c0) / 2;
      std::pair<int, int> keep, give;
      if (((v >> k) & 1) == 0) {
        keep = {c0, c0 + h};
        give = {c0 + h, c1};
      } else {
        keep = {c0 + h, c1};
        give = {c0, c0 + h};
      }
      nseg[v] = keep;
      const auto [lo, hi] = elems(give.first, give.second);
      const int wire = (k > 0 || folded[real[v]]) ? sm.e_acc : sm.e_in;
      Msg m = sm.msg(real[v], real[w], hi - lo, true, wire, "halving", lo, lo, chunk_list(give.first, give.second));
      m.pieces.push_back({&acc[real[v]], lo, &acc[real[w]], lo, hi - lo});
      ms.push_back(std::move(m));
      const int own = (k > 0 || folded[real[w]]) ? sm.e_acc : sm.e_in;
      sm.rw(hi - lo, {own, wire, k == L - 1 ? sm.e_out : sm.e_acc});
    }
    sm.run_step(step++, ms);
    seg = nseg;
  }
  for (int j = 0; j < L; ++j) {
    const int d = 1 << (L - 1 - j);
    std::vector<Msg> ms;
    std::vector<std::pair<int, int>> nseg = seg;
    for (int v = 0; v < P; ++v) {
      const int w = v ^ d;
      const auto [c0, c1] = seg[v];
      const auto [lo, hi] = elems(c0, c1);
      Msg m = sm.msg(real[v], real[w], hi - lo, false, sm.e_out, "doubling", lo, lo, chunk_list(c0, c1));
      m.pieces.push_back({&acc[real[v]], lo, &acc[real[w]], lo, hi - lo});
      ms.push_back(std::move(m));
      sm.rw(hi - lo, {sm.e_out, sm.e_out});
      nseg[v] = {std::min(c0, seg[w].first), std::max(c1, seg[w].second)};
    }
    sm.run_step(step++, ms);
    seg = nseg;
  }
  if (rr) {
    std::vector<Msg> ms;
    for (int i = 0; i < rr; ++i) {
      Msg m = sm.msg(2 * i, 2 * i + 1, count, false, sm.e_out, "unfold", 0, 0);
      m.pieces.push_back({&acc[2 * i], 0, &acc[2 * i + 1], 0, count});
      ms.push_back(std::move(m));
      sm.rw(count, {sm.e_out, sm.e_out});
    }
    sm.run_step(step++, ms);
  }
  narrow_all(sm, acc, count, o);
}

// Double Binary Tree ([Latency-formula page] section "Double Binary Tree",
// eq. model-algo-dbt-ar).  Tree A is the [hccl article]'s heap on the ranks
// (section "Tree算法"): node i has children 2i+1 and 2i+2, and adds its left
// child's subtree sum, then its right child's, to its own value,
// S(i) = (x_i + S(2i+1)) + S(2i+2).  Tree B (reading: the page asks for two
// trees with different parent/child relations but does not build them) is
// the mirror, heap node i on rank N-1-i, so every rank is interior in at most
// one tree.  Tree A carries part 0 of a two-way split of the buffer, tree B
// part 1.  Reduce one tree level per step, deepest first; then broadcast one
// level per step, root first; the root broadcasts its sum (the article's
// code broadcasts its receive buffer, which at the root holds the last
// child's data: a garble; reading taken).
int heap_level(int i) {
  int d = 0;
  while ((2 << d) <= i + 1) ++d;
  return d;
}

void allreduce_dbt(Sim& sm, const In& in, int64_t count, Out& o) {
  const int N = static_cast<int>(in.size());
  if (N == 1) return self_copy(sm, in, count, o);
  const int es = esize_of(sm.dt);
  std::vector<Buf> acc;
  for (int r = 0; r < N; ++r) acc.push_back(lane_buf(in[r], count, sm.dt));
  const int D = heap_level(N - 1);
  struct Tree {
    const char* name;
    bool mirror;
    int64_t lo, hi;
  };
  const auto a = part_range(0, count, 2, es), b = part_range(1, count, 2, es);
  const Tree trees[2] = {{"A", false, a.first, a.second}, {"B", true, b.first, b.second}};
  auto rank_of = [&](const Tree& t, int i) { return t.mirror ? N - 1 - i : i; };
  int step = 0;
  for (int t = 0; t < D; ++t) {
    const int depth = D - 1 - t;
    std::vector<Msg> ms;
    for (const Tree& tr : trees) {
      const std::string phase = std::string("reduce") + tr.name;
      for (int i = 0; i < N; ++i) {
        if (heap_level(i) != depth) continue;
        std::vector<int> kids;
        for (int c : {2 * i + 1, 2 * i + 2})
          if (c < N) kids.push_back(c);
        if (kids.empty()) continue;
        const int v = rank_of(tr, i);
        std::vector<int> reads{sm.e_in};
        for (int c : kids) {
          const bool leaf = 2 * c + 1 >= N;
          const int wire = leaf ? sm.e_in : sm.e_acc;
          reads.push_back(wire);
          const int u = rank_of(tr, c);
          Msg m = sm.msg(u, v, tr.hi - tr.lo, true, wire, phase.c_str(), tr.lo, tr.lo);
          m.pieces.push_back({&acc[u], tr.lo, &acc[v], tr.lo, tr.hi - tr.lo});
          ms.push_back(std::move(m));
        }
        reads.push_back(i == 0 ? sm.e_out : sm.e_acc);
        sm.rw(tr.hi - tr.lo, reads);
      }
    }
    sm.run_step(step++, ms);
  }
  for (int t = 0; t < D; ++t) {
    const int depth = t + 1;
    std::vector<Msg> ms;
    for (const Tree& tr : trees) {
      const std::string phase = std::string("bcast") + tr.name;
      for (int i = 0; i < N; ++i) {
        if (heap_level(i) != depth) continue;
        const int u = rank_of(tr, (i - 1) / 2), v = rank_of(tr, i);
        Msg m = sm.msg(u, v, tr.hi - tr.lo, false, sm.e_out, phase.c_str(), tr.lo, tr.lo);
        m.pieces.push_back({&acc[u], tr.lo, &acc[v], tr.lo, tr.hi - tr.lo});
        ms.push_back(std::move(m));
        sm.rw(tr.hi - tr.lo, {sm.e_out, sm.e_out});
      }
    }
    sm.run_step(step++, ms);
  }
  narrow_all(sm, acc, count, o);
}

void allreduce(Sim& sm, const In& in, int64_t count, const std::string& algo, bool inplace, Out& o) {
  const int N = static_cast<int>(in.size());
  if (algo != "fused" && algo != "ring" && algo != "rhd" && algo != "dbt" && algo != "mesh" && algo != "ring_hop")
    throw Unsupported("allreduce/" + algo);
  if (N == 1 && inplace) {  // one rank, in place: the result is already there
    o.outputs.emplace_back(in[0], in[0] + count * sm.e_in);
    return;
  }
  if (algo == "fused") return allreduce_fused(sm, in, count, o);
  if (algo == "ring") return allreduce_ring(sm, in, count, o, false);
  if (algo == "ring_hop") return allreduce_ring(sm, in, count, o, true);
  if (algo == "rhd") return allreduce_rhd(sm, in, count, o);
  if (algo == "dbt") return allreduce_dbt(sm, in, count, o);
  return allreduce_mesh(sm, in, count, o);
}

// ---------------------------------------------------------------------------
// ReduceScatter and AllGather alone ([Latency-formula page] sections "Ring
// ReduceScatter" and "Ring AllGather", eqs. model-algo-ring-reducescatter,
// model-algo-ring-allgather)
// ---------------------------------------------------------------------------

// Each input holds N blocks of rc elements; rank r ends with block r of the
// reduction.  Ring (reading: block ownership is left open; rank r owns block
// r): the AllReduce ReduceScatter shifted by one block -- at step s rank r
// sends block (r - s - 1) mod N to r + 1, which adds it; block c is summed
// x_{c+1} + x_{c+2} + ... + x_{c+N}.
void reduce_scatter(Sim& sm, const In& in, int64_t total, const std::string& algo, Out& o) {
  const int N = static_cast<int>(in.size());
  if (total % N) throw BadArg("reduce_scatter: input length not a multiple of N");
  const int64_t rc = total / N;
  const int es = esize_of(sm.dt);
  const bool fl = lanes_are_float(sm.dt);
  if (algo == "fused") {
    for (int r = 0; r < N; ++r) {
      std::vector<Lane> acc = widen_buf(in[0] + r * rc * es, rc, sm.dt);
      for (int q = 1; q < N; ++q) {
        const std::vector<Lane> x = widen_buf(in[q] + r * rc * es, rc, sm.dt);
        combine_into(acc.data(), x.data(), rc, sm.op, fl);
      }
      for (int q = 0; q < N; ++q)
        if (q != r) sm.log.push_back(Record{0, q, r, rc, 1, es, r * rc, 0, "fused", {}});
      o.outputs.push_back(narrow_buf(acc.data(), rc, sm.dt));
      std::vector<int> sizes(N, sm.e_in);
      sizes.push_back(sm.e_out);
      sm.rw(rc, sizes);
    }
    return;
  }
  if (algo != "ring") throw Unsupported("reduce_scatter/" + algo);
  if (N == 1) {
    sm.rw(rc, {sm.e_in, sm.e_out});
    o.outputs.emplace_back(in[0], in[0] + total * es);
    return;
  }
  std::vector<Buf> acc;
  for (int r = 0; r < N; ++r) acc.push_back(lane_buf(in[r], total, sm.dt));
  for (int s = 0; s < N - 1; ++s) {
    std::vector<Msg> ms;
    for (int r = 0; r < N; ++r) {
      const int c = mod(r - s - 1, N);
      const int64_t lo = c * rc;
      const int dst = (r + 1) % N;
      const int wire = s == 0 ? sm.e_in : sm.e_acc;
      Msg m = sm.msg(r, dst, rc, true, wire, "rs", lo, lo, {c});
      m.pieces.push_back({&acc[r], lo, &acc[dst], lo, rc});
      ms.push_back(std::move(m));
      sm.rw(rc, {sm.e_in, wire, s == N - 2 ? sm.e_out : sm.e_acc});
    }
    sm.run_step(s, ms);
  }
  for (int r = 0; r < N; ++r) o.outputs.push_back(narrow_buf(acc[r].l.data() + r * rc, rc, sm.dt));
}

// Each rank contributes sc elements; every rank ends with all N blocks,
// block q from rank q.  Ring: each rank first places its own block (a local
// copy), then at step s rank r forwards block (r - s) mod N to r + 1.
void allgather(Sim& sm, const In& in, int64_t sc, const std::string& algo, Out& o) {
  const int N = static_cast<int>(in.size());
  const int es = esize_of(sm.dt);
  if (algo == "fused") {
    std::vector<uint8_t> all;
    for (int q = 0; q < N; ++q) all.insert(all.end(), in[q], in[q] + sc * es);
    for (int r = 0; r < N; ++r) o.outputs.push_back(all);
    for (int q = 0; q < N; ++q)
      for (int r = 0; r < N; ++r)
        if (q != r) sm.log.push_back(Record{0, q, r, sc, 0, sm.e_in, 0, q * sc, "fused", {}});
    sm.rw(sc * N, {sm.e_in});
    sm.rw(sc * N * N, {sm.e_out});
    return;
  }
  if (algo != "ring") throw Unsupported("allgather/" + algo);
  std::vector<Buf> out;
  for (int r = 0; r < N; ++r) {
    out.push_back(byte_buf(N * sc, es));
    std::memcpy(out[r].b.data() + r * sc * es, in[r], static_cast<size_t>(sc * es));
    sm.rw(sc, {sm.e_in, sm.e_out});
  }
  for (int s = 0; s < N - 1; ++s) {
    std::vector<Msg> ms;
    for (int r = 0; r < N; ++r) {
      const int c = mod(r - s, N);
      const int dst = (r + 1) % N;
      Msg m = sm.msg(r, dst, sc, false, sm.e_out, "ag", c * sc, c * sc, {c});
      m.pieces.push_back({&out[r], c * sc, &out[dst], c * sc, sc});
      ms.push_back(std::move(m));
      sm.rw(sc, {sm.e_out, sm.e_out});
    }
    sm.run_step(s, ms);
  }
  for (Buf& b : out) o.outputs.push_back(std::move(b.b));
}

// ---------------------------------------------------------------------------
// Broadcast, Scatter, Gather, Reduce ([Bcast/Scatter page]; [Latency-formula
// page] section "Broadcast / Reduce 怎么用 Tree 算法")
// ---------------------------------------------------------------------------

// Binomial distances, one per step: 2^(L-1), ..., 2, 1 with L = ceil(log2 N)
// ([Bcast/Scatter page] section "二叉树（Binomial Tree）" and its 8-node table:
// 0->4; 0->2, 4->6; 0->1, 2->3, 4->5, 6->7).  At distance d every relative
// rank v = (r - root) mod N with v mod 2d == 0 and v + d < N sends to v + d.
std::vector<int> binomial_distances(int N) {
  const int L = ceil_log2(N);
  std::vector<int> d;
  for (int s = 0; s < L; ++s) d.push_back(1 << (L - 1 - s));
  return d;
}

// Binomial Scatter steps: at distance d, relative rank v hands the chunks of
// relative ranks [v + d, min(v + 2d, N)) to v + d, so the steps move M/2,
// M/4, ... ([Bcast/Scatter page] section "二叉树 Scatter", its 8-node table).
// hold[r] holds chunk c at range(c); a message carries its chunks as pieces.
template <class Range>
int binomial_scatter_steps(Sim& sm, int N, int root, Range range, std::vector<Buf>& hold, int step0) {
  const std::vector<int> ds = binomial_distances(N);
  for (size_t s = 0; s < ds.size(); ++s) {
    const int d = ds[s];
    std::vector<Msg> ms;
    for (int v = 0; v < N; v += 2 * d) {
      if (v + d >= N) continue;
      const int src = (v + root) % N, dst = (v + d + root) % N;
      std::vector<int64_t> chunks;
      int64_t n = 0;
      for (int q = v + d; q < std::min(v + 2 * d, N); ++q) {
        const int c = (q + root) % N;
        chunks.push_back(c);
        const auto [lo, hi] = range(c);
        n += hi - lo;
      }
      Msg m = sm.msg(src, dst, n, false, sm.e_in, "scatter", -1, -1, chunks);
      for (int64_t c : chunks) {
        const auto [lo, hi] = range(static_cast<int>(c));
        m.pieces.push_back({&hold[src], lo, &hold[dst], lo, hi - lo});
      }
      ms.push_back(std::move(m));
      sm.rw(n, {sm.e_in, sm.e_out});
    }
    sm.run_step(step0 + static_cast<int>(s), ms);
  }
  return step0 + static_cast<int>(ds.size());
}

// B_i = A_root on every rank ([Bcast/Scatter page] eq. onetoall-bcast-semantic).
void broadcast(Sim& sm, const uint8_t* A, int N, int64_t count, int root, const std::string& algo, bool inplace,
               Out& o) {
  const int es = esize_of(sm.dt);
  if (algo == "fused") {
    for (int r = 0; r < N; ++r) o.outputs.emplace_back(A, A + count * es);
    for (int r = 0; r < N; ++r)
      if (r != root) sm.log.push_back(Record{0, root, r, count, 0, es, 0, 0, "fused", {}});
    const int ndst = inplace ? N - 1 : N;
    if (ndst) {
      std::vector<int> sizes{sm.e_in};
      sizes.insert(sizes.end(), ndst, sm.e_out);
      sm.rw(count, sizes);
    }
    return;
  }
  if (algo == "binomial") {
    // ceil(log2 N) steps; each holder sends the whole message to one new rank
    // per step ([Bcast/Scatter page] eq. binomial-bcast; [Latency-formula
    // page] eq. model-algo-bcast-tree)
    std::vector<Buf> have;
    for (int r = 0; r < N; ++r) have.push_back(r == root ? byte_copy(A, count, es) : byte_buf(count, es));
    if (!inplace) sm.rw(count, {sm.e_in, sm.e_out});
    const std::vector<int> ds = binomial_distances(N);
    for (size_t s = 0; s < ds.size(); ++s) {
      const int d = ds[s];
      std::vector<Msg> ms;
      for (int v = 0; v < N; v += 2 * d) {
        if (v + d >= N) continue;
        const int src = (v + root) % N, dst = (v + d + root) % N;
        Msg m = sm.msg(src, dst, count, false, sm.e_in, "bcast", 0, 0);
        m.pieces.push_back({&have[src], 0, &have[dst], 0, count});
        ms.push_back(std::move(m));
        sm.rw(count, {sm.e_out, sm.e_out});
      }
      sm.run_step(static_cast<int>(s), ms);
    }
    for (Buf& b : have) o.outputs.push_back(std::move(b.b));
    return;
  }
  if (algo == "scatter_allgather") {
    // a binomial Scatter of the message's N chunks, then a Ring AllGather
    // ([Bcast/Scatter page] section "Broadcast 与 Scatter 的关系")
    auto range = [&](int c) { return part_range(c, count, N, es); };
    std::vector<Buf> hold;
    for (int r = 0; r < N; ++r) hold.push_back(r == root ? byte_copy(A, count, es) : byte_buf(count, es));
    const auto rl = range(root);
    if (!inplace) sm.rw(rl.second - rl.first, {sm.e_in, sm.e_out});
    const int step = binomial_scatter_steps(sm, N, root, range, hold, 0);
    std::vector<Buf> out;
    for (int r = 0; r < N; ++r) {
      out.push_back(byte_buf(count, es));
      const auto [lo, hi] = range(r);
      std::memcpy(out[r].b.data() + lo * es, hold[r].b.data() + lo * es, static_cast<size_t>((hi - lo) * es));
    }
    if (inplace) std::memcpy(out[root].b.data(), A, static_cast<size_t>(count * es));
    for (int s = 0; s < N - 1; ++s) {
      std::vector<Msg> ms;
      for (int r = 0; r < N; ++r) {
        const int c = mod(r - s, N);
        const auto [lo, hi] = range(c);
        const int dst = (r + 1) % N;
        Msg m = sm.msg(r, dst, hi - lo, false, sm.e_out, "ag", lo, lo, {c});
        m.pieces.push_back({&out[r], lo, &out[dst], lo, hi - lo});
        ms.push_back(std::move(m));
        sm.rw(hi - lo, {sm.e_out, sm.e_out});
      }
      sm.run_step(step + s, ms);
    }
    for (Buf& b : out) o.outputs.push_back(std::move(b.b));
    return;
  }
  throw Unsupported("broadcast/" + algo);
}

// Chunked (pipelined) Broadcasts ([Bcast/Scatter page] sections "分块链式流水线"
// and "分块二叉树流水线", eqs. pipe-chain-bcast and pipe-tree-bcast): the
// message is cut into k chunks and chunk j takes the unpipelined route
// delayed by j steps (reading: the pages give only step counts and chunk
// sizes).  Chain: relative rank v forwards chunk j to v + 1 at step v + j,
// N + k - 2 steps.  Tree: chunk j takes binomial step s at step j + s,
// ceil(log2 N) + k - 1 steps.
void broadcast_pipelined(Sim& sm, const uint8_t* A, int N, int64_t count, int root, const std::string& algo, int k,
                         bool inplace, Out& o) {
  if (k < 1) throw BadArg("nchunks must be >= 1");
  const int es = esize_of(sm.dt);
  std::vector<Buf> have;
  for (int r = 0; r < N; ++r) have.push_back(r == root ? byte_copy(A, count, es) : byte_buf(count, es));
  if (!inplace) sm.rw(count, {sm.e_in, sm.e_out});
  const std::vector<int> ds = binomial_distances(N);
  int nsteps = 0;
  if (algo == "pipe_chain")
    nsteps = N > 1 ? N + k - 2 : 0;
  else if (algo == "pipe_tree")
    nsteps = N > 1 ? static_cast<int>(ds.size()) + k - 1 : 0;
  else
    throw Unsupported("broadcast/" + algo);
  for (int t = 0; t < nsteps; ++t) {
    std::vector<Msg> ms;
    for (int j = 0; j < k; ++j) {
      const auto [lo, hi] = part_range(j, count, k, es);
      std::vector<std::pair<int, int>> hops;
      if (algo == "pipe_chain") {
        if (t - j >= 0 && t - j < N - 1) hops.push_back({t - j, t - j + 1});
      } else {
        const int s = t - j;
        if (s >= 0 && s < static_cast<int>(ds.size())) {
          const int d = ds[s];
          for (int v = 0; v < N; v += 2 * d)
            if (v + d < N) hops.push_back({v, v + d});
        }
      }
      for (const auto& [v, w] : hops) {
        const int src = (v + root) % N, dst = (w + root) % N;
        Msg m = sm.msg(src, dst, hi - lo, false, sm.e_in, algo.c_str(), lo, lo, {j});
        m.pieces.push_back({&have[src], lo, &have[dst], lo, hi - lo});
        ms.push_back(std::move(m));
        sm.rw(hi - lo, {sm.e_out, sm.e_out});
      }
    }
    sm.run_step(t, ms);
  }
  for (Buf& b : have) o.outputs.push_back(std::move(b.b));
}

// The root holds [A_0, ..., A_{N-1}]; rank i receives A_i ([Bcast/Scatter
// page] eq. onetoall-scatter-semantic).
void scatter(Sim& sm, const uint8_t* A, int N, int64_t total, int root, const std::string& algo, Out& o) {
  if (total % N) throw BadArg("scatter: input length not a multiple of N");
  const int64_t rc = total / N;
  const int es = esize_of(sm.dt);
  if (algo == "fused") {
    for (int r = 0; r < N; ++r) o.outputs.emplace_back(A + r * rc * es, A + (r + 1) * rc * es);
    for (int r = 0; r < N; ++r)
      if (r != root) sm.log.push_back(Record{0, root, r, rc, 0, sm.e_in, r * rc, 0, "fused", {r}});
    sm.rw(rc * N, {sm.e_in, sm.e_out});
    return;
  }
  if (algo != "binomial") throw Unsupported("scatter/" + algo);
  auto range = [&](int c) { return std::make_pair(c * rc, (c + 1) * rc); };
  std::vector<Buf> hold;
  for (int r = 0; r < N; ++r) hold.push_back(r == root ? byte_copy(A, total, es) : byte_buf(total, es));
  sm.rw(rc, {sm.e_in, sm.e_out});  // the root's own block
  binomial_scatter_steps(sm, N, root, range, hold, 0);
  for (int r = 0; r < N; ++r)
    o.outputs.emplace_back(hold[r].b.begin() + r * rc * es, hold[r].b.begin() + (r + 1) * rc * es);
}

// The dual of Scatter ([Bcast/Scatter page] section "对偶性：Scatter 与
// Gather", eq. onetoall-gather-scatter-duality: reverse the data flow).
// binomial (reading): distances 1, 2, 4, ...; at distance d relative rank v
// with v mod 2d == d hands everything it holds -- the chunks of relative
// ranks [v, min(v + d, N)) -- to v - d.
void gather(Sim& sm, const In& in, int64_t rc, int root, const std::string& algo, Out& o) {
  const int N = static_cast<int>(in.size());
  const int es = esize_of(sm.dt);
  if (algo == "fused") {
    std::vector<uint8_t> all;
    for (int q = 0; q < N; ++q) all.insert(all.end(), in[q], in[q] + rc * es);
    for (int r = 0; r < N; ++r)
      if (r != root) sm.log.push_back(Record{0, r, root, rc, 0, sm.e_in, 0, r * rc, "fused", {r}});
    sm.rw(rc * N, {sm.e_in, sm.e_out});
    o.outputs.push_back(std::move(all));
    return;
  }
  if (algo != "binomial") throw Unsupported("gather/" + algo);
  std::vector<Buf> hold;
  for (int r = 0; r < N; ++r) {
    hold.push_back(byte_buf(N * rc, es));
    std::memcpy(hold[r].b.data() + r * rc * es, in[r], static_cast<size_t>(rc * es));
  }
  sm.rw(rc, {sm.e_in, sm.e_out});  // the root's own block
  const int L = ceil_log2(N);
  for (int s = 0; s < L; ++s) {
    const int d = 1 << s;
    std::vector<Msg> ms;
    for (int u = 0; u < N; u += 2 * d) {
      const int v = u + d;
      if (v >= N) continue;
      const int src = (v + root) % N, dst = (u + root) % N;
      std::vector<int64_t> chunks;
      for (int q = v; q < std::min(v + d, N); ++q) chunks.push_back((q + root) % N);
      const int64_t n = rc * static_cast<int64_t>(chunks.size());
      Msg m = sm.msg(src, dst, n, false, sm.e_in, "gather", -1, -1, chunks);
      for (int64_t c : chunks) m.pieces.push_back({&hold[src], c * rc, &hold[dst], c * rc, rc});
      ms.push_back(std::move(m));
      sm.rw(n, {sm.e_in, sm.e_out});
    }
    sm.run_step(s, ms);
  }
  o.outputs.push_back(std::move(hold[root].b));
}

// Reduce to one root ([Latency-formula page] section "Broadcast / Reduce 怎么用
// Tree 算法", eq. model-algo-reduce-tree: the Tree Broadcast run backwards).
// binomial (reading): distances 1, 2, 4, ...; at distance d relative rank u
// with u mod 2d == 0 adds the partial sum of u + d to its own, so the
// association is the balanced tree over adjacent relative ranks.  fused: rank
// order, as the fused AllReduce.
void reduce(Sim& sm, const In& in, int64_t count, int root, const std::string& algo, bool inplace, Out& o) {
  const int N = static_cast<int>(in.size());
  if (algo != "fused" && algo != "binomial") throw Unsupported("reduce/" + algo);
  if (N == 1) {
    if (!inplace) sm.rw(count, {sm.e_in, sm.e_out});
    o.outputs.emplace_back(in[0], in[0] + count * sm.e_in);
    return;
  }
  const bool fl = lanes_are_float(sm.dt);
  if (algo == "fused") {
    std::vector<Lane> acc = widen_buf(in[0], count, sm.dt);
    for (int q = 1; q < N; ++q) {
      const std::vector<Lane> x = widen_buf(in[q], count, sm.dt);
      combine_into(acc.data(), x.data(), count, sm.op, fl);
    }
    for (int q = 0; q < N; ++q)
      if (q != root) sm.log.push_back(Record{0, q, root, count, 1, sm.e_in, 0, 0, "fused", {}});
    std::vector<int> sizes(N, sm.e_in);
    sizes.push_back(sm.e_out);
    sm.rw(count, sizes);
    o.outputs.push_back(narrow_buf(acc.data(), count, sm.dt));
    return;
  }
  std::vector<Buf> acc;
  for (int r = 0; r < N; ++r) acc.push_back(lane_buf(in[r], count, sm.dt));
  std::vector<bool> partial(N, false);  // relative rank holds a partial sum
  const int L = ceil_log2(N);
  for (int s = 0; s < L; ++s) {
    const int d = 1 << s;
    std::vector<Msg> ms;
    for (int u = 0; u < N; u += 2 * d) {
      const int v = u + d;
      if (v >= N) continue;
      const int src = (v + root) % N, dst = (u + root) % N;
      const int wire = partial[v] ? sm.e_acc : sm.e_in;
      Msg m = sm.msg(src, dst, count, true, wire, "reduce", 0, 0);
      m.pieces.push_back({&acc[src], 0, &acc[dst], 0, count});
      ms.push_back(std::move(m));
      const bool last = u == 0 && s == L - 1;
      sm.rw(count, {partial[u] ? sm.e_acc : sm.e_in, wire, last ? sm.e_out : sm.e_acc});
      partial[u] = true;
    }
    sm.run_step(s, ms);
  }
  o.outputs.push_back(narrow_buf(acc[root].l.data(), count, sm.dt));
}

// ---------------------------------------------------------------------------
// AllToAll: with N blocks of B elements per buffer, out_j[block i] =
// in_i[block j] ([Latency-formula page] section "AllToAll 算法怎么选")
// ---------------------------------------------------------------------------
void alltoall(Sim& sm, const In& in, int64_t total, const std::string& algo, Out& o) {
  const int N = static_cast<int>(in.size());
  if (total % N) throw BadArg("alltoall: input length not a multiple of N");
  const int64_t B = total / N;
  const int es = esize_of(sm.dt);
  auto block_of = [&](int i, int j) { return in[i] + j * B * es; };
  if (algo == "fused") {
    for (int j = 0; j < N; ++j) {
      std::vector<uint8_t> out;
      for (int i = 0; i < N; ++i) out.insert(out.end(), block_of(i, j), block_of(i, j) + B * es);
      o.outputs.push_back(std::move(out));
    }
    for (int i = 0; i < N; ++i)
      for (int j = 0; j < N; ++j)
        if (i != j) sm.log.push_back(Record{0, i, j, B, 0, sm.e_in, j * B, i * B, "fused", {}});
    sm.rw(total * N, {sm.e_in, sm.e_out});
    return;
  }
  if (algo == "pairwise") {
    // [Latency-formula page] eq. model-algo-a2a-pairwise: in round k = 1 ..
    // N-1 rank i sends its block for rank (i + k) mod N there (reading: and so
    // receives from (i - k) mod N).  Round 0 is the local block.
    std::vector<Buf> src, out;
    for (int i = 0; i < N; ++i) {
      src.push_back(byte_copy(in[i], total, es));
      out.push_back(byte_buf(total, es));
      std::memcpy(out[i].b.data() + i * B * es, block_of(i, i), static_cast<size_t>(B * es));
      sm.rw(B, {sm.e_in, sm.e_out});
    }
    for (int k = 1; k < N; ++k) {
      std::vector<Msg> ms;
      for (int i = 0; i < N; ++i) {
        const int j = (i + k) % N;
        Msg m = sm.msg(i, j, B, false, sm.e_in, "round", j * B, i * B);
        m.pieces.push_back({&src[i], j * B, &out[j], i * B, B});
        ms.push_back(std::move(m));
        sm.rw(B, {sm.e_in, sm.e_out});
      }
      sm.run_step(k, ms);
    }
    sm.local_steps = N > 1 ? 1 : 0;
    for (Buf& b : out) o.outputs.push_back(std::move(b.b));
    return;
  }
  if (algo == "ring") {
    // [Latency-formula page] eq. model-algo-a2a-ring: N-1 rounds between ring
    // neighbours.  Reading: store and forward -- in round k every rank passes
    // to i + 1 every block it holds that is not addressed to itself, nearest
    // destination first; a block from s for d travels (d - s) mod N hops.
    std::vector<Buf> out;
    for (int i = 0; i < N; ++i) {
      out.push_back(byte_buf(total, es));
      std::memcpy(out[i].b.data() + i * B * es, block_of(i, i), static_cast<size_t>(B * es));
      sm.rw(B, {sm.e_in, sm.e_out});
    }
    // blocks in transit at each rank: (source, destination, data); one slot
    // per (source, destination) in each rank's transit buffer
    struct Held {
      int s, d;
    };
    std::vector<std::vector<Held>> held(N);
    std::vector<Buf> tr, nx;
    for (int i = 0; i < N; ++i) {
      tr.push_back(byte_buf(static_cast<int64_t>(N) * N * B, es));
      nx.push_back(byte_buf(static_cast<int64_t>(N) * N * B, es));
      for (int d = 0; d < N; ++d)
        if (d != i) {
          held[i].push_back({i, d});
          std::memcpy(tr[i].b.data() + (static_cast<int64_t>(i) * N + d) * B * es, block_of(i, d),
                      static_cast<size_t>(B * es));
        }
    }
    for (int k = 1; k < N; ++k) {
      std::vector<Msg> ms;
      std::vector<std::vector<Held>> next(N);
      for (int i = 0; i < N; ++i) {
        const int dst = (i + 1) % N;
        std::vector<Held> keys = held[i];
        std::stable_sort(keys.begin(), keys.end(),
                         [&](const Held& a, const Held& b) { return mod(a.d - dst, N) < mod(b.d - dst, N); });
        std::vector<int64_t> chunks;
        for (const Held& h : keys) chunks.push_back(static_cast<int64_t>(h.s) * N + h.d);
        Msg m = sm.msg(i, dst, static_cast<int64_t>(keys.size()) * B, false, sm.e_in, "ring", -1, -1, chunks);
        for (const Held& h : keys) {
          const int64_t slot = (static_cast<int64_t>(h.s) * N + h.d) * B;
          if (h.d == dst)
            m.pieces.push_back({&tr[i], slot, &out[dst], h.s * B, B});
          else {
            m.pieces.push_back({&tr[i], slot, &nx[dst], slot, B});
            next[dst].push_back(h);
          }
        }
        ms.push_back(std::move(m));
        sm.rw(static_cast<int64_t>(keys.size()) * B, {sm.e_in, sm.e_out});
      }
      sm.run_step(k, ms);
      std::swap(tr, nx);
      held = next;
    }
    sm.local_steps = N > 1 ? 1 : 0;
    for (Buf& b : out) o.outputs.push_back(std::move(b.b));
    return;
  }
  if (algo == "bruck") {
    // [Latency-formula page] eq. model-algo-a2a-bruck; the algorithm of Bruck
    // et al. (1997) that the page cites.  Rank i rotates its blocks so that
    // position p holds its block for rank (i + p) mod N; in round k it sends
    // every position p with bit k set to rank (i + 2^k) mod N, which stores it
    // at the same position; after all rounds position p of rank j holds the
    // block from rank (j - p) mod N, which a final inverse rotation puts at
    // block (j - p) mod N.  Bytes: every round rewrites each rank's working
    // buffer once, the rotations folded into the first and last rounds.
    const int L = ceil_log2(N);
    if (N == 1) {
      sm.rw(B, {sm.e_in, sm.e_out});
      o.outputs.emplace_back(in[0], in[0] + total * es);
      return;
    }
    std::vector<Buf> W;
    for (int i = 0; i < N; ++i) {
      W.push_back(byte_buf(total, es));
      for (int p = 0; p < N; ++p)
        std::memcpy(W[i].b.data() + p * B * es, block_of(i, (i + p) % N), static_cast<size_t>(B * es));
    }
    for (int k = 0; k < L; ++k) {
      std::vector<Msg> ms;
      for (int i = 0; i < N; ++i) {
        const int dst = (i + (1 << k)) % N;
        std::vector<int64_t> pos;
        for (int p = 0; p < N; ++p)
          if ((p >> k) & 1) pos.push_back(p);
        Msg m = sm.msg(i, dst, static_cast<int64_t>(pos.size()) * B, false, sm.e_in, "round", -1, -1, pos);
        for (int64_t p : pos) m.pieces.push_back({&W[i], p * B, &W[dst], p * B, B});
        ms.push_back(std::move(m));
      }
      sm.run_step(k, ms);
      sm.rw(static_cast<int64_t>(N) * N * B, {sm.e_in, sm.e_out});
    }
    for (int j = 0; j < N; ++j) {
      std::vector<uint8_t> out;
      for (int i = 0; i < N; ++i) {
        const int p = mod(j - i, N);
        out.insert(out.end(), W[j].b.begin() + p * B * es, W[j].b.begin() + (p + 1) * B * es);
      }
      o.outputs.push_back(std::move(out));
    }
    return;
  }
  throw Unsupported("alltoall/" + algo);
}

// ---------------------------------------------------------------------------
// closed-form association trees ([hccl article] "Mesh算法", "Ring算法",
// "Tree算法"; [Latency-formula page] "Recursive Halving-Doubling", "Double
// Binary Tree"), stated directly from the step descriptions and evaluated
// per element; independent of the simulation above
// ---------------------------------------------------------------------------
// A tree over ranks as a node list: leaf nodes name a rank, inner nodes two
// earlier nodes (left operand, right operand); the last node is the root.
struct Node {
  int rank;  // >= 0: a leaf
  int a, b;
};
using Tree = std::vector<Node>;

int t_leaf(Tree& t, int rank) {
  t.push_back({rank, -1, -1});
  return static_cast<int>(t.size()) - 1;
}
int t_join(Tree& t, int a, int b) {
  t.push_back({-1, a, b});
  return static_cast<int>(t.size()) - 1;
}

// ((r0 + r1) + r2) + ...
Tree fold_tree(const std::vector<int>& ranks) {
  Tree t;
  int acc = t_leaf(t, ranks[0]);
  for (size_t i = 1; i < ranks.size(); ++i) acc = t_join(t, acc, t_leaf(t, ranks[i]));
  return t;
}

// Recursive halving pairs adjacent participants first (distance 1, then 2,
// 4, ...), so P participants form a balanced tree in their order.  A
// participant that absorbed a folded-in partner contributes (x_2i + x_2i+1).
int balanced(Tree& t, const std::vector<int>& leaves, size_t lo, size_t hi) {
  if (hi - lo == 1) return leaves[lo];
  const size_t mid = lo + (hi - lo) / 2;
  const int a = balanced(t, leaves, lo, mid);
  const int b = balanced(t, leaves, mid, hi);
  return t_join(t, a, b);
}
Tree halving_tree(int N) {
  int P = 1;
  while (2 * P <= N) P *= 2;
  const int extra = N - P;  // ranks 0..2*extra-1 pair off first: 2i+1 into 2i
  Tree t;
  std::vector<int> leaves;
  for (int i = 0; i < extra; ++i) leaves.push_back(t_join(t, t_leaf(t, 2 * i), t_leaf(t, 2 * i + 1)));
  for (int r = 2 * extra; r < N; ++r) leaves.push_back(t_leaf(t, r));
  balanced(t, leaves, 0, leaves.size());
  return t;
}

// heap node h on rank rank_of(h): S(h) = (x + S(2h+1)) + S(2h+2)
int heap_sum(Tree& t, int h, int N, bool mirror) {
  int acc = t_leaf(t, mirror ? N - 1 - h : h);
  for (int c : {2 * h + 1, 2 * h + 2})
    if (c < N) acc = t_join(t, acc, heap_sum(t, c, N, mirror));
  return acc;
}
Tree heap_tree(int N, bool mirror) {
  Tree t;
  heap_sum(t, 0, N, mirror);
  return t;
}

// Evaluate tree t on the lanes of element i of every rank; with round_hop
// every inner value is rounded to the data type (a schedule that stores its
// partials in the data type).
Lane eval_tree(const Tree& t, const std::vector<const uint8_t*>& vals, int64_t i, int dt, int op, bool round_hop,
               std::vector<Lane>& tmp) {
  tmp.resize(t.size());
  const int es = esize_of(dt);
  const bool fl = lanes_are_float(dt);
  for (size_t k = 0; k < t.size(); ++k) {
    const Node& n = t[k];
    if (n.rank >= 0) {
      tmp[k] = widen_elem(vals[n.rank] + i * es, dt);
    } else {
      Lane v = combine1(tmp[n.a], tmp[n.b], op, fl);
      if (round_hop) {
        uint8_t b[4];
        narrow_elem(v, dt, b);
        v = widen_elem(b, dt);
      }
      tmp[k] = v;
    }
  }
  return tmp.back();
}

void copy_err(const std::string& m, char* err, int errlen) {
  if (err && errlen > 0) std::snprintf(err, static_cast<size_t>(errlen), "%s", m.c_str());
}

}  // namespace

struct vo_result {
  Out out;
  std::vector<Record> log;
  int64_t hbm = 0;
  int local_steps = 0;
};

extern "C" {

int vo_run(const char* coll_c, const char* algo_c, int N, const void* const* inputs, int64_t n_in, int dtype, int op,
           int root, int inplace, int nchunks, vo_result** out, char* err, int errlen) {
  try {
    if (!coll_c || !algo_c || !out) throw BadArg("null argument");
    if (N < 1) throw BadArg("nranks must be >= 1");
    if (dtype < 0 || dtype > 3) throw BadArg("unknown dtype");
    if (op < 0 || op > 2) throw BadArg("unknown op");
    if (n_in < 0) throw BadArg("negative count");
    const std::string coll(coll_c), algo(algo_c);
    const bool rooted_in = coll == "broadcast" || coll == "scatter";
    const int nin = rooted_in ? 1 : N;
    In in;
    for (int r = 0; r < nin; ++r) {
      if (!inputs || (!inputs[r] && n_in > 0)) throw BadArg("null input");
      in.push_back(static_cast<const uint8_t*>(inputs[r]));
    }
    if ((rooted_in || coll == "gather" || coll == "reduce") && (root < 0 || root >= N))
      throw BadArg("root outside [0, N)");
    Sim sm(dtype, op);
    auto res = new vo_result;
    try {
      if (coll == "allreduce")
        allreduce(sm, in, n_in, algo, inplace != 0, res->out);
      else if (coll == "reduce_scatter")
        reduce_scatter(sm, in, n_in, algo, res->out);
      else if (coll == "allgather")
        allgather(sm, in, n_in, algo, res->out);
      else if (coll == "broadcast") {
        if (algo == "pipe_chain" || algo == "pipe_tree")
          broadcast_pipelined(sm, in[0], N, n_in, root, algo, nchunks, inplace != 0, res->out);
        else
          broadcast(sm, in[0], N, n_in, root, algo, inplace != 0, res->out);
      } else if (coll == "scatter")
        scatter(sm, in[0], N, n_in, root, algo, res->out);
      else if (coll == "gather")
        gather(sm, in, n_in, root, algo, res->out);
      else if (coll == "reduce")
        reduce(sm, in, n_in, root, algo, inplace != 0, res->out);
      else if (coll == "alltoall")
        alltoall(sm, in, n_in, algo, res->out);
      else
        throw BadArg("unknown collective " + coll);
    } catch (...) {
      delete res;
      throw;
    }
    res->log = std::move(sm.log);
    res->hbm = sm.hbm;
    res->local_steps = sm.local_steps;
    *out = res;
    return 0;
  } catch (const Unsupported& e) {
    copy_err(e.what(), err, errlen);
    return 1;
  } catch (const std::exception& e) {
    copy_err(e.what(), err, errlen);
    return 2;
  }
}

int vo_noutputs(const vo_result* r) { return static_cast<int>(r->out.outputs.size()); }
int64_t vo_output_elems(const vo_result* r, int i) { return static_cast<int64_t>(r->out.outputs[i].size()); }
void vo_output_copy(const vo_result* r, int i, void* dst) {
  const auto& v = r->out.outputs[i];
  if (!v.empty()) std::memcpy(dst, v.data(), v.size());
}
int64_t vo_hbm_bytes(const vo_result* r) { return r->hbm; }
int vo_local_steps(const vo_result* r) { return r->local_steps; }
int64_t vo_nrecords(const vo_result* r) { return static_cast<int64_t>(r->log.size()); }
void vo_records(const vo_result* r, int64_t* f) {
  for (const Record& x : r->log) {
    const int64_t v[9] = {x.step, x.src, x.dst, x.n, x.reduce, x.esize, x.src_off, x.dst_off,
                          static_cast<int64_t>(x.chunks.size())};
    std::memcpy(f, v, sizeof(v));
    f += 9;
  }
}
int64_t vo_nchunks_total(const vo_result* r) {
  int64_t n = 0;
  for (const Record& x : r->log) n += static_cast<int64_t>(x.chunks.size());
  return n;
}
void vo_record_chunks(const vo_result* r, int64_t* c) {
  for (const Record& x : r->log)
    for (int64_t v : x.chunks) *c++ = v;
}
const char* vo_record_phase(const vo_result* r, int64_t i) { return r->log[static_cast<size_t>(i)].phase.c_str(); }
void vo_free(vo_result* r) { delete r; }

void vo_set_fault(int kind, int step) {
  g_fault_kind = kind;
  g_fault_step = step;
}

int vo_allreduce_at(const void* const* values, int N, const char* algo_c, int64_t count, int dtype,
                    const int64_t* idx, int64_t nidx, int op, void* out, char* err, int errlen) {
  try {
    if (N < 1 || !values || !algo_c || (nidx > 0 && (!idx || !out))) throw BadArg("bad argument");
    if (dtype < 0 || dtype > 3 || op < 0 || op > 2) throw BadArg("unknown dtype or op");
    const std::string algo(algo_c);
    const int es = esize_of(dtype);
    for (int64_t i = 0; i < nidx; ++i)
      if (idx[i] < 0 || idx[i] >= count) throw BadArg("index outside the buffer");
    std::vector<const uint8_t*> vals;
    for (int r = 0; r < N; ++r) vals.push_back(static_cast<const uint8_t*>(values[r]));
    // group key -> tree: ring: the element's chunk; dbt: its half; else one tree
    std::vector<Tree> trees;
    std::vector<int> which(static_cast<size_t>(std::max<int64_t>(nidx, 0)));
    bool hop = false;
    if (algo == "fused" || algo == "mesh") {
      std::vector<int> ranks;
      for (int r = 0; r < N; ++r) ranks.push_back(r);
      trees.push_back(fold_tree(ranks));
    } else if (algo == "ring" || algo == "ring_hop") {
      // chunk c of element e, then x_c + x_{c+1} + ... + x_{c+N-1}
      hop = algo == "ring_hop";
      for (int c = 0; c < N; ++c) {
        std::vector<int> ranks;
        for (int j = 0; j < N; ++j) ranks.push_back((c + j) % N);
        trees.push_back(fold_tree(ranks));
      }
      const int64_t align = 16 / es;
      int64_t ce = count > 0 ? (count + N - 1) / N : 0;
      ce = (ce + align - 1) / align * align;
      for (int64_t i = 0; i < nidx; ++i) which[i] = static_cast<int>(idx[i] / ce);
    } else if (algo == "rhd") {
      trees.push_back(halving_tree(N));
    } else if (algo == "dbt") {
      // the first part of a two-way split on tree A, the rest on tree B
      trees.push_back(heap_tree(N, false));
      trees.push_back(heap_tree(N, true));
      const int64_t align = 16 / es;
      int64_t half = count > 0 ? (count + 1) / 2 : 0;
      half = std::min((half + align - 1) / align * align, count);
      for (int64_t i = 0; i < nidx; ++i) which[i] = idx[i] < half ? 0 : 1;
    } else {
      throw Unsupported("allreduce/" + algo);
    }
    std::vector<Lane> tmp;
    uint8_t* o = static_cast<uint8_t*>(out);
    for (int64_t i = 0; i < nidx; ++i) {
      const Lane v = eval_tree(trees[which[i]], vals, i, dtype, op, hop, tmp);
      narrow_elem(v, dtype, o + i * es);
    }
    return 0;
  } catch (const Unsupported& e) {
    copy_err(e.what(), err, errlen);
    return 1;
  } catch (const std::exception& e) {
    copy_err(e.what(), err, errlen);
    return 2;
  }
}

int vo_reduce_scatter_at(const void* const* values, int N, const char* algo_c, int64_t rc, int dtype,
                         const int64_t* idx, int64_t nidx, int op, void* out, char* err, int errlen) {
  try {
    if (N < 1 || !values || !algo_c || (nidx > 0 && (!idx || !out))) throw BadArg("bad argument");
    if (dtype < 0 || dtype > 3 || op < 0 || op > 2) throw BadArg("unknown dtype or op");
    const std::string algo(algo_c);
    const int es = esize_of(dtype);
    std::vector<const uint8_t*> vals;
    for (int r = 0; r < N; ++r) vals.push_back(static_cast<const uint8_t*>(values[r]));
    std::vector<Tree> trees;
    const bool ring = algo == "ring";
    if (algo == "fused") {
      std::vector<int> ranks;
      for (int r = 0; r < N; ++r) ranks.push_back(r);
      trees.push_back(fold_tree(ranks));
    } else if (ring) {
      // block c (on rank c): x_{c+1} + x_{c+2} + ... + x_{c+N}
      for (int c = 0; c < N; ++c) {
        std::vector<int> ranks;
        for (int j = 1; j <= N; ++j) ranks.push_back((c + j) % N);
        trees.push_back(fold_tree(ranks));
      }
    } else {
      throw Unsupported("reduce_scatter/" + algo);
    }
    std::vector<Lane> tmp;
    uint8_t* o = static_cast<uint8_t*>(out);
    for (int64_t i = 0; i < nidx; ++i) {
      if (idx[i] < 0 || idx[i] >= rc * N) throw BadArg("index outside the buffer");
      const Tree& t = trees[ring ? static_cast<size_t>(idx[i] / rc) : 0];
      narrow_elem(eval_tree(t, vals, i, dtype, op, false, tmp), dtype, o + i * es);
    }
    return 0;
  } catch (const Unsupported& e) {
    copy_err(e.what(), err, errlen);
    return 1;
  } catch (const std::exception& e) {
    copy_err(e.what(), err, errlen);
    return 2;
  }
}

void vo_bf16_from_f32(const float* x, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = narrow_bf16(bits_of(x[i]));
}
void vo_f32_from_bf16(const uint16_t* x, float* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = float_of(widen_bf16(x[i]));
}
void vo_f16_from_f32(const float* x, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = narrow_f16(bits_of(x[i]));
}
void vo_f32_from_f16(const uint16_t* x, float* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = float_of(widen_f16(x[i]));
}

}  // extern "C"
