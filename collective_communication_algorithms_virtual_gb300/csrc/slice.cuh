// Device code of the sliced form (sm_103a): a whole fp32 / int32 AllReduce
// plan in one launch over the GPU, each thread carrying its 16-byte group of
// every rank buffer through every step.  Uses the plan description and the
// helpers of kernels.cuh.
#pragma once

#include "kernels.cuh"

namespace vc {
namespace dev {

// -- element-sliced plans ---------------------------------------------------------
// A plan whose every operation maps element e of each source to element e of
// each destination, at the same byte offset in every rank buffer (the fp32 /
// int32 AllReduce schedules: Ring, RHD, DBT, Mesh), can run with its step
// barrier kept per element instead of per launch.  The buffers are cut into
// slices of U * BT 16-byte groups; thread i of a block owns groups i, i + BT,
// ... of its slice -- the same bytes of every rank's send and receive buffer
// -- for the whole launch.  The thread walks the plan's steps in order and, in each,
// applies every operation that covers its group: sources combined in the
// plan's order, the result stored to every destination.  Whatever a step
// reads at a position was written there by an earlier step, by this same
// thread, so program order is the step barrier and no thread reads what
// another wrote (loads go to L2 with .cg; a thread's own earlier store to the
// address is ordered before them).  Steps, operations, operands and every
// element's association are the plan's; only positions far apart run out of
// step with each other, as when a ring is pipelined in slices.  The
// operation's first element is its operands' common offset / 4; the element
// after its last group whole is handled by the owner of that group.
template <int RMODE, int OP>
__device__ __forceinline__ uint4 cmb4(uint4 a, uint4 w) {
  if constexpr (RMODE == kF32) {
    a.x = __float_as_uint(cmb<OP>(__uint_as_float(a.x), __uint_as_float(w.x)));
    a.y = __float_as_uint(cmb<OP>(__uint_as_float(a.y), __uint_as_float(w.y)));
    a.z = __float_as_uint(cmb<OP>(__uint_as_float(a.z), __uint_as_float(w.z)));
    a.w = __float_as_uint(cmb<OP>(__uint_as_float(a.w), __uint_as_float(w.w)));
  } else {
    a.x = cmbi<OP>(a.x, w.x);
    a.y = cmbi<OP>(a.y, w.y);
    a.z = cmbi<OP>(a.z, w.z);
    a.w = cmbi<OP>(a.w, w.w);
  }
  return a;
}

// Shared memory of a block: the plan description (16-byte words), the call's
// buffer bases, then two tables the block derives once: each operation's
// element range [e0, e1) and each operand's address (base + offset).  Every
// buffer of a sliced call holds fewer than 2^29 elements (checked on the
// host), so element and byte offsets within it fit 32 bits.
__host__ __device__ constexpr size_t slice_smem_bytes(uint32_t words, uint32_t nbases, uint32_t nops,
                                                      uint32_t nrefs) {
  return size_t(words) * 16 + size_t(nbases) * 8 + size_t(nops) * 8 + size_t(nrefs) * 8;
}

// BT threads a block; U groups a thread, BT apart (slices of U * BT groups);
// the loads of a thread's groups in a step are issued together.
template <int RMODE, int OP, int U, int BT>
__global__ void __launch_bounds__(BT) slice_kernel(const __grid_constant__ PlanParams p) {
  static_assert(RMODE == kF32 || RMODE == kI32, "sliced plans are fp32 or int32");
  extern __shared__ uint4 sm[];
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (uint32_t i = threadIdx.x; i < p.words; i += BT) sm[i] = ld16(p.plan + i);
  const void** sbase = reinterpret_cast<const void**>(sm + p.words);
  for (uint32_t i = threadIdx.x; i < p.nbases; i += BT) sbase[i] = p.base[i];
  __syncthreads();
  const PlanHeader h = *reinterpret_cast<const PlanHeader*>(sm);
  const PlanStep* steps = reinterpret_cast<const PlanStep*>(sm + 1);
  const OpDesc* ops = reinterpret_cast<const OpDesc*>(sm + 1 + h.nsteps);
  const OperandRef* refs = reinterpret_cast<const OperandRef*>(ops + h.nops);
  int2* rng = reinterpret_cast<int2*>(sbase + p.nbases);             // per operation: e0, e1
  char** addr = reinterpret_cast<char**>(rng + h.nops);              // per operand: its address
  for (uint32_t i = threadIdx.x; i < h.nops; i += BT) {
    const int e0 = static_cast<int>(refs[ops[i].p0].off >> 2);
    rng[i] = make_int2(e0, e0 + static_cast<int>(ops[i].n));
  }
  for (uint32_t i = threadIdx.x; i < h.nrefs; i += BT)
    addr[i] = static_cast<char*>(const_cast<void*>(sbase[refs[i].base])) + refs[i].off;
  __syncthreads();
  asm volatile("griddepcontrol.wait;" ::: "memory");
  constexpr int kSlice = U * BT;
  const int groups = static_cast<int>(p.groups);
  const int nslices = (groups + kSlice - 1) / kSlice;
  for (int sl = blockIdx.x; sl < nslices; sl += gridDim.x) {
    const int g0 = sl * kSlice + static_cast<int>(threadIdx.x);  // this thread's groups: g0 + u * BT
    if (g0 >= groups) break;
    const int ea = g0 * 4, eb = (g0 + (U - 1) * BT) * 4 + 4;     // elements its groups span
    for (uint32_t s = 0; s < h.nsteps; ++s) {
      const PlanStep st = steps[s];
      // Each thread looks for the next operation of the step that covers one
      // of its groups, then applies it.  Threads of a warp can be in different
      // operations (small chunks); searching first and applying after keeps
      // the warp together, so their loads go out at once instead of one
      // operation's chain after another.
      // The step's operations are listed by position (ascending first
      // element), so none after one that starts past this thread's groups
      // can cover them.  Stopping there measured faster where a thread
      // carries 4 or more groups (4 MiB per rank: ring 24.5 -> 20.4 us) and
      // slower where it carries 1 or 2 (up to 2 MiB: ring 10.7 -> 13.4 us at
      // 4 KiB), so only the former stop early.
      uint32_t k = st.op0;
      const uint32_t kend = st.op0 + st.nops;
      for (;;) {
        int2 r = make_int2(0, 0);
        for (; k < kend; ++k) {
          r = rng[k];
          if constexpr (U >= 4) {
            if (r.x >= eb) {
              k = kend;
              break;
            }
          }
          if (ea < r.y && eb > r.x) break;  // covers one of the groups
        }
        if (k >= kend) break;
        const OpDesc& o = ops[k++];
        char* const* P = addr + o.p0;  // sources, then destinations
        const int ns = o.ns, nd = o.nd;
        bool whole[U];
        int off[U];  // bytes into every operand
        uint4 acc[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int e = (g0 + u * BT) * 4;
          whole[u] = e >= r.x && e + 4 <= r.y;
          off[u] = (e - r.x) * 4;
          if (whole[u]) acc[u] = ld16_cg(P[0] + off[u]);
        }
        if (st.mode != kCopy) {
          for (int q = 1; q < ns; ++q) {
            const char* src = P[q];
            uint4 w[U];
#pragma unroll
            for (int u = 0; u < U; ++u)
              if (whole[u]) w[u] = ld16_cg(src + off[u]);
#pragma unroll
            for (int u = 0; u < U; ++u)
              if (whole[u]) acc[u] = cmb4<RMODE, OP>(acc[u], w[u]);
          }
        }
        for (int d = 0; d < nd; ++d) {
          char* dp = P[ns + d];
#pragma unroll
          for (int u = 0; u < U; ++u)
            if (whole[u]) st16_wb(dp + off[u], acc[u]);
        }
        // the operation ends inside a group: its last elements one by one
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int e = (g0 + u * BT) * 4;
          if (whole[u] || e < r.x || e >= r.y) continue;
          for (int x = e; x < r.y; ++x) {
            const int xo = (x - r.x) * 4;
            uint32_t a = ld32<true>(P[0] + xo);
            if (st.mode != kCopy)
              for (int q = 1; q < ns; ++q) {
                const uint32_t w = ld32<true>(P[q] + xo);
                if constexpr (RMODE == kF32) a = __float_as_uint(cmb<OP>(__uint_as_float(a), __uint_as_float(w)));
                else a = cmbi<OP>(a, w);
              }
            for (int d = 0; d < nd; ++d) *reinterpret_cast<uint32_t*>(P[ns + d] + xo) = a;
          }
        }
      }
    }
  }
}

}  // namespace dev
}  // namespace vc
