// Device code of the sliced form (sm_103a): a whole AllReduce plan in one
// launch over the GPU, each thread carrying its 16-byte group of every rank
// buffer through every step.  Uses the plan description and the helpers of
// kernels.cuh.
#pragma once

#include "kernels.cuh"

namespace vc {
namespace dev {

// -- element-sliced plans ---------------------------------------------------------
// A plan whose every operation maps element position e of each source to
// position e of each destination, each buffer holding position e at one fixed
// place (the AllReduce schedules: Ring, RHD, DBT, Mesh), can run with its
// step barrier kept per element instead of per launch.  The buffers are cut
// into slices of U * BT groups of 16 bytes of the data type (4 fp32 / int32
// elements, 8 bf16 / fp16 ones); thread i of a block owns groups i, i + BT,
// ... of its slice -- the same positions of every rank's send and receive
// buffer, and of the fp32 partial sums that 16-bit plans keep in scratch --
// for the whole launch.  The thread walks the plan's steps in order and, in
// each, applies every operation that covers its group: sources combined in
// the plan's order, the result stored to every destination.  Whatever a step
// reads at a position was written there by an earlier step, by this same
// thread, so program order is the step barrier and no thread reads what
// another wrote (a thread's own earlier store to an address is ordered before
// its later loads of it, whatever the cache path; see the loads below).
// Steps, operations, operands and every
// element's association are the plan's; only positions far apart run out of
// step with each other, as when a ring is pipelined in slices.  The host
// checks that every position has one place in each buffer; the positions
// after an operation's last whole group are handled, one by one, by the
// owner of that group.
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

// Loads of the sliced form.  A thread reads what it stored earlier in the
// launch -- receive buffers and scratch, which the host checks are written at
// every position before they are read -- through L1 (.ca): its own store is
// visible to its own later load, and the line is near.  Measured on 8 ranks:
// fp32 4 KiB - 4 MiB per rank 0.4-1.6 us faster than through L2 alone (.cg).
// Send buffers hold data from before the launch, which another grid may have
// written while this one waited on it, so they are read at L2 (.cg), never
// from an L1 line of an overlapping grid.  Their operand addresses carry a
// tag in bit 0 (addresses are 16-byte aligned).
__device__ __forceinline__ uint4 ld16_ca(const void* p) {
  uint4 v;
  asm volatile("ld.global.ca.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}
__device__ __forceinline__ W8 ldv32_ca(const void* p) {
  W8 v;
  asm volatile("ld.global.ca.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]), "=r"(v.w[5]), "=r"(v.w[6]),
                 "=r"(v.w[7])
               : "l"(p)
               : "memory");
  return v;
}
// An operand's address with its tag removed; *pre: a send buffer.
__device__ __forceinline__ const char* slice_src(const char* tagged, bool* pre) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(tagged);
  *pre = (a & 1) != 0;
  return reinterpret_cast<const char*>(a & ~uintptr_t(1));
}
// Loads the whole groups of one operand (offsets in bytes).  With several
// groups a thread the cache path is chosen once for all of them (measured on
// 8 ranks, 512 KiB - 4 MiB per rank: 0.2-1 us faster than choosing per load);
// with one, per load (up to 256 KiB: 0.1-0.5 us faster than a branch).
template <int U>
__device__ __forceinline__ void ld16_groups(uint4 (&v)[U], const char* p, bool pre, const bool (&whole)[U],
                                            const int (&off)[U]) {
  if constexpr (U == 1) {
    if (whole[0]) v[0] = pre ? ld16_cg(p + off[0]) : ld16_ca(p + off[0]);
  } else if (pre) {
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (whole[u]) v[u] = ld16_cg(p + off[u]);
  } else {
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (whole[u]) v[u] = ld16_ca(p + off[u]);
  }
}
// The address table entry of operand i (tagged when it is a send buffer,
// base index below N).
__device__ __forceinline__ char* slice_addr(const OperandRef& r, const void* const* sbase, uint32_t nranks) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(sbase[r.base]) + static_cast<uintptr_t>(r.off);
  return reinterpret_cast<char*>(a | (r.base < nranks ? 1 : 0));
}

// Shared memory of a block: the plan description (16-byte words), the call's
// buffer bases, then two tables: each operation's element range [e0, e1)
// and each operand's address (base + offset).  (Kernels that take the ranges
// the host lists read them as part of the description: the same size, up to
// 8 bytes.)  Every buffer
// of a sliced call holds fewer than 2^29 elements (checked on the host), so
// element and byte offsets within it fit 32 bits.
__host__ __device__ constexpr size_t slice_smem_bytes(uint32_t words, uint32_t nbases, uint32_t nops,
                                                      uint32_t nrefs) {
  return size_t(words) * 16 + size_t(nbases) * 8 + size_t(nops) * 8 + size_t(nrefs) * 8;
}

// BT threads a block; U groups a thread, BT apart (slices of U * BT groups);
// the loads of a thread's groups in a step are issued together.  HR: the
// operations' element ranges are the ones the host lists after the
// description; otherwise each is derived from its first operand's offset,
// which the host allows only where every operand region has origin 0 (the
// AllReduce schedules, the Broadcasts).
template <int RMODE, int OP, int U, int BT, bool HR>
__global__ void __launch_bounds__(BT) slice_kernel(const __grid_constant__ PlanParams p) {
  static_assert(RMODE == kF32 || RMODE == kI32, "4-byte sliced plans are fp32 or int32");
  extern __shared__ uint4 sm[];
  for (uint32_t i = threadIdx.x; i < p.words; i += BT) sm[i] = ld16(p.plan + i);
  const void** sbase = reinterpret_cast<const void**>(sm + p.words);
  for (uint32_t i = threadIdx.x; i < p.nbases; i += BT) sbase[i] = p.base[i];
  __syncthreads();
  const PlanHeader h = *reinterpret_cast<const PlanHeader*>(sm);
  const PlanStep* steps = reinterpret_cast<const PlanStep*>(sm + 1);
  const OpDesc* ops = reinterpret_cast<const OpDesc*>(sm + 1 + h.nsteps);
  const OperandRef* refs = reinterpret_cast<const OperandRef*>(ops + h.nops);
  int2* rng;    // per operation: e0, e1
  char** addr;  // per operand: its address
  if constexpr (HR) {
    rng = const_cast<int2*>(reinterpret_cast<const int2*>(refs + h.nrefs));
    addr = reinterpret_cast<char**>(const_cast<void**>(sbase + p.nbases));
  } else {
    rng = reinterpret_cast<int2*>(sbase + p.nbases);
    addr = reinterpret_cast<char**>(rng + h.nops);
    // absolute positions: every operand in a send or receive buffer at byte 4 e0
    for (uint32_t i = threadIdx.x; i < h.nops; i += BT) {
      const int e0 = static_cast<int>(refs[ops[i].p0].off >> 2);
      rng[i] = make_int2(e0, e0 + static_cast<int>(ops[i].n));
    }
  }
  for (uint32_t i = threadIdx.x; i < h.nrefs; i += BT)
    addr[i] = slice_addr(refs[i], sbase, (p.nbases - 1) / 2);
  __syncthreads();
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // at most one grid ahead (plan_kernel)
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
        bool pre0;
        const char* const s0 = slice_src(P[0], &pre0);
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int e = (g0 + u * BT) * 4;
          whole[u] = e >= r.x && e + 4 <= r.y;
          off[u] = (e - r.x) * 4;
        }
        ld16_groups<U>(acc, s0, pre0, whole, off);
        if (st.mode != kCopy) {
          for (int q = 1; q < ns; ++q) {
            bool pre;
            const char* const src = slice_src(P[q], &pre);
            uint4 w[U];
            ld16_groups<U>(w, src, pre, whole, off);
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
            uint32_t a = ld32<true>(s0 + xo);
            if (st.mode != kCopy)
              for (int q = 1; q < ns; ++q) {
                bool pre;
                const uint32_t w = ld32<true>(slice_src(P[q], &pre) + xo);
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

// 16-bit plans: copies the description -- here with the operations' element
// ranges after the operand table, which the host lists because fp32 partials
// in scratch sit at other offsets than the data -- and the bases to shared
// memory, and derives each operand's address (after the bases).
template <int BT>
__device__ __forceinline__ void slice_prologue(const PlanParams& p, uint4* sm) {
  for (uint32_t i = threadIdx.x; i < p.words; i += BT) sm[i] = ld16(p.plan + i);
  const void** sbase = reinterpret_cast<const void**>(sm + p.words);
  for (uint32_t i = threadIdx.x; i < p.nbases; i += BT) sbase[i] = p.base[i];
  __syncthreads();
  const PlanHeader h = *reinterpret_cast<const PlanHeader*>(sm);
  const OpDesc* ops = reinterpret_cast<const OpDesc*>(sm + 1 + h.nsteps);
  const OperandRef* refs = reinterpret_cast<const OperandRef*>(ops + h.nops);
  char** addr = reinterpret_cast<char**>(const_cast<void**>(sbase + p.nbases));
  for (uint32_t i = threadIdx.x; i < h.nrefs; i += BT)
    addr[i] = slice_addr(refs[i], sbase, (p.nbases - 1) / 2);
  __syncthreads();
}

// The search of slice_kernel as a function: the next operation of the step,
// from k on, that covers one of the groups spanning elements [ea, eb);
// returns its index, or kend.
template <int U>
__device__ __forceinline__ uint32_t slice_next_op(const int2* rng, uint32_t k, uint32_t kend, int ea, int eb,
                                                  int2* r) {
  for (; k < kend; ++k) {
    *r = rng[k];
    if constexpr (U >= 4) {
      if (r->x >= eb) return kend;
    }
    if (ea < r->y && eb > r->x) return k;  // covers one of the groups
  }
  return kend;
}

// bf16 / fp16 plans: a group is 8 elements, 16 bytes of a buffer in the data
// type or 32 of an fp32 partial-sum buffer (smask / dmask bit set).  Every
// source is widened to fp32 (exact) and combined in the plan's order; a
// destination in the data type takes the fp32 result rounded to nearest even,
// once, exactly as the per-step kernels do.  Copies move the data type.
// Against the form of slice_kernel (ranges derived in the block, the search
// inline), this one measured 0.2-1 us faster on 16-bit plans (8 ranks, 4 KiB
// to 4 MiB per rank); on 4-byte plans it measured up to 0.5 us slower at up
// to 256 KiB, so each keeps the form that measured faster for it.
template <bool F16, int OP, int U, int BT>
__global__ void __launch_bounds__(BT) slice16_kernel(const __grid_constant__ PlanParams p) {
  extern __shared__ uint4 sm[];
  slice_prologue<BT>(p, sm);
  const PlanHeader h = *reinterpret_cast<const PlanHeader*>(sm);
  const PlanStep* steps = reinterpret_cast<const PlanStep*>(sm + 1);
  const OpDesc* ops = reinterpret_cast<const OpDesc*>(sm + 1 + h.nsteps);
  const int2* rng = reinterpret_cast<const int2*>(reinterpret_cast<const OperandRef*>(ops + h.nops) + h.nrefs);
  char* const* addr = reinterpret_cast<char* const*>(reinterpret_cast<void* const*>(sm + p.words) + p.nbases);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");  // at most one grid ahead (plan_kernel)
  constexpr int kSlice = U * BT;
  const int groups = static_cast<int>(p.groups);
  const int nslices = (groups + kSlice - 1) / kSlice;
  for (int sl = blockIdx.x; sl < nslices; sl += gridDim.x) {
    const int g0 = sl * kSlice + static_cast<int>(threadIdx.x);  // this thread's groups: g0 + u * BT
    if (g0 >= groups) break;
    const int ea = g0 * 8, eb = (g0 + (U - 1) * BT) * 8 + 8;     // elements its groups span
    for (uint32_t s = 0; s < h.nsteps; ++s) {
      const PlanStep st = steps[s];
      const uint32_t kend = st.op0 + st.nops;
      int2 r = make_int2(0, 0);
      for (uint32_t k = slice_next_op<U>(rng, st.op0, kend, ea, eb, &r); k < kend;
           k = slice_next_op<U>(rng, k + 1, kend, ea, eb, &r)) {
        const OpDesc& o = ops[k];
        char* const* P = addr + o.p0;  // sources, then destinations
        const int ns = o.ns, nd = o.nd;
        bool whole[U];
        int rel[U];  // elements into every operand
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int e = (g0 + u * BT) * 8;
          whole[u] = e >= r.x && e + 8 <= r.y;
          rel[u] = e - r.x;
        }
        bool pre0;
        const char* const s0 = slice_src(P[0], &pre0);
        int off2[U];  // bytes into the operands in the data type
#pragma unroll
        for (int u = 0; u < U; ++u) off2[u] = rel[u] * 2;
        if (st.mode == kCopy) {
          uint4 v[U];
          ld16_groups<U>(v, s0, pre0, whole, off2);
          for (int d = 0; d < nd; ++d) {
            char* dp = P[ns + d];
#pragma unroll
            for (int u = 0; u < U; ++u)
              if (whole[u]) st16_wb(dp + rel[u] * 2, v[u]);
          }
        } else {
          float acc[U][8];
          for (int q = 0; q < ns; ++q) {
            bool pre;
            const char* const src = slice_src(P[q], &pre);
            if ((o.smask >> q) & 1) {  // fp32 partials (scratch): one 32-byte access a group
              W8 a[U];
#pragma unroll
              for (int u = 0; u < U; ++u)
                if (whole[u]) a[u] = ldv32_ca(src + rel[u] * 4);
#pragma unroll
              for (int u = 0; u < U; ++u)
                if (whole[u]) {
                  float f[8];
#pragma unroll
                  for (int i = 0; i < 8; ++i) f[i] = __uint_as_float(a[u].w[i]);
                  accumulate8<OP>(acc[u], f, q == 0);
                }
            } else {
              uint4 w[U];
              ld16_groups<U>(w, src, pre, whole, off2);
#pragma unroll
              for (int u = 0; u < U; ++u)
                if (whole[u]) {
                  float f[8];
                  widen8<F16>(w[u], f);
                  accumulate8<OP>(acc[u], f, q == 0);
                }
            }
          }
          for (int d = 0; d < nd; ++d) {
            char* dp = P[ns + d];
            if ((o.dmask >> d) & 1) {
#pragma unroll
              for (int u = 0; u < U; ++u)
                if (whole[u]) {
                  W8 w;
#pragma unroll
                  for (int i = 0; i < 8; ++i) w.w[i] = __float_as_uint(acc[u][i]);
                  stv32<true>(dp + rel[u] * 4, w);
                }
            } else {
#pragma unroll
              for (int u = 0; u < U; ++u)
                if (whole[u])
                  st16_wb(dp + rel[u] * 2, make_uint4(pack2<F16>(acc[u][0], acc[u][1]), pack2<F16>(acc[u][2], acc[u][3]),
                                                      pack2<F16>(acc[u][4], acc[u][5]), pack2<F16>(acc[u][6], acc[u][7])));
            }
          }
        }
        // the operation ends inside a group: its last elements one by one
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int e = (g0 + u * BT) * 8;
          if (whole[u] || e < r.x || e >= r.y) continue;
          for (int x = e; x < r.y; ++x) {
            const int xr = x - r.x;
            if (st.mode == kCopy) {
              const uint16_t v = ld16b<true>(s0 + xr * 2);
              for (int d = 0; d < nd; ++d) *reinterpret_cast<uint16_t*>(P[ns + d] + xr * 2) = v;
              continue;
            }
            float a = 0.f;
            for (int q = 0; q < ns; ++q) {
              bool pre;
              const char* const src = slice_src(P[q], &pre);
              const float v = ((o.smask >> q) & 1) ? __uint_as_float(ld32<true>(src + xr * 4))
                                                    : widen1<F16>(ld16b<true>(src + xr * 2));
              a = q == 0 ? v : cmb<OP>(a, v);
            }
            for (int d = 0; d < nd; ++d) {
              if ((o.dmask >> d) & 1) *reinterpret_cast<float*>(P[ns + d] + xr * 4) = a;
              else *reinterpret_cast<uint16_t*>(P[ns + d] + xr * 2) = narrow1<F16>(a);
            }
          }
        }
      }
    }
  }
}

}  // namespace dev
}  // namespace vc
