// Device code of the virtual-rank collectives (sm_103a): the step kernel
// that runs one step of a plan per launch, and the plan kernel that runs a
// whole small plan in one launch of one thread-block cluster.
//
// A plan (plan.h) is a list of steps; a step is a list of independent
// operations.  A persistent grid walks "tiles" (groups of 16-byte groups of
// one run of one operation); each thread loads its groups from every source
// with 128-bit loads, combines them in the order the plan lists them (fp32
// registers; 16-bit types widened exactly; int32 wrapping), and stores the
// result to every destination with 128-bit stores.  Copy steps move raw
// 16-byte groups; a copy to several destinations stages the tile in shared
// memory and writes it out with bulk asynchronous (TMA) stores.  Distinct
// elements are the only thing split across threads, so each element's
// association is exactly the plan's.
//
// Nothing here is a dense contraction: the kernels are HBM-streaming and use
// no tensor cores.  No kernel spins on a flag: between steps the order is
// stream order (one launch per step) or a hardware cluster barrier that
// every block of the cluster meets once per step (one launch per plan).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <type_traits>

#include "vc.h"

namespace vc {
namespace dev {


constexpr int kThreads = 256;
constexpr int kUnroll = 4;           // 16-byte groups per thread per tile (vector path)
constexpr int kScalarPerThread = 4;  // elements per thread per tile (element path)
constexpr int kTileGroups = kThreads * kUnroll;
constexpr int kTileElems = kThreads * kScalarPerThread;
// A tile is worked by kThreads threads: a whole block of the per-step kernel,
// or one of the sub-blocks of a one-launch plan's larger blocks.
__device__ __forceinline__ int lane() { return static_cast<int>(threadIdx.x) & (kThreads - 1); }

// Kernel modes: copy; fp32 / int32 reductions; 16-bit float reductions whose
// sources mix the data type with fp32 partial sums, or are all of the data
// type ("P": pure), for bf16 and fp16.
enum : int { kCopy = 0, kF32 = 1, kI32 = 2, kBF16 = 3, kBF16P = 4, kF16 = 5, kF16P = 6 };
// Reduction ops.  max / min keep the first operand unless the second is
// larger / smaller or the first is NaN (so NaN is passed over while a number
// is present and of +0 / -0 the first seen is kept); int32 compares signed.
enum : int { kSum = 0, kMax = 1, kMin = 2 };

struct __align__(16) OpDesc {
  int64_t n;        // elements per run (copy: elements of esz bytes)
  int64_t nb;       // runs
  int64_t sstride;  // bytes between runs, sources
  int64_t dstride;  // bytes between runs, destinations
  int64_t groups;   // vector path: 16-byte groups per run (fp32 bf16-mode operands: 32 bytes)
  uint64_t smask;   // bf16 mode: bit s set -> source s is stored as fp32
  uint64_t dmask;   // bf16 mode: bit d set -> destination d is stored as fp32
  uint32_t tile0;   // first tile of this operation within the launch
  uint32_t tpr;     // tiles per run
  uint16_t p0;      // first pointer (sources, then destinations)
  uint8_t ns, nd;
  uint8_t vec;      // 1: vector path
  uint8_t esz;      // copy: element size in bytes
  uint8_t upt;      // vector path: groups per thread in one tile (1, 2, 4; 8 in the bulk-copy pipeline)
  uint8_t keep;     // the next step reads the results: store them with the default L2 policy
};

template <int OPS, int PTRS>
struct __align__(16) LaunchParams {
  uint32_t nops;    // operations in use
  uint32_t ntiles;  // tiles of the launch
  uint32_t rev;     // walk the launch's tiles last to first (the previous step's latest writes first)
  uint32_t late;    // 1: the grid leaves room on the GPU; let the next grid in only after the wait
  OpDesc op[OPS];
  const void* ptr[PTRS];
};
using SmallParams = LaunchParams<16, 64>;
using LargeParams = LaunchParams<128, 512>;
static_assert(sizeof(OpDesc) % 16 == 0, "plan descriptions are copied in 16-byte words");

// -- memory access --------------------------------------------------------------
// Per-step launches (COH = false): the sources of a launch are never written
// during it, so loads take the non-coherent path and skip L1; stores are
// streaming (evict-first in L2).  One-launch plans (COH = true) read in a step
// what other blocks of the cluster wrote in an earlier one: loads go to L2
// (.cg, never a stale L1 line) after the step barrier, stores are plain.
__device__ __forceinline__ uint4 ld16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint4 ld16_cg(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}
// Streaming store (evict-first in L2): measured 2-3% faster than a plain
// store on the write-heavy steps (fused AllReduce / AllToAll, tree levels)
// and neutral on the ring steps whose outputs the next step reads.
__device__ __forceinline__ void st16(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void st16_wb(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
// 32-byte accesses (one fp32 partial group: 8 floats) as single 256-bit
// loads and stores, so that a warp's access is one contiguous kilobyte.  As
// two 16-byte accesses 32 bytes apart, each instruction used half of every
// sector it touched and the second fetched the same sectors from L2 again.
// A 256-bit access must be 32-byte aligned; the vector path only guarantees
// 16, so callers check the operand's base (group offsets are multiples of
// 32) and otherwise take two 16-byte accesses.
struct __align__(32) W8 {
  uint32_t w[8];
};
template <bool COH>
__device__ __forceinline__ W8 ldv32(const void* p) {
  W8 v;
  if constexpr (COH)
    asm volatile("ld.global.cg.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]), "=r"(v.w[5]), "=r"(v.w[6]),
                   "=r"(v.w[7])
                 : "l"(p)
                 : "memory");
  else
    asm volatile("ld.global.nc.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]), "=r"(v.w[5]), "=r"(v.w[6]),
                   "=r"(v.w[7])
                 : "l"(p));
  return v;
}
template <bool COH, bool KEEP = false>
__device__ __forceinline__ void stv32(void* p, const W8& v) {
  if constexpr (COH || KEEP)
    asm volatile("st.global.v8.u32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]),
                 "r"(v.w[3]), "r"(v.w[4]), "r"(v.w[5]), "r"(v.w[6]), "r"(v.w[7])
                 : "memory");
  else
    asm volatile("st.global.cs.v8.u32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]),
                 "r"(v.w[3]), "r"(v.w[4]), "r"(v.w[5]), "r"(v.w[6]), "r"(v.w[7])
                 : "memory");
}
template <bool COH>
__device__ __forceinline__ uint4 ldv(const void* p) {
  if constexpr (COH) return ld16_cg(p);
  else return ld16(p);
}
// Loads whose lines are not read again (the mixed 16-bit kernel's sources:
// each partial is consumed once) marked evict-first in L2, leaving room for
// the results a step keeps for the next one.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t pol;
  asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
template <bool COH>
__device__ __forceinline__ uint4 ldv_once(const void* p) {
  if constexpr (COH) return ld16_cg(p);
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(l2_evict_first()));
  return v;
}
template <bool COH>
__device__ __forceinline__ W8 ldv32_once(const void* p) {
  if constexpr (COH) return ldv32<COH>(p);
  W8 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8], %9;"
               : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]), "=r"(v.w[5]), "=r"(v.w[6]),
                 "=r"(v.w[7])
               : "l"(p), "l"(l2_evict_first()));
  return v;
}
// KEEP: results the next step reads take the default L2 policy instead of
// streaming (evict-first), so that they can still be in L2 when it does.
template <bool COH, bool KEEP = false>
__device__ __forceinline__ void stv(void* p, uint4 v) {
  if constexpr (COH || KEEP) st16_wb(p, v);
  else st16(p, v);
}
// Runs f with the store policy as a compile-time flag, chosen once per tile
// (a uniform branch).  Chosen per store, as a store pair under a predicate,
// each store took two issue slots: the fused AllReduce (eight destinations)
// measured 0.5 us slower at 1 KiB per rank and 12% at 4 MiB.  Coherent
// kernels have one form.
// FAN: kernels with the bulk-store path run the fused one-step calls, whose
// results nothing reads again: one streaming form (with both, that kernel's
// schedule changed and the fused AllReduce measured 2% slower).
template <bool COH, bool FAN = false, class F>
__device__ __forceinline__ void keep_stores(bool keep, F&& f) {
  if constexpr (COH || FAN) f(std::false_type{});
  else if (keep) f(std::true_type{});
  else f(std::false_type{});
}

template <int OP>
__device__ __forceinline__ float cmb(float a, float b) {
  if constexpr (OP == kSum) return __fadd_rn(a, b);
  else if constexpr (OP == kMax) return (b > a || a != a) ? b : a;
  else return (b < a || a != a) ? b : a;
}
template <int OP>
__device__ __forceinline__ uint32_t cmbi(uint32_t a, uint32_t b) {
  if constexpr (OP == kSum) return a + b;  // two's-complement wrap-around
  else if constexpr (OP == kMax) return static_cast<int32_t>(b) > static_cast<int32_t>(a) ? b : a;
  else return static_cast<int32_t>(b) < static_cast<int32_t>(a) ? b : a;
}

// 16-bit float formats: widening is exact; narrowing rounds to nearest even.
template <bool F16>
__device__ __forceinline__ float widen1(uint16_t h) {
  if constexpr (F16) return __half2float(__ushort_as_half(h));
  else return __uint_as_float(static_cast<uint32_t>(h) << 16);
}
template <bool F16>
__device__ __forceinline__ uint16_t narrow1(float x) {
  if constexpr (F16) return __half_as_ushort(__float2half_rn(x));
  else return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}
template <bool F16>
__device__ __forceinline__ void widen2(uint32_t w, float* f) {
  if constexpr (F16) {
    const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&w));
    f[0] = v.x;
    f[1] = v.y;
  } else {
    f[0] = __uint_as_float(w << 16);
    f[1] = __uint_as_float(w & 0xffff0000u);
  }
}
template <bool F16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {  // lo in the low half
  if constexpr (F16) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}
template <bool F16>
__device__ __forceinline__ void widen8(uint4 v, float* f) {
  widen2<F16>(v.x, f);
  widen2<F16>(v.y, f + 2);
  widen2<F16>(v.z, f + 4);
  widen2<F16>(v.w, f + 6);
}

// -- vector path -------------------------------------------------------------
// A tile is the groups [gbeg, gend) of one run of one operation; thread i
// takes groups gbeg + i, gbeg + i + kThreads, ...  `ptr` is the operation's
// pointer table (sources, then destinations): an array of addresses, or a
// table that forms them from buffer bases.
//
// Fan-out copies (one source, several destinations: fused AllGather and
// Broadcast): the tile is loaded into shared memory and thread 0 issues one
// bulk asynchronous store per destination (cp.async.bulk, the TMA engine),
// which writes it out in 16 KB bursts.  Measured 3-4.5% faster than eight
// 128-bit stores per thread on the fused Broadcast and AllGather at 8 x 256
// MiB; single-destination copies keep the plain path (no gain there).  The
// next tile's loads are issued before waiting until the previous tile's bulk
// stores have read the buffer (wait_group.read), so the two overlap; the
// kernel waits for the stores' completion before it exits.
template <class PT>
__device__ __forceinline__ void tile_copy_fanout(const OpDesc& o, const PT& ptr, int64_t run, int64_t gbeg,
                                                 int64_t gend) {
  __shared__ alignas(128) uint4 stage[kTileGroups];
  const int ng = static_cast<int>(gend - gbeg);
  const char* s = static_cast<const char*>(ptr[0]) + run * o.sstride;
  uint4 v[kUnroll];
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const int64_t g = gbeg + u * kThreads + threadIdx.x;
    if (g < gend) v[u] = ld16(s + g * 16);
  }
  if (threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
  __syncthreads();
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const int64_t g = gbeg + u * kThreads + threadIdx.x;
    if (g < gend) stage[g - gbeg] = v[u];
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // make the tile visible to the bulk copies
  __syncthreads();
  if (threadIdx.x == 0 && ng > 0) {
    const uint32_t saddr = static_cast<uint32_t>(__cvta_generic_to_shared(stage));
    for (int d = 0; d < o.nd; ++d) {
      char* dp = static_cast<char*>(const_cast<void*>(ptr[o.ns + d])) + run * o.dstride + gbeg * 16;
      asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dp), "r"(saddr), "r"(ng * 16)
                   : "memory");
    }
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  }
}

// FAN: the kernel has the bulk-store path for multi-destination operations
// compiled in (copies here, fp32 / int32 sums in tile_4b); without it the
// copy kernel needs 32 registers instead of 44 and keeps 8 blocks per SM
// resident instead of 5.
template <bool COH, bool FAN, class PT>
__device__ __forceinline__ void tile_copy(const OpDesc& o, const PT& ptr, int64_t run, int64_t gbeg, int64_t gend) {
  const bool keep = o.keep;  // read before the loads (see tile_4b)
  if constexpr (FAN && !COH) {
    if (o.nd > 1) {
      tile_copy_fanout(o, ptr, run, gbeg, gend);
      return;
    }
  }
  // slot u of this thread is group gbeg + lane() + u * kThreads; it
  // exists while u * kThreads < lim
  const int lim = static_cast<int>(gend - gbeg) - lane();
  const int64_t off = (gbeg + lane()) * 16;
  const char* s = static_cast<const char*>(ptr[0]) + run * o.sstride + off;
  uint4 v[kUnroll];
#pragma unroll
  for (int u = 0; u < kUnroll; ++u)
    if (u * kThreads < lim) v[u] = ldv<COH>(s + u * kThreads * 16);
  keep_stores<COH, FAN>(keep, [&](auto k) {
    for (int d = 0; d < o.nd; ++d) {
      char* dp = static_cast<char*>(const_cast<void*>(ptr[o.ns + d])) + run * o.dstride + off;
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        if (u * kThreads < lim) stv<COH, decltype(k)::value>(dp + u * kThreads * 16, v[u]);
    }
  });
}

// fp32 and int32: 4 elements per 16-byte group.  The loads of SB sources are
// issued together, then combined one after another in source order, so an
// operation with many sources waits for ceil(ns / SB) memory round trips
// rather than ns.  SB = 1 (fewest registers, most resident blocks) for
// launches that fill the GPU; SB = 4 for small launches of many-source
// operations, where the round trips are the time: measured on 8 ranks, the
// fused AllReduce of 1 MiB per rank takes 3.6 instead of 5.6 us, while at
// 256 MiB per rank SB = 4 is 2% slower than SB = 1.
// Writes a finished fp32 / int32 tile to every destination of a
// multi-destination operation (fused AllReduce) with one bulk asynchronous
// store per destination from shared memory, as the fan-out copies do, instead
// of one 128-bit store per thread per destination: 8 ranks, 256 MiB per rank,
// 658 -> 650 us.  The stores carry an L2 evict-first policy (as the streaming
// stores of the other paths): without it the written lines linger in L2 and
// the next kernel pays for writing them back (the next launch measured 3%
// slower).
template <class PT>
__device__ __forceinline__ void store_tile_bulk(const OpDesc& o, const PT& ptr, int64_t run, int64_t gbeg,
                                                int64_t gend, const uint4 (&acc)[kUnroll]) {
  __shared__ alignas(128) uint4 rstage[kTileGroups];
  const int ng = static_cast<int>(gend - gbeg);
  const int lim = ng - lane();
  if (threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
  __syncthreads();
#pragma unroll
  for (int u = 0; u < kUnroll; ++u)
    if (u * kThreads < lim) rstage[lane() + u * kThreads] = acc[u];
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();
  if (threadIdx.x == 0 && ng > 0) {
    const uint32_t saddr = static_cast<uint32_t>(__cvta_generic_to_shared(rstage));
    uint64_t pol;
    if (o.keep) asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
    else asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    for (int d = 0; d < o.nd; ++d) {
      char* dp = static_cast<char*>(const_cast<void*>(ptr[o.ns + d])) + run * o.dstride + gbeg * 16;
      asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(dp), "r"(saddr), "r"(ng * 16), "l"(pol)
                   : "memory");
    }
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  }
}

template <bool FLOAT, int OP, bool COH, int SB, bool FAN, class PT>
__device__ __forceinline__ void tile_4b(const OpDesc& o, const PT& ptr, int64_t run, int64_t gbeg, int64_t gend) {
  // The store policy is read before the loads: read at the stores, it kept the
  // operation's parameter address live across them (44 -> 56 registers).  The
  // kernel with the bulk-store path reads it at the stores (hoisted there, it
  // reshaped that kernel's schedule and the fused AllReduce measured 1.4% slower).
  [[maybe_unused]] const bool keep_early = FAN ? false : static_cast<bool>(o.keep);
  const int lim = static_cast<int>(gend - gbeg) - lane();  // slots as in tile_copy
  const int64_t soff = run * o.sstride + (gbeg + lane()) * 16;
  // The first source loads straight into the accumulator (a register copy of
  // a pending load would stall until it arrives, holding back the next loads).
  uint4 acc[kUnroll];
  {
    const char* s = static_cast<const char*>(ptr[0]) + soff;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (u * kThreads < lim) acc[u] = ldv<COH>(s + u * kThreads * 16);
  }
  for (int k0 = 1; k0 < o.ns; k0 += SB) {
    uint4 v[SB][kUnroll];
#pragma unroll
    for (int j = 0; j < SB; ++j) {
      if (k0 + j < o.ns) {
        const char* s = static_cast<const char*>(ptr[k0 + j]) + soff;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
          if (u * kThreads < lim) v[j][u] = ldv<COH>(s + u * kThreads * 16);
      }
    }
#pragma unroll
    for (int j = 0; j < SB; ++j) {
      if (k0 + j < o.ns) {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          if (u * kThreads < lim) {
            const uint4 w = v[j][u];
            if constexpr (FLOAT) {
              acc[u].x = __float_as_uint(cmb<OP>(__uint_as_float(acc[u].x), __uint_as_float(w.x)));
              acc[u].y = __float_as_uint(cmb<OP>(__uint_as_float(acc[u].y), __uint_as_float(w.y)));
              acc[u].z = __float_as_uint(cmb<OP>(__uint_as_float(acc[u].z), __uint_as_float(w.z)));
              acc[u].w = __float_as_uint(cmb<OP>(__uint_as_float(acc[u].w), __uint_as_float(w.w)));
            } else {
              acc[u].x = cmbi<OP>(acc[u].x, w.x);
              acc[u].y = cmbi<OP>(acc[u].y, w.y);
              acc[u].z = cmbi<OP>(acc[u].z, w.z);
              acc[u].w = cmbi<OP>(acc[u].w, w.w);
            }
          }
        }
      }
    }
  }
  if constexpr (FAN && !COH) {
    if (o.nd > 1) {
      store_tile_bulk(o, ptr, run, gbeg, gend, acc);
      return;
    }
  }
  const bool keep = FAN ? static_cast<bool>(o.keep) : keep_early;
  const int64_t doff = run * o.dstride + (gbeg + lane()) * 16;
  keep_stores<COH, FAN>(keep, [&](auto k) {
    for (int d = 0; d < o.nd; ++d) {
      char* dp = static_cast<char*>(const_cast<void*>(ptr[o.ns + d])) + doff;
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        if (u * kThreads < lim) stv<COH, decltype(k)::value>(dp + u * kThreads * 16, acc[u]);
    }
  });
}

// Adds one loaded group of 8 values to the accumulator (or starts it).
template <int OP>
__device__ __forceinline__ void accumulate8(float* acc, const float* f, bool first) {
  if (first) {
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = f[i];
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = cmb<OP>(acc[i], f[i]);
  }
}

template <bool F16, int U, bool COH, bool KEEP, class PT>
__device__ __forceinline__ void store_half_mode(const OpDesc& o, const PT& ptr, int64_t run, int64_t g0, int64_t gend,
                                                float (&acc)[U][8]) {
  for (int d = 0; d < o.nd; ++d) {
    char* dp = static_cast<char*>(const_cast<void*>(ptr[o.ns + d])) + run * o.dstride;
    const bool f32 = (o.dmask >> d) & 1;
    const bool a32 = (reinterpret_cast<uintptr_t>(dp) & 31) == 0;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t g = g0 + u * kThreads;
      if (g < gend) {
        if (f32) {
          if (a32) {
            W8 v;
#pragma unroll
            for (int i = 0; i < 8; ++i) v.w[i] = __float_as_uint(acc[u][i]);
            stv32<COH, KEEP>(dp + g * 32, v);
          } else {
            stv<COH, KEEP>(dp + g * 32, make_uint4(__float_as_uint(acc[u][0]), __float_as_uint(acc[u][1]),
                                                   __float_as_uint(acc[u][2]), __float_as_uint(acc[u][3])));
            stv<COH, KEEP>(dp + g * 32 + 16, make_uint4(__float_as_uint(acc[u][4]), __float_as_uint(acc[u][5]),
                                                        __float_as_uint(acc[u][6]), __float_as_uint(acc[u][7])));
          }
        } else {
          stv<COH, KEEP>(dp + g * 16, make_uint4(pack2<F16>(acc[u][0], acc[u][1]), pack2<F16>(acc[u][2], acc[u][3]),
                                                 pack2<F16>(acc[u][4], acc[u][5]), pack2<F16>(acc[u][6], acc[u][7])));
        }
      }
    }
  }
}

// 16-bit data with fp32 partial sums among the sources: kBatchBF sources'
// loads are in flight together before they are combined, one after another
// in source order.  A group is 16 bytes of a 16-bit source or 32 of an fp32
// one, loaded as one access either way.
constexpr int kUnrollBF = 2;  // groups per thread per pass
constexpr int kBatchBF = 2;
template <bool F16, int OP, bool COH, class PT>
__device__ __forceinline__ void tile_half_mixed(const OpDesc& o, const PT& ptr, int64_t run, int64_t gbeg,
                                                int64_t gend) {
  const bool keep = o.keep;  // read before the loads (see tile_4b)
  // A tile is covered in passes of kUnrollBF groups per thread.
#pragma unroll 1
  for (int pass = 0; pass < kUnroll / kUnrollBF; ++pass) {
    const int64_t pbeg = gbeg + pass * kUnrollBF * kThreads;
    if (pbeg >= gend) break;
    const int64_t g0 = pbeg + lane();
    float acc[kUnrollBF][8];
    for (int k = 0; k < o.ns; k += kBatchBF) {
      W8 raw[kBatchBF][kUnrollBF];
#pragma unroll
      for (int j = 0; j < kBatchBF; ++j) {
        if (k + j < o.ns) {
          const char* s = static_cast<const char*>(ptr[k + j]) + run * o.sstride;
          const bool f32 = (o.smask >> (k + j)) & 1;
          const bool a32 = (reinterpret_cast<uintptr_t>(s) & 31) == 0;
#pragma unroll
          for (int u = 0; u < kUnrollBF; ++u) {
            const int64_t g = g0 + u * kThreads;
            if (g < gend) {
              if (f32 && a32) {
                raw[j][u] = ldv32_once<COH>(s + g * 32);
              } else if (f32) {
                const uint4 a = ldv_once<COH>(s + g * 32), b = ldv_once<COH>(s + g * 32 + 16);
                raw[j][u].w[0] = a.x; raw[j][u].w[1] = a.y; raw[j][u].w[2] = a.z; raw[j][u].w[3] = a.w;
                raw[j][u].w[4] = b.x; raw[j][u].w[5] = b.y; raw[j][u].w[6] = b.z; raw[j][u].w[7] = b.w;
              } else {
                const uint4 v = ldv_once<COH>(s + g * 16);
                raw[j][u].w[0] = v.x; raw[j][u].w[1] = v.y; raw[j][u].w[2] = v.z; raw[j][u].w[3] = v.w;
              }
            }
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kBatchBF; ++j) {
        if (k + j < o.ns) {
          const bool f32 = (o.smask >> (k + j)) & 1;
#pragma unroll
          for (int u = 0; u < kUnrollBF; ++u) {
            const int64_t g = g0 + u * kThreads;
            if (g < gend) {
              float f[8];
              if (f32) {
#pragma unroll
                for (int i = 0; i < 8; ++i) f[i] = __uint_as_float(raw[j][u].w[i]);
              } else {
                widen8<F16>(make_uint4(raw[j][u].w[0], raw[j][u].w[1], raw[j][u].w[2], raw[j][u].w[3]), f);
              }
              accumulate8<OP>(acc[u], f, k + j == 0);
            }
          }
        }
      }
    }
    keep_stores<COH>(keep, [&](auto k) { store_half_mode<F16, kUnrollBF, COH, decltype(k)::value>(o, ptr, run, g0, gend, acc); });
  }
}

// Every source stored in the 16-bit type (fused AllReduce / ReduceScatter,
// first ring and halving steps): kBatchBP sources' loads are in flight
// together before they are combined, still one after another in source
// order.  Measured on the fused bf16 AllReduce at 8 x 128 MiB: 5811 -> 6516
// GB/s; kept apart from the mixed kernel because its extra registers lower
// that kernel's occupancy.
constexpr int kUnrollBP = 4;
constexpr int kBatchBP = 2;
template <bool F16, int OP, bool COH, class PT>
__device__ __forceinline__ void tile_half_pure(const OpDesc& o, const PT& ptr, int64_t run, int64_t gbeg,
                                               int64_t gend) {
  const bool keep = o.keep;  // read before the loads (see tile_4b)
#pragma unroll 1
  for (int pass = 0; pass < kUnroll / kUnrollBP; ++pass) {
    const int64_t pbeg = gbeg + pass * kUnrollBP * kThreads;
    if (pbeg >= gend) break;
    const int64_t g0 = pbeg + lane();
    float acc[kUnrollBP][8];
    for (int k = 0; k < o.ns; k += kBatchBP) {
      uint4 raw[kBatchBP][kUnrollBP];
#pragma unroll
      for (int j = 0; j < kBatchBP; ++j) {
        if (k + j < o.ns) {
          const char* s = static_cast<const char*>(ptr[k + j]) + run * o.sstride;
#pragma unroll
          for (int u = 0; u < kUnrollBP; ++u) {
            const int64_t g = g0 + u * kThreads;
            if (g < gend) raw[j][u] = ldv<COH>(s + g * 16);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kBatchBP; ++j) {
        if (k + j < o.ns) {
#pragma unroll
          for (int u = 0; u < kUnrollBP; ++u) {
            const int64_t g = g0 + u * kThreads;
            if (g < gend) {
              float f[8];
              widen8<F16>(raw[j][u], f);
              accumulate8<OP>(acc[u], f, k + j == 0);
            }
          }
        }
      }
    }
    keep_stores<COH>(keep, [&](auto k) { store_half_mode<F16, kUnrollBP, COH, decltype(k)::value>(o, ptr, run, g0, gend, acc); });
  }
}

template <int MODE, int OP, bool COH, int SB, bool FAN, class PT>
__device__ __forceinline__ void tile_vec(const OpDesc& o, const PT& ptr, int64_t run, int64_t gbeg, int64_t gend) {
  if constexpr (MODE == kCopy) tile_copy<COH, FAN>(o, ptr, run, gbeg, gend);
  else if constexpr (MODE == kF32) tile_4b<true, OP, COH, SB, FAN>(o, ptr, run, gbeg, gend);
  else if constexpr (MODE == kI32) tile_4b<false, OP, COH, SB, FAN>(o, ptr, run, gbeg, gend);
  else if constexpr (MODE == kBF16) tile_half_mixed<false, OP, COH>(o, ptr, run, gbeg, gend);
  else if constexpr (MODE == kF16) tile_half_mixed<true, OP, COH>(o, ptr, run, gbeg, gend);
  else if constexpr (MODE == kBF16P) tile_half_pure<false, OP, COH>(o, ptr, run, gbeg, gend);
  else tile_half_pure<true, OP, COH>(o, ptr, run, gbeg, gend);
}

// -- element path (unaligned operands and the tails of vector runs) ---------
// Scalar loads: plain, or through L2 (.cg) for one-launch plans (see ldv).
template <bool COH>
__device__ __forceinline__ uint32_t ld32(const void* p) {
  if constexpr (COH) {
    uint32_t v;
    asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
  } else {
    return *static_cast<const uint32_t*>(p);
  }
}
template <bool COH>
__device__ __forceinline__ uint16_t ld16b(const void* p) {
  if constexpr (COH) {
    uint16_t v;
    asm volatile("ld.global.cg.u16 %0, [%1];" : "=h"(v) : "l"(p) : "memory");
    return v;
  } else {
    return *static_cast<const uint16_t*>(p);
  }
}

template <int MODE, int OP, bool COH, class PT>
__device__ __forceinline__ void elem(const OpDesc& o, const PT& ptr, int64_t soff, int64_t doff, int64_t e) {
  if constexpr (MODE == kCopy) {
    const char* s = static_cast<const char*>(ptr[0]) + soff + e * o.esz;
    if (o.esz == 2) {
      const uint16_t v = ld16b<COH>(s);
      for (int d = 0; d < o.nd; ++d)
        *reinterpret_cast<uint16_t*>(static_cast<char*>(const_cast<void*>(ptr[o.ns + d])) + doff + e * 2) = v;
    } else {
      const uint32_t v = ld32<COH>(s);
      for (int d = 0; d < o.nd; ++d)
        *reinterpret_cast<uint32_t*>(static_cast<char*>(const_cast<void*>(ptr[o.ns + d])) + doff + e * 4) = v;
    }
  } else if constexpr (MODE == kF32) {
    float acc = __uint_as_float(ld32<COH>(static_cast<const char*>(ptr[0]) + soff + e * 4));
    for (int k = 1; k < o.ns; ++k)
      acc = cmb<OP>(acc, __uint_as_float(ld32<COH>(static_cast<const char*>(ptr[k]) + soff + e * 4)));
    for (int d = 0; d < o.nd; ++d)
      *reinterpret_cast<float*>(static_cast<char*>(const_cast<void*>(ptr[o.ns + d])) + doff + e * 4) = acc;
  } else if constexpr (MODE == kI32) {
    uint32_t acc = ld32<COH>(static_cast<const char*>(ptr[0]) + soff + e * 4);
    for (int k = 1; k < o.ns; ++k) acc = cmbi<OP>(acc, ld32<COH>(static_cast<const char*>(ptr[k]) + soff + e * 4));
    for (int d = 0; d < o.nd; ++d)
      *reinterpret_cast<uint32_t*>(static_cast<char*>(const_cast<void*>(ptr[o.ns + d])) + doff + e * 4) = acc;
  } else {
    constexpr bool F16 = MODE == kF16 || MODE == kF16P;
    float acc = 0.f;
    for (int k = 0; k < o.ns; ++k) {
      const char* s = static_cast<const char*>(ptr[k]) + soff;
      const float v = ((o.smask >> k) & 1) ? __uint_as_float(ld32<COH>(s + e * 4)) : widen1<F16>(ld16b<COH>(s + e * 2));
      acc = k == 0 ? v : cmb<OP>(acc, v);
    }
    for (int d = 0; d < o.nd; ++d) {
      char* dp = static_cast<char*>(const_cast<void*>(ptr[o.ns + d])) + doff;
      if ((o.dmask >> d) & 1) *reinterpret_cast<float*>(dp + e * 4) = acc;
      else *reinterpret_cast<uint16_t*>(dp + e * 2) = narrow1<F16>(acc);
    }
  }
}

template <int MODE>
__device__ __forceinline__ int64_t group_elems(const OpDesc& o) {
  return MODE == kCopy ? 16 / o.esz : (MODE == kF32 || MODE == kI32 ? 4 : 8);
}

// Tile lt of operation o (tiles of one operation are numbered run by run).
// ELEM: the launch has operations that take the element path (unaligned, or
// a tail after the last whole group).  Launches without them use the kernel
// compiled without that path: inlined, its registers count against the
// vector path (58 instead of 46 for fp32), costing a resident block per SM.
template <int MODE, int OP, bool COH, int SB, bool ELEM, bool FAN, class PT>
__device__ __forceinline__ void run_tile(const OpDesc& o, const PT& ptr, uint32_t lt) {
  const uint32_t run32 = lt / o.tpr;  // tiles of a launch number below 2^32
  const int64_t run = run32;
  const int64_t tr = lt - run32 * o.tpr;
  if (!ELEM || o.vec) {
    const int64_t tg = static_cast<int64_t>(o.upt) * kThreads;
    const int64_t gbeg = tr * tg;
    const int64_t gend = gbeg + tg < o.groups ? gbeg + tg : o.groups;
    tile_vec<MODE, OP, COH, SB, FAN>(o, ptr, run, gbeg, gend);
  }
  if constexpr (ELEM) {
    const int64_t soff = run * o.sstride, doff = run * o.dstride;
    if (o.vec) {
      if (tr == o.tpr - 1) {  // elements after the last whole group (single-run operations only)
        for (int64_t e = o.groups * group_elems<MODE>(o) + lane(); e < o.n; e += kThreads)
          elem<MODE, OP, COH>(o, ptr, soff, doff, e);
      }
    } else {
      const int64_t e0 = tr * kTileElems;
      const int64_t e1 = e0 + kTileElems < o.n ? e0 + kTileElems : o.n;
      for (int64_t e = e0 + lane(); e < e1; e += kThreads) elem<MODE, OP, COH>(o, ptr, soff, doff, e);
    }
  }
}

// The operation holding tile t: the last of op[0, nops) whose tile0 <= t.
__device__ __forceinline__ int find_op(const OpDesc* op, int nops, uint32_t t) {
  int lo = 0, hi = nops - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (op[mid].tile0 <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// One launch of one step.  The operation lookup (a binary search on each
// operation's first tile) reads a shared-memory copy of the first-tile
// column, made before waiting on the previous grid; the operations' fields
// and pointers are read from the parameter block in the constant bank (a
// shared-memory copy of those measured 5-9% slower on the bf16 ring steps:
// the per-source loops then wait on a shared-memory load for each source's
// pointer).  Programmatic dependent launch: this grid may be scheduled while
// the previous step's grid drains; it lets the next step be scheduled the
// same way, then waits until the previous grid has completed and its writes
// are visible before touching the buffers.  Without the launch attribute
// both are no-ops and stream order applies.  A grid that covers the GPU
// keeps the next one from running ahead of it.  One that leaves room (late:
// fewer tiles than resident blocks) lets the next grid in only after its wait,
// as the one-launch kernels do (see plan_kernel).  After the wait for every
// grid, the 256 MiB per rank Ring and RHD measured 4% and 2% slower; for none,
// per-step Rings of 512 KiB - 1 MiB per rank 12-28% slower.
template <int MODE, int OP, class P, int SB, bool ELEM, bool FAN>
__global__ void __launch_bounds__(kThreads) step_kernel(const __grid_constant__ P p) {
  __shared__ uint32_t s_tile0[sizeof(P::op) / sizeof(OpDesc)];
  const bool late = p.late != 0;
  if (!late) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int nops = static_cast<int>(p.nops);
  for (int i = threadIdx.x; i < nops; i += kThreads) s_tile0[i] = p.op[i].tile0;
  __syncthreads();
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (late) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // (kernels with the bulk-store path, which serve fused and fan-out
  // operations, keep the forward walk: their code stays as it was, and the
  // fused AllReduce measured 2% slower with the direction select in it)
  const bool rev = !FAN && p.rev != 0;
  for (uint32_t t0 = blockIdx.x; t0 < p.ntiles; t0 += gridDim.x) {
    const uint32_t t = rev ? p.ntiles - 1 - t0 : t0;
    int lo = 0, hi = nops - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_tile0[mid] <= t) lo = mid; else hi = mid - 1;
    }
    const OpDesc& o = p.op[lo];
    run_tile<MODE, OP, false, SB, ELEM, FAN>(o, p.ptr + o.p0, t - o.tile0);
  }
  // outstanding bulk stores of fan-out copies finish before the block exits
  if (FAN && threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// -- bulk-copy (TMA) kernel ------------------------------------------------------
// Copy steps whose operations are all 16-byte aligned with no element tail run
// as a pipeline of bulk asynchronous copies: in each block one thread loads a
// tile of up to 32 KB global -> shared (cp.async.bulk with mbarrier
// completion), keeping kCopyStages tiles in flight, and writes each landed
// tile to every destination with bulk stores (cp.async.bulk shared -> global);
// a stage is refilled once the stores of the tile it held have read it.  One
// block per SM.  Measured on a 1 GiB copy: 6835 GB/s against 6385 for 128-bit
// loads and stores through registers (8 blocks per SM); 256 MiB: 6517 vs 6206.
// The host takes it for launches that write at least 128 MiB in calls without
// 16-bit reduction steps; other copy launches keep the register kernel.
// Waits on an mbarrier are bounded: one that gives up sets the device error
// word, stops issuing, waits (bounded) for the loads it issued and returns.
constexpr int kCopyStages = 3;
constexpr int kCopyTileBytes = 32 << 10;  // largest tile: 2048 groups (tile groups = upt * kThreads, upt <= 8)
constexpr int kCopyThreads = 32;
constexpr uint32_t kMbarWaitLimit = 1u << 21;

__device__ uint32_t g_device_error;  // bit 1: a bulk-copy wait gave up

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

// Polls the mbarrier phase with test_wait (never blocks: try_wait may suspend
// the thread for a system-dependent time per call, which would leave the
// total unbounded), backing off with a short sleep after the first polls:
// at most kMbarWaitLimit polls of at most ~0.1 us sleep each, well under a
// second, while a tile's load lands in a few microseconds.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (uint32_t it = 0; it < kMbarWaitLimit; ++it) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    if (ok) return true;
    if (it >= 32) __nanosleep(64);
  }
  return false;
}

template <class P, bool DRILL = false>
__global__ void __launch_bounds__(kCopyThreads) tma_copy_kernel(const __grid_constant__ P p) {
  extern __shared__ __align__(128) unsigned char stage[];  // kCopyStages * kCopyTileBytes, then the mbarriers
  __shared__ uint32_t s_tile0[sizeof(P::op) / sizeof(OpDesc)];
  uint64_t* bars = reinterpret_cast<uint64_t*>(stage + kCopyStages * kCopyTileBytes);
  const bool late = p.late != 0;  // as in step_kernel
  if (!late) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int nops = static_cast<int>(p.nops);
  for (int i = threadIdx.x; i < nops; i += kCopyThreads) s_tile0[i] = p.op[i].tile0;
  if (threadIdx.x == 0) {
    for (int k = 0; k < kCopyStages; ++k)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(bars + k)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (late) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x != 0) return;
  // tile i of this block is global tile blockIdx.x + i * gridDim.x
  const int64_t n = p.ntiles > blockIdx.x ? (p.ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  struct Tile {
    const OpDesc* o;
    int64_t run, gbeg;
    uint32_t bytes;
  };
  auto tile = [&](int64_t i) {
    const uint32_t t0 = static_cast<uint32_t>(blockIdx.x + i * gridDim.x);
    const uint32_t t = p.rev ? p.ntiles - 1 - t0 : t0;
    int lo = 0, hi = nops - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_tile0[mid] <= t) lo = mid; else hi = mid - 1;
    }
    const OpDesc& o = p.op[lo];
    const uint32_t lt = t - o.tile0, run = lt / o.tpr, tr = lt - run * o.tpr;
    const int64_t tg = int64_t(o.upt) * kThreads;
    const int64_t gbeg = tr * tg, gend = gbeg + tg < o.groups ? gbeg + tg : o.groups;
    return Tile{&o, run, gbeg, static_cast<uint32_t>((gend - gbeg) * 16)};
  };
  // stores: evict first in L2, as the streaming stores of the other paths,
  // unless the next step reads them (keep); loads: read once, evict first
  uint64_t evict_first, evict_normal;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(evict_first));
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(evict_normal));
  auto load = [&](int64_t i) {
    const int k = static_cast<int>(i % kCopyStages);
    const Tile x = tile(i);
    const char* src = static_cast<const char*>(p.ptr[x.o->p0]) + x.run * x.o->sstride + x.gbeg * 16;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bars + k)), "r"(x.bytes)
                 : "memory");
    if (DRILL && i == 0) return;
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
                     smem_addr(stage + k * kCopyTileBytes)),
                 "l"(src), "r"(x.bytes), "r"(smem_addr(bars + k)), "l"(evict_first)
                 : "memory");
  };

  int64_t issued = 0;
  for (; issued < n && issued < kCopyStages; ++issued) load(issued);
  int64_t i = 0;
  bool ok = true;
  for (; i < n; ++i) {
    const int k = static_cast<int>(i % kCopyStages);
    if (!mbar_wait(smem_addr(bars + k), static_cast<uint32_t>((i / kCopyStages) & 1))) {
      ok = false;
      break;
    }
    const Tile x = tile(i);
    const uint64_t policy = x.o->keep ? evict_normal : evict_first;
    for (int d = 0; d < x.o->nd; ++d) {
      char* dst = static_cast<char*>(const_cast<void*>(p.ptr[x.o->p0 + x.o->ns + d])) + x.run * x.o->dstride + x.gbeg * 16;
      asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(dst),
                   "r"(smem_addr(stage + k * kCopyTileBytes)), "r"(x.bytes), "l"(policy)
                   : "memory");
    }
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    if (i >= 1 && issued < n) {  // refill the stage of tile i - 1 once its stores have read it
      asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
      load(issued++);
    }
  }
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  if (!ok) {
    atomicOr(&g_device_error, 2u);
    // loads issued and not consumed land before the block's shared memory is released
    for (int64_t j = i; j < issued; ++j)
      mbar_wait(smem_addr(bars + j % kCopyStages), static_cast<uint32_t>((j / kCopyStages) & 1));
  }
}

// -- one-launch plans ------------------------------------------------------------
// A plan can run as one launch of one thread-block cluster: the blocks walk
// the tiles of step 0, meet at a cluster barrier (release / acquire: every
// write of the step is visible to every block before any block starts the
// next), walk step 1, and so on.  The operations, their order and each
// element's association are those of the per-step launches; only the launch
// and grid drain between steps are gone.  The plan's description lives in
// device memory (written once per plan shape): a header, the steps, the
// operations (tile numbers relative to their step, pointer indices into the
// operand table) and the operand table, whose entries name a buffer base
// (send r, recv r, scratch) and a byte offset.  The call passes only the
// bases.  Every block copies the description and the bases to shared memory
// before waiting on the previous grid, so the lookups of the step walk are
// shared-memory reads.
struct __align__(16) PlanHeader {
  uint32_t nsteps, nops, nrefs, pad;
};
struct __align__(16) PlanStep {
  uint32_t op0;     // first operation of the step
  uint32_t nops;    // its operations
  uint32_t ntiles;  // its tiles
  uint32_t mode;    // kCopy or the plan's reduction mode
};
struct __align__(16) OperandRef {
  uint32_t base;  // index into the bases: send r = r, recv r = N + r, scratch = 2N
  uint32_t pad;
  int64_t off;    // bytes from the base
};
struct RefPtrs {
  const OperandRef* ref;
  const void* const* base;
  __device__ __forceinline__ const void* operator[](int k) const {
    return static_cast<const char*>(base[ref[k].base]) + ref[k].off;
  }
};
struct __align__(16) PlanParams {
  const uint4* plan;  // the description, 16-byte words
  uint32_t words;
  uint32_t nbases;
  int64_t groups;     // sliced plans: 16-byte groups per rank buffer that the plan covers
  const void* base[2 * VC_MAX_RANKS + 1];
};

// Blocks of kPlanSubs sub-blocks of kThreads threads; each sub-block walks
// its own tiles (tile functions index by lane()).  Measured on 8 ranks: two
// sub-blocks double the bandwidth of mid-size plans (16 MB per rank ring:
// 962 -> 599 us) but add about 0.2 us per step to small ones (1 KB ring:
// 18.0 -> 20.9 us), and single launches are only chosen for small ones.
constexpr int kPlanSubs = 1;
constexpr int kPlanThreads = kThreads * kPlanSubs;

template <int RMODE, int OP>
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const __grid_constant__ PlanParams p) {
  extern __shared__ uint4 sm[];
  for (uint32_t i = threadIdx.x; i < p.words; i += kPlanThreads) sm[i] = ld16(p.plan + i);
  const void** sbase = reinterpret_cast<const void**>(sm + p.words);
  for (uint32_t i = threadIdx.x; i < p.nbases; i += kPlanThreads) sbase[i] = p.base[i];
  __syncthreads();
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // The next grid may be scheduled once every block of this one is past its
  // wait: at most one grid ahead.  Triggered as the first instruction (as a
  // step grid does), each waiting grid admitted the next, a run of small
  // back-to-back launches filled the SMs with waiting blocks, and the time
  // per launch grew with the run.  The sliced form, 8 ranks, fp32 Ring at 1
  // MiB per rank: 12.2 us a call at 10 calls in a graph, 19.7 at 400; with the
  // trigger here, 11.1 at both.  This form: 28.8 -> 22.7 us at 1 MiB.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const PlanHeader h = *reinterpret_cast<const PlanHeader*>(sm);
  const PlanStep* steps = reinterpret_cast<const PlanStep*>(sm + 1);
  const OpDesc* ops = reinterpret_cast<const OpDesc*>(sm + 1 + h.nsteps);
  const OperandRef* refs = reinterpret_cast<const OperandRef*>(ops + h.nops);
  // Every block runs every iteration of this loop (the step count is the
  // same for all), so each meets each barrier exactly once.
  for (uint32_t s = 0; s < h.nsteps; ++s) {
    const PlanStep st = steps[s];
    const OpDesc* sop = ops + st.op0;
    const uint32_t first = blockIdx.x * kPlanSubs + threadIdx.x / kThreads, stride = gridDim.x * kPlanSubs;
    for (uint32_t t = first; t < st.ntiles; t += stride) {
      const OpDesc& o = sop[find_op(sop, static_cast<int>(st.nops), t)];
      const RefPtrs ptr{refs + o.p0, sbase};
      if (st.mode == kCopy) run_tile<kCopy, OP, true, 1, true, false>(o, ptr, t - o.tile0);
      else run_tile<RMODE, OP, true, 4, true, false>(o, ptr, t - o.tile0);
    }
    if (s + 1 < h.nsteps)
      asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
  }
}

}  // namespace dev
}  // namespace vc
