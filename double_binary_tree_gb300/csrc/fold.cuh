// The reduction of one unit over the emulated ranks, in the schedule's order.
//
// All R ranks' buffers sit in one GPU's memory, so every "message" of the
// ring or tree schedule stays on chip: a thread takes the R ranks' copies of
// one 16-byte unit (or one element), folds them in exactly the order the
// schedule reduces them, narrows once, and the kernel stores the result to
// every rank that receives it.
//
// Reduction orders (sources: [Interview] "all-reduce 每张卡要发多少数据? ring 和
// tree 有什么区别?", section "手撕代码(NumPy 模拟 ring all-reduce)" and Figure 1;
// [Course13] "NCCL 专家课程 13：Tree、双树、层次化连接与真实交叉区间", sections
// "先固定方向", "runTreeSplit 如何流水", "每种 rank 的操作"):
//   ring AllReduce  element in block j of its loop: ranks j, j+1, ..., j-1
//   ReduceScatter   element of block b: ranks b+1, ..., b
//   tree AllReduce  post-order over the channel's tree, local input first,
//                   children in down[] order (the FoldProg stream)
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#ifndef __CUDACC_RTC__  // run-time compilation (jit.cc) has no host headers
#include <cuda_runtime.h>
#include <stdint.h>
#endif

#include "bounds.cuh"
#include "common.h"

namespace vr {

// Programmatic dependent launch.  A kernel launched with programmatic
// stream serialisation may start while the previous kernel on its stream is
// still running: pdl_launch lets the next kernel start early in the same
// way, pdl_wait blocks until the previous kernel has finished and its memory
// is visible.  Every kernel here calls pdl_wait after its prologue and
// before touching global memory, so stream order is kept; for a kernel
// launched without the attribute both are no-ops.
__device__ __forceinline__ void pdl_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <bool C, class A, class B> struct Select { typedef A type; };
template <class A, class B> struct Select<false, A, B> { typedef B type; };

constexpr int kBatch = 8;  // rank loads issued together before they are folded

// ------------------------------------------------------------ element types
template <typename T> struct Ty;
template <> struct Ty<float> {
  static constexpr int U = 4;  // elements per 16 bytes
  typedef unsigned Bits;
  static __device__ __forceinline__ float widen(Bits b) { return __uint_as_float(b); }
  static __device__ __forceinline__ Bits narrow(float x) { return __float_as_uint(x); }
};
template <> struct Ty<__half> {
  static constexpr int U = 8;
  typedef unsigned short Bits;
  static __device__ __forceinline__ float widen(Bits b) { return __half2float(__ushort_as_half(b)); }
  static __device__ __forceinline__ Bits narrow(float x) { return __half_as_ushort(__float2half_rn(x)); }
};
template <> struct Ty<__nv_bfloat16> {
  static constexpr int U = 8;
  typedef unsigned short Bits;
  static __device__ __forceinline__ float widen(Bits b) {
    return __bfloat162float(__ushort_as_bfloat16(b));
  }
  static __device__ __forceinline__ Bits narrow(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
  }
};

// ---------------------------------------------------------- memory access
// Every global access below goes through these helpers (or a bulk copy),
// each checked in the bounds-checked build (bounds.cuh): a refused load
// reads zeros, a refused store is dropped.
__device__ __forceinline__ uint4 ld_global_v4(const void* p) {
  uint4 v;
  if (!VR_ACCESS_OK(p, 16, false)) return make_uint4(0, 0, 0, 0);
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}
__device__ __forceinline__ void st_global_v4(void* p, uint4 v) {
  if (!VR_ACCESS_OK(p, 16, true)) return;
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}
// Plain (coherent) load and store of one value of type V.
template <typename V> __device__ __forceinline__ V ld_plain(const void* p) {
  if (!VR_ACCESS_OK(p, sizeof(V), false)) return V();
  return *reinterpret_cast<const V*>(p);
}
// Read-only (non-coherent cache) load of one value of type V.
template <typename V> __device__ __forceinline__ V ld_ro(const void* p) {
  if (!VR_ACCESS_OK(p, sizeof(V), false)) return V();
  return __ldg(reinterpret_cast<const V*>(p));
}
template <typename V> __device__ __forceinline__ void st_plain(void* p, V v) {
  if (!VR_ACCESS_OK(p, sizeof(V), true)) return;
  *reinterpret_cast<V*>(p) = v;
}
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// A unit is one 16-byte vector (NV = Ty<T>::U elements) or one element.
template <typename T, int NV> struct Unit {
  typedef typename Ty<T>::Bits Bits;
  typedef typename Select<NV == 1, Bits, uint4>::type Raw;

  static __device__ __forceinline__ void store(char* p, Raw v) {
    if constexpr (NV == 1) st_plain<Bits>(p, v);
    else st_global_v4(p, v);
  }
  static __device__ __forceinline__ void unpack(Raw v, float (&x)[NV]) {
    if constexpr (NV == 1) {
      x[0] = Ty<T>::widen(v);
    } else if constexpr (sizeof(T) == 4) {
      x[0] = Ty<T>::widen(v.x); x[1] = Ty<T>::widen(v.y);
      x[2] = Ty<T>::widen(v.z); x[3] = Ty<T>::widen(v.w);
    } else {
      const unsigned w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        x[2 * i] = Ty<T>::widen((Bits)(w[i] & 0xFFFFu));
        x[2 * i + 1] = Ty<T>::widen((Bits)(w[i] >> 16));
      }
    }
  }
  static __device__ __forceinline__ Raw pack(const float (&x)[NV]) {
    if constexpr (NV == 1) {
      return Ty<T>::narrow(x[0]);
    } else if constexpr (sizeof(T) == 4) {
      return make_uint4(Ty<T>::narrow(x[0]), Ty<T>::narrow(x[1]), Ty<T>::narrow(x[2]),
                        Ty<T>::narrow(x[3]));
    } else {
      unsigned w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        w[i] = (unsigned)Ty<T>::narrow(x[2 * i]) | ((unsigned)Ty<T>::narrow(x[2 * i + 1]) << 16);
      return make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
};

// Where rank r's copy of the unit being folded lives.
struct GlobalSrc {              // ptr[r] + off, global memory
  const char* const* ptr;
  long long off;
};
struct SharedSrc {              // base + r * stride, shared memory
  const unsigned char* base;    // plain loads: the compiler may schedule them freely,
  uint32_t stride;              // but not across the mbarrier wait (a memory clobber)
};

template <typename T, int NV>
__device__ __forceinline__ typename Unit<T, NV>::Raw load_unit(const GlobalSrc& s, int r) {
  const char* p = s.ptr[r] + s.off;
  if constexpr (NV == 1) {
    if (!VR_ACCESS_OK(p, sizeof(typename Ty<T>::Bits), false)) return 0;
    return __ldg(reinterpret_cast<const typename Ty<T>::Bits*>(p));
  } else {
    return ld_global_v4(p);
  }
}
template <typename T, int NV>
__device__ __forceinline__ typename Unit<T, NV>::Raw load_unit(const SharedSrc& s, int r) {
  return *reinterpret_cast<const typename Unit<T, NV>::Raw*>(s.base + (uint32_t)r * s.stride);
}

// ----------------------------------------------------------- reduction op
// Sum: IEEE fp32 addition of the exactly widened inputs, never contracted.
__device__ __forceinline__ float add_rn(float a, float b) { return __fadd_rn(a, b); }

// Max: the larger value in the IEEE total order of non-NaN floats (-0 below
// +0).  Widening is exact and monotone, so the order of the widened fp32
// values is the order of the element type's own values; Max therefore runs
// on order-preserving integer keys of the raw bits -- sign-magnitude mapped
// to unsigned (negative: all bits flipped, positive: sign bit flipped) --
// and needs no float conversion.  16-bit keys are compared two per 32-bit
// word.
__device__ __forceinline__ unsigned key32(unsigned b) {
  return b ^ ((unsigned)((int)b >> 31) | 0x80000000u);
}
__device__ __forceinline__ unsigned unkey32(unsigned k) {
  return k ^ (~(unsigned)((int)k >> 31) | 0x80000000u);
}
// 0xFFFF in every 16-bit lane whose top bit is set, else 0: a byte permute
// that replicates the sign of bytes 1 and 3 (selector nibbles 8 | byte).
__device__ __forceinline__ unsigned lane_signs16x2(unsigned w) {
  unsigned m;
  asm("prmt.b32 %0, %1, %2, 0xBB99;" : "=r"(m) : "r"(w), "r"(0u));
  return m;
}
__device__ __forceinline__ unsigned key16x2(unsigned w) {
  return w ^ (lane_signs16x2(w) | 0x80008000u);  // negative lanes: all bits flipped
}
__device__ __forceinline__ unsigned unkey16x2(unsigned k) {
  return k ^ (~lane_signs16x2(k) | 0x80008000u);  // lanes >= +0 have the top bit set
}
__device__ __forceinline__ unsigned max_u16x2(unsigned a, unsigned b) {
  unsigned d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// The fold's working lanes for one unit: fp32 values for Sum, integer keys
// for Max.
template <typename T, int OP, int NV, bool IS_SUM = (OP == VR_SUM)> struct Lanes;

template <typename T, int NV> struct Lanes<T, VR_SUM, NV, true> {
  typedef float L;
  static constexpr int N = NV;
  typedef Unit<T, NV> Un;
  static __device__ __forceinline__ void decode(typename Un::Raw v, L (&x)[N]) { Un::unpack(v, x); }
  static __device__ __forceinline__ typename Un::Raw encode(const L (&x)[N]) { return Un::pack(x); }
  static __device__ __forceinline__ L op(L a, L b) { return add_rn(a, b); }
};

template <typename T, int NV> struct Lanes<T, VR_MAX, NV, false> {
  typedef unsigned L;
  typedef Unit<T, NV> Un;
  static constexpr bool kWide = sizeof(T) == 4;
  static constexpr int N = NV == 1 ? 1 : 4;  // 32-bit words per unit
  static __device__ __forceinline__ void decode(typename Un::Raw v, L (&x)[N]) {
    if constexpr (NV == 1) {
      x[0] = kWide ? key32((unsigned)v) : key16x2((unsigned)v);
    } else {
      const unsigned w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) x[i] = kWide ? key32(w[i]) : key16x2(w[i]);
    }
  }
  static __device__ __forceinline__ typename Un::Raw encode(const L (&x)[N]) {
    if constexpr (NV == 1) {
      return (typename Un::Raw)(kWide ? unkey32(x[0]) : (unkey16x2(x[0]) & 0xFFFFu));
    } else {
      unsigned w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) w[i] = kWide ? unkey32(x[i]) : unkey16x2(x[i]);
      return make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
  static __device__ __forceinline__ L op(L a, L b) {
    if constexpr (kWide) return max(a, b);
    else return max_u16x2(a, b);
  }
};

// ------------------------------------------------------------------ folds
// Ranks j, j+1, ..., j+R-1 (mod R), left to right.  The first batch is
// peeled so that no step has to ask whether it is the first.
template <typename T, int OP, int NV, class Src, int B = kBatch>
__device__ __forceinline__ typename Unit<T, NV>::Raw ring_fold(const Src& src, int R, int j) {
  typedef Unit<T, NV> Un;
  typedef Lanes<T, OP, NV> Ln;
  typename Ln::L acc[Ln::N];
  for (int k0 = 0; k0 < R; k0 += B) {
    typename Un::Raw v[B];
#pragma unroll
    for (int i = 0; i < B; ++i) {
      const int k = k0 + i;
      if (k < R) {
        int r = j + k;
        r -= r >= R ? R : 0;
        v[i] = load_unit<T, NV>(src, r);
      }
    }
    int i0 = 0;
    if (k0 == 0) {
      Ln::decode(v[0], acc);
      i0 = 1;
    }
#pragma unroll
    for (int i = 0; i < B; ++i) {
      const int k = k0 + i;
      if (i >= i0 && k < R) {
        typename Ln::L x[Ln::N];
        Ln::decode(v[i], x);
#pragma unroll
        for (int e = 0; e < Ln::N; ++e) acc[e] = Ln::op(acc[e], x[e]);
      }
    }
  }
  return Ln::encode(acc);
}

// ring_fold with two batches of loads in flight: the loads of batch b + 1
// are issued before batch b is folded, so a fold over many ranks waits for
// memory about half as often (the same operations in the same order).
template <typename T, int OP, int NV, class Src, int B = kBatch>
__device__ __forceinline__ typename Unit<T, NV>::Raw ring_fold_2(const Src& src, int R, int j) {
  typedef Unit<T, NV> Un;
  typedef Lanes<T, OP, NV> Ln;
  typename Ln::L acc[Ln::N];
  typename Un::Raw v[2][B];
  auto issue = [&](int buf, int k0) {
#pragma unroll
    for (int i = 0; i < B; ++i) {
      const int k = k0 + i;
      if (k < R) {
        int r = j + k;
        r -= r >= R ? R : 0;
        v[buf][i] = load_unit<T, NV>(src, r);
      }
    }
  };
  auto fold = [&](int buf, int k0) {
#pragma unroll
    for (int i = 0; i < B; ++i) {
      const int k = k0 + i;
      if (k < R) {
        typename Ln::L x[Ln::N];
        Ln::decode(v[buf][i], x);
        if (k == 0) {
#pragma unroll
          for (int e = 0; e < Ln::N; ++e) acc[e] = x[e];
        } else {
#pragma unroll
          for (int e = 0; e < Ln::N; ++e) acc[e] = Ln::op(acc[e], x[e]);
        }
      }
    }
  };
  issue(0, 0);
  for (int k0 = 0; k0 < R; k0 += 2 * B) {
    if (k0 + B < R) issue(1, k0 + B);
    fold(0, k0);
    if (k0 + B < R) {
      if (k0 + 2 * B < R) issue(0, k0 + 2 * B);
      fold(1, k0 + B);
    }
  }
  return Ln::encode(acc);
}

// A unit whose elements [0, split) lie in ring block j and [split, NV) in
// block j+1 (the next block of the same loop): the first folds ranks
// j, j+1, ..., j-1, the second j+1, ..., j-1, j -- the same loads, one rank
// later.  Both folds run over one pass of vector loads (rank j's value is
// kept and folded last into the second), and each element takes its own.
template <typename T, int OP, class Src>
__device__ __forceinline__ uint4 ring_fold_split(const Src& src, int R, int j, int split) {
  constexpr int NV = Ty<T>::U;
  typedef Unit<T, NV> Un;
  typedef Lanes<T, OP, NV> Ln;
  typename Ln::L a[Ln::N], b[Ln::N], first[Ln::N];
#pragma unroll
  for (int e = 0; e < Ln::N; ++e) a[e] = b[e] = first[e] = 0;
  for (int k0 = 0; k0 < R; k0 += kBatch) {
    uint4 v[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int k = k0 + i;
      if (k < R) {
        int r = j + k;
        r -= r >= R ? R : 0;
        v[i] = load_unit<T, NV>(src, r);
      }
    }
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int k = k0 + i;
      if (k < R) {
        typename Ln::L x[Ln::N];
        Ln::decode(v[i], x);
#pragma unroll
        for (int e = 0; e < Ln::N; ++e) {
          if (k == 0) {
            a[e] = x[e];
            first[e] = x[e];
          } else {
            a[e] = Ln::op(a[e], x[e]);
            b[e] = k == 1 ? x[e] : Ln::op(b[e], x[e]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int e = 0; e < Ln::N; ++e) b[e] = R == 1 ? first[e] : Ln::op(b[e], first[e]);
  const uint4 ra = Ln::encode(a), rb = Ln::encode(b);
  // element e of the unit occupies bytes [e*E, (e+1)*E): keep ra's bytes below split*E
  const int cut = split * (int)sizeof(T);
  unsigned w[4];
  const unsigned wa[4] = {ra.x, ra.y, ra.z, ra.w}, wb[4] = {rb.x, rb.y, rb.z, rb.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int lo = 4 * i;  // first byte of word i
    const unsigned keepA = cut >= lo + 4 ? 0xFFFFFFFFu : (cut <= lo ? 0u : (1u << (8 * (cut - lo))) - 1u);
    w[i] = (wa[i] & keepA) | (wb[i] & ~keepA);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Partials of a tree fold.  The top partial lives in fixed registers, so
// the common step -- fold a loaded value into the top -- is straight-line
// code; only a push (a second child's subtree begins) or a pop (it ends)
// touches the slots below, through a switch on the depth.  The depth is the
// same for every lane that follows the same program, so the switches are
// uniform branches, and naming each slot statically keeps them in registers.
template <typename Ln, int S> struct Below {
  static_assert(S == 4 || S == 8, "4 or 8 partials");
  static constexpr int N = Ln::N;
  typename Ln::L b0[N], b1[N], b2[N], b3[N], b4[N], b5[N], b6[N];
};
#define VR_BELOW_SLOTS(X) X(0, b0) X(1, b1) X(2, b2) X(3, b3) X(4, b4) X(5, b5) X(6, b6)

// below[d] = top
template <typename Ln, int S>
__device__ __forceinline__ void below_store(Below<Ln, S>& bl, int d, const typename Ln::L (&top)[Ln::N]) {
  switch (d) {
#define VR_CASE(i, m)                                                       \
  case i:                                                                   \
    if constexpr (i < S - 1) {                                              \
      _Pragma("unroll") for (int e = 0; e < Ln::N; ++e) bl.m[e] = top[e];   \
    }                                                                       \
    break;
    VR_BELOW_SLOTS(VR_CASE)
#undef VR_CASE
  }
}
// top = below[d] (op) top
template <typename Ln, int S>
__device__ __forceinline__ void below_fold(const Below<Ln, S>& bl, int d, typename Ln::L (&top)[Ln::N]) {
  switch (d) {
#define VR_CASE(i, m)                                                                  \
  case i:                                                                              \
    if constexpr (i < S - 1) {                                                         \
      _Pragma("unroll") for (int e = 0; e < Ln::N; ++e) top[e] = Ln::op(bl.m[e], top[e]); \
    }                                                                                  \
    break;
    VR_BELOW_SLOTS(VR_CASE)
#undef VR_CASE
  }
}
#undef VR_BELOW_SLOTS

template <typename T, int OP, int NV, int S, class Src, int B = kBatch>
__device__ __forceinline__ typename Unit<T, NV>::Raw tree_fold(const Src& src, const FoldProg& p,
                                                              int R) {
  typedef Unit<T, NV> Un;
  typedef Lanes<T, OP, NV> Ln;
  typename Ln::L top[Ln::N];
#pragma unroll
  for (int e = 0; e < Ln::N; ++e) top[e] = 0;
  Below<Ln, S> below;
  int sp = 0;  // live partials, the top included
  for (int k0 = 0; k0 < R; k0 += B) {
    typename Un::Raw v[B];
#pragma unroll
    for (int i = 0; i < B; ++i) {
      const int k = k0 + i;
      if (k < R) v[i] = load_unit<T, NV>(src, p.rank[k]);
    }
#pragma unroll
    for (int i = 0; i < B; ++i) {
      const int k = k0 + i;
      if (k < R) {
        const int c = p.ctl[k];
        for (int q = c & 15; q > 0; --q) below_fold<Ln, S>(below, --sp - 1, top);
        typename Ln::L x[Ln::N];
        Ln::decode(v[i], x);
        if (c & 16) {
          if (sp > 0) below_store<Ln, S>(below, sp - 1, top);
#pragma unroll
          for (int e = 0; e < Ln::N; ++e) top[e] = x[e];
          ++sp;
        } else {
#pragma unroll
          for (int e = 0; e < Ln::N; ++e) top[e] = Ln::op(top[e], x[e]);
        }
      }
    }
  }
  for (int q = p.tail; q > 0; --q) below_fold<Ln, S>(below, --sp - 1, top);
  return Ln::encode(top);
}

#ifdef VR_JIT_TREE
// Defined by the run-time compiled source (jit.cc): the straight-line fold of
// program t of the call's programs.
template <typename T, int OP, int NV, class Src>
__device__ __forceinline__ typename Unit<T, NV>::Raw jit_tree_fold(const Src& src, int t);
#endif

// The tree fold of program t: interpreted from its stream, or in a kernel
// compiled at run time for this call's programs (VR_JIT_TREE), the same
// steps as straight-line code -- the same operations in the same order.
template <typename T, int OP, int NV, int S, class Src, int B = kBatch>
__device__ __forceinline__ typename Unit<T, NV>::Raw tree_fold_t(const Src& src,
                                                                const FoldProg* progs, int t,
                                                                int R) {
#ifdef VR_JIT_TREE
  return jit_tree_fold<T, OP, NV, Src>(src, t);
#else
  return tree_fold<T, OP, NV, S, Src, B>(src, progs[t], R);
#endif
}

#ifdef VR_JIT_RING
// Defined by the run-time compiled source (jit.cc) for one rank count: the
// ranks' units loaded in rank order, folded in the rotation of block j.
template <typename T, int OP, int NV, class Src>
__device__ __forceinline__ typename Unit<T, NV>::Raw jit_ring_fold(const Src& src, int j);
#endif

// The ring fold of block j (ranks j, j+1, ..., j-1): the loop above, or in a
// kernel compiled at run time for the call's rank count (VR_JIT_RING), the
// same folds with the loads' ranks fixed at compile time.
template <typename T, int OP, int NV, class Src, int B = kBatch>
__device__ __forceinline__ typename Unit<T, NV>::Raw ring_fold_t(const Src& src, int R, int j) {
#ifdef VR_JIT_RING
  return jit_ring_fold<T, OP, NV, Src>(src, j);
#else
  return ring_fold<T, OP, NV, Src, B>(src, R, j);
#endif
}

// --------------------------------------------------------- partition math
// Where element e sits: its channel range [lo, hi) and, for the ring, its
// block [lo, hi) inside the loop with block number j.  Channels hold 16-byte
// grains split with array_split semantics; ring loops hold R*C elements, the
// last one shorter, each cut into R blocks with array_split semantics.
struct Cursor {
  long long lo, hi;
  int j;  // ring block number
  int t;  // tree index of the channel
  // ring: the current loop's end and block sizes (q + 1 for the first m)
  long long loopEnd, q;
  int m;
};

// a / b for 0 <= a, 0 < b: 32-bit division when both fit (any message under
// 4 Gi elements per rank), the much longer 64-bit sequence otherwise.
__device__ __forceinline__ long long udiv(long long a, long long b) {
  return ((unsigned long long)(a | b) >> 32) == 0 ? (long long)((unsigned)a / (unsigned)b)
                                                  : a / b;
}

// n / d with d's reciprocal M (KArgs): one high multiply when both fit in
// 32 bits (exact there: Lemire, Kaser and Kurz, "Faster remainder by direct
// computation", 2019), a 64-bit division otherwise.
__device__ __forceinline__ long long div_by(long long n, long long d, unsigned long long M) {
  if (((unsigned long long)(n | d) >> 32) == 0)
    return d == 1 ? n : (long long)__umul64hi(M, (unsigned long long)n);
  return n / d;
}

template <int U>
__device__ __forceinline__ void locate_channel(const KArgs& a, long long e, int& k,
                                               long long& cs, long long& ce) {
  const long long g = e / U;
  const long long big = a.gm * (a.gq + 1);
  long long gs;
  if (g < big) {
    k = (int)div_by(g, a.gq + 1, a.mGq1);
    gs = (long long)k * (a.gq + 1);
  } else {
    k = (int)(a.gm + div_by(g - big, a.gq, a.mGq));
    gs = big + (long long)(k - a.gm) * a.gq;
  }
  const long long len = a.gq + (k < a.gm ? 1 : 0);
  cs = gs * U;
  ce = min(a.count, (gs + len) * U);
}

template <int U, int MODE>
__device__ __forceinline__ void locate(const KArgs& a, long long e, Cursor& c) {
  int k;
  long long cs, ce;
  locate_channel<U>(a, e, k, cs, ce);
  if constexpr (MODE == kTreeAllReduce) {
    c.lo = cs;
    c.hi = ce;
    c.t = a.chanProg[k];
    c.j = 0;
  } else {
    const long long R = a.R;
    const long long LC = R * a.chunk;
    const long long off = e - cs;
    const long long ls = div_by(off, LC, a.mLC) * LC;
    const long long L = min(LC, (ce - cs) - ls);
    const long long w = off - ls;
    const long long q = div_by(L, R, a.mR), m = L - q * R;
    long long j, bs, bl;
    if (w < m * (q + 1)) {
      j = udiv(w, q + 1);
      bs = j * (q + 1);
      bl = q + 1;
    } else {
      // a full loop has blocks of exactly `chunk` elements
      const long long rest = w - m * (q + 1);
      j = m + (q == a.chunk ? div_by(rest, q, a.mC) : udiv(rest, q));
      bs = m * (q + 1) + (j - m) * q;
      bl = q;
    }
    c.lo = cs + ls + bs;
    c.hi = c.lo + bl;
    c.j = (int)j;
    c.t = 0;
    c.loopEnd = cs + ls + L;
    c.q = q;
    c.m = (int)m;
  }
}

// Move the cursor to element e.  A thread walks the message forwards, so
// stepping through the following blocks of the same ring loop (adds and
// compares) is the common case; anything else is located from scratch.
template <int U, int MODE>
__device__ __forceinline__ void seek(const KArgs& a, long long e, Cursor& c) {
  if (e >= c.lo && e < c.hi) return;
  if constexpr (MODE != kTreeAllReduce) {
    if (e >= c.hi && e < c.loopEnd) {
      do {
        ++c.j;
        c.lo = c.hi;
        c.hi = c.lo + c.q + (c.j < c.m ? 1 : 0);
      } while (e >= c.hi);
      return;
    }
  }
  locate<U, MODE>(a, e, c);
}

// One element of an AllReduce: its fold in the schedule of element e.
template <typename T, int OP, int MODE, int S, class Src>
__device__ __forceinline__ typename Ty<T>::Bits fold_element(const KArgs& a, const Src& src,
                                                            const FoldProg* progs, long long e,
                                                            Cursor& cur) {
  seek<Ty<T>::U, MODE>(a, e, cur);
  if constexpr (MODE == kTreeAllReduce) return tree_fold<T, OP, 1, S>(src, progs[cur.t], a.R);
  else return ring_fold<T, OP, 1>(src, a.R, cur.j);
}

// Out-of-line copies of the rare paths (a unit cut by a block boundary,
// single elements) for the register-path kernels, whose occupancy depends on
// the streaming loop's registers.  The cursor is taken by value: a reference
// would pin the caller's cursor to local memory for its whole loop.  The
// shared-memory-staged kernels, which run one CTA per SM, inline them.
template <typename T, int OP, class Src>
__device__ __noinline__ uint4 ring_fold_split_rare(const Src src, int R, int j, int split) {
  return ring_fold_split<T, OP>(src, R, j, split);
}
template <typename T, int OP, int MODE, int S, class Src>
__device__ __noinline__ typename Ty<T>::Bits fold_element_rare(const KArgs& a, const Src src,
                                                              const FoldProg* progs, long long e,
                                                              Cursor cur) {
  return fold_element<T, OP, MODE, S>(a, src, progs, e, cur);
}

}  // namespace vr
