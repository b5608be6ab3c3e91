// Collective kernels of the emulated ranks (sm_103a).
//
// All R ranks' buffers sit in one GPU's memory, so every "message" of the
// ring or tree schedule stays on chip: a thread loads the R ranks' copies of
// one 16-byte unit, folds them in fp32 registers in exactly the order the
// schedule reduces them, narrows once, and stores the result to every rank
// that receives it.  HBM traffic is the minimum: each input read once, each
// output written once.
//
// Reduction orders (sources: [Interview] "all-reduce 每张卡要发多少数据? ring 和
// tree 有什么区别?", section "手撕代码(NumPy 模拟 ring all-reduce)" and Figure 1;
// [Course13] "NCCL 专家课程 13：Tree、双树、层次化连接与真实交叉区间", sections
// "先固定方向", "runTreeSplit 如何流水", "每种 rank 的操作"):
//   ring AllReduce  element in block j of its loop: ranks j, j+1, ..., j-1
//   ReduceScatter   element of block b: ranks b+1, ..., b
//   tree AllReduce  post-order over the channel's tree, local input first,
//                   children in down[] order (the FoldProg stream)
// Reduce-up and broadcast-down of the tree are fused per unit: the root's
// value is stored to all R ranks as soon as it is folded.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "common.h"

namespace vr {

constexpr int kBlock = 256;  // threads per CTA
constexpr int kBatch = 8;    // rank loads kept in flight per thread

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
__device__ __forceinline__ uint4 ld_v4(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}
__device__ __forceinline__ void st_v4(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// A unit is one 16-byte vector (NV = Ty<T>::U elements) or one element.
template <typename T, int NV> struct Unit {
  typedef typename Ty<T>::Bits Bits;
  typedef typename std::conditional<NV == 1, Bits, uint4>::type Raw;

  static __device__ __forceinline__ Raw load(const char* p) {
    if constexpr (NV == 1) return __ldg(reinterpret_cast<const Bits*>(p));
    else return ld_v4(p);
  }
  static __device__ __forceinline__ void store(char* p, Raw v) {
    if constexpr (NV == 1) *reinterpret_cast<Bits*>(p) = v;
    else st_v4(p, v);
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

// ----------------------------------------------------------- reduction op
// Sum: IEEE fp32 addition, never contracted.  Max: the larger value; for
// equal values the bitwise AND keeps +0 over -0 (and is the identity
// otherwise), so Max is commutative and associative bit-for-bit.
template <int OP> __device__ __forceinline__ float combine(float a, float b) {
  if constexpr (OP == VR_SUM) {
    return __fadd_rn(a, b);
  } else {
    return b > a ? b : (b == a ? __int_as_float(__float_as_int(a) & __float_as_int(b)) : a);
  }
}

// ------------------------------------------------------------------ folds
// Ranks j, j+1, ..., j+R-1 (mod R), left to right.
template <typename T, int OP, int NV>
__device__ __forceinline__ typename Unit<T, NV>::Raw ring_fold(const char* const* src,
                                                              long long off, int R, int j) {
  typedef Unit<T, NV> Un;
  float acc[NV];
#pragma unroll
  for (int e = 0; e < NV; ++e) acc[e] = 0.f;
  for (int k0 = 0; k0 < R; k0 += kBatch) {
    typename Un::Raw v[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int k = k0 + i;
      if (k < R) {
        int r = j + k;
        r -= r >= R ? R : 0;
        v[i] = Un::load(src[r] + off);
      }
    }
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int k = k0 + i;
      if (k < R) {
        float x[NV];
        Un::unpack(v[i], x);
#pragma unroll
        for (int e = 0; e < NV; ++e) acc[e] = k == 0 ? x[e] : combine<OP>(acc[e], x[e]);
      }
    }
  }
  return Un::pack(acc);
}

// Partial-sum stack of a tree fold, kMaxStack named slots.  `sp` is the same
// for every lane that follows the same program, so the switches below are
// uniform branches; each case names its slots statically, which keeps the
// whole stack in registers (an array indexed by `sp` would go to local
// memory).
template <int NV, int S> struct Stack {
  static_assert(S == 4 || S == 8, "stack of 4 or 8 slots");
  float s0[NV], s1[NV], s2[NV], s3[NV], s4[NV], s5[NV], s6[NV], s7[NV];
};
static_assert(kMaxStack == 8, "Stack has at most eight slots");
#define VR_STACK_SLOTS(X) X(0, s0) X(1, s1) X(2, s2) X(3, s3) X(4, s4) X(5, s5) X(6, s6) X(7, s7)

template <int OP, int NV, int S>
__device__ __forceinline__ void stack_push(Stack<NV, S>& st, int sp, const float (&x)[NV]) {
  switch (sp) {
#define VR_CASE(i, m)                                                  \
  case i:                                                              \
    if constexpr (i < S) {                                             \
      _Pragma("unroll") for (int e = 0; e < NV; ++e) st.m[e] = x[e];   \
    }                                                                  \
    break;
    VR_STACK_SLOTS(VR_CASE)
#undef VR_CASE
  }
}
template <int OP, int NV, int S>
__device__ __forceinline__ void stack_add(Stack<NV, S>& st, int sp, const float (&x)[NV]) {
  switch (sp - 1) {
#define VR_CASE(i, m)                                                                         \
  case i:                                                                                     \
    if constexpr (i < S) {                                                                    \
      _Pragma("unroll") for (int e = 0; e < NV; ++e) st.m[e] = combine<OP>(st.m[e], x[e]);    \
    }                                                                                         \
    break;
    VR_STACK_SLOTS(VR_CASE)
#undef VR_CASE
  }
}
// Fold the top partial into the one below it.
template <int OP, int NV, int S>
__device__ __forceinline__ void stack_pop_add(Stack<NV, S>& st, int sp) {
  switch (sp - 1) {
#define VR_CASE(i, lo, hi)                                                                       \
  case i:                                                                                        \
    if constexpr (i < S) {                                                                       \
      _Pragma("unroll") for (int e = 0; e < NV; ++e) st.lo[e] = combine<OP>(st.lo[e], st.hi[e]); \
    }                                                                                            \
    break;
    VR_CASE(1, s0, s1) VR_CASE(2, s1, s2) VR_CASE(3, s2, s3) VR_CASE(4, s3, s4)
    VR_CASE(5, s4, s5) VR_CASE(6, s5, s6) VR_CASE(7, s6, s7)
#undef VR_CASE
  }
}
#undef VR_STACK_SLOTS

template <typename T, int OP, int NV, int S>
__device__ __forceinline__ typename Unit<T, NV>::Raw tree_fold(const char* const* src,
                                                              long long off, const FoldProg& p,
                                                              int R) {
  typedef Unit<T, NV> Un;
  Stack<NV, S> st;
  int sp = 0;
  for (int k0 = 0; k0 < R; k0 += kBatch) {
    typename Un::Raw v[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int k = k0 + i;
      if (k < R) v[i] = Un::load(src[p.rank[k]] + off);
    }
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int k = k0 + i;
      if (k < R) {
        const int c = p.ctl[k];
        for (int q = c & 15; q > 0; --q) {
          stack_pop_add<OP, NV, S>(st, sp);
          --sp;
        }
        float x[NV];
        Un::unpack(v[i], x);
        if (c & 16) {
          stack_push<OP, NV, S>(st, sp, x);
          ++sp;
        } else {
          stack_add<OP, NV, S>(st, sp, x);
        }
      }
    }
  }
  for (int q = p.tail; q > 0; --q) {
    stack_pop_add<OP, NV, S>(st, sp);
    --sp;
  }
  return Un::pack(st.s0);
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
};

template <int U>
__device__ __forceinline__ void locate_channel(const KArgs& a, long long e, int& k,
                                               long long& cs, long long& ce) {
  const long long g = e / U;
  const long long big = a.gm * (a.gq + 1);
  long long gs;
  if (g < big) {
    k = (int)(g / (a.gq + 1));
    gs = (long long)k * (a.gq + 1);
  } else {
    k = (int)(a.gm + (g - big) / a.gq);
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
    c.t = k < a.treeSplit ? 0 : 1;
    c.j = 0;
  } else {
    const long long R = a.R;
    const long long LC = R * a.chunk;
    const long long off = e - cs;
    const long long ls = (off / LC) * LC;
    const long long L = min(LC, (ce - cs) - ls);
    const long long w = off - ls;
    const long long q = L / R, m = L % R;
    long long j, bs, bl;
    if (w < m * (q + 1)) {
      j = w / (q + 1);
      bs = j * (q + 1);
      bl = q + 1;
    } else {
      j = m + (w - m * (q + 1)) / q;
      bs = m * (q + 1) + (j - m) * q;
      bl = q;
    }
    c.lo = cs + ls + bs;
    c.hi = c.lo + bl;
    c.j = (int)j;
    c.t = 0;
  }
}

// ---------------------------------------------------------------- kernels
// Shared-memory copies of the rank pointers (and tree programs): indexed by
// a runtime rank, they must not live in the parameter bank.
template <int MODE>
__device__ __forceinline__ void stage_args(const KArgs& a, const char** s_src, char** s_dst,
                                           FoldProg* s_prog) {
  for (int i = threadIdx.x; i < a.R; i += blockDim.x) {
    s_src[i] = static_cast<const char*>(a.src[i]);
    s_dst[i] = static_cast<char*>(a.dst[i]);
  }
  if constexpr (MODE == kTreeAllReduce) {
    const unsigned* from = reinterpret_cast<const unsigned*>(a.prog);
    unsigned* to = reinterpret_cast<unsigned*>(s_prog);
    for (int i = threadIdx.x; i < (int)(2 * sizeof(FoldProg) / 4); i += blockDim.x) to[i] = from[i];
  }
  __syncthreads();
}

// AllReduce, ring or tree.  Persistent grid: CTA b owns a contiguous run of
// units, its threads stride through it so a warp touches 512 contiguous bytes
// of each rank per access.
// S: partial-sum slots of the tree fold (4 or 8; unused by the ring).
template <typename T, int OP, int MODE, bool VEC, int S>
__global__ void __launch_bounds__(kBlock) allreduce_kernel(const __grid_constant__ KArgs a) {
  constexpr int U = Ty<T>::U;
  constexpr int NV = VEC ? U : 1;
  constexpr long long E = sizeof(T);
  __shared__ const char* s_src[kMaxRanks];
  __shared__ char* s_dst[kMaxRanks];
  __shared__ __align__(16) FoldProg s_prog[2];
  stage_args<MODE>(a, s_src, s_dst, s_prog);

  const int R = a.R;
  const long long count = a.count;
  const long long units = (count + NV - 1) / NV;
  const long long ub = units * blockIdx.x / gridDim.x;
  const long long ue = units * (blockIdx.x + 1) / gridDim.x;
  Cursor cur{0, -1, 0, 0};
  for (long long u = ub + threadIdx.x; u < ue; u += blockDim.x) {
    const long long e0 = u * NV;
    const int n = (int)min((long long)NV, count - e0);
    if (e0 < cur.lo || e0 >= cur.hi) locate<U, MODE>(a, e0, cur);
    if (n == NV && e0 + NV <= cur.hi) {
      typename Unit<T, NV>::Raw o;
      if constexpr (MODE == kTreeAllReduce) o = tree_fold<T, OP, NV, S>(s_src, e0 * E, s_prog[cur.t], R);
      else o = ring_fold<T, OP, NV>(s_src, e0 * E, R, cur.j);
      for (int r = 0; r < R; ++r) Unit<T, NV>::store(s_dst[r] + e0 * E, o);
    } else {
      // a unit cut by the end of the message or by a ring block boundary
      for (int i = 0; i < n; ++i) {
        const long long e = e0 + i;
        if (e < cur.lo || e >= cur.hi) locate<U, MODE>(a, e, cur);
        typename Unit<T, 1>::Raw o;
        if constexpr (MODE == kTreeAllReduce) o = tree_fold<T, OP, 1, S>(s_src, e * E, s_prog[cur.t], R);
        else o = ring_fold<T, OP, 1>(s_src, e * E, R, cur.j);
        for (int r = 0; r < R; ++r) Unit<T, 1>::store(s_dst[r] + e * E, o);
      }
    }
  }
}

// ReduceScatter: unit (b, p) folds block b at offset p over ranks b+1, ..., b
// and stores it to rank b only.
template <typename T, int OP, bool VEC>
__global__ void __launch_bounds__(kBlock) reduce_scatter_kernel(const __grid_constant__ KArgs a) {
  constexpr int NV = VEC ? Ty<T>::U : 1;
  constexpr long long E = sizeof(T);
  __shared__ const char* s_src[kMaxRanks];
  __shared__ char* s_dst[kMaxRanks];
  stage_args<kReduceScatter>(a, s_src, s_dst, nullptr);

  const int R = a.R;
  const long long rc = a.count;
  const long long per = (rc + NV - 1) / NV;
  const long long units = per * R;
  const long long ub = units * blockIdx.x / gridDim.x;
  const long long ue = units * (blockIdx.x + 1) / gridDim.x;
  for (long long u = ub + threadIdx.x; u < ue; u += blockDim.x) {
    const int b = (int)(u / per);
    const long long p0 = (u - (long long)b * per) * NV;
    const int n = (int)min((long long)NV, rc - p0);
    const int j = b + 1 == R ? 0 : b + 1;
    if (n == NV) {
      Unit<T, NV>::store(s_dst[b] + p0 * E,
                         ring_fold<T, OP, NV>(s_src, ((long long)b * rc + p0) * E, R, j));
    } else {
      for (int i = 0; i < n; ++i)
        Unit<T, 1>::store(s_dst[b] + (p0 + i) * E,
                          ring_fold<T, OP, 1>(s_src, ((long long)b * rc + p0 + i) * E, R, j));
    }
  }
}

// AllGather as bytes: unit (r, p) copies 16 bytes (or one byte) of rank r's
// buffer into block r of every rank's output; the copy onto itself of an
// in-place AllGather is skipped.
template <bool VEC>
__global__ void __launch_bounds__(kBlock) allgather_kernel(const __grid_constant__ KArgs a) {
  constexpr int NB = VEC ? 16 : 1;
  __shared__ const char* s_src[kMaxRanks];
  __shared__ char* s_dst[kMaxRanks];
  stage_args<kAllGather>(a, s_src, s_dst, nullptr);

  const int R = a.R;
  const long long bytes = a.count;
  const long long per = (bytes + NB - 1) / NB;
  const long long units = per * R;
  const long long ub = units * blockIdx.x / gridDim.x;
  const long long ue = units * (blockIdx.x + 1) / gridDim.x;
  for (long long u = ub + threadIdx.x; u < ue; u += blockDim.x) {
    const int r = (int)(u / per);
    const long long off = (u - (long long)r * per) * NB;
    const char* from = s_src[r] + off;
    if constexpr (VEC) {
      const uint4 v = ld_v4(from);
      for (int q = 0; q < R; ++q) {
        char* to = s_dst[q] + (long long)r * bytes + off;
        if (to != from) st_v4(to, v);
      }
    } else {
      const unsigned char v = __ldg(reinterpret_cast<const unsigned char*>(from));
      for (int q = 0; q < R; ++q) {
        char* to = s_dst[q] + (long long)r * bytes + off;
        if (to != from) *reinterpret_cast<unsigned char*>(to) = v;
      }
    }
  }
}

}  // namespace vr
