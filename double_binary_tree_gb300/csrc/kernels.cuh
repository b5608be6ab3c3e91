// Register-path collective kernels (sm_103a).
//
// Each thread loads the R ranks' copies of a unit straight from global
// memory (up to kBatch loads in flight), folds them (fold.cuh) and stores the
// result to every receiving rank.  They serve AllReduce under 16 MiB per
// rank (under 32 MiB for 2-7 ranks) and the rings of 2 and 6 ranks, the tree
// when run-time specialisation is off, ReduceScatter outside the staged
// kernel's range (16-bit types, more than 8 ranks, under 16 MiB sent per
// rank), and buffers that are not 16-byte aligned (element units).  Larger
// aligned AllReduce runs the TMA-staged kernel of staged.cuh.
//
// Persistent grid: CTA b owns a contiguous run of units and its threads
// stride through it, so a warp touches 512 contiguous bytes of each rank per
// access.  Reduce-up and broadcast-down of the tree are fused per unit: the
// root's value is stored to all R ranks as soon as it is folded.
#pragma once

#include "fold.cuh"

namespace vr {

constexpr int kBlock = 256;  // threads per CTA of the register-path kernels
// Resident CTAs per SM the register-path kernels are compiled for (up to
// 128 registers each): measured faster than 3 CTAs at up to 85 registers,
// which made the ring kernels spill.
#ifndef VR_MIN_BLOCKS_RING
#define VR_MIN_BLOCKS_RING 2
#endif
constexpr int kMinBlocksTree = 2;
constexpr int kMinBlocksRing = VR_MIN_BLOCKS_RING;
constexpr int kMinBlocksSmall = 3;
// Kernels compiled at run time may ask for more resident CTAs (jit.cc).
#ifdef VR_JIT_MIN_BLOCKS
constexpr int kMinBlocksJit = VR_JIT_MIN_BLOCKS;
#else
constexpr int kMinBlocksJit = 0;
#endif

// Rank pointers (and tree programs) copied to shared memory: they are indexed
// by a runtime rank.
// (Also the programmatic-launch handshake: the next kernel may start now,
// and nothing below this call touches global memory before the previous
// kernel is done.)
template <int MODE>
__device__ __forceinline__ void stage_args(const KArgs& a, const char** s_src, char** s_dst,
                                           FoldProg* s_prog) {
  pdl_launch();
  for (int i = threadIdx.x; i < a.R; i += blockDim.x) {
    s_src[i] = static_cast<const char*>(a.src[i]);
    s_dst[i] = static_cast<char*>(a.dst[i]);
  }
  if constexpr (MODE == kTreeAllReduce) {
    const unsigned* from = reinterpret_cast<const unsigned*>(a.prog);
    unsigned* to = reinterpret_cast<unsigned*>(s_prog);
    const int words = a.nProgs * (int)(sizeof(FoldProg) / 4);
    for (int i = threadIdx.x; i < words; i += blockDim.x) to[i] = from[i];
  }
  VR_BOUNDS_SETUP(a);
  __syncthreads();
  pdl_wait();
}

// AllReduce, ring or tree.  VEC: 16-byte units (aligned buffers), else one
// element per unit.  SMALL (at most 4 ranks): a 4-load batch is enough, so
// the kernel fits 3 CTAs per SM (85 registers) -- with few ranks a thread
// has few loads in flight, and only more resident threads make up for it.
template <typename T, int OP, int MODE, bool VEC, int S, bool SMALL>
__global__ void __launch_bounds__(kBlock, kMinBlocksJit ? kMinBlocksJit
                                          : SMALL ? kMinBlocksSmall
                                          : (MODE == kTreeAllReduce ? kMinBlocksTree
                                                                    : kMinBlocksRing))
    allreduce_kernel(const __grid_constant__ KArgs a) {
  constexpr int U = Ty<T>::U;
  constexpr int NV = VEC ? U : 1;
  constexpr long long E = sizeof(T);
  constexpr int B = SMALL ? 4 : kBatch;
  __shared__ const char* s_src[kMaxRanks];
  __shared__ char* s_dst[kMaxRanks];
  __shared__ __align__(16) FoldProg s_prog[kMaxProgs];
  stage_args<MODE>(a, s_src, s_dst, s_prog);

  const int R = a.R;
  const long long count = a.hi;  // end of this launch's range of the message
  const long long u0 = a.lo / NV;
  const long long units = (count + NV - 1) / NV - u0;
  const long long ub = u0 + udiv(units * blockIdx.x, gridDim.x);
  const long long ue = u0 + udiv(units * (blockIdx.x + 1), gridDim.x);
  // The trailing partial unit of a vector call (count % NV elements) is not
  // one thread's work: its elements go to the first threads of the CTA that
  // owns it, before that CTA's main loop, which stops short of it.
  const long long fullU = count / NV;  // (the element path has no partial unit)
  if (VEC && count % NV && fullU >= ub && fullU < ue && threadIdx.x < count - fullU * NV) {
    const long long e = fullU * NV + threadIdx.x;
    const GlobalSrc src{s_src, e * E};
    const typename Ty<T>::Bits o = fold_element_rare<T, OP, MODE, S>(
        a, src, s_prog, e, Cursor{0, -1, 0, 0, 0, 0, 0});
    for (int r = 0; r < R; ++r) Unit<T, 1>::store(s_dst[r] + e * E, o);
  }
  const long long uEnd = VEC && ue > fullU ? fullU : ue;
  Cursor cur{0, -1, 0, 0, 0, 0, 0};
  for (long long u = ub + threadIdx.x; u < uEnd; u += blockDim.x) {
    const long long e0 = u * NV;
    const int n = (int)min((long long)NV, count - e0);
    seek<U, MODE>(a, e0, cur);
    if (n == NV && e0 + NV <= cur.hi) {
      const GlobalSrc src{s_src, e0 * E};
      typename Unit<T, NV>::Raw o;
      if constexpr (MODE == kTreeAllReduce)
        o = tree_fold_t<T, OP, NV, S, GlobalSrc, B>(src, s_prog, cur.t, R);
      else
        o = ring_fold_t<T, OP, NV, GlobalSrc, B>(src, R, cur.j);
      for (int r = 0; r < R; ++r) Unit<T, NV>::store(s_dst[r] + e0 * E, o);
    } else if (MODE == kRingAllReduce && VEC && n == NV && e0 + NV <= cur.loopEnd &&
               e0 + NV <= cur.hi + cur.q + (cur.j + 1 < cur.m ? 1 : 0)) {
      // a unit cut by one ring block boundary inside a loop
      const GlobalSrc src{s_src, e0 * E};
      const uint4 o = ring_fold_split_rare<T, OP>(src, R, cur.j, (int)(cur.hi - e0));
      for (int r = 0; r < R; ++r) st_global_v4(s_dst[r] + e0 * E, o);
    } else {
      // a unit cut by several block boundaries (or, on the element path,
      // the one element of the unit)
      for (int i = 0; i < n; ++i) {
        const long long e = e0 + i;
        const GlobalSrc src{s_src, e * E};
        const typename Ty<T>::Bits o = fold_element_rare<T, OP, MODE, S>(a, src, s_prog, e, cur);
        for (int r = 0; r < R; ++r) Unit<T, 1>::store(s_dst[r] + e * E, o);
      }
    }
  }
}

// ReduceScatter: unit (b, p) folds block b at offset p over ranks b+1, ..., b
// and stores it to rank b only.
template <typename T, int OP, bool VEC>
__global__ void __launch_bounds__(kBlock, kMinBlocksRing)
    reduce_scatter_kernel(const __grid_constant__ KArgs a) {
  constexpr int NV = VEC ? Ty<T>::U : 1;
  constexpr long long E = sizeof(T);
  __shared__ const char* s_src[kMaxRanks];
  __shared__ char* s_dst[kMaxRanks];
  stage_args<kReduceScatter>(a, s_src, s_dst, nullptr);

  const int R = a.R;
  const long long rc = a.count;
  const long long per = (rc + NV - 1) / NV;
  const long long units = per * R;
  const long long ub = udiv(units * blockIdx.x, gridDim.x);
  const long long ue = udiv(units * (blockIdx.x + 1), gridDim.x);
  for (long long u = ub + threadIdx.x; u < ue; u += blockDim.x) {
    const int b = (int)(u / per);
    const long long p0 = (u - (long long)b * per) * NV;
    const int n = (int)min((long long)NV, rc - p0);
    const int j = b + 1 == R ? 0 : b + 1;
    if (n == NV) {
      const GlobalSrc src{s_src, ((long long)b * rc + p0) * E};
      Unit<T, NV>::store(s_dst[b] + p0 * E, ring_fold_2<T, OP, NV>(src, R, j));
    } else {
      for (int i = 0; i < n; ++i) {
        const GlobalSrc src{s_src, ((long long)b * rc + p0 + i) * E};
        Unit<T, 1>::store(s_dst[b] + (p0 + i) * E, ring_fold<T, OP, 1>(src, R, j));
      }
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
  const long long ub = udiv(units * blockIdx.x, gridDim.x);
  const long long ue = udiv(units * (blockIdx.x + 1), gridDim.x);
  for (long long u = ub + threadIdx.x; u < ue; u += blockDim.x) {
    const int r = (int)(u / per);
    const long long off = (u - (long long)r * per) * NB;
    const char* from = s_src[r] + off;
    if constexpr (VEC) {
      const uint4 v = ld_global_v4(from);
      for (int q = 0; q < R; ++q) {
        char* to = s_dst[q] + (long long)r * bytes + off;
        if (to != from) st_global_v4(to, v);
      }
    } else {
      const unsigned char v = ld_ro<unsigned char>(from);
      for (int q = 0; q < R; ++q) {
        char* to = s_dst[q] + (long long)r * bytes + off;
        if (to != from) st_plain<unsigned char>(to, v);
      }
    }
  }
}

}  // namespace vr
