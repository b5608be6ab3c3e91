// Non-fused variants of the AllReduce schedules (sm_103a), kept to measure
// what fusing the schedule into one pass buys.
//
// Two-phase tree ([Course13] "当前环境命中哪个 device 实现": runTreeUpDown
// reduces the whole message up the tree, then broadcasts it down, where
// runTreeSplit overlaps the two): tree_up_kernel folds every unit over its
// channel's tree and stores the value to the tree root's receive buffer only;
// tree_down_kernel then copies it from there to every other rank.  Same fold
// order as the fused kernel, so the same bits; one more read and write of
// the message.
//
// Stepwise ring ([Interview] "手撕代码(NumPy 模拟 ring all-reduce)";
// [Internals] "Ring：带宽友好，但启动步骤会随规模增长"): every reduce-scatter
// and all-gather step of the ring runs as its own pair of launches, and every
// message crosses HBM: the send kernel copies each rank's outgoing block of
// every loop into a FIFO, the receive kernel folds the FIFO into the
// receiving rank's block (or overwrites it, in the all-gather half).  Each
// rank's working copy is its receive buffer, in the element type, so 16-bit
// partials are rounded to the element type at every hop, as messages that
// travel in that type are.
#pragma once

#include "kernels.cuh"

namespace vr {

// ----------------------------------------------------------- two-phase tree
template <typename T, int OP, bool VEC, int S>
__global__ void __launch_bounds__(kBlock, kMinBlocksTree) tree_up_kernel(const __grid_constant__ KArgs a) {
  constexpr int U = Ty<T>::U;
  constexpr int NV = VEC ? U : 1;
  constexpr long long E = sizeof(T);
  __shared__ const char* s_src[kMaxRanks];
  __shared__ char* s_dst[kMaxRanks];
  __shared__ __align__(16) FoldProg s_prog[kMaxProgs];
  stage_args<kTreeAllReduce>(a, s_src, s_dst, s_prog);

  const int R = a.R;
  const long long count = a.count;
  const long long units = (count + NV - 1) / NV;
  const long long ub = udiv(units * blockIdx.x, gridDim.x);
  const long long ue = udiv(units * (blockIdx.x + 1), gridDim.x);
  Cursor cur{0, -1, 0, 0, 0, 0, 0};
  for (long long u = ub + threadIdx.x; u < ue; u += blockDim.x) {
    const long long e0 = u * NV;
    const int n = (int)min((long long)NV, count - e0);
    seek<U, kTreeAllReduce>(a, e0, cur);
    char* root = s_dst[s_prog[cur.t].root];
    if (n == NV) {
      const GlobalSrc src{s_src, e0 * E};
      Unit<T, NV>::store(root + e0 * E, tree_fold<T, OP, NV, S>(src, s_prog[cur.t], R));
    } else {
      for (int i = 0; i < n; ++i) {
        const GlobalSrc src{s_src, (e0 + i) * E};
        Unit<T, 1>::store(root + (e0 + i) * E, tree_fold<T, OP, 1, S>(src, s_prog[cur.t], R));
      }
    }
  }
}

template <typename T, bool VEC>
__global__ void __launch_bounds__(kBlock) tree_down_kernel(const __grid_constant__ KArgs a) {
  constexpr int U = Ty<T>::U;
  constexpr int NV = VEC ? U : 1;
  constexpr long long E = sizeof(T);
  __shared__ const char* s_src[kMaxRanks];
  __shared__ char* s_dst[kMaxRanks];
  __shared__ __align__(16) FoldProg s_prog[kMaxProgs];
  stage_args<kTreeAllReduce>(a, s_src, s_dst, s_prog);

  const int R = a.R;
  const long long count = a.count;
  const long long units = (count + NV - 1) / NV;
  const long long ub = udiv(units * blockIdx.x, gridDim.x);
  const long long ue = udiv(units * (blockIdx.x + 1), gridDim.x);
  Cursor cur{0, -1, 0, 0, 0, 0, 0};
  for (long long u = ub + threadIdx.x; u < ue; u += blockDim.x) {
    const long long e0 = u * NV;
    const int n = (int)min((long long)NV, count - e0);
    seek<U, kTreeAllReduce>(a, e0, cur);
    const int root = s_prog[cur.t].root;
    if (n == NV) {
      const typename Unit<T, NV>::Raw v = ld_plain<typename Unit<T, NV>::Raw>(s_dst[root] + e0 * E);
      for (int r = 0; r < R; ++r)
        if (r != root) Unit<T, NV>::store(s_dst[r] + e0 * E, v);
    } else {
      for (int i = 0; i < n; ++i) {
        const typename Ty<T>::Bits v = ld_plain<typename Ty<T>::Bits>(s_dst[root] + (e0 + i) * E);
        for (int r = 0; r < R; ++r)
          if (r != root) Unit<T, 1>::store(s_dst[r] + (e0 + i) * E, v);
      }
    }
  }
}

// ------------------------------------------------------------ stepwise ring
// Element e of block b: at reduce-scatter step s the block leaves rank b+s
// for rank b+s+1; at all-gather step s it leaves rank b+s-1 for rank b+s.
__device__ __forceinline__ void step_ranks(int R, int phase, int step, int b, int& from,
                                           int& to) {
  from = (b + step + (phase == kStepCopy ? R - 1 : 0)) % R;
  to = from + 1 == R ? 0 : from + 1;
}

// One phase of one ring step over the whole message: kStepSend (of the
// reduce-scatter half, or of the all-gather half when `gather`), then
// kStepReduce or kStepCopy.  The working copies are the receive buffers.
template <typename T, int OP, bool VEC>
__global__ void __launch_bounds__(kBlock)
    ring_step_kernel(const __grid_constant__ KArgs a, int phase, int step, int gather) {
  constexpr int U = Ty<T>::U;
  constexpr int NV = VEC ? U : 1;
  constexpr long long E = sizeof(T);
  typedef Lanes<T, OP, NV> Ln;
  typedef Lanes<T, OP, 1> L1;
  __shared__ const char* s_src[kMaxRanks];
  __shared__ char* s_dst[kMaxRanks];
  stage_args<kRingAllReduce>(a, s_src, s_dst, nullptr);

  const int R = a.R;
  // the send phase of the all-gather half uses the all-gather sender
  const int routing = phase == kStepSend ? (gather ? kStepCopy : kStepReduce) : phase;
  char* fifo = static_cast<char*>(a.scratch);
  const long long count = a.count;
  const long long units = (count + NV - 1) / NV;
  const long long ub = udiv(units * blockIdx.x, gridDim.x);
  const long long ue = udiv(units * (blockIdx.x + 1), gridDim.x);
  Cursor cur{0, -1, 0, 0, 0, 0, 0};
  for (long long u = ub + threadIdx.x; u < ue; u += blockDim.x) {
    const long long e0 = u * NV;
    const int n = (int)min((long long)NV, count - e0);
    seek<U, kRingAllReduce>(a, e0, cur);
    if (n == NV && e0 + NV <= cur.hi) {
      int from, to;
      step_ranks(R, routing, step, cur.j, from, to);
      char* m = fifo + e0 * E;
      typedef typename Unit<T, NV>::Raw Raw;  // 16 bytes, or one element
      if (phase == kStepSend) {
        Unit<T, NV>::store(m, ld_plain<Raw>(s_dst[from] + e0 * E));
      } else if (phase == kStepCopy) {
        Unit<T, NV>::store(s_dst[to] + e0 * E, ld_plain<Raw>(m));
      } else {
        typename Ln::L x[Ln::N], y[Ln::N];
        Ln::decode(ld_plain<Raw>(s_dst[to] + e0 * E), x);
        Ln::decode(ld_plain<Raw>(m), y);
#pragma unroll
        for (int e = 0; e < Ln::N; ++e) x[e] = Ln::op(x[e], y[e]);
        Unit<T, NV>::store(s_dst[to] + e0 * E, Ln::encode(x));
      }
    } else {
      for (int i = 0; i < n; ++i) {
        const long long e = e0 + i;
        seek<U, kRingAllReduce>(a, e, cur);
        int from, to;
        step_ranks(R, routing, step, cur.j, from, to);
        typedef typename Ty<T>::Bits Bits;
        char* m = fifo + e * E;
        if (phase == kStepSend) {
          st_plain<Bits>(m, ld_plain<Bits>(s_dst[from] + e * E));
        } else if (phase == kStepCopy) {
          st_plain<Bits>(s_dst[to] + e * E, ld_plain<Bits>(m));
        } else {
          typename L1::L x[1], y[1];
          L1::decode(ld_plain<Bits>(s_dst[to] + e * E), x);
          L1::decode(ld_plain<Bits>(m), y);
          x[0] = L1::op(x[0], y[0]);
          st_plain<Bits>(s_dst[to] + e * E, L1::encode(x));
        }
      }
    }
  }
}

// recv[r] = send[r] for every rank whose buffers differ (the stepwise ring's
// working copies start as the inputs).
template <bool VEC>
__global__ void __launch_bounds__(kBlock) copy_ranks_kernel(const __grid_constant__ KArgs a) {
  constexpr int NB = VEC ? 16 : 1;
  __shared__ const char* s_src[kMaxRanks];
  __shared__ char* s_dst[kMaxRanks];
  stage_args<kAllGather>(a, s_src, s_dst, nullptr);
  const int R = a.R;
  const long long bytes = a.count;  // per rank
  const long long per = (bytes + NB - 1) / NB;
  const long long units = per * R;
  const long long ub = udiv(units * blockIdx.x, gridDim.x);
  const long long ue = udiv(units * (blockIdx.x + 1), gridDim.x);
  for (long long u = ub + threadIdx.x; u < ue; u += blockDim.x) {
    const int r = (int)(u / per);
    if (s_src[r] == s_dst[r]) continue;
    const long long off = (u - (long long)r * per) * NB;
    if constexpr (VEC) {
      if (off + 16 <= bytes) {
        st_global_v4(s_dst[r] + off, ld_global_v4(s_src[r] + off));
      } else {  // the buffer's last bytes, short of a whole 16-byte unit
        for (long long b = off; b < bytes; ++b)
          st_plain<char>(s_dst[r] + b, ld_plain<char>(s_src[r] + b));
      }
    } else {
      st_plain<char>(s_dst[r] + off, ld_plain<char>(s_src[r] + off));
    }
  }
}

}  // namespace vr
