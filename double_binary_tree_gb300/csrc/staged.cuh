// TMA-staged collective kernels (sm_103a): AllReduce (ring, tree) and
// ReduceScatter on 16-byte aligned buffers.
//
// One CTA per SM.  The message is cut into tiles of tileUnits 16-byte units
// per rank.  Warp 0 (the producer) moves each tile's R rank slices into a
// stage of shared memory with bulk asynchronous copies (cp.async.bulk, one
// copy of tileBytes per rank, completion counted on the stage's "full"
// mbarrier); the consumer warps wait for the stage, fold its units from
// shared memory in the schedule's order (fold.cuh), each thread a strided
// share of the tile, store the results to every receiving rank straight from
// registers, and hand the stage back on its "empty" mbarrier.  The copies in
// flight depend on the stages, not on registers, which is what bounded the
// register-path kernels.
//
// Reduce-up and broadcast-down of the tree overlap the way the pages'
// runTreeSplit overlaps them ([Course13] "runTreeSplit 如何流水": different
// chunks are in different phases at once): while one stage is folded and
// broadcast, the following stages' inputs are already being reduced into
// shared memory.
//
// Every wait is bounded: after KArgs::timeoutNs the waiting warp records
// VR_ERR_TIMEOUT in the status word and raises the CTA's abort flag; the
// others leave their loops, and the producer still waits (bounded) for every
// copy it issued before the CTA exits, so no copy lands in freed shared
// memory.
#pragma once

#include "fold.cuh"

namespace vr {


__device__ __forceinline__ void mbar_init(uint32_t bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, unsigned bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint32_t bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Completes `bytes` of the barrier's expected transaction count without a
// copy (a bulk load the bounds-checked build refused).
__device__ __forceinline__ void mbar_complete_tx(uint32_t bar, unsigned bytes) {
  asm volatile("mbarrier.complete_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, unsigned bytes,
                                          uint32_t bar) {
  if (!VR_ACCESS_OK(src, bytes, false)) {
    mbar_complete_tx(bar, bytes);
    return;
  }
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait until the phase of `bar` with parity `parity` has completed.  Gives
// up (false) after limit_ns, or as soon as *abort is raised when honor_abort.
__device__ __forceinline__ bool wait_phase(uint32_t bar, unsigned parity, const volatile int* abort,
                                           bool honor_abort, unsigned long long limit_ns) {
  if (mbar_test(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (unsigned it = 1;; ++it) {
    if (mbar_test(bar, parity)) return true;
    if ((it & 15) == 0) {
      if (honor_abort && *abort) return false;
      if (global_ns() - t0 > limit_ns) return false;
    }
  }
}

__device__ __forceinline__ void raise_error(unsigned* status, volatile int* abort, unsigned code) {
  if (status) atomicCAS(status, 0u, code);
  *abort = 1;
}

// ------------------------------------------------------------ tile scheduler
// A staged AllReduce given a scheduler slot (KArgs::sched) does not cut the
// message into one fixed run of tiles per CTA: its producers draw tiles from
// a counter, so that CTAs on SMs that drain faster take more of them.
// With few pipeline stages (many ranks, or few ranks with large tiles) the
// SMs' rates differ by up to a fifth within one launch, and a fixed split
// waits for the slowest.
//
// A slot is four words of global memory: the owning launch (its %gridid,
// which is the same for every CTA of one launch and for every replay of one
// instantiated graph node, and differs between concurrent launches), the next
// tile, and the counts of CTAs that joined and left (32 bits each).  The host
// gives each stream its own slot and each launch captured into a graph a
// slot of its own, so that the launches sharing a slot run one after the
// other; the owner word checks it.  A producer joins after the previous
// kernel on the stream has finished (pdl_wait), and the last CTA to leave
// clears the slot for the next launch.  A slot held by another launch is
// waited for, bounded: a CTA that cannot join reports VR_ERR_TIMEOUT and
// takes no tile; one that finds more joins than the grid has CTAs (a slot
// left behind by an execution of this launch that did not complete) reports
// VR_ERR_INTERNAL and takes none.
constexpr long long kSchedChunkBytes = 64 << 10;  // traffic of the tiles of one draw

// A drawn ring tile's place in the ring schedule, found by the producer (one
// search per tile) and handed to the consumers with the tile: the ring
// block of the tile's first element, that block's loop, and the loop's block
// sizes.  The consumers step forwards from it inside the tile.
struct RingMark {
  long long lo, loopEnd, q;
  int j, m;
};
__device__ __forceinline__ unsigned long long grid_id() {
  unsigned long long g;
  asm volatile("mov.u64 %0, %%gridid;" : "=l"(g));
  return g | (1ull << 63);  // never 0, the free slot's owner
}

// Lane 0 of a producer warp: VR_SUCCESS once this CTA has joined the slot.
__device__ __forceinline__ unsigned sched_join(unsigned long long* slot, unsigned ctas,
                                               unsigned long long limit_ns) {
  const unsigned long long gid = grid_id();
  unsigned long long t0 = 0;
  for (unsigned it = 0;; ++it) {
    const unsigned long long prev = atomicCAS(slot, 0ull, gid);
    if (prev == 0ull || prev == gid) break;
    const unsigned long long now = global_ns();
    if (it == 0) t0 = now;
    else if (now - t0 > limit_ns) return VR_ERR_TIMEOUT;
    __nanosleep(256);
  }
  __threadfence();  // the previous owner's clearing is seen before the counter is used
  return atomicAdd(reinterpret_cast<unsigned*>(slot + 2), 1u) < ctas ? VR_SUCCESS
                                                                     : VR_ERR_INTERNAL;
}

// Lane 0 of a producer warp that joined, after its last draw: the last CTA
// to leave clears the counters, then frees the slot.
__device__ __forceinline__ void sched_leave(unsigned long long* slot, unsigned ctas) {
  __threadfence();
  if (atomicAdd(reinterpret_cast<unsigned*>(slot + 2) + 1, 1u) == ctas - 1) {
    atomicExch(slot + 1, 0ull);
    atomicExch(slot + 2, 0ull);
    __threadfence();
    atomicExch(slot, 0ull);
  }
}

// Tile i of a CTA's work: the byte offset of its slice inside each source
// rank's buffer, the bytes the producer copies, and the units it covers.
// AllReduce: every CTA owns a run [cub, cue) of whole tiles of the message
// (the last tile of the message shorter) and takes them in turn.
// ReduceScatter: tile t (= tb + i) of the whole call, tiles not crossing a
// block.
struct TileGeom {
  long long srcOff;   // bytes from each source buffer's start
  unsigned bytes;     // bytes copied per rank (full 16-byte units only)
  long long u0;       // first unit (AllReduce: of the message; ReduceScatter: of block b)
  int units;          // units in the tile, a trailing partial unit included
  int b;              // ReduceScatter: the block (and receiving rank)
};

template <int MODE>
__device__ __forceinline__ TileGeom tile_geom(const KArgs& a, long long t, long long cub,
                                              long long cue) {
  const int TU = a.tileUnits;
  TileGeom g;
  if constexpr (MODE == kReduceScatter) {
    const long long perB = a.unitsFull;           // units of one block (all full)
    const long long tilesB = (perB + TU - 1) / TU;
    g.b = (int)(t / tilesB);
    const long long tt = t - (long long)g.b * tilesB;
    g.u0 = tt * TU;
    g.units = (int)min((long long)TU, perB - g.u0);
    g.bytes = (unsigned)g.units * 16u;
    g.srcOff = (long long)g.b * perB * 16 + g.u0 * 16;
  } else {
    g.b = 0;
    g.u0 = cub + t * TU;
    g.units = (int)min((long long)TU, cue - g.u0);
    const long long full = min((long long)g.units, max(0LL, a.unitsFull - g.u0));
    g.bytes = (unsigned)full * 16u;
    g.srcOff = g.u0 * 16;
  }
  return g;
}

// DRAWN (AllReduce): the CTAs draw their tiles through the scheduler slot
// KArgs::sched instead of taking fixed runs.
template <typename T, int OP, int MODE, int S, bool DRAWN = false>
__global__ void __launch_bounds__(kWarpSize * (kStagedMaxConsumers + 1), 1)
    staged_kernel(const __grid_constant__ KArgs a) {
  constexpr int U = Ty<T>::U;
  constexpr long long E = sizeof(T);
  extern __shared__ __align__(128) unsigned char smem[];
  const int NS = a.stages;
  const int R = a.R;
  const uint32_t TB = a.tileBytes;                   // bytes per rank per tile
  const uint32_t stageBytes = a.stageBytes;          // R * TB, 128-byte multiple
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);  // full[s] = bars[s], empty[s] = bars[16 + s]
  volatile int* abort = reinterpret_cast<volatile int*>(smem + 16 * kStagedMaxStages);
  const char** s_src = reinterpret_cast<const char**>(smem + 16 * kStagedMaxStages + 16);
  char** s_dst = reinterpret_cast<char**>(smem + 16 * kStagedMaxStages + 16 + 8 * kMaxRanks);
  FoldProg* s_prog = reinterpret_cast<FoldProg*>(s_dst + kMaxRanks);
  // the tile each stage holds, when tiles are drawn at run time (-1: no more),
  // and a drawn ring tile's place in the ring schedule
  volatile long long* s_tile = reinterpret_cast<volatile long long*>(s_prog + kMaxProgs);
  RingMark* s_mark = reinterpret_cast<RingMark*>(
      const_cast<long long*>(s_tile + kStagedMaxStages));
  static_assert(16 * kStagedMaxStages + 16 + 16 * kMaxRanks + kMaxProgs * sizeof(FoldProg) +
                        (8 + sizeof(RingMark)) * kStagedMaxStages <=
                    kStagedHeader,
                "shared-memory header overflows");
  static_assert((16 * kStagedMaxStages + 16 + 16 * kMaxRanks + kMaxProgs * sizeof(FoldProg)) % 8 ==
                0, "tile slots misaligned");
  const uint32_t data = smem_addr(smem + kStagedHeader);
  const unsigned char* stage0 = smem + kStagedHeader;
  const uint32_t full0 = smem_addr(bars), empty0 = smem_addr(bars + kStagedMaxStages);

  const int warp = threadIdx.x / kWarpSize, lane = threadIdx.x % kWarpSize;
  pdl_launch();
  for (int i = threadIdx.x; i < R; i += blockDim.x) {
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
  if (threadIdx.x == 0) {
    *abort = 0;
    for (int s = 0; s < NS; ++s) {
      mbar_init(full0 + 8 * s, 1);   // the producer's arrive (plus the copies' bytes)
      mbar_init(empty0 + 8 * s, a.consumers);  // one release per consumer warp
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();
  pdl_wait();  // the previous kernel on the stream is done

  // this CTA's work: tiles [tb, tb + n) of the call (ReduceScatter), or the
  // units [cub, cue), n tiles (AllReduce); with a scheduler slot, the tiles
  // of the whole range that its producer draws
  long long tb = 0, n = 0, cub = 0, cue = 0;
  constexpr bool dyn = MODE != kReduceScatter && DRAWN;
  if constexpr (MODE == kReduceScatter) {
    tb = udiv(a.tiles * blockIdx.x, gridDim.x);
    n = udiv(a.tiles * (blockIdx.x + 1), gridDim.x) - tb;
  } else if (dyn) {
    cub = a.unitLo;
    cue = a.unitsAll;
    n = a.tiles;
  } else {
    // whole tiles per CTA, on the tile grid of the message: measured 0.5-1.5 %
    // faster than equal runs of units (R = 4, 8 and 64), whose copies do not
    // start on the tile grid (and 1-3 % more when those do not start on
    // 32-byte sectors either)
    const long long tb2 = udiv(a.tiles * blockIdx.x, gridDim.x);
    const long long te2 = udiv(a.tiles * (blockIdx.x + 1), gridDim.x);
    cub = a.unitLo + tb2 * a.tileUnits;
    cue = min(a.unitsAll, a.unitLo + te2 * a.tileUnits);
    n = te2 - tb2;
  }

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const long long stallAt = blockIdx.x == 0 ? a.injectStall : -1;
    long long issued = 0;
    // run-time tiles: draws of K tiles, the next draw made when a draw's
    // first tile is issued (lane 0 holds its result)
    bool joined = false;
    int sent = -1;  // the stage that carried the end mark to the consumers
    long long K = 1, cb = 0, left = 0;
    unsigned long long nb = 0;
    Cursor pcur{0, -1, 0, 0, 0, 0, 0};  // drawn ring: lane 0's place in the schedule
    if (dyn) {
      unsigned e = VR_SUCCESS;
      if (lane == 0) e = sched_join(a.sched, gridDim.x, a.timeoutNs);
      e = __shfl_sync(~0u, e, 0);
      joined = e == VR_SUCCESS;
      if (!joined && lane == 0) raise_error(a.status, abort, e);  // the consumers leave too
      K = max(1LL, kSchedChunkBytes / (2LL * R * TB));
      if (joined && lane == 0) nb = atomicAdd(a.sched + 1, (unsigned long long)K);
    }
    for (long long i = 0; dyn || i < n; ++i) {
      const int s = (int)(i % NS);
      const long long k = i / NS;
      if (k > 0) {
        const bool ok = __any_sync(
            ~0u, wait_phase(empty0 + 8 * s, (unsigned)((k - 1) & 1), abort, true, a.timeoutNs));
        if (!ok) {
          if (lane == 0 && !*abort) raise_error(a.status, abort, VR_ERR_TIMEOUT);
          break;
        }
      }
      if (__shfl_sync(~0u, *abort, 0)) break;
      long long t = tb + i;
      if (dyn) {
        if (left == 0) {
          cb = (long long)__shfl_sync(~0u, nb, 0);
          left = K;
          if (cb < a.tiles && lane == 0) nb = atomicAdd(a.sched + 1, (unsigned long long)K);
        }
        t = cb + (K - left);
        --left;
        if (t >= a.tiles) {  // none left: the consumers stop at this stage
          if (lane == 0) {
            s_tile[s] = -1;
            mbar_arrive(full0 + 8 * s);
          }
          __syncwarp();
          sent = s;
          break;
        }
      }
      const TileGeom g = tile_geom<MODE>(a, t, cub, cue);
      // (a drawn ring tile: the copies are issued first and the tile's mark
      // found while they fly; the producer's arrival, after the mark, ends
      // the stage's phase)
      constexpr bool mark = dyn && MODE == kRingAllReduce;
      if (lane == 0) {
        if (dyn) s_tile[s] = t;
        if (mark) mbar_expect_tx(full0 + 8 * s, (unsigned)R * g.bytes);
        else mbar_arrive_expect_tx(full0 + 8 * s, (unsigned)R * g.bytes);
      }
      __syncwarp();
      issued = i + 1;
      if (i == stallAt) continue;  // test hook: this fill never lands
      if (g.bytes)
        for (int r = lane; r < R; r += kWarpSize)
          bulk_load(data + s * stageBytes + r * TB, s_src[r] + g.srcOff, g.bytes, full0 + 8 * s);
      if constexpr (mark) {
        if (lane == 0) {
          seek<U, MODE>(a, g.u0 * U, pcur);
          s_mark[s] = RingMark{pcur.lo, pcur.loopEnd, pcur.q, pcur.j, pcur.m};
          mbar_arrive(full0 + 8 * s);
        }
      }
    }
    // Drain: every copy issued must have landed before the CTA may exit.
    // (The stage that carried the end mark was waited for as empty, so its
    // last copies have landed; its barrier has moved a phase past them.)
    for (int s = 0; s < NS && s < issued; ++s) {
      const long long last = s + ((issued - 1 - s) / NS) * NS;  // last tile index of stage s
      if (last == stallAt || s == sent) continue;
      const bool ok = __any_sync(
          ~0u, wait_phase(full0 + 8 * s, (unsigned)((last / NS) & 1), abort, false, a.timeoutNs));
      if (!ok && lane == 0) raise_error(a.status, abort, VR_ERR_TIMEOUT);
    }
    if (joined && lane == 0) sched_leave(a.sched, gridDim.x);
    return;
  }

  // ------------------------------------------------------------ consumers
  // Every consumer warp takes part in every tile: thread ct folds the units
  // ct, ct + 32 * NC, ... of the tile.
  const int NC = a.consumers;
  if (warp > NC) return;
  const int ct = threadIdx.x - kWarpSize;
  const int nct = kWarpSize * NC;
  Cursor cur{0, -1, 0, 0, 0, 0, 0};
  for (long long i = 0; dyn || i < n; ++i) {
    const int s = (int)(i % NS);
    const bool ok =
        __any_sync(~0u, wait_phase(full0 + 8 * s, (unsigned)((i / NS) & 1), abort, true, a.timeoutNs));
    if (!ok) {
      if (lane == 0 && !*abort) raise_error(a.status, abort, VR_ERR_TIMEOUT);
      break;
    }
    long long t = tb + i;
    if (dyn) {
      t = s_tile[s];
      if (t < 0) break;
    }
    if constexpr (dyn && MODE == kRingAllReduce) {
      const RingMark mk = s_mark[s];
      cur.lo = mk.lo;
      cur.j = mk.j;
      cur.m = mk.m;
      cur.q = mk.q;
      cur.loopEnd = mk.loopEnd;
      cur.hi = mk.lo + mk.q + (mk.j < mk.m ? 1 : 0);
    }
    const TileGeom g = tile_geom<MODE>(a, t, cub, cue);
    const unsigned char* base = stage0 + (size_t)s * stageBytes;
    for (int lu = ct; lu < g.units; lu += nct) {
      if constexpr (MODE == kReduceScatter) {
        const int j = g.b + 1 == R ? 0 : g.b + 1;
        const SharedSrc src{base + 16 * lu, TB};
        Unit<T, U>::store(s_dst[g.b] + (g.u0 + lu) * 16, ring_fold<T, OP, U>(src, R, j));
      } else {
        const long long u = g.u0 + lu;
        const long long e0 = u * U;
        if (u < a.unitsFull) {
          seek<U, MODE>(a, e0, cur);
          if (e0 + U <= cur.hi) {
            const SharedSrc src{base + 16 * lu, TB};
            typename Unit<T, U>::Raw o;
            if constexpr (MODE == kTreeAllReduce) o = tree_fold_t<T, OP, U, S>(src, s_prog, cur.t, R);
            else o = ring_fold_t<T, OP, U>(src, R, cur.j);
            for (int r = 0; r < R; ++r) Unit<T, U>::store(s_dst[r] + e0 * E, o);
          } else if (MODE == kRingAllReduce && e0 + U <= cur.loopEnd &&
                     e0 + U <= cur.hi + cur.q + (cur.j + 1 < cur.m ? 1 : 0)) {
            // a unit cut by one ring block boundary inside a loop
            const SharedSrc src{base + 16 * lu, TB};
            const uint4 o = ring_fold_split<T, OP>(src, R, cur.j, (int)(cur.hi - e0));
            for (int r = 0; r < R; ++r) st_global_v4(s_dst[r] + e0 * E, o);
          } else {
            // a unit cut by several ring block boundaries: element by element
            for (int x = 0; x < U; ++x) {
              const SharedSrc src{base + 16 * lu + x * E, TB};
              const typename Ty<T>::Bits o =
                  fold_element<T, OP, MODE, S>(a, src, s_prog, e0 + x, cur);
              for (int r = 0; r < R; ++r) Unit<T, 1>::store(s_dst[r] + (e0 + x) * E, o);
            }
          }
        }
        // (the partial unit at the end of the message: below, after the tiles)
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);
  }
  // The partial unit at the end of the message (not copied): its elements,
  // read from global memory, go to different consumer threads of the CTA
  // that owns it, so their loads are not waited for in turn.
  if constexpr (MODE != kReduceScatter) {
    if ((dyn ? blockIdx.x == 0 : cue == a.unitsAll) && a.unitsAll > a.unitsFull &&
        ct < a.hi - a.unitsFull * U) {
      const long long e = a.unitsFull * U + ct;
      const GlobalSrc src{s_src, e * E};
      const typename Ty<T>::Bits o = fold_element<T, OP, MODE, S>(a, src, s_prog, e, cur);
      for (int r = 0; r < R; ++r) Unit<T, 1>::store(s_dst[r] + e * E, o);
    }
  }
}

}  // namespace vr
