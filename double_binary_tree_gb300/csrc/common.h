// Internal types shared by the host planner and the kernels.
#pragma once

#ifdef __CUDACC_RTC__  // run-time compilation (jit.cc): no C library headers
typedef unsigned char uint8_t;
typedef unsigned short uint16_t;
typedef unsigned int uint32_t;
typedef unsigned long long uint64_t;
typedef long long int64_t;
typedef unsigned long long uintptr_t;
#else
#include <stdint.h>
#endif

#include "../../include/vr.h"

namespace vr {

constexpr int kWarpSize = 32;
constexpr int kMaxRanks = VR_MAX_RANKS;
constexpr int kMaxChannels = VR_MAX_CHANNELS;
constexpr int kGrainBytes = 16;      // channel ranges are cut in 16-byte grains
constexpr int kMaxStack = 8;         // partial sums a tree fold keeps live at once
constexpr int kStagedMaxStages = 16; // shared-memory stages of a staged kernel
constexpr int kStagedMaxConsumers = 7;  // its consumer warps (8 warps per CTA: 2 per SM sub-partition)
constexpr int kStagedHeader = 4096;  // its barriers, flags, pointer tables and programs
constexpr int kMaxProgs = 16;        // distinct tree fold programs per call
// Tile scheduler slots (staged.cuh): 4 words each, one slot per stream and
// one per launch captured into a graph.
constexpr int kSchedSlots = 4096;
constexpr int kSchedStreamSlots = 1024;  // slots [0, 1024) serve streams, the rest captures

// A tree's reduction order as a stream of rank loads.  Slot i loads rank
// rank[i]; before it, ctl[i] & 15 "pop-add" steps fold the top partial into
// the one below it; then the loaded value is pushed as a new partial
// (ctl[i] & 16) or folded into the top partial.  `tail` pop-adds close the
// stream, leaving the root's value as the only partial.
struct alignas(4) FoldProg {
  uint8_t rank[kMaxRanks];
  uint8_t ctl[kMaxRanks];
  uint8_t n;      // == R
  uint8_t tail;
  uint8_t depth;  // deepest partial stack the stream needs
  uint8_t root;   // the tree's root rank
};

enum Mode : int { kRingAllReduce = 0, kTreeAllReduce = 1, kReduceScatter = 2, kAllGather = 3 };

// Phases of one step of the stepwise ring (ablation.cuh).
enum StepPhase : int { kStepSend = 0, kStepReduce = 1, kStepCopy = 2 };

// Everything a collective kernel needs, passed by value as the kernel
// parameter (about 1.2 KB).
struct KArgs {
  const void* src[kMaxRanks];
  void* dst[kMaxRanks];
  long long count;      // AllReduce: elements per rank; ReduceScatter: recvcount;
                        // AllGather: sendcount in bytes
  long long grains;     // AllReduce: 16-byte grains of the message
  long long gq, gm;     // grains / nChannels, grains % nChannels
  long long chunk;      // C, elements per rank per ring loop block
  // 64-bit reciprocals of the partition's divisors (gq + 1, gq, R * chunk, R,
  // chunk): n / d = high 64 bits of M * n for 32-bit n and d, M =
  // floor((2^64 - 1) / d) + 1 (0 for d = 1, which divides trivially).
  unsigned long long mGq1, mGq, mLC, mR, mC;
  long long lo, hi;     // AllReduce: the elements [lo, hi) this launch folds, a piece of the
                        // count-element message whose partition the fields above describe
                        // (lo at a 16-byte boundary); [0, count) for a whole message
  int R;
  int nCh;
  int nProgs;           // fold programs in prog[]
  int pad;
  unsigned* status;     // this device's status word
  void* scratch;        // stepwise ring: the message FIFO (count elements)
  // The call's buffers for the bounds-checked build (bounds.cuh): bytes of
  // every send buffer, of every receive buffer and of the scratch FIFO, and
  // the device word that records the first access outside them.
  unsigned long long srcBytes, dstBytes, scratchBytes;
  unsigned long long* boundsWhere;
  // Staged AllReduce: this launch's tile scheduler slot (tiles drawn at
  // run time), or null (every CTA takes a fixed run of tiles).
  unsigned long long* sched;
  // TMA-staged kernels (staged.cuh)
  long long unitLo;     // AllReduce: first 16-byte unit of the range
  long long unitsAll;   // AllReduce: end unit of the range, a trailing partial one included
  long long unitsFull;  // AllReduce: end of the full units of the range; ReduceScatter: units
                        // per block
  long long tiles;      // tiles of tileUnits units
  unsigned long long timeoutNs;  // limit of every bounded wait
  long long injectStall;         // test hook: CTA 0 never loads its tile of this index (-1: off)
  int stages;           // shared-memory stages
  int consumers;        // consumer warps
  int tileUnits;        // 16-byte units per rank per tile
  unsigned tileBytes;   // bytes per rank per tile (16 * tileUnits)
  unsigned stageBytes;  // R * tileBytes
  uint8_t chanProg[kMaxChannels];  // channel c folds with prog[chanProg[c]]
  FoldProg prog[kMaxProgs];
};

// CUDA's classic limit on a kernel's parameter block.
static_assert(sizeof(KArgs) <= 4096, "kernel arguments exceed 4 KB");

}  // namespace vr
