// Host-side planning functions and kernel launchers (internal).
#pragma once

#include <cuda_runtime.h>

#include "common.h"

namespace vr {

// Tuning and test options (options.cc): the environment's values at the
// first use, then whatever vr_set_option stored.  -1: the call site's
// default applies.
enum Option : int {
  kOptKernelPath,      // 0 auto, 1 register path, 2 staged kernel
  kOptJit,             // 0: interpreting folds only
  kOptJitRing,         // 0 never, 1 also staged, 2 register path only
  kOptJitOcc,          // 0 never, 4 always, else by rounds
  kOptSmallRanks,      // 0: no few-rank register-path variant
  kOptPdl,             // 0: no programmatic stream serialisation
  kOptSpread,          // 0: no CTA shrinking for small calls
  kOptStagedMinBytes,  // staged kernel from this many bytes per rank
  kOptStagedTileBytes, // 0: the built-in tile
  kOptStagedMinStages, // -1: by rank count
  kOptStagedStages,    // 0: as many as fit
  kOptAgTile,          // -1: gather_tile_bytes()
  kOptAgStages,        // -1: gather_stages()
  kOptAgCtas,          // -1: gather_ctas_per_sm()
  kOptAgOrder,         // 0 by source size, 1 source-major, 2 destination-major
  kOptSched,           // staged trees' tiles: 0 fixed runs, 1 drawn where faster, 2 always drawn
  kOptDebug,           // bit set of kDebug* subsystems
  kOptCount
};
constexpr long long kDebugGraph = 1;  // print tree, ring and partition tables
long long option(Option o);
long long option_or(Option o, long long dflt);

// The argument and buffer checks of the stepwise ring AllReduce, its
// scratch aside (api.cc): VR_SUCCESS or the code the call returns.
vr_result_t check_stepwise_args(const void* const* sendbufs, void* const* recvbufs, int R,
                                size_t count, int dtype, int op, int nChannels,
                                size_t chunkBytes);

// The option VR_DEBUG=GRAPH (graphlog.cc): tree and ring tables, and a
// collective call's plan the first time the process sees it (its channel
// partition when `partitioned`), printed to stderr; no-ops otherwise.
bool graph_logging();
void log_trees(const vr_tree_t* trees, int R, int nCh);
void log_ring(const int* next, int R, int nCh);
void log_plan(const char* kind, int algo, int R, int L, size_t count, int dtype, int nCh,
              size_t chunkBytes, const vr_tree_t* trees, bool partitioned);

void build_ring(int R, int nCh, int* next, int* prev);
void btree(int n, int r, int* up, int* d0, int* d1, int* childType);
void dtree(int n, int r, int t[2][4]);
int channel_tree(int c, int nCh);
vr_result_t build_dtree(int nNodes, int L, int nCh, vr_tree_t* out);
vr_result_t build_dtree_ex(int nNodes, int L, int nCh, int pattern, const int* orders,
                           vr_tree_t* out);
bool valid_tree(const vr_tree_t* tree, int R);
vr_result_t compile_fold(const vr_tree_t* tree, int R, FoldProg* prog);
vr_result_t dtree_programs(int nNodes, int L, FoldProg out[2]);

// Tree kernel specialised at run time for a call's fold programs (jit.cc):
// the shared-memory-staged one when `staged` (drawing its tiles through
// KArgs::sched when `drawn`), else the register-path one (16-byte units; the
// few-rank variant when `small`; compiled for at least `minBlocks` resident
// CTAs per SM when it is above 0).
bool jit_enabled();
vr_result_t jit_tree_kernel(int dtype, int op, int stack, bool small, bool staged,
                            const FoldProg* progs, int nProgs, const void** out,
                            int minBlocks = 0, bool drawn = false);
// The ring AllReduce kernel specialised for R ranks (the same variants).
vr_result_t jit_ring_kernel(int dtype, int op, int R, bool small, bool staged, const void** out,
                            int minBlocks = 0);
void jit_counts(long long* compiled, long long* failed);
vr_result_t jit_compile_dtree(int nNodes, int L, int dtype, int op, int arch,
                              size_t* cubinBytes, char* log, size_t logBytes);
vr_result_t jit_compile_ring(int R, int dtype, int op, int arch, size_t* cubinBytes, char* log,
                             size_t logBytes);

// Kernel entry points, one getter per element type: `mode` is a Mode,
// `vec` selects the 16-byte vector path (all buffers and block offsets
// 16-byte aligned), else the element path; `stack` is the deepest partial
// stack of the tree programs (selects the 4- or 8-slot tree kernel).
// `small`: the register-path variant for at most 4 ranks (vector path).
const void* kernel_ptr_f32(int mode, int op, bool vec, int stack, bool small);
const void* kernel_ptr_f16(int mode, int op, bool vec, int stack, bool small);
const void* kernel_ptr_bf16(int mode, int op, bool vec, int stack, bool small);
const void* kernel_ptr_allgather(bool vec);
// TMA AllGather (16-byte aligned buffers): one warp per CTA.
const void* kernel_ptr_allgather_tma(int tile, int stages);
// The destination-major one (sources small enough to stay in L2).
const void* kernel_ptr_allgather_tma_dest(int tile, int stages);
int gather_tile_bytes();
int gather_stages();
int gather_ctas_per_sm();
// `drawn` (AllReduce): the variant whose CTAs draw tiles through KArgs::sched.
const void* staged_kernel_ptr_f32(int mode, int op, int stack, bool drawn);
const void* staged_kernel_ptr_f16(int mode, int op, int stack, bool drawn);
const void* staged_kernel_ptr_bf16(int mode, int op, int stack, bool drawn);

// Non-fused variants (kernels_ablation.cu).
enum AblationKernel : int { kTreeUp = 0, kTreeDown = 1, kRingStep = 2, kCopyRanks = 3 };
const void* ablation_kernel_ptr(int which, int dtype, int op, bool vec, int stack);

// The current device's status word: its address, and read-and-clear.
cudaError_t status_word_address(unsigned** p);
cudaError_t read_and_clear_status(unsigned* value);
// The word where the bounds-checked build records the first refused
// address: its address, and read-and-clear.
cudaError_t bounds_word_address(unsigned long long** p);
cudaError_t read_and_clear_bounds(unsigned long long* value);
// The current device's tile scheduler slots (kSchedSlots x 4 words).
cudaError_t sched_table_address(unsigned long long** p);

}  // namespace vr
