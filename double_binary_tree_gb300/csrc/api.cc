// The C ABI of include/vr.h: argument checks, host planning and the kernel
// launches of each collective call (one for the fused collectives).
#include <algorithm>
#include <array>
#include <atomic>
#include <climits>
#include <cstdint>
#include <cstdlib>
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <thread>
#include <tuple>
#include <utility>

#include "host.h"

namespace vr {
namespace {

constexpr int kBlockThreads = 256;  // must equal kBlock of kernels.cuh

std::atomic<unsigned long long> g_launches{0};
std::mutex g_mu;

struct DeviceInfo {
  int sms = 0;
  int l2Bytes = 0;
  int smemOptin = 0;  // largest dynamic shared memory a CTA may opt into
  unsigned* status = nullptr;
  unsigned long long* boundsWhere = nullptr;  // first refused address (bounds-checked build)
  unsigned long long* sched = nullptr;        // tile scheduler slots (kSchedSlots x 4 words)
};
std::map<int, DeviceInfo> g_devices;                             // by device ordinal
std::map<std::pair<const void*, int>, int> g_occupancy;          // (kernel, device)
std::map<std::pair<int, int>, std::array<FoldProg, 2>> g_progs;  // (nNodes, localRanks)
std::map<std::pair<const void*, int>, int> g_smemSet;            // (kernel, device) -> bytes
std::map<std::pair<const void*, int>, int> g_staticSmem;         // (kernel, device) -> bytes
// Tile scheduler slots handed out: one per stream (per host thread for the
// per-thread default stream) and one per launch captured into a graph.
std::map<std::tuple<int, cudaStream_t, std::thread::id>, int> g_streamSlots;
std::map<int, int> g_streamSlotsUsed, g_captureSlotsUsed;  // by device
std::atomic<long long> g_stallNext{-1};                          // test hook
std::atomic<long long> g_shrinkNext{0};                          // test hook (bounds-checked build)
std::atomic<int> g_shrinkWhich{0};

// Test hook of the bounds-checked build: the next launch's recorded buffer
// extents (send 1, receive 2, FIFO 4 in `which`) end `n` bytes early -- the
// buffers themselves are untouched, so its last accesses are refused without
// any access outside real memory.
void shrink_extents(KArgs& a) {
  const long long n = g_shrinkNext.exchange(0);
  const int which = g_shrinkWhich.load();
  if (n <= 0) return;
  const unsigned long long k = (unsigned long long)n;
  auto cut = [k](unsigned long long x) { return x > k ? x - k : 0ull; };
  if (which & 1) a.srcBytes = cut(a.srcBytes);
  if (which & 2) a.dstBytes = cut(a.dstBytes);
  if (which & 4) a.scratchBytes = cut(a.scratchBytes);
}

unsigned long long wait_timeout_ns() {
  static const unsigned long long ns = [] {
    const char* v = std::getenv("VR_WAIT_TIMEOUT_NS");
    const unsigned long long x = v ? std::strtoull(v, nullptr, 10) : 0;
    return x ? x : 1000000000ull;  // 1 s
  }();
  return ns;
}

// Test and tuning option VR_KERNEL_PATH: 1 (register) or 2 (staged) forces
// aligned AllReduce / ReduceScatter onto one kernel family.
int forced_path() { return (int)option(kOptKernelPath); }

size_t elem_size(int dtype) {
  switch (dtype) {
    case VR_FLOAT32: return 4;
    case VR_FLOAT16:
    case VR_BFLOAT16: return 2;
    default: return 0;
  }
}

vr_result_t device_info(DeviceInfo* out, int* device) {
  if (cudaGetDevice(device) != cudaSuccess) return VR_ERR_CUDA;
  std::lock_guard<std::mutex> g(g_mu);
  auto it = g_devices.find(*device);
  if (it == g_devices.end()) {
    DeviceInfo d;
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, *device) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.smemOptin, cudaDevAttrMaxSharedMemoryPerBlockOptin, *device) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&d.l2Bytes, cudaDevAttrL2CacheSize, *device) != cudaSuccess)
      return VR_ERR_CUDA;
    if (status_word_address(&d.status) != cudaSuccess ||
        bounds_word_address(&d.boundsWhere) != cudaSuccess ||
        sched_table_address(&d.sched) != cudaSuccess)
      return VR_ERR_CUDA;
    it = g_devices.emplace(*device, d).first;
  }
  *out = it->second;
  return VR_SUCCESS;
}

int blocks_per_sm(const void* fn, int device) {
  std::lock_guard<std::mutex> g(g_mu);
  auto key = std::make_pair(fn, device);
  auto it = g_occupancy.find(key);
  if (it != g_occupancy.end()) return it->second;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kBlockThreads, 0) != cudaSuccess || n < 1)
    n = 1;
  g_occupancy[key] = n;
  return n;
}

vr_result_t tree_programs(int nNodes, int L, std::array<FoldProg, 2>* out) {
  std::lock_guard<std::mutex> g(g_mu);
  auto key = std::make_pair(nNodes, L);
  auto it = g_progs.find(key);
  if (it == g_progs.end()) {
    std::array<FoldProg, 2> p;
    const vr_result_t e = dtree_programs(nNodes, L, p.data());
    if (e != VR_SUCCESS) return e;
    it = g_progs.emplace(key, p).first;
  }
  *out = it->second;
  return VR_SUCCESS;
}

// The double tree's two programs; channels [0, ceil(nCh/2)) fold with tree
// 0, the others with tree 1.
void set_dtree_programs(KArgs& a, const std::array<FoldProg, 2>& p, int nCh) {
  a.prog[0] = p[0];
  a.prog[1] = p[1];
  a.nProgs = 2;
  for (int c = 0; c < nCh; ++c) a.chanProg[c] = (uint8_t)channel_tree(c, nCh);
}

bool overlap(uintptr_t a, size_t an, uintptr_t b, size_t bn) {
  return an && bn && a < b + bn && b < a + an;
}

// Buffer rules shared by the collectives.  recv[r] may not touch another
// rank's send or recv buffer; against its own send buffer it is either
// disjoint or in the collective's in-place position: recv == send + recvAt
// (AllReduce: 0, ReduceScatter: r * recvBytes) or send == recv + sendAt
// (AllGather: r * sendBytes).
// Every buffer must also be aligned to the element size E: the element
// path accesses whole elements.
enum Kind { kAR, kRS, kAG };
vr_result_t check_buffers(const void* const* send, void* const* recv, int R, size_t sendBytes,
                          size_t recvBytes, Kind kind, size_t E, bool nullRecvOk = false) {
  if (!send || !recv) return VR_ERR_INVALID_ARGUMENT;
  for (int r = 0; r < R; ++r) {
    if ((sendBytes && !send[r]) || (recvBytes && !recv[r] && !nullRecvOk))
      return VR_ERR_INVALID_ARGUMENT;
    if (((uintptr_t)send[r] | (uintptr_t)recv[r]) % E) return VR_ERR_INVALID_ARGUMENT;
  }
  if (!recvBytes) return VR_SUCCESS;
  // Receive buffers (all recvBytes long) sorted by address must be pairwise
  // disjoint: each one ends before the next begins.
  struct Iv {
    uintptr_t lo;
    int r;
  };
  Iv rv[kMaxRanks];
  int n = 0;
  for (int r = 0; r < R; ++r)
    if (recv[r]) rv[n++] = Iv{(uintptr_t)recv[r], r};  // NULL: nothing received
  std::sort(rv, rv + n, [](const Iv& x, const Iv& y) { return x.lo < y.lo; });
  for (int i = 1; i < n; ++i)
    if (rv[i].lo - rv[i - 1].lo < recvBytes) return VR_ERR_INVALID_ARGUMENT;
  if (!sendBytes) return VR_SUCCESS;
  // A send buffer may touch no receive buffer but its own rank's, and that
  // one only in the collective's in-place position.  The receive buffers
  // that overlap send[q] are consecutive in address order (equal lengths,
  // disjoint): the first one ending after send[q] begins, and those after it
  // that begin before send[q] ends.
  for (int q = 0; q < R; ++q) {
    const uintptr_t s = (uintptr_t)send[q];
    int i = (int)(std::lower_bound(rv, rv + n, s,
                                   [&](const Iv& x, uintptr_t v) { return x.lo + recvBytes <= v; }) -
                  rv);
    for (; i < n && rv[i].lo < s + sendBytes; ++i) {
      if (rv[i].r != q) return VR_ERR_INVALID_ARGUMENT;
      const uintptr_t d = rv[i].lo;
      bool inPlace = false;
      if (kind == kAR) inPlace = d == s;
      if (kind == kRS) inPlace = d == s + (uintptr_t)q * recvBytes;
      if (kind == kAG) inPlace = s == d + (uintptr_t)q * sendBytes;
      if (!inPlace) return VR_ERR_INVALID_ARGUMENT;
    }
  }
  return VR_SUCCESS;
}

// Optional (VR_VALIDATE_POINTERS=1): every buffer must be reachable from the
// current device.  Off by default: it costs a driver query per buffer.
vr_result_t check_reachable(const void* const* ptrs, int R, int device) {
  static const bool on = [] {
    const char* v = std::getenv("VR_VALIDATE_POINTERS");
    return v && v[0] == '1';
  }();
  if (!on) return VR_SUCCESS;
  for (int r = 0; r < R; ++r) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, ptrs[r]) != cudaSuccess) {
      cudaGetLastError();
      return VR_ERR_INVALID_ARGUMENT;
    }
    if (at.type == cudaMemoryTypeUnregistered) return VR_ERR_INVALID_ARGUMENT;
    if (at.type == cudaMemoryTypeDevice && at.device != device) return VR_ERR_INVALID_ARGUMENT;
    if (at.type == cudaMemoryTypeHost && at.devicePointer == nullptr) return VR_ERR_INVALID_ARGUMENT;
  }
  return VR_SUCCESS;
}

bool aligned16(const void* const* p, int R, size_t extraStride) {
  for (int r = 0; r < R; ++r)
    if (((uintptr_t)p[r] | extraStride) & 15) return false;
  return true;
}

const void* pick_staged(int dtype, int mode, int op, int stack = 0, bool drawn = false) {
  switch (dtype) {
    case VR_FLOAT32: return staged_kernel_ptr_f32(mode, op, stack, drawn);
    case VR_FLOAT16: return staged_kernel_ptr_f16(mode, op, stack, drawn);
    case VR_BFLOAT16: return staged_kernel_ptr_bf16(mode, op, stack, drawn);
    default: return nullptr;
  }
}

// Register-path kernel; fp32 with at most 4 ranks takes the variant compiled
// for 3 CTAs per SM (1.2-1.5x faster from 16 MiB per rank; slower for 16-bit
// types, which keep the general kernel).  Rings below 8 MiB per rank keep
// the general kernel too: measured at 4 ranks, 17 % faster at 1 MiB and 2 %
// at 4 MiB, 7 % slower at 16 and 24 MiB (trees: no difference).  The option
// VR_SMALL_RANKS=0 turns it off for tuning.
bool use_small(int dtype, int mode, bool vec, int stack, int R, size_t bytesPerRank) {
  return dtype == VR_FLOAT32 && vec && R <= 4 && stack <= 4 && mode != kReduceScatter &&
         (mode != kRingAllReduce || bytesPerRank >= (8u << 20)) && option(kOptSmallRanks) != 0;
}
const void* pick_kernel(int dtype, int mode, int op, bool vec, int stack = 0, int R = 64,
                        size_t bytesPerRank = 0) {
  const bool small = use_small(dtype, mode, vec, stack, R, bytesPerRank);
  switch (dtype) {
    case VR_FLOAT32: return kernel_ptr_f32(mode, op, vec, stack, small);
    case VR_FLOAT16: return kernel_ptr_f16(mode, op, vec, stack, small);
    case VR_BFLOAT16: return kernel_ptr_bf16(mode, op, vec, stack, small);
    default: return nullptr;
  }
}

// Launches `fn`.  With programmatic stream serialisation (`pdl`, unless
// VR_PDL=0) the kernel may start while the previous kernel on the stream
// drains -- every kernel here waits for it (pdl_wait) before touching global
// memory.  Measured on GB300: 4-15% faster back-to-back AllReduce of 64 KiB -
// 4 MiB per rank, 0.6-1.4% from 64 MiB, neutral for ReduceScatter; 10%
// slower for the TMA AllGather, which therefore launches without it.
cudaError_t launch_kernel(const void* fn, dim3 grid, dim3 block, void** args, size_t smem,
                          void* stream, bool pdl = true) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[1];
  if (pdl && option(kOptPdl)) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelExC(&cfg, fn, args);
}

vr_result_t launch(const void* fn, KArgs& a, long long units, void* stream,
                   void** extra = nullptr, int nExtra = 0) {
  if (!fn) return VR_ERR_INTERNAL;
  DeviceInfo di;
  int device = 0;
  vr_result_t e = device_info(&di, &device);
  if (e != VR_SUCCESS) return e;
  if ((e = check_reachable(a.src, a.R, device)) != VR_SUCCESS) return e;
  if ((e = check_reachable(const_cast<const void* const*>(a.dst), a.R, device)) != VR_SUCCESS)
    return e;
  a.status = di.status;
  a.boundsWhere = di.boundsWhere;
  shrink_extents(a);
  const long long resident = (long long)di.sms * blocks_per_sm(fn, device);
  const long long wanted = (units + kBlockThreads - 1) / kBlockThreads;
  // Fewer units than 256-thread CTAs to cover every SM: smaller CTAs (a
  // warp multiple), so that the work spreads over all SMs instead of
  // queueing on a few (each SM's load bandwidth bounds a small call).
  int block = kBlockThreads;
  if (wanted < di.sms && option(kOptSpread)) {
    const long long perSm = (units + di.sms - 1) / di.sms;
    block = (int)std::min<long long>(kBlockThreads, std::max<long long>(32, (perSm + 31) / 32 * 32));
  }
  const long long grid =
      std::max(1LL, std::min(resident, (units + block - 1) / block));
  void* args[4] = {&a, nullptr, nullptr, nullptr};
  for (int i = 0; i < nExtra && i < 3; ++i) args[1 + i] = extra[i];
  if (launch_kernel(fn, dim3((unsigned)grid), dim3(block), args, 0, stream) != cudaSuccess)
    return VR_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return VR_SUCCESS;
}

// Staged geometry of an AllReduce of 2-7 ranks: bytes per rank per tile and
// stages (0: no staged kernel).  Measured on GB300 (fp32, 16 / 64 / 256 MiB
// per rank, cold buffers, graph replays, tiles of 4-14 KB per rank and 3-5
// stages): the best stages hold 20-43 KB, three to five of them -- a short
// pipeline of large copies, where 8 and more ranks do best with many small
// stages.  With 2-5 ranks the register path keeps every thread's few loads
// waiting in turn and reaches 0.67-0.91 of the copy bandwidth; these tiles
// reach 0.93-0.99 from 64 MiB per rank (2 ranks: tree 0.86-0.93).  The ring
// of 2 ranks and of 6 ranks keeps the register path (the staged ring was
// slower there); from 16 to 64 MiB the gain grows from none to 4-10 %.
struct SmallGeometry {
  unsigned tile;
  int stages;
};
// `drawn`: the geometry of a launch that draws its tiles, where it differs --
// the 4-rank ring: 12 KB x 3 (0.965 of the copy bandwidth at 64 MiB per rank
// against 0.92 with 8 KB x 4 drawn and 0.93 with fixed runs; 12 KB x 3 with
// fixed runs 0.86).
SmallGeometry small_geometry(int mode, int R, bool drawn = false) {
  if (drawn && mode == kRingAllReduce && R == 4) return {12288, 3};
  static const SmallGeometry ring[8] = {{0, 0},    {0, 0},    {0, 0},    {14336, 3},
                                        {8192, 4}, {6144, 3}, {0, 0},    {4096, 4}};
  static const SmallGeometry tree[8] = {{0, 0},    {0, 0},    {14336, 4}, {8192, 4},
                                        {7168, 3}, {6144, 3}, {4096, 4},  {4096, 3}};
  if (R < 2 || R > 7) return {0, 0};
  return mode == kRingAllReduce ? ring[R] : mode == kTreeAllReduce ? tree[R] : SmallGeometry{0, 0};
}
constexpr size_t kSmallStagedMinBytes = 32u << 20;  // per rank, 2-7 ranks

// Whether a staged AllReduce of R ranks of `dtype` draws its tiles at run
// time (VR_SCHED=1).  Measured against fixed runs on one GB300 (16-256 MiB
// per rank): trees 1-5 % faster for 4-7 ranks, 12-16 % for 9-16 (4 KB
// tiles), 10-12 % for 17-64; rings 12-15 % faster for 16-33 ranks, 8 % for
// 48 and 1 % for 64 (whose fold, a loop over 64 rotated ranks in 3 consumer
// warps, bounds it), and for 9-15 ranks 13-19 % in fp32 but within 2 % in
// fp16 (each 16-byte unit twice the elements to widen and add: the
// consumers, not the SMs' copy rates, bound those); the 4-rank fp32 ring,
// with larger tiles (small_geometry), 4-5 % at 32-256 MiB per rank.
// Slower: 2-3 rank trees (9 %), 8 ranks (trees 7-13 %, rings 22-24 %: the
// one geometry with both 2 KB tiles and a deep pipeline, 13 stages, where the
// SMs' rates stay even and each tile's drawn index costs the consumers a
// shared-memory round trip on one unit of work per thread); 3, 5 and 7 rank
// rings are within 2 % either way with their fixed-run geometry.
bool sched_tiles(int mode, int R, int dtype) {
  const long long o = option(kOptSched);
  if (o == 0) return false;
  if (o >= 2) return true;
  if (mode == kTreeAllReduce) return R >= 4 && R != 8;
  return R >= 16 || ((R == 4 || R >= 9) && dtype == VR_FLOAT32);
}

// Which kernel family serves an aligned AllReduce.  Below 16 MiB per rank
// the staged kernel's pipeline does not fill.  Measured on GB300: from 16 MiB
// per rank the staged kernel beats the register path for the ring of 8-64
// ranks and, with its fold specialised at run time (jit.cc), for the tree of
// 8-64 ranks (the interpreting staged tree is 2-3x slower than the register
// path); with 2-7 ranks it wins from 32 MiB per rank with the geometry above.
bool use_staged(int mode, int R, size_t bytesPerRank) {
  const size_t minBytes = (size_t)option(kOptStagedMinBytes);
  // Trees that draw their tiles beat the register path earlier: above 8
  // ranks from half the threshold (R = 12 / 16 bf16 at 8 MiB per rank: 0 /
  // 5 % faster, at 12 MiB 9 / 12 %), and 5-7 ranks from 24 MiB (2-6 %
  // faster there, 0-2 % slower at 16 MiB; 4 ranks stay 2-14 % slower below
  // 32 MiB).
  // (the trees' drawing rule does not depend on the element type)
  const bool drawnTree = mode == kTreeAllReduce && sched_tiles(mode, R, VR_FLOAT32);
  if (R < 8) {
    const size_t small =
        drawnTree && R >= 5 ? kSmallStagedMinBytes * 3 / 4 : kSmallStagedMinBytes;
    if (small_geometry(mode, R).tile == 0 || bytesPerRank < std::max(minBytes, small))
      return false;
  } else if (bytesPerRank < (drawnTree ? minBytes / 2 : minBytes)) {
    return false;
  }
  if (mode == kRingAllReduce) return true;
  if (mode == kTreeAllReduce) return jit_enabled();
  return false;
}

// ReduceScatter: one store per unit leaves the staged consumers little work
// per tile, so their per-tile overhead shows unless tiles are large (64 KB
// stages, see staged_tile_bytes).  Measured on GB300 from 16 MiB sent per
// rank, fp32: 20% (8 ranks) to 37% (2 ranks) faster than the register path.
// Above 8 ranks such tiles do not fit three stages, and for 16-bit types the
// consumers' widening work makes the staged kernel slower (R = 8 bf16: 128
// against 101 us): both stay on the register path.
bool use_staged_rs(int R, int dtype, size_t sendBytesPerRank) {
  return dtype == VR_FLOAT32 && R >= 2 && R <= 8 &&
         sendBytesPerRank >= (size_t)option(kOptStagedMinBytes);
}

// Per-rank tile bytes of the staged kernel (bulk copies below 2 KB lose
// throughput; 4 KB measured best for 9..16 ranks; ReduceScatter: 64 KB stages
// up to 16 KB per rank).
unsigned staged_tile_bytes(int R, int mode, bool drawn) {
  if (mode == kReduceScatter) return std::min(16384u, (65536u / (unsigned)R) & ~15u);
  if (R < 8 && small_geometry(mode, R, drawn).tile) return small_geometry(mode, R, drawn).tile;
  return R > 8 && R <= 16 ? 4096u : 2048u;
}

// The tile scheduler slot of a staged AllReduce launch on `stream` (staged.cuh):
// the stream's own slot, or a fresh one for a launch being captured into a
// graph (each captured launch runs as its own graph node, whose replays CUDA
// runs one after another); -1 when none is left or the stream's capture
// state cannot be read -- the launch then splits its tiles in fixed runs.
int sched_slot(int device, void* stream) {
  const cudaStream_t s = (cudaStream_t)stream;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  std::lock_guard<std::mutex> g(g_mu);
  if (cap == cudaStreamCaptureStatusActive) {
    int& used = g_captureSlotsUsed[device];
    if (used >= kSchedSlots - kSchedStreamSlots) return -1;
    return kSchedStreamSlots + used++;
  }
  if (cap != cudaStreamCaptureStatusNone) return -1;
  const std::thread::id tid = s == cudaStreamPerThread ? std::this_thread::get_id()
                                                        : std::thread::id();
  const auto key = std::make_tuple(device, s, tid);
  auto it = g_streamSlots.find(key);
  if (it != g_streamSlots.end()) return it->second;
  int& used = g_streamSlotsUsed[device];
  if (used >= kSchedStreamSlots) return -1;
  g_streamSlots.emplace(key, used);
  return used++;
}

// Staged geometry: tiles of tileUnits 16-byte units per rank; as many stages
// (at most 16) as fit in the opt-in shared memory; up to 7 consumer warps.
// a.unitsAll / a.unitsFull describe the message (AllReduce) or one block
// (ReduceScatter); the tile count follows from the geometry.
vr_result_t launch_staged(const void* fn, KArgs& a, int mode, void* stream) {
  if (!fn) return VR_ERR_INTERNAL;
  DeviceInfo di;
  int device = 0;
  vr_result_t e = device_info(&di, &device);
  if (e != VR_SUCCESS) return e;
  if ((e = check_reachable(a.src, a.R, device)) != VR_SUCCESS) return e;
  if ((e = check_reachable(const_cast<const void* const*>(a.dst), a.R, device)) != VR_SUCCESS)
    return e;
  a.status = di.status;
  a.boundsWhere = di.boundsWhere;
  shrink_extents(a);
  // Largest per-rank tile (fewer, larger bulk copies) that still leaves
  // at least kMinStages stages in the opt-in shared memory.
  // (the bounds-checked build adds a table in static shared memory)
  int staticSmem = 0;
  {
    std::lock_guard<std::mutex> g(g_mu);
    auto key = std::make_pair(fn, device);
    auto it = g_staticSmem.find(key);
    if (it == g_staticSmem.end()) {
      cudaFuncAttributes fa;
      if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess) return VR_ERR_CUDA;
      it = g_staticSmem.emplace(key, (int)fa.sharedSizeBytes).first;
    }
    staticSmem = it->second;
  }
  const int room = di.smemOptin - staticSmem - kStagedHeader;
  unsigned tb = (unsigned)option(kOptStagedTileBytes);
  // Above 32 ranks two stages with larger tiles (more consumer warps) beat
  // three smaller ones: measured 2.5% (tree) to 20% (ring) faster at 64.
  int minStages = (int)option_or(kOptStagedMinStages, a.R > 32 ? 2 : 3);
  if (!tb) {
    tb = staged_tile_bytes(a.R, mode, a.sched != nullptr);
    if (a.R > 32 && mode != kReduceScatter)  // the largest 512-byte multiple that fits
      tb = std::max(512u, ((unsigned)(room / (minStages * a.R))) & ~511u);
    while (tb > 512 && (long long)a.R * tb * minStages > room) tb -= 512;
  }
  a.tileBytes = tb;
  a.tileUnits = (int)(tb / 16);
  const long long TU = a.tileUnits;
  a.tiles = mode == kReduceScatter ? (long long)a.R * ((a.unitsFull + TU - 1) / TU)
                                   : (a.unitsAll - a.unitLo + TU - 1) / TU;
  a.stageBytes = ((unsigned)a.R * a.tileBytes + 127u) & ~127u;
  const int fit = room / (int)a.stageBytes;
  a.stages = std::min(kStagedMaxStages, fit);
  int cap = (int)option(kOptStagedStages);
  const SmallGeometry sg = small_geometry(mode, a.R, a.sched != nullptr);
  if (!cap && a.R < 8 && mode != kReduceScatter && (unsigned)tb == sg.tile)
    cap = sg.stages;  // the few-rank geometry's short pipeline
  if (cap) a.stages = std::min(a.stages, cap);
  if (a.stages < 2) return VR_ERR_INTERNAL;
  a.consumers = std::max(1, std::min(kStagedMaxConsumers, a.tileUnits / 32));
  const size_t smem = kStagedHeader + (size_t)a.stages * a.stageBytes;
  {
    std::lock_guard<std::mutex> g(g_mu);
    int& set = g_smemSet[std::make_pair(fn, device)];
    if (set < (int)smem) {
      if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               di.smemOptin - staticSmem) != cudaSuccess)
        return VR_ERR_CUDA;
      set = di.smemOptin - staticSmem;
    }
  }
  a.timeoutNs = wait_timeout_ns();
  a.injectStall = g_stallNext.exchange(-1);
  const int grid = (int)std::max(1LL, std::min<long long>(di.sms, a.tiles));
  void* args[] = {&a};
  // (Overlapped launch measured neutral to 5% slower above 32 ranks.)
  if (launch_kernel(fn, dim3(grid), dim3(32 * (a.consumers + 1)), args, smem, stream,
                    a.R <= 32) != cudaSuccess)
    return VR_ERR_CUDA;
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return VR_SUCCESS;
}

// A buffer of `count` elements of E bytes, `mult` blocks of it (the R blocks
// of a ReduceScatter send or an AllGather receive buffer): its byte count
// must fit the kernels' signed 64-bit offsets, and every count * E below is
// computed only after this check.
bool bytes_fit(size_t count, size_t E, size_t mult = 1) {
  return E && mult && count <= (size_t)LLONG_MAX / E / mult;
}

bool valid_common(int R, int dtype, int nChannels, size_t chunkBytes) {
  return R >= 1 && R <= kMaxRanks && elem_size(dtype) && nChannels >= 1 &&
         nChannels <= kMaxChannels && chunkBytes > 0 && chunkBytes % kGrainBytes == 0;
}

void fill_partition(KArgs& a, size_t count, size_t E, int nCh, size_t chunkBytes) {
  a.count = (long long)count;
  const long long U = kGrainBytes / (long long)E;
  a.grains = ((long long)count + U - 1) / U;
  a.gq = a.grains / nCh;
  a.gm = a.grains % nCh;
  a.chunk = (long long)(chunkBytes / E);
  a.nCh = nCh;
  a.lo = 0;
  a.hi = (long long)count;
  // reciprocals of the cursor's divisors (a.R is set by the caller)
  auto recip = [](long long d) -> unsigned long long {
    return d > 1 ? ~0ull / (unsigned long long)d + 1 : 0ull;
  };
  a.mGq1 = recip(a.gq + 1);
  a.mGq = recip(a.gq);
  a.mLC = recip((long long)a.R * a.chunk);
  a.mR = recip(a.R);
  a.mC = recip(a.chunk);
}

// A register-path call is a few rounds per thread, each R loads of one unit
// waited for together (a DRAM round trip), over a persistent grid of every
// resident thread.  While a tree call takes at most three rounds it is
// bound by those round trips, and when the specialised kernel compiled for
// four CTAs per SM (at most 64 registers) takes a whole round off every
// thread, that kernel is used.  Measured on GB300 (R = 4, 7, 8; fp32 and
// bf16): 9-17% faster at 2 MiB per rank, 2-8% at 4 MiB; 2-5% slower from
// 6 MiB (four rounds or more), and 4-21% slower for every ring, which keep
// their kernels.  VR_JIT_OCC=0 never switches, =4 always does (rings too).
const void* more_resident(const void* special, long long units, int dtype, int op, int mode,
                          int stack, const KArgs& a) {
  const long long occ = option(kOptJitOcc);
  if (occ == 0 || (occ != 4 && mode != kTreeAllReduce)) return special;
  DeviceInfo di;
  int device = 0;
  if (device_info(&di, &device) != VR_SUCCESS) return special;
  const int now = blocks_per_sm(special, device);
  if (now >= 4) return special;
  const long long oneCtaPerSm = (long long)kBlockThreads * di.sms;  // threads
  const long long roundsNow = (units + oneCtaPerSm * now - 1) / (oneCtaPerSm * now);
  const long long roundsFour = (units + oneCtaPerSm * 4 - 1) / (oneCtaPerSm * 4);
  if (occ != 4 && (roundsNow > 3 || roundsFour >= roundsNow)) return special;
  const bool small = use_small(dtype, mode, true, stack, a.R, (size_t)a.count * elem_size(dtype));
  const void* four = nullptr;
  const vr_result_t e =
      mode == kTreeAllReduce
          ? jit_tree_kernel(dtype, op, stack, small, false, a.prog, a.nProgs, &four, 4)
          : jit_ring_kernel(dtype, op, a.R, small, false, &four, 4);
  if (e != VR_SUCCESS || blocks_per_sm(four, device) < 4) return special;
  return four;
}

// The AllReduce kernel over the elements [lo, hi) of the message `a`
// describes (lo at a 16-byte boundary): the staged kernel, or the register
// kernel (16-byte units when `vec`, else elements).  Every element's fold
// reads only that element of each rank, and its order comes from the whole
// message's partition, so pieces give the whole message's bits.
vr_result_t launch_allreduce_range(KArgs& a, int dtype, int mode, int op, int stack, bool vec,
                                   bool staged, long long lo, long long hi, void* stream) {
  const long long E = (long long)elem_size(dtype);
  const size_t bytes = (size_t)a.count * (size_t)E;  // per rank, the whole message
  a.lo = lo;
  a.hi = hi;
  // Trees on 16-byte units: the kernels specialised for this call's programs
  // when they can be had (jit.cc), else the interpreting ones.
  // (The specialised register-path kernel measured slower than the
  // interpreting one at 64 ranks: above 32 only the staged one is used.)
  // A staged AllReduce draws its tiles through its stream's scheduler slot
  // where that measured faster (staged.cuh).
  a.sched = nullptr;
  if (staged && sched_tiles(mode, a.R, dtype)) {
    DeviceInfo di;
    int device = 0;
    const vr_result_t e = device_info(&di, &device);
    if (e != VR_SUCCESS) return e;
    const int slot = sched_slot(device, stream);
    if (slot >= 0) a.sched = di.sched + 4 * (size_t)slot;
  }
  const bool drawn = a.sched != nullptr;
  const void* special = nullptr;
  if (mode == kTreeAllReduce && vec && (staged || a.R <= 32) && jit_enabled() &&
      jit_tree_kernel(dtype, op, stack, use_small(dtype, mode, vec, stack, a.R, bytes), staged,
                      a.prog, a.nProgs, &special, 0, drawn) != VR_SUCCESS)
    special = nullptr;
  // The ring specialised for R ranks: measured 6-12% faster on the register
  // path for 3-16 ranks, neutral on the staged one (VR_JIT_RING=1 also takes
  // it there, 0 turns it off).
  const long long jr = option(kOptJitRing);
  if (mode == kRingAllReduce && vec && a.R >= 3 && a.R <= 16 && jr != 0 &&
      (!staged || (jr == 1 && !drawn)) && jit_enabled() &&
      jit_ring_kernel(dtype, op, a.R, use_small(dtype, mode, vec, stack, a.R, bytes), staged,
                      &special) != VR_SUCCESS)
    special = nullptr;
  if (staged) {
    a.unitLo = lo * E / 16;
    a.unitsAll = (hi * E + 15) / 16;
    a.unitsFull = hi * E / 16;
    return launch_staged(special ? special : pick_staged(dtype, mode, op, stack, drawn), a, mode,
                         stream);
  }
  const long long NV = vec ? kGrainBytes / E : 1;
  const long long units = (hi + NV - 1) / NV - lo / NV;
  if (special) special = more_resident(special, units, dtype, op, mode, stack, a);
  return launch(special ? special : pick_kernel(dtype, mode, op, vec, stack, a.R, bytes), a,
                units, stream);
}

// Per device: the two copy streams and three events of vr_allreduce_host,
// created on first use with that device current.
struct HostPipe {
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, loaded = nullptr, folded = nullptr, stored = nullptr;
};
std::map<int, HostPipe> g_pipes;
std::mutex g_pipeMu;  // held for a whole vr_allreduce_host enqueue (the events are shared)

vr_result_t host_pipe(int device, HostPipe** out) {
  auto it = g_pipes.find(device);
  if (it == g_pipes.end()) {
    HostPipe p;
    if (cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.start, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.loaded, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.folded, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.stored, cudaEventDisableTiming) != cudaSuccess)
      return VR_ERR_CUDA;
    it = g_pipes.emplace(device, p).first;
  }
  *out = &it->second;
  return VR_SUCCESS;
}

}  // namespace
}  // namespace vr

using namespace vr;

extern "C" {

vr_result_t vr_build_ring(int R, int nChannels, int* next, int* prev) {
  if (R < 1 || R > kMaxRanks || nChannels < 1 || nChannels > kMaxChannels || !next || !prev)
    return VR_ERR_INVALID_ARGUMENT;
  build_ring(R, nChannels, next, prev);
  log_ring(next, R, nChannels);
  return VR_SUCCESS;
}

vr_result_t vr_build_dtree(int nNodes, int localRanks, int nChannels, vr_tree_t* trees) {
  if (nNodes < 1 || localRanks < 1 || nNodes > kMaxRanks || localRanks > kMaxRanks ||
      nNodes * localRanks > kMaxRanks || nChannels < 1 || nChannels > kMaxChannels || !trees)
    return VR_ERR_INVALID_ARGUMENT;
  const vr_result_t e = build_dtree(nNodes, localRanks, nChannels, trees);
  if (e == VR_SUCCESS) log_trees(trees, nNodes * localRanks, nChannels);
  return e;
}

vr_result_t vr_build_dtree_ex(int nNodes, int localRanks, int nChannels,
                              vr_tree_pattern_t pattern, const int* intraOrders,
                              vr_tree_t* trees) {
  if (nNodes < 1 || localRanks < 1 || nNodes > kMaxRanks || localRanks > kMaxRanks ||
      nNodes * localRanks > kMaxRanks || nChannels < 1 || nChannels > kMaxChannels || !trees ||
      (pattern != VR_PATTERN_TREE && pattern != VR_PATTERN_SPLIT_TREE &&
       pattern != VR_PATTERN_BALANCED_TREE))
    return VR_ERR_INVALID_ARGUMENT;
  const vr_result_t e =
      build_dtree_ex(nNodes, localRanks, nChannels, pattern, intraOrders, trees);
  if (e == VR_SUCCESS) log_trees(trees, nNodes * localRanks, nChannels);
  return e;
}

vr_result_t vr_partition(size_t count, vr_dtype_t dtype, int nChannels, int channel,
                         size_t* offset, size_t* channelCount) {
  const size_t E = elem_size(dtype);
  if (!E || nChannels < 1 || nChannels > kMaxChannels || channel < 0 || channel >= nChannels ||
      !offset || !channelCount)
    return VR_ERR_INVALID_ARGUMENT;
  const size_t U = kGrainBytes / E;
  const size_t grains = (count + U - 1) / U;
  const size_t q = grains / nChannels, m = grains % nChannels;
  const size_t gs = channel * q + std::min<size_t>(channel, m);
  const size_t gl = q + ((size_t)channel < m ? 1 : 0);
  const size_t s = std::min(count, gs * U), e = std::min(count, (gs + gl) * U);
  *offset = s;
  *channelCount = e - s;
  return VR_SUCCESS;
}

vr_result_t vr_ring_block(size_t count, vr_dtype_t dtype, int R, int nChannels,
                          size_t chunkBytes, size_t elem, int* channel, int* block) {
  if (!valid_common(R, dtype, nChannels, chunkBytes) || elem >= count || !channel || !block)
    return VR_ERR_INVALID_ARGUMENT;
  const size_t E = elem_size(dtype), C = chunkBytes / E;
  for (int c = 0; c < nChannels; ++c) {
    size_t s, n;
    vr_partition(count, dtype, nChannels, c, &s, &n);
    if (elem < s || elem >= s + n) continue;
    const size_t LC = (size_t)R * C, off = elem - s;
    const size_t ls = off / LC * LC, L = std::min(LC, n - ls), w = off - ls;
    const size_t q = L / R, m = L % R;
    *channel = c;
    *block = (int)(w < m * (q + 1) ? w / (q + 1) : m + (w - m * (q + 1)) / q);
    return VR_SUCCESS;
  }
  return VR_ERR_INTERNAL;
}

}  // extern "C"

namespace vr {
namespace {

// Validates an AllReduce and fills `a` (ranks, partition, tree programs),
// `mode` and `stack`.  AUTO resolves through the current cost model.
vr_result_t plan_allreduce(const void* const* sendbufs, void* const* recvbufs, int R,
                           size_t count, vr_dtype_t dtype, vr_op_t op, vr_algo_t algo,
                           int nChannels, size_t chunkBytes, int localRanks, KArgs& a, int& mode,
                           int& stack) {
  if (algo == VR_ALGO_AUTO && valid_common(R, dtype, nChannels, chunkBytes) && localRanks >= 1 &&
      R % localRanks == 0 && bytes_fit(count, elem_size(dtype)) &&
      vr_select_algo(R, localRanks, count * elem_size(dtype), nullptr, &algo) != VR_SUCCESS)
    return VR_ERR_INTERNAL;
  if (!valid_common(R, dtype, nChannels, chunkBytes) || (op != VR_SUM && op != VR_MAX) ||
      (algo != VR_ALGO_RING && algo != VR_ALGO_TREE) || localRanks < 1 || R % localRanks ||
      !bytes_fit(count, elem_size(dtype)))
    return VR_ERR_INVALID_ARGUMENT;
  const size_t E = elem_size(dtype);
  vr_result_t e = check_buffers(sendbufs, recvbufs, R, count * E, count * E, kAR, E);
  if (e != VR_SUCCESS) return e;
  std::memset(&a, 0, sizeof(a));
  a.R = R;
  for (int r = 0; r < R; ++r) { a.src[r] = sendbufs[r]; a.dst[r] = recvbufs[r]; }
  a.srcBytes = a.dstBytes = count * E;
  fill_partition(a, count, E, nChannels, chunkBytes);
  mode = kRingAllReduce;
  stack = 0;
  // Two ranks: the ring folds every element as x_j (op) x_(j+1), and for two
  // operands both orders give the same bits (IEEE addition and the Max of
  // the total order commute), so it is also the two-rank tree's fold, local
  // input first.  The ring of two ranks runs the tree kernels (with the
  // few-rank staged geometry of the tree): measured on GB300, 5.2 against
  // 8.0 us at 4 MiB per rank and 0.86 against 0.66 of the copy bandwidth at
  // 64 MiB.
  const bool twoRankRing = algo == VR_ALGO_RING && R == 2;
  if ((algo == VR_ALGO_TREE || twoRankRing) && count > 0) {
    mode = kTreeAllReduce;
    std::array<FoldProg, 2> p;
    if ((e = tree_programs(twoRankRing ? 2 : R / localRanks, twoRankRing ? 1 : localRanks,
                           &p)) != VR_SUCCESS)
      return e;
    set_dtree_programs(a, p, nChannels);
    stack = std::max(p[0].depth, p[1].depth);
  }
  if (count > 0 && graph_logging()) {
    static vr_tree_t trees[kMaxRanks * kMaxChannels];  // under the log's own lock below
    static std::mutex mu;
    std::lock_guard<std::mutex> g(mu);
    const bool tree = algo == VR_ALGO_TREE &&
                      build_dtree(R / localRanks, localRanks, nChannels, trees) == VR_SUCCESS;
    log_plan("allreduce", algo, R, localRanks, count, dtype, nChannels, chunkBytes,
             tree ? trees : nullptr, true);
  }
  return VR_SUCCESS;
}

// Host memory (page-locked or not) for the host buffers, memory of the
// current device for the workspace.
bool is_device_memory(const void* p, int device) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) &&
         at.device == device;
}
bool is_host_memory(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeHost || at.type == cudaMemoryTypeUnregistered;
}

}  // namespace

vr_result_t check_stepwise_args(const void* const* sendbufs, void* const* recvbufs, int R,
                                size_t count, int dtype, int op, int nChannels,
                                size_t chunkBytes) {
  if (!valid_common(R, dtype, nChannels, chunkBytes) || (op != VR_SUM && op != VR_MAX) ||
      !bytes_fit(count, elem_size(dtype)))
    return VR_ERR_INVALID_ARGUMENT;
  const size_t E = elem_size(dtype);
  return check_buffers(sendbufs, recvbufs, R, count * E, count * E, kAR, E);
}

}  // namespace vr

extern "C" {

vr_result_t vr_allreduce_ex(const void* const* sendbufs, void* const* recvbufs, int R,
                            size_t count, vr_dtype_t dtype, vr_op_t op, vr_algo_t algo,
                            int nChannels, size_t chunkBytes, int localRanks, void* stream) {
  KArgs a;
  int mode = 0, stack = 0;
  vr_result_t e = plan_allreduce(sendbufs, recvbufs, R, count, dtype, op, algo, nChannels,
                                 chunkBytes, localRanks, a, mode, stack);
  if (e != VR_SUCCESS || count == 0) return e;
  const size_t E = elem_size(dtype);
  // Small rings run the element kernel, one element per thread (same order,
  // same bits).  A latency-bound call lasts as long as its slowest thread,
  // and in the vector path that is a thread whose unit a ring block boundary
  // cuts (folded out of line, element by element when blocks are shorter
  // than a unit).  Measured on GB300: faster up to 64 Ki elements per rank
  // (R = 4 fp32, R = 8 bf16), slower from 128 Ki.
  const bool tinyBlocks = mode == kRingAllReduce && (a.gq < R || count <= 65536);
  const bool vec = aligned16(sendbufs, R, 0) && aligned16(recvbufs, R, 0) && !tinyBlocks;
  const int forced = forced_path();
  const bool staged = vec && forced != 1 && (forced == 2 || use_staged(mode, R, count * E));
  return launch_allreduce_range(a, dtype, mode, op, stack, vec, staged, 0, (long long)count,
                                stream);
}

vr_result_t vr_allreduce_host(const void* const* sendbufs, void* const* recvbufs, int R,
                              size_t count, vr_dtype_t dtype, vr_op_t op, vr_algo_t algo,
                              int nChannels, size_t chunkBytes, int localRanks,
                              void* const* workbufs, size_t pieceBytes, void* stream) {
  if (pieceBytes == 0) pieceBytes = VR_HOST_PIECE_BYTES;
  if (pieceBytes % kGrainBytes || !sendbufs || !recvbufs || !workbufs ||
      !valid_common(R, dtype, nChannels, chunkBytes) || !bytes_fit(count, elem_size(dtype)))
    return VR_ERR_INVALID_ARGUMENT;
  const size_t E = elem_size(dtype);
  // the host side: distinct buffers, in place allowed, NULL receive buffers skipped
  vr_result_t e = check_buffers(sendbufs, recvbufs, R, count * E, count * E, kAR, E, true);
  if (e != VR_SUCCESS) return e;
  // the device side: the workspace, folded in place
  KArgs a;
  int mode = 0, stack = 0;
  e = plan_allreduce(const_cast<const void* const*>(workbufs), workbufs, R, count, dtype, op,
                     algo, nChannels, chunkBytes, localRanks, a, mode, stack);
  if (e != VR_SUCCESS || count == 0) return e;
  DeviceInfo di;
  int device = 0;
  if ((e = device_info(&di, &device)) != VR_SUCCESS) return e;
  for (int r = 0; r < R; ++r)
    if (!is_device_memory(workbufs[r], device) || !is_host_memory(sendbufs[r]) ||
        (recvbufs[r] && !is_host_memory(recvbufs[r])))
      return VR_ERR_INVALID_ARGUMENT;
  const bool vec = aligned16(const_cast<const void* const*>(workbufs), R, 0);
  const int forced = forced_path();
  const bool staged = vec && forced != 1 && (forced == 2 || use_staged(mode, R, count * E));
  const long long piece = (long long)(pieceBytes / E);
  const cudaStream_t s = (cudaStream_t)stream;

  std::lock_guard<std::mutex> g(g_pipeMu);
  HostPipe* hp = nullptr;
  {
    std::lock_guard<std::mutex> g2(g_mu);
    if ((e = host_pipe(device, &hp)) != VR_SUCCESS) return e;
  }
  // Nothing is copied in before the caller's earlier work on `stream` is done.
  if (cudaEventRecord(hp->start, s) != cudaSuccess ||
      cudaStreamWaitEvent(hp->in, hp->start, 0) != cudaSuccess)
    return VR_ERR_CUDA;
  for (long long lo = 0; lo < (long long)count; lo += piece) {
    const long long hi = std::min((long long)count, lo + piece);
    const size_t off = (size_t)lo * E, bytes = (size_t)(hi - lo) * E;
    for (int r = 0; r < R; ++r)
      if (cudaMemcpyAsync((char*)workbufs[r] + off, (const char*)sendbufs[r] + off, bytes,
                          cudaMemcpyHostToDevice, hp->in) != cudaSuccess)
        return VR_ERR_CUDA;
    // a wait takes the event's latest record, so one event serves every piece
    if (cudaEventRecord(hp->loaded, hp->in) != cudaSuccess ||
        cudaStreamWaitEvent(s, hp->loaded, 0) != cudaSuccess)
      return VR_ERR_CUDA;
    if ((e = launch_allreduce_range(a, dtype, mode, op, stack, vec, staged, lo, hi, stream)) !=
        VR_SUCCESS)
      return e;
    if (cudaEventRecord(hp->folded, s) != cudaSuccess ||
        cudaStreamWaitEvent(hp->out, hp->folded, 0) != cudaSuccess)
      return VR_ERR_CUDA;
    for (int r = 0; r < R; ++r)
      if (recvbufs[r] &&
          cudaMemcpyAsync((char*)recvbufs[r] + off, (const char*)workbufs[r] + off, bytes,
                          cudaMemcpyDeviceToHost, hp->out) != cudaSuccess)
        return VR_ERR_CUDA;
  }
  // Work enqueued on `stream` after this call runs after the last copy out.
  if (cudaEventRecord(hp->stored, hp->out) != cudaSuccess ||
      cudaStreamWaitEvent(s, hp->stored, 0) != cudaSuccess)
    return VR_ERR_CUDA;
  return VR_SUCCESS;
}


vr_result_t vr_allreduce(const void* const* sendbufs, void* const* recvbufs, int R, size_t count,
                         vr_dtype_t dtype, vr_op_t op, vr_algo_t algo, int nChannels,
                         size_t chunkBytes, void* stream) {
  return vr_allreduce_ex(sendbufs, recvbufs, R, count, dtype, op, algo, nChannels, chunkBytes, 1,
                         stream);
}

vr_result_t vr_allreduce_trees(const void* const* sendbufs, void* const* recvbufs, int R,
                               size_t count, vr_dtype_t dtype, vr_op_t op, int nChannels,
                               size_t chunkBytes, const vr_tree_t* trees, void* stream) {
  if (!valid_common(R, dtype, nChannels, chunkBytes) || (op != VR_SUM && op != VR_MAX) || !trees ||
      !bytes_fit(count, elem_size(dtype)))
    return VR_ERR_INVALID_ARGUMENT;
  for (int c = 0; c < nChannels; ++c)
    if (!valid_tree(trees + (size_t)c * R, R)) return VR_ERR_INVALID_ARGUMENT;
  const size_t E = elem_size(dtype);
  vr_result_t e = check_buffers(sendbufs, recvbufs, R, count * E, count * E, kAR, E);
  if (e != VR_SUCCESS || count == 0) return e;
  log_plan("allreduce", VR_ALGO_TREE, R, 0, count, dtype, nChannels, chunkBytes, trees, true);
  KArgs a;
  std::memset(&a, 0, sizeof(a));
  a.R = R;
  for (int r = 0; r < R; ++r) { a.src[r] = sendbufs[r]; a.dst[r] = recvbufs[r]; }
  a.srcBytes = a.dstBytes = count * E;
  fill_partition(a, count, E, nChannels, chunkBytes);
  // one program per distinct tree
  int stack = 0;
  for (int c = 0; c < nChannels; ++c) {
    const vr_tree_t* tc = trees + (size_t)c * R;
    int found = -1;
    for (int q = 0; q < c && found < 0; ++q)
      if (std::memcmp(tc, trees + (size_t)q * R, sizeof(vr_tree_t) * R) == 0)
        found = a.chanProg[q];
    if (found < 0) {
      if (a.nProgs == kMaxProgs) return VR_ERR_UNSUPPORTED;
      if (compile_fold(tc, R, &a.prog[a.nProgs]) != VR_SUCCESS) return VR_ERR_UNSUPPORTED;
      stack = std::max(stack, (int)a.prog[a.nProgs].depth);
      found = a.nProgs++;
    }
    a.chanProg[c] = (uint8_t)found;
  }
  const bool vec = aligned16(sendbufs, R, 0) && aligned16(recvbufs, R, 0);
  const int forced = forced_path();
  const bool staged =
      vec && forced != 1 && (forced == 2 || use_staged(kTreeAllReduce, R, count * E));
  return launch_allreduce_range(a, dtype, kTreeAllReduce, op, stack, vec, staged, 0,
                                (long long)count, stream);
}

vr_result_t vr_reduce_scatter(const void* const* sendbufs, void* const* recvbufs, int R,
                              size_t recvcount, vr_dtype_t dtype, vr_op_t op, vr_algo_t algo,
                              int nChannels, size_t chunkBytes, void* stream) {
  if (!valid_common(R, dtype, nChannels, chunkBytes) || (op != VR_SUM && op != VR_MAX) ||
      (algo != VR_ALGO_RING && algo != VR_ALGO_TREE) ||
      !bytes_fit(recvcount, elem_size(dtype), (size_t)R))
    return VR_ERR_INVALID_ARGUMENT;
  if (algo == VR_ALGO_TREE) return VR_ERR_UNSUPPORTED;
  const size_t E = elem_size(dtype);
  vr_result_t e = check_buffers(sendbufs, recvbufs, R, (size_t)R * recvcount * E, recvcount * E, kRS, E);
  if (e != VR_SUCCESS || recvcount == 0) return e;
  log_plan("reduce_scatter", VR_ALGO_RING, R, 1, recvcount, dtype, nChannels, chunkBytes,
           nullptr, false);
  KArgs a;
  std::memset(&a, 0, sizeof(a));
  a.R = R;
  for (int r = 0; r < R; ++r) { a.src[r] = sendbufs[r]; a.dst[r] = recvbufs[r]; }
  a.count = (long long)recvcount;
  a.nCh = nChannels;
  a.chunk = (long long)(chunkBytes / E);
  a.srcBytes = (size_t)R * recvcount * E;
  a.dstBytes = recvcount * E;
  const bool vec = aligned16(sendbufs, R, recvcount * E) && aligned16(recvbufs, R, 0);
  const int forced = forced_path();
  if (vec && forced != 1 && (forced == 2 || use_staged_rs(R, dtype, recvcount * E * R))) {
    a.unitsFull = (long long)(recvcount * E / 16);
    a.unitsAll = a.unitsFull;
    return launch_staged(pick_staged(dtype, kReduceScatter, op), a, kReduceScatter, stream);
  }
  const long long NV = vec ? kGrainBytes / (long long)E : 1;
  const long long units = (long long)R * (((long long)recvcount + NV - 1) / NV);
  return launch(pick_kernel(dtype, kReduceScatter, op, vec), a, units, stream);
}

vr_result_t vr_allgather(const void* const* sendbufs, void* const* recvbufs, int R,
                         size_t sendcount, vr_dtype_t dtype, vr_algo_t algo, int nChannels,
                         size_t chunkBytes, void* stream) {
  if (!valid_common(R, dtype, nChannels, chunkBytes) ||
      (algo != VR_ALGO_RING && algo != VR_ALGO_TREE) ||
      !bytes_fit(sendcount, elem_size(dtype), (size_t)R))
    return VR_ERR_INVALID_ARGUMENT;
  if (algo == VR_ALGO_TREE) return VR_ERR_UNSUPPORTED;
  const size_t bytes = sendcount * elem_size(dtype);
  vr_result_t e = check_buffers(sendbufs, recvbufs, R, bytes, (size_t)R * bytes, kAG,
                                elem_size(dtype));
  if (e != VR_SUCCESS || sendcount == 0) return e;
  log_plan("allgather", VR_ALGO_RING, R, 1, sendcount, dtype, nChannels, chunkBytes, nullptr,
           false);
  KArgs a;
  std::memset(&a, 0, sizeof(a));
  a.R = R;
  for (int r = 0; r < R; ++r) { a.src[r] = sendbufs[r]; a.dst[r] = recvbufs[r]; }
  a.count = (long long)bytes;
  a.nCh = nChannels;
  a.srcBytes = bytes;
  a.dstBytes = (size_t)R * bytes;
  const bool vec = aligned16(sendbufs, R, bytes) && aligned16(recvbufs, R, 0);
  if (vec && forced_path() != 1) {
    // the TMA copy: one warp per CTA, tiles of gather_tile_bytes() of one rank
    DeviceInfo di;
    int device = 0;
    if ((e = device_info(&di, &device)) != VR_SUCCESS) return e;
    // Destination-major (one store per loaded tile, the sources re-read from
    // L2) when the R sources together take at most a quarter of L2, with
    // 32 KB tiles in 3 stages.  Measured on GB300 (graph replays): R=64 x
    // 16 MiB fp16 152-153 us against 166 us source-major (7.2 TB/s: the
    // writes dominate, so this passes the read+write copy bandwidth), R=16
    // 40.6 against 42.8 us, R=4 and R=8 equal to 2 %; with larger sources
    // (R=8 x 128 MiB, R=64 x 64 MiB) source-major was 2-6 % faster.
    const long long order = option(kOptAgOrder);
    const bool destMajor =
        order == 2 || (order == 0 && (size_t)R * bytes <= (size_t)di.l2Bytes / 4);
    // geometry: tuning overrides VR_AG_TILE / VR_AG_STAGES / VR_AG_CTAS
    const int tile = (int)option_or(kOptAgTile, destMajor ? 32768 : gather_tile_bytes());
    const int stages = (int)option_or(kOptAgStages, destMajor ? 3 : gather_stages());
    const int ctas = (int)std::max(1LL, option_or(kOptAgCtas, gather_ctas_per_sm()));
    const void* fn = destMajor ? kernel_ptr_allgather_tma_dest(tile, stages)
                               : kernel_ptr_allgather_tma(tile, stages);
    if (!fn) return VR_ERR_INVALID_ARGUMENT;
    const size_t smem = (size_t)tile * stages;
    {
      std::lock_guard<std::mutex> g(g_mu);
      int& set = g_smemSet[std::make_pair(fn, device)];
      if (set < (int)smem) {
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
          return VR_ERR_CUDA;
        set = (int)smem;
      }
    }
    a.tiles = (long long)R * (((long long)bytes + tile - 1) / tile) * (destMajor ? R : 1);
    a.status = di.status;
    a.boundsWhere = di.boundsWhere;
    shrink_extents(a);
    a.timeoutNs = wait_timeout_ns();
    a.injectStall = g_stallNext.exchange(-1);
    const long long grid = std::min<long long>(a.tiles, (long long)di.sms * ctas);
    void* args[] = {&a};
    if (launch_kernel(fn, dim3((unsigned)grid), dim3(32), args, smem, stream, false) !=
        cudaSuccess)
      return VR_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return VR_SUCCESS;
  }
  const long long NB = vec ? kGrainBytes : 1;
  const long long units = (long long)R * (((long long)bytes + NB - 1) / NB);
  return launch(kernel_ptr_allgather(vec), a, units, stream);
}

size_t vr_ring_stepwise_scratch_bytes(size_t count, vr_dtype_t dtype) {
  const size_t E = elem_size(dtype);
  return bytes_fit(count, E) ? (count * E + 15) / 16 * 16 : 0;
}

vr_result_t vr_allreduce_ring_stepwise(const void* const* sendbufs, void* const* recvbufs, int R,
                                       size_t count, vr_dtype_t dtype, vr_op_t op,
                                       int nChannels, size_t chunkBytes, void* scratch,
                                       size_t scratchBytes, void* stream) {
  vr_result_t e = check_stepwise_args(sendbufs, recvbufs, R, count, dtype, op, nChannels,
                                      chunkBytes);
  if (e != VR_SUCCESS || count == 0) return e;
  const size_t E = elem_size(dtype);
  const size_t need = vr_ring_stepwise_scratch_bytes(count, dtype);
  if (!scratch || scratchBytes < need || (uintptr_t)scratch % E) return VR_ERR_INVALID_ARGUMENT;
  for (int r = 0; r < R; ++r)
    if (overlap((uintptr_t)scratch, need, (uintptr_t)sendbufs[r], count * E) ||
        overlap((uintptr_t)scratch, need, (uintptr_t)recvbufs[r], count * E))
      return VR_ERR_INVALID_ARGUMENT;
  KArgs a;
  std::memset(&a, 0, sizeof(a));
  a.R = R;
  for (int r = 0; r < R; ++r) { a.src[r] = sendbufs[r]; a.dst[r] = recvbufs[r]; }
  a.scratch = scratch;
  a.srcBytes = a.dstBytes = count * E;
  a.scratchBytes = need;
  const bool vec = aligned16(sendbufs, R, 0) && aligned16(recvbufs, R, 0) &&
                   (((uintptr_t)scratch & 15) == 0);
  // working copies: recv = send
  a.count = (long long)(count * E);
  const long long NB = vec ? 16 : 1;
  if ((e = launch(ablation_kernel_ptr(kCopyRanks, dtype, op, vec, 0), a,
                  (long long)R * ((a.count + NB - 1) / NB), stream)) != VR_SUCCESS)
    return e;
  fill_partition(a, count, E, nChannels, chunkBytes);
  const void* step = ablation_kernel_ptr(kRingStep, dtype, op, vec, 0);
  const long long NV = vec ? kGrainBytes / (long long)E : 1;
  const long long units = ((long long)count + NV - 1) / NV;
  for (int half = 0; half < 2; ++half) {
    int gather = half;
    for (int s = 0; s < R - 1; ++s) {
      int phase = kStepSend;
      void* extra[3] = {&phase, &s, &gather};
      if ((e = launch(step, a, units, stream, extra, 3)) != VR_SUCCESS) return e;
      phase = half ? kStepCopy : kStepReduce;
      if ((e = launch(step, a, units, stream, extra, 3)) != VR_SUCCESS) return e;
    }
  }
  return VR_SUCCESS;
}

vr_result_t vr_allreduce_tree_updown(const void* const* sendbufs, void* const* recvbufs, int R,
                                     size_t count, vr_dtype_t dtype, vr_op_t op, int nChannels,
                                     size_t chunkBytes, int localRanks, void* stream) {
  if (!valid_common(R, dtype, nChannels, chunkBytes) || (op != VR_SUM && op != VR_MAX) ||
      localRanks < 1 || R % localRanks || !bytes_fit(count, elem_size(dtype)))
    return VR_ERR_INVALID_ARGUMENT;
  const size_t E = elem_size(dtype);
  vr_result_t e = check_buffers(sendbufs, recvbufs, R, count * E, count * E, kAR, E);
  if (e != VR_SUCCESS || count == 0) return e;
  KArgs a;
  std::memset(&a, 0, sizeof(a));
  a.R = R;
  for (int r = 0; r < R; ++r) { a.src[r] = sendbufs[r]; a.dst[r] = recvbufs[r]; }
  a.srcBytes = a.dstBytes = count * E;
  fill_partition(a, count, E, nChannels, chunkBytes);
  std::array<FoldProg, 2> p;
  if ((e = tree_programs(R / localRanks, localRanks, &p)) != VR_SUCCESS) return e;
  set_dtree_programs(a, p, nChannels);
  const int stack = std::max(p[0].depth, p[1].depth);
  const bool vec = aligned16(sendbufs, R, 0) && aligned16(recvbufs, R, 0);
  const long long NV = vec ? kGrainBytes / (long long)E : 1;
  const long long units = ((long long)count + NV - 1) / NV;
  if ((e = launch(ablation_kernel_ptr(kTreeUp, dtype, op, vec, stack), a, units, stream)) !=
      VR_SUCCESS)
    return e;
  return launch(ablation_kernel_ptr(kTreeDown, dtype, op, vec, stack), a, units, stream);
}

vr_result_t vr_stream_status(void* stream) {
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return VR_ERR_CUDA;
  unsigned v = 0;
  if (read_and_clear_status(&v) != cudaSuccess) return VR_ERR_CUDA;
  return (vr_result_t)v;
}

unsigned long long vr_launch_count(void) { return g_launches.load(); }

vr_result_t vr_debug_shrink_next(long long bytes, int which) {
  if (bytes < 0 || which < 0 || which > 7) return VR_ERR_INVALID_ARGUMENT;
  g_shrinkWhich.store(which);
  g_shrinkNext.store(bytes);
  return VR_SUCCESS;
}

vr_result_t vr_debug_stall_next(long long tile) {
  if (tile < -1) return VR_ERR_INVALID_ARGUMENT;
  g_stallNext.store(tile);
  return VR_SUCCESS;
}

vr_result_t vr_debug_sched_slot(void* stream, unsigned long long* words, int write) {
  if (!words) return VR_ERR_INVALID_ARGUMENT;
  DeviceInfo di;
  int device = 0;
  vr_result_t e = device_info(&di, &device);
  if (e != VR_SUCCESS) return e;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing((cudaStream_t)stream, &cap) != cudaSuccess ||
      cap != cudaStreamCaptureStatusNone)
    return VR_ERR_INVALID_ARGUMENT;
  const int slot = sched_slot(device, stream);
  if (slot < 0) return VR_ERR_UNSUPPORTED;
  unsigned long long* p = di.sched + 4 * (size_t)slot;
  const cudaStream_t s = (cudaStream_t)stream;
  const cudaError_t c = write ? cudaMemcpyAsync(p, words, 4 * sizeof(*words),
                                                cudaMemcpyHostToDevice, s)
                              : cudaMemcpyAsync(words, p, 4 * sizeof(*words),
                                                cudaMemcpyDeviceToHost, s);
  if (c != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess) return VR_ERR_CUDA;
  return VR_SUCCESS;
}

const char* vr_get_error_string(vr_result_t result) {
  switch (result) {
    case VR_SUCCESS: return "success";
    case VR_ERR_INVALID_ARGUMENT: return "invalid argument";
    case VR_ERR_UNSUPPORTED: return "unsupported combination";
    case VR_ERR_CUDA: return "CUDA runtime error";
    case VR_ERR_TIMEOUT: return "device-side wait timed out";
    case VR_ERR_INTERNAL: return "internal error";
    default: return "unknown result";
  }
}

vr_result_t vr_jit_status(int* enabled, long long* compiled, long long* failed) {
  if (!enabled || !compiled || !failed) return VR_ERR_INVALID_ARGUMENT;
  *enabled = jit_enabled() ? 1 : 0;
  jit_counts(compiled, failed);
  return VR_SUCCESS;
}

vr_result_t vr_jit_compile_dtree(int nNodes, int localRanks, vr_dtype_t dtype, vr_op_t op,
                                 int smArch, size_t* cubinBytes, char* log, size_t logBytes) {
  if (!cubinBytes || !elem_size(dtype) || (op != VR_SUM && op != VR_MAX) || smArch < 90)
    return VR_ERR_INVALID_ARGUMENT;
  return jit_compile_dtree(nNodes, localRanks, dtype, op, smArch, cubinBytes, log, logBytes);
}

vr_result_t vr_jit_compile_ring(int R, vr_dtype_t dtype, vr_op_t op, int smArch,
                                size_t* cubinBytes, char* log, size_t logBytes) {
  if (!cubinBytes || !elem_size(dtype) || (op != VR_SUM && op != VR_MAX) || smArch < 90)
    return VR_ERR_INVALID_ARGUMENT;
  return jit_compile_ring(R, dtype, op, smArch, cubinBytes, log, logBytes);
}

void vr_finalize(void) {
  {
    std::lock_guard<std::mutex> gp(g_pipeMu);
    int current = 0;
    const bool haveDevice = cudaGetDevice(&current) == cudaSuccess;
    for (auto& kv : g_pipes) {
      if (cudaSetDevice(kv.first) != cudaSuccess) continue;
      HostPipe& p = kv.second;
      cudaStreamSynchronize(p.in);
      cudaStreamSynchronize(p.out);
      cudaStreamDestroy(p.in);
      cudaStreamDestroy(p.out);
      for (cudaEvent_t ev : {p.start, p.loaded, p.folded, p.stored}) cudaEventDestroy(ev);
    }
    g_pipes.clear();
    if (haveDevice) cudaSetDevice(current);
  }
  std::lock_guard<std::mutex> g(g_mu);
  g_progs.clear();
  g_occupancy.clear();
  g_devices.clear();
  g_smemSet.clear();
  g_staticSmem.clear();
}

}  // extern "C"
