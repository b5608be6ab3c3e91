// Bounds-checked build (VR_DEBUG_BOUNDS defined): every global-memory access
// of a kernel is checked against the buffers of its launch before it is
// made.
//
// The library's calls return at enqueue, so a fault in a kernel surfaces
// later and asynchronously ([Internals] "API 返回只意味着提交边界"); with no
// memory checker at hand, this build makes each kernel its own: an access
// outside every buffer of the call (a store outside every writable one)
// records VR_ERR_INTERNAL in the device status word (read by
// vr_stream_status) and the first such address in a second word
// (vr_debug_bounds_fault), and is skipped -- a skipped bulk copy still
// completes its barrier's byte count, so nothing waits for it.  In the
// normal build the checks compile to nothing.
#pragma once

#include "common.h"

namespace vr {

// One buffer of a launch: [lo, lo + bytes), writable or not.
struct Extent {
  const char* lo;
  unsigned long long bytes;
  int writable;
};

// Does [p, p + n) lie inside one extent (a writable one for a store)?  The
// same predicate runs on the device and, for the host's self-test, on the
// CPU (vr_debug_access_ok).
__host__ __device__ inline bool access_in(const Extent* ext, int nExt, const char* p,
                                          unsigned long long n, bool store) {
  const unsigned long long a = (unsigned long long)(uintptr_t)p;
  for (int i = 0; i < nExt; ++i) {
    const Extent& e = ext[i];
    if (!e.lo || (store && !e.writable)) continue;
    const unsigned long long lo = (unsigned long long)(uintptr_t)e.lo;
    if (a >= lo && n <= e.bytes && a - lo <= e.bytes - n) return true;
  }
  return false;
}

#ifdef VR_DEBUG_BOUNDS
struct BoundsTable {
  Extent ext[2 * kMaxRanks + 1];  // src[r], dst[r], then the scratch FIFO
  int n;
  unsigned* status;
  unsigned long long* where;
};
// One per CTA: the buffers of the running launch (filled by bounds_setup).
__shared__ BoundsTable g_bounds;

// Fills the table from the launch's arguments; every thread of the CTA
// calls it, and the caller's barrier publishes it.
__device__ __forceinline__ void bounds_setup(const KArgs& a) {
  for (int i = threadIdx.x; i < a.R; i += blockDim.x) {
    g_bounds.ext[2 * i] = Extent{static_cast<const char*>(a.src[i]), a.srcBytes, 0};
    g_bounds.ext[2 * i + 1] = Extent{static_cast<const char*>(a.dst[i]), a.dstBytes, 1};
  }
  if (threadIdx.x == 0) {
    g_bounds.ext[2 * a.R] = Extent{static_cast<const char*>(a.scratch), a.scratchBytes, 1};
    g_bounds.n = 2 * a.R + 1;
    g_bounds.status = a.status;
    g_bounds.where = a.boundsWhere;
  }
}

static __device__ __noinline__ bool access_ok(const void* p, unsigned long long n, bool store) {
  if (access_in(g_bounds.ext, g_bounds.n, static_cast<const char*>(p), n, store)) return true;
  if (g_bounds.status) atomicCAS(g_bounds.status, 0u, (unsigned)VR_ERR_INTERNAL);
  if (g_bounds.where) atomicCAS(g_bounds.where, 0ull, (unsigned long long)(uintptr_t)p);
  return false;
}
#define VR_ACCESS_OK(p, n, store) ::vr::access_ok((p), (n), (store))
#define VR_BOUNDS_SETUP(a) ::vr::bounds_setup(a)
#else
#define VR_ACCESS_OK(p, n, store) true
#define VR_BOUNDS_SETUP(a) ((void)0)
#endif

}  // namespace vr
