// AllGather kernel instantiations and the per-device status word.
#include "gather.cuh"
#include "host.h"
#include "kernels.cuh"

namespace vr {

// First device-side error recorded by any kernel of this library on this
// device since it was last read (0 = none).
__device__ unsigned g_status_word = 0;
// First address the bounds-checked build refused on this device since it
// was last read (0 = none).
__device__ unsigned long long g_bounds_word = 0;
// Tile scheduler slots of the staged AllReduce kernels (staged.cuh), 4 words
// each, all zero when free.
__device__ unsigned long long g_sched[kSchedSlots * 4];

const void* kernel_ptr_allgather(bool vec) {
  return vec ? (const void*)allgather_kernel<true> : (const void*)allgather_kernel<false>;
}

// TMA AllGather variants: (tile bytes, stages); nullptr for other pairs.
const void* kernel_ptr_allgather_tma(int tile, int stages) {
#define VR_AG(T, S) \
  if (tile == T && stages == S) return (const void*)allgather_tma_kernel<T, S>;
  VR_AG(8192, 4) VR_AG(8192, 8) VR_AG(16384, 4) VR_AG(16384, 6) VR_AG(32768, 3) VR_AG(4096, 8)
#undef VR_AG
  return nullptr;
}
// Destination-major TMA AllGather variants (small sources).
const void* kernel_ptr_allgather_tma_dest(int tile, int stages) {
#define VR_AG(T, S) \
  if (tile == T && stages == S) return (const void*)allgather_tma_dest_kernel<T, S>;
  VR_AG(8192, 4) VR_AG(8192, 8) VR_AG(16384, 4) VR_AG(16384, 6) VR_AG(32768, 3) VR_AG(4096, 8)
#undef VR_AG
  return nullptr;
}
int gather_tile_bytes() { return (int)kGatherTile; }
int gather_stages() { return kGatherStages; }
int gather_ctas_per_sm() { return kGatherCtasPerSm; }

cudaError_t read_and_clear_status(unsigned* value) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_status_word, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  const unsigned zero = 0;
  return cudaMemcpyToSymbol(g_status_word, &zero, sizeof(unsigned));
}

cudaError_t status_word_address(unsigned** p) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(p), g_status_word);
}

cudaError_t bounds_word_address(unsigned long long** p) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(p), g_bounds_word);
}

cudaError_t sched_table_address(unsigned long long** p) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(p), g_sched);
}

cudaError_t read_and_clear_bounds(unsigned long long* value) {
  cudaError_t e = cudaMemcpyFromSymbol(value, g_bounds_word, sizeof(*value));
  if (e != cudaSuccess) return e;
  const unsigned long long zero = 0;
  return cudaMemcpyToSymbol(g_bounds_word, &zero, sizeof(zero));
}

}  // namespace vr

using namespace vr;

extern "C" {

int vr_debug_bounds_checked(void) {
#ifdef VR_DEBUG_BOUNDS
  return 1;
#else
  return 0;
#endif
}

vr_result_t vr_debug_bounds_fault(unsigned long long* address) {
  if (!address) return VR_ERR_INVALID_ARGUMENT;
  if (read_and_clear_bounds(address) != cudaSuccess) return VR_ERR_CUDA;
  return VR_SUCCESS;
}

int vr_debug_access_ok(const void* const* lo, const unsigned long long* bytes,
                       const int* writable, int n, const void* p, unsigned long long size,
                       int store) {
  if (n < 0 || n > 2 * kMaxRanks + 1 || (n > 0 && (!lo || !bytes || !writable))) return -1;
  Extent ext[2 * kMaxRanks + 1];
  for (int i = 0; i < n; ++i)
    ext[i] = Extent{static_cast<const char*>(lo[i]), bytes[i], writable[i]};
  return access_in(ext, n, static_cast<const char*>(p), size, store != 0) ? 1 : 0;
}

}  // extern "C"
