// AllGather kernel instantiations and the per-device status word.
#include "gather.cuh"
#include "host.h"
#include "kernels.cuh"

namespace vr {

// First device-side error recorded by any kernel of this library on this
// device since it was last read (0 = none).
__device__ unsigned g_status_word = 0;

const void* kernel_ptr_allgather(bool vec) {
  return vec ? (const void*)allgather_kernel<true> : (const void*)allgather_kernel<false>;
}

const void* kernel_ptr_allgather_tma() { return (const void*)allgather_tma_kernel; }
int gather_tile_bytes() { return (int)kGatherTile; }
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

}  // namespace vr
