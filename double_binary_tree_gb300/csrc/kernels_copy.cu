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

// TMA AllGather variants: (tile bytes, stages); nullptr for other pairs.
const void* kernel_ptr_allgather_tma(int tile, int stages) {
#define VR_AG(T, S) \
  if (tile == T && stages == S) return (const void*)allgather_tma_kernel<T, S>;
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

}  // namespace vr
