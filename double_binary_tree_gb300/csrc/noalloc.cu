// Stepwise ring AllReduce for callers that cannot allocate device memory.
//
// vr_allreduce_ring_stepwise needs a scratch FIFO in device memory.  Some
// callers cannot provide one: a runtime that has handed all of the GPU's
// memory to its own allocator, or code on a latency-critical path that may
// not call cudaMalloc / cudaFree (they can synchronise the device).  This
// entry point runs the same kernels with the FIFO in a file-scope device
// array instead, so it allocates nothing.
#include <cuda_runtime.h>

#include <map>
#include <mutex>

#include "host.h"

namespace {

// The FIFO.  Every GPU that loads this file's module holds these
// VR_NOALLOC_SCRATCH_BYTES bytes until the process exits; all calls share
// them.  CUDA loads modules lazily by default, so on a device the array
// comes into being at the first call there (the address lookup below).
static __device__ __align__(256) unsigned char g_noalloc_fifo[VR_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
std::map<int, void*> g_fifo;  // device ordinal -> device address of g_noalloc_fifo

// The device address of the FIFO on the current device.  In host code the
// array's name only stands in for the symbol; the address comes from the
// runtime, once per device, with that device current.
vr_result_t fifo_address(void** out) {
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return VR_ERR_CUDA;
  std::lock_guard<std::mutex> g(g_mu);
  auto it = g_fifo.find(device);
  if (it == g_fifo.end()) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_fifo) != cudaSuccess || p == nullptr)
      return VR_ERR_CUDA;
    it = g_fifo.emplace(device, p).first;
  }
  *out = it->second;
  return VR_SUCCESS;
}

}  // namespace

extern "C" vr_result_t vr_allreduce_ring_stepwise_noalloc(const void* const* sendbufs,
                                                          void* const* recvbufs, int R,
                                                          size_t count, vr_dtype_t dtype,
                                                          vr_op_t op, int nChannels,
                                                          size_t chunkBytes, void* stream) {
  // the arguments first: a bad call is INVALID_ARGUMENT whatever its size
  const vr_result_t bad = vr::check_stepwise_args(sendbufs, recvbufs, R, count, dtype, op,
                                                  nChannels, chunkBytes);
  if (bad != VR_SUCCESS) return bad;
  const size_t need = vr_ring_stepwise_scratch_bytes(count, dtype);
  if (need > VR_NOALLOC_SCRATCH_BYTES) return VR_ERR_UNSUPPORTED;
  void* fifo = nullptr;
  if (count > 0 && need > 0) {
    const vr_result_t e = fifo_address(&fifo);
    if (e != VR_SUCCESS) return e;
  }
  return vr_allreduce_ring_stepwise(sendbufs, recvbufs, R, count, dtype, op, nChannels,
                                    chunkBytes, fifo, VR_NOALLOC_SCRATCH_BYTES, stream);
}
