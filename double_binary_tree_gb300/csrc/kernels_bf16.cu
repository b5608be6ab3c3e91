// Instantiations of the AllReduce / ReduceScatter kernels for element type
// __nv_bfloat16 (one translation unit per type, compiled in parallel).
#include "host.h"
#include "kernels.cuh"
#include "staged.cuh"

namespace vr {

// Register-path kernels: `vec` = 16-byte units, else element units.  The
// few-rank variant (`small`) is fp32-only: for 16-bit types it measured
// slower than the general kernel at 2-4 ranks, so `small` is ignored here.
const void* kernel_ptr_bf16(int mode, int op, bool vec, int stack, bool /*small*/) {
#define VR_PICK(OP, VEC, SMALL)                                                                   \
  switch (mode) {                                                                                 \
    case kRingAllReduce:                                                                          \
      return (const void*)allreduce_kernel<__nv_bfloat16, OP, kRingAllReduce, VEC, 4, SMALL>;              \
    case kTreeAllReduce:                                                                          \
      return stack <= 4 ? (const void*)allreduce_kernel<__nv_bfloat16, OP, kTreeAllReduce, VEC, 4, SMALL>  \
                        : (const void*)allreduce_kernel<__nv_bfloat16, OP, kTreeAllReduce, VEC, 8, false>; \
    case kReduceScatter: return (const void*)reduce_scatter_kernel<__nv_bfloat16, OP, VEC>;                \
    default: return nullptr;                                                                      \
  }
  if (op == VR_SUM) {
    if (vec) { VR_PICK(VR_SUM, true, false) } else { VR_PICK(VR_SUM, false, false) }
  } else {
    if (vec) { VR_PICK(VR_MAX, true, false) } else { VR_PICK(VR_MAX, false, false) }
  }
#undef VR_PICK
}

// TMA-staged kernels (16-byte aligned buffers only).
const void* staged_kernel_ptr_bf16(int mode, int op, int stack, bool drawn) {
#define VR_PICK(OP)                                                                       \
  switch (mode) {                                                                         \
    case kRingAllReduce:                                                                  \
      return drawn ? (const void*)staged_kernel<__nv_bfloat16, OP, kRingAllReduce, 4, true>           \
                   : (const void*)staged_kernel<__nv_bfloat16, OP, kRingAllReduce, 4>;                \
    case kTreeAllReduce:                                                                  \
      if (drawn)                                                                          \
        return stack <= 4 ? (const void*)staged_kernel<__nv_bfloat16, OP, kTreeAllReduce, 4, true>     \
                          : (const void*)staged_kernel<__nv_bfloat16, OP, kTreeAllReduce, 8, true>;    \
      return stack <= 4 ? (const void*)staged_kernel<__nv_bfloat16, OP, kTreeAllReduce, 4>          \
                        : (const void*)staged_kernel<__nv_bfloat16, OP, kTreeAllReduce, 8>;         \
    case kReduceScatter: return (const void*)staged_kernel<__nv_bfloat16, OP, kReduceScatter, 4>;  \
    default: return nullptr;                                                              \
  }
  if (op == VR_SUM) { VR_PICK(VR_SUM) } else { VR_PICK(VR_MAX) }
#undef VR_PICK
}

}  // namespace vr
