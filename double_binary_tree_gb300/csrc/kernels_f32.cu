// Instantiations of the AllReduce / ReduceScatter kernels for element type
// float (one translation unit per type, compiled in parallel).
#include "host.h"
#include "kernels.cuh"
#include "staged.cuh"

namespace vr {

// Register-path kernels: `vec` = 16-byte units, else element units;
// `small`: the variant for at most 4 ranks.
const void* kernel_ptr_f32(int mode, int op, bool vec, int stack, bool small) {
#define VR_PICK(OP, VEC, SMALL)                                                                   \
  switch (mode) {                                                                                 \
    case kRingAllReduce:                                                                          \
      return (const void*)allreduce_kernel<float, OP, kRingAllReduce, VEC, 4, SMALL>;              \
    case kTreeAllReduce:                                                                          \
      return stack <= 4 ? (const void*)allreduce_kernel<float, OP, kTreeAllReduce, VEC, 4, SMALL>  \
                        : (const void*)allreduce_kernel<float, OP, kTreeAllReduce, VEC, 8, false>; \
    case kReduceScatter: return (const void*)reduce_scatter_kernel<float, OP, VEC>;                \
    default: return nullptr;                                                                      \
  }
  if (op == VR_SUM) {
    if (vec && small) { VR_PICK(VR_SUM, true, true) }
    else if (vec) { VR_PICK(VR_SUM, true, false) } else { VR_PICK(VR_SUM, false, false) }
  } else {
    if (vec && small) { VR_PICK(VR_MAX, true, true) }
    else if (vec) { VR_PICK(VR_MAX, true, false) } else { VR_PICK(VR_MAX, false, false) }
  }
#undef VR_PICK
}

// TMA-staged kernels (16-byte aligned buffers only).
const void* staged_kernel_ptr_f32(int mode, int op, int stack, bool drawn) {
#define VR_PICK(OP)                                                                       \
  switch (mode) {                                                                         \
    case kRingAllReduce:                                                                  \
      return drawn ? (const void*)staged_kernel<float, OP, kRingAllReduce, 4, true>           \
                   : (const void*)staged_kernel<float, OP, kRingAllReduce, 4>;                \
    case kTreeAllReduce:                                                                  \
      if (drawn)                                                                          \
        return stack <= 4 ? (const void*)staged_kernel<float, OP, kTreeAllReduce, 4, true>     \
                          : (const void*)staged_kernel<float, OP, kTreeAllReduce, 8, true>;    \
      return stack <= 4 ? (const void*)staged_kernel<float, OP, kTreeAllReduce, 4>          \
                        : (const void*)staged_kernel<float, OP, kTreeAllReduce, 8>;         \
    case kReduceScatter: return (const void*)staged_kernel<float, OP, kReduceScatter, 4>;  \
    default: return nullptr;                                                              \
  }
  if (op == VR_SUM) { VR_PICK(VR_SUM) } else { VR_PICK(VR_MAX) }
#undef VR_PICK
}

}  // namespace vr
