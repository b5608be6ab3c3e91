// Instantiations of the AllReduce / ReduceScatter kernels for element type
// float (one translation unit per type, compiled in parallel).
#include "host.h"
#include "kernels.cuh"

namespace vr {

const void* kernel_ptr_f32(int mode, int op, bool vec, int stack) {
#define VR_PICK(OP, VEC)                                                         \
  switch (mode) {                                                                \
    case kRingAllReduce: return (const void*)allreduce_kernel<float, OP, kRingAllReduce, VEC, 4>; \
    case kTreeAllReduce:                                                         \
      return stack <= 4 ? (const void*)allreduce_kernel<float, OP, kTreeAllReduce, VEC, 4>  \
                        : (const void*)allreduce_kernel<float, OP, kTreeAllReduce, VEC, 8>;  \
    case kReduceScatter: return (const void*)reduce_scatter_kernel<float, OP, VEC>;  \
    default: return nullptr;                                                     \
  }
  if (op == VR_SUM) {
    if (vec) { VR_PICK(VR_SUM, true) } else { VR_PICK(VR_SUM, false) }
  } else {
    if (vec) { VR_PICK(VR_MAX, true) } else { VR_PICK(VR_MAX, false) }
  }
#undef VR_PICK
}

}  // namespace vr
