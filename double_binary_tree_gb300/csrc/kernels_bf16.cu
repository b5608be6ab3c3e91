// Instantiations of the AllReduce / ReduceScatter kernels for element type
// __nv_bfloat16 (one translation unit per type, compiled in parallel).
#include "host.h"
#include "kernels.cuh"
#include "staged.cuh"

namespace vr {

// Register-path kernels: `vec` = 16-byte units, else element units.
const void* kernel_ptr_bf16(int mode, int op, bool vec, int stack, bool pair) {
#define VR_PICK(OP, VEC, PAIR)                                                                   \
  switch (mode) {                                                                                \
    case kRingAllReduce:                                                                         \
      return (const void*)allreduce_kernel<__nv_bfloat16, OP, kRingAllReduce, VEC, 4, (VEC && PAIR) ? 2 : 1>; \
    case kTreeAllReduce:                                                                         \
      if (PAIR)                                                                                  \
        return (const void*)allreduce_kernel<__nv_bfloat16, OP, kTreeAllReduce, VEC, 4, (VEC && PAIR) ? 2 : 1>; \
      return stack <= 4 ? (const void*)allreduce_kernel<__nv_bfloat16, OP, kTreeAllReduce, VEC, 4, 1>     \
                        : (const void*)allreduce_kernel<__nv_bfloat16, OP, kTreeAllReduce, VEC, 8, 1>;    \
    case kReduceScatter: return (const void*)reduce_scatter_kernel<__nv_bfloat16, OP, VEC>;               \
    default: return nullptr;                                                                     \
  }
  // two units per step: vector path, at most 4 ranks (trees of <= 4 ranks
  // fold with at most 4 partials)
  if (op == VR_SUM) {
    if (vec && pair) { VR_PICK(VR_SUM, true, true) }
    else if (vec) { VR_PICK(VR_SUM, true, false) } else { VR_PICK(VR_SUM, false, false) }
  } else {
    if (vec && pair) { VR_PICK(VR_MAX, true, true) }
    else if (vec) { VR_PICK(VR_MAX, true, false) } else { VR_PICK(VR_MAX, false, false) }
  }
#undef VR_PICK
}

// TMA-staged kernels (16-byte aligned buffers only).
const void* staged_kernel_ptr_bf16(int mode, int op, int stack) {
#define VR_PICK(OP)                                                                       \
  switch (mode) {                                                                         \
    case kRingAllReduce: return (const void*)staged_kernel<__nv_bfloat16, OP, kRingAllReduce, 4>;  \
    case kTreeAllReduce:                                                                  \
      return stack <= 4 ? (const void*)staged_kernel<__nv_bfloat16, OP, kTreeAllReduce, 4>          \
                        : (const void*)staged_kernel<__nv_bfloat16, OP, kTreeAllReduce, 8>;         \
    case kReduceScatter: return (const void*)staged_kernel<__nv_bfloat16, OP, kReduceScatter, 4>;  \
    default: return nullptr;                                                              \
  }
  if (op == VR_SUM) { VR_PICK(VR_SUM) } else { VR_PICK(VR_MAX) }
#undef VR_PICK
}

}  // namespace vr
