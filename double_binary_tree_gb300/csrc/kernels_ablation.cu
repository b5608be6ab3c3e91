// Instantiations of the non-fused variants (two-phase tree, stepwise ring)
// for every element type.
#include "ablation.cuh"
#include "host.h"

namespace vr {

namespace {
template <typename T>
const void* pick(int which, int op, bool vec, int stack) {
#define VR_ONE(OP, VEC)                                                                        \
  switch (which) {                                                                             \
    case kTreeUp:                                                                              \
      return stack <= 4 ? (const void*)tree_up_kernel<T, OP, VEC, 4>                          \
                        : (const void*)tree_up_kernel<T, OP, VEC, 8>;                         \
    case kTreeDown: return (const void*)tree_down_kernel<T, VEC>;                              \
    case kRingStep: return (const void*)ring_step_kernel<T, OP, VEC>;                          \
    default: return nullptr;                                                                   \
  }
  if (op == VR_SUM) {
    if (vec) { VR_ONE(VR_SUM, true) } else { VR_ONE(VR_SUM, false) }
  } else {
    if (vec) { VR_ONE(VR_MAX, true) } else { VR_ONE(VR_MAX, false) }
  }
#undef VR_ONE
}
}  // namespace

const void* ablation_kernel_ptr(int which, int dtype, int op, bool vec, int stack) {
  if (which == kCopyRanks)
    return vec ? (const void*)copy_ranks_kernel<true> : (const void*)copy_ranks_kernel<false>;
  switch (dtype) {
    case VR_FLOAT32: return pick<float>(which, op, vec, stack);
    case VR_FLOAT16: return pick<__half>(which, op, vec, stack);
    case VR_BFLOAT16: return pick<__nv_bfloat16>(which, op, vec, stack);
    default: return nullptr;
  }
}

}  // namespace vr
