// Speculative single-pass instances for float gradients.
#include "k_spec.cuh"

namespace zg {
const void* spec_kernel_f32(int comm_dtype, int param_dtype, int world) {
  return spec_kernel_for<float, false>(comm_dtype, param_dtype, world);
}
}  // namespace zg
