// Speculative single-pass instances for __half gradients.
#include "k_spec.cuh"

namespace zg {
const void* spec_kernel_f16(int comm_dtype, int param_dtype, int world) {
  return spec_kernel_for<__half, false>(comm_dtype, param_dtype, world);
}
}  // namespace zg
