// Speculative single-pass instances for __nv_bfloat16 gradients.
#include "k_spec.cuh"

namespace zg {
const void* spec_kernel_bf16(int comm_dtype, int param_dtype, int world) {
  return spec_kernel_for<__nv_bfloat16, false>(comm_dtype, param_dtype, world);
}
}  // namespace zg
