// Speculative single-pass instances for __half gradients in stage 1 (ZeRO-1),
// which also write the W all-reduce outputs (compiled apart from the other
// stages' instances so that the build runs them in parallel).
#include "k_spec.cuh"

namespace zg {
const void* spec_kernel_s1_f16(int comm_dtype, int param_dtype, int world) {
  return spec_kernel_for<__half, true>(comm_dtype, param_dtype, world);
}
}  // namespace zg
