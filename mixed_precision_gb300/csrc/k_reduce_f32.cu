// K1 instances for float gradients (split by gradient dtype to compile in parallel).
#include "k_reduce.cuh"

namespace zg {
const void* reduce_kernel_f32(int comm_dtype, int world, int stage, int variant) {
  return reduce_kernel_for<float>(comm_dtype, world, stage, variant);
}
}  // namespace zg
