// K1 instances for __half gradients (split by gradient dtype to compile in parallel).
#include "k_reduce.cuh"

namespace zg {
const void* reduce_kernel_f16(int comm_dtype, int world, int stage, int variant) {
  return reduce_kernel_for<__half>(comm_dtype, world, stage, variant);
}
}  // namespace zg
