// K1 instances for __nv_bfloat16 gradients (split by gradient dtype to compile in parallel).
#include "k_reduce.cuh"

namespace zg {
const void* reduce_kernel_bf16(int comm_dtype, int world, int stage, int variant) {
  return reduce_kernel_for<__nv_bfloat16>(comm_dtype, world, stage, variant);
}
}  // namespace zg
