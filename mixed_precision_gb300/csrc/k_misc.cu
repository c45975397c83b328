// Gradient accumulation into fp32 main gradients, and the self-test of the
// bounded-wait path.
#include "bulk.cuh"
#include "vec.cuh"
#include "zero.h"

namespace zg {

// main[w][i] = (first ? +0 : main[w][i]) + fp32(micro[w][i]) over real elements.
// leetllm "Deep dive: Megatron", "Distributed optimizer": BF16 parameters
// with FP32 main gradients; "3.7 ...", "Initializing a DeepSpeed Engine":
// the reduction fires only on boundary micro-steps, so gradients accumulate
// in between.
template <typename MT>
__global__ void __launch_bounds__(kThreads) k_accumulate(const __grid_constant__ AccArgs a) {
  for (int t = blockIdx.x; t < a.n_tiles; t += gridDim.x) {
    const Tile tl = a.tiles[t];
    const int nvec = tl.len >> 3;
    for (int w = 0; w < a.world; ++w) {
      const MT* src = static_cast<const MT*>(a.micro[w]) + tl.flat;
      float* dst = a.main[w] + tl.flat;
      for (int v = threadIdx.x; v < nvec; v += kThreads) {
        float x[8], s[8];
        load8(src + v * 8, x);
        if (a.first) {
#pragma unroll
          for (int j = 0; j < 8; ++j) s[j] = 0.0f;
        } else {
          load8_f32(dst + v * 8, s);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) s[j] = __fadd_rn(s[j], x[j]);
        store8_f32(dst + v * 8, s);
      }
      const int rem = tl.len & 7;
      if (threadIdx.x < rem) {
        const int i = nvec * 8 + threadIdx.x;
        const float base = a.first ? 0.0f : dst[i];
        dst[i] = __fadd_rn(base, DT<MT>::to_f32(src[i]));
      }
    }
  }
}

cudaError_t launch_accumulate(const AccArgs& a, int grid, cudaStream_t s) {
  const void* f = nullptr;
  switch (a.micro_dtype) {
    case kF32: f = reinterpret_cast<const void*>(&k_accumulate<float>); break;
    case kF16: f = reinterpret_cast<const void*>(&k_accumulate<__half>); break;
    case kBF16: f = reinterpret_cast<const void*>(&k_accumulate<__nv_bfloat16>); break;
    default: return cudaErrorInvalidValue;
  }
  void* args[] = {const_cast<AccArgs*>(&a)};
  return cudaLaunchKernel(f, dim3(grid), dim3(kThreads), args, 0, s);
}

// Self-test: an mbarrier armed for 16 bytes that never arrive; the bounded
// wait must give up and record the timeout, in the module's own word or (err
// not NULL) OR-ed into a layout's device error word as the step kernels do.
// Nothing is copied, so nothing is in flight when the block exits.
static __device__ unsigned g_selftest_error;

__global__ void k_selftest_wait(uint32_t limit, unsigned* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_init_fence();
    mbar_arrive_expect_tx(&bar, 16);
    const unsigned code = mbar_wait(&bar, 0, limit) ? 0u : kErrWaitTimeout;
    g_selftest_error = code;
    if (err != nullptr && code != 0u) atomicOr(err, code);
  }
}

cudaError_t launch_selftest_wait(uint32_t limit, unsigned* err, cudaStream_t s) {
  k_selftest_wait<<<1, 32, 0, s>>>(limit, err);
  return cudaGetLastError();
}

}  // namespace zg

using namespace zg;

extern "C" int zero_selftest_wait_timeout(uint32_t spin_limit, void* stream) {
  if (spin_limit < 1 || spin_limit > kSpinLimit)
    return zero_internal_fail(ZERO_ERR_INVALID, "spin_limit outside 1..2^22");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned err = 0;
  cudaError_t e = launch_selftest_wait(spin_limit, nullptr, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&err, g_selftest_error, sizeof(err));
  if (e != cudaSuccess) return zero_internal_fail(ZERO_ERR_CUDA, cudaGetErrorString(e));
  if (err != 0) return zero_internal_fail(ZERO_ERR_TIMEOUT, "bounded wait gave up (self-test)");
  return ZERO_OK;
}
