// Bulk asynchronous copies (global -> shared) completed on mbarriers, for the
// streaming kernels' shared-memory pipelines. Inline PTX for sm_90+ /
// sm_103a: cp.async.bulk with mbarrier::complete_tx, mbarrier try_wait with a
// bounded retry count. Every wait here gives up after kSpinLimit tries and
// reports it, so no kernel can spin forever.
#pragma once

#include <cstdint>

#include "internal.h"  // kSpinLimit, kErrWaitTimeout

namespace zg {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make the barrier initialisation visible to the async (bulk copy) proxy.
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// The single arrival of a phase, announcing `bytes` of incoming bulk data.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// The single arrival of a phase with no data (completes the phase at once).
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// bytes (a multiple of 16, both addresses 16-byte aligned) from global to this
// CTA's shared memory; completion is counted on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete; false after `limit`
// unsuccessful tries (kSpinLimit by default).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          uint32_t limit = kSpinLimit) {
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// Programmatic dependent launch (sm_90+). A kernel launched with the
// programmatic-stream-serialization attribute may start before the kernel
// ahead of it in the stream has finished; griddep_wait() then blocks until
// that kernel has completed and its memory is visible, exactly the ordering
// of a plain launch. Every step kernel calls it before its first global
// access, then griddep_trigger(): once every block of this kernel has
// started, the next kernel's blocks may be scheduled (into the slots this
// kernel's finishing blocks free) and run up to their own wait. Without the
// attribute both instructions do nothing.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace zg
