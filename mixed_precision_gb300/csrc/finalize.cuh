// The finalize step's arithmetic, shared by the one-block finalize kernels
// and by the streaming kernels that finish it in their last block.
// "3.7 Megatron-LM, DeepSpeed & Parallelism in Practice", "ZeRO-Offload and
// ZeRO-Infinity": gradient_clipping, and fp16 loss_scale 0 (dynamic) with a
// loss_scale_window. "nano-deepspeed (Teaching Edition)", "2. Current Feature
// Range": FP16 dynamic loss scaling. The pages print no formula; the reading:
//   inv = 1 / (S * D), norm = inv * sqrt(sum r^2),
//   clip = min(1, max_norm / (norm + 1e-6)) (1 when max_norm <= 0);
//   overflow -> skip, S <- max(S * backoff, min_scale) (dynamic), counter <- 0;
//   clean    -> t += 1, counter += 1, S <- S * growth when counter == N.
#pragma once

#include "vec.cuh"

namespace zg {

// Pieces shared by both finalizes (one thread each).

// The step's norm report; returns inv = 1 / (S * D).
__device__ inline double record_norm(double sumsq, unsigned any, int world, const Hparams& hp,
                                     DevState* st) {
  const double D = hp.grad_divisor > 0.0 ? hp.grad_divisor : (double)world;
  const double inv = 1.0 / (st->scale * D);
  st->need_fallback = 0;
  st->restore_params = 0;
  st->fast_path = 0;
  st->norm_sq_raw = sumsq;
  st->grad_norm = inv * sqrt(sumsq);
  st->overflow = any ? 1 : 0;
  return inv;
}

__device__ inline double clip_coef(const Hparams& hp, const DevState* st) {
  if (!(hp.max_grad_norm > 0.0)) return 1.0;
  const double c = hp.max_grad_norm / (st->grad_norm + 1e-6);
  return c > 1.0 ? 1.0 : c;
}

// Overflow: the step is skipped, the scale backs off, the clean count restarts.
__device__ inline void skip_step(DevState* st) {
  st->steps += 1;
  st->skipped = 1;
  st->skip = 1;
  st->clip_coef = 0.0;
  if (st->dynamic) {
    const double s2 = st->scale * st->backoff_factor;
    st->scale = s2 < st->min_scale ? st->min_scale : s2;
  }
  st->counter = 0;
}

// A clean step: t advances, the update's scalars for clip coefficient c, and
// the scale grows after growth_interval clean steps.
__device__ inline void apply_step(const Hparams& hp, double inv, double c, DevState* st) {
  st->steps += 1;
  st->skipped = 0;
  st->clip_coef = c;
  double b1t, b2t;
  bias_powers(hp, st, b1t, b2t);
  st->t += 1;
  st->beta1_pow = b1t;
  st->beta2_pow = b2t;
  st->beta1_pow_of = hp.beta1;
  st->beta2_pow_of = hp.beta2;
  const AdamScalars a = derive_adam_scalars(hp, inv, c, b1t, b2t);
  st->gscale = a.gs;
  st->lr_wd = a.lr_wd;
  st->step_size = a.step;
  st->inv_sqrt_bc2 = a.isb2;
  st->beta1 = a.b1;
  st->one_minus_beta1 = a.omb1;
  st->beta2 = a.b2;
  st->one_minus_beta2 = a.omb2;
  st->eps = a.eps;
  st->counter += 1;
  if (st->dynamic && st->counter == st->growth_interval) {
    st->scale = st->scale * st->growth_factor;
    st->counter = 0;
  }
}

// The clip predictor, copied to the host word the library reads before the
// next speculative step (a hint for which kernels to launch; every path
// computes the same step).
__device__ inline void publish_prediction(const DevState* st) {
  if (st->hint != nullptr) *reinterpret_cast<volatile int*>(st->hint) = st->predict_fallback;
}

// The scaler state machine and the update's scalars from the global sum of
// squares and overflow flag (one thread).
__device__ inline void finalize_state(double sumsq, unsigned any, int world, const Hparams& hp,
                                      DevState* st) {
  const double inv = record_norm(sumsq, any, world, hp, st);
  if (any) {
    skip_step(st);
    return;
  }
  const double c = clip_coef(hp, st);
  st->skip = 0;
  st->predict_fallback = c < 1.0 ? 1 : 0;
  publish_prediction(st);
  apply_step(hp, inv, c, st);
}

// The speculative step's finalize (one thread): skip on overflow (and ask for
// the parameters back), ask for the two-pass kernels when clipping is active,
// else commit the single pass (flip the current state set).
__device__ inline void finalize_spec_state(double sumsq, unsigned any, int world, const Hparams& hp,
                                           DevState* st) {
  const double inv = record_norm(sumsq, any, world, hp, st);
  if (any) {
    skip_step(st);
    st->restore_params = 1;
    return;
  }
  if (clip_coef(hp, st) < 1.0) {  // clipping active: the guarded two-pass kernels redo the step
    st->need_fallback = 1;
    st->skip = 1;
    st->predict_fallback = 1;
    publish_prediction(st);
    return;
  }
  st->skip = 1;  // the update already happened
  st->cur ^= 1;
  st->fast_path = 1;
  apply_step(hp, inv, 1.0, st);
}

// The speculative finalize when the single pass did not run (the last step
// clipped): go straight to the two-pass kernels.
__device__ inline void spec_predicted_state(DevState* st) {
  st->need_fallback = 1;
  st->restore_params = 0;
  st->fast_path = 0;
  st->skip = 1;
}

// The end of a streaming pass that produces norm partials, called by each of
// the block's NC consumer warps with its lane's sum of squares and
// non-finite flag. The warp's total (a fixed shuffle tree) goes to a shared
// slot; the block's last warp to arrive (a shared counter) adds the slots in
// warp order and writes the block's partial. With `blocks_done` (the fused
// finalize), that warp then publishes the partial and counts the block in on
// the device counter, which wraps to 0 after the last block. Returns, in
// every lane, whether this warp counted in the grid's last block: that warp
// then sums all partials and runs the finalize.
template <int NC>
__device__ inline bool publish_block_partial(double x, unsigned bad, double* s_part,
                                             unsigned* s_flag, unsigned* s_done,
                                             double* part_sumsq, unsigned* part_ovf,
                                             unsigned* blocks_done) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_down_sync(0xffffffffu, x, o);
  const unsigned any = __any_sync(0xffffffffu, bad != 0u) ? 1u : 0u;
  unsigned last = 0u;
  if (lane == 0) {
    s_part[warp] = x;
    s_flag[warp] = any;
    __threadfence_block();
    if (atomicAdd(s_done, 1u) == NC - 1) {
      __threadfence_block();
      double total = 0.0;
      unsigned f = 0u;
      for (int w = 0; w < NC; ++w) {
        total += *reinterpret_cast<volatile double*>(&s_part[w]);
        f |= *reinterpret_cast<volatile unsigned*>(&s_flag[w]);
      }
      part_sumsq[blockIdx.x] = total;
      part_ovf[blockIdx.x] = f;
      if (blocks_done != nullptr) {
        __threadfence();
        last = atomicInc(blocks_done, gridDim.x - 1) == gridDim.x - 1 ? 1u : 0u;
      }
    }
  }
  return __shfl_sync(0xffffffffu, last, 0) != 0u;
}

// Sum and OR of n block partials by one warp, in a fixed order (lane-strided,
// then a fixed shuffle tree), so the result is the same on every run. Reads
// through L2: other blocks wrote the partials during this kernel.
__device__ inline void warp_sum_partials(const double* part, const unsigned* ovf, int n,
                                         double& sum, unsigned& any) {
  const int lane = threadIdx.x & 31;
  double acc = 0.0;
  unsigned o = 0u;
  // Sixteen independent loads in flight per lane, then the adds in index
  // order (lane, lane + 32, ...): one L2 round trip per sixteen partials.
  constexpr int U = 16;
  for (int base = lane; base < n; base += 32 * U) {
    double v[U];
    unsigned f[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + 32 * u;
      v[u] = i < n ? __ldcg(part + i) : 0.0;
      f[u] = i < n ? __ldcg(ovf + i) : 0u;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      acc += v[u];
      o |= f[u];
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    acc += __shfl_down_sync(0xffffffffu, acc, off);
    o |= __shfl_down_sync(0xffffffffu, o, off);
  }
  sum = __shfl_sync(0xffffffffu, acc, 0);
  any = __shfl_sync(0xffffffffu, o, 0);
}

}  // namespace zg
