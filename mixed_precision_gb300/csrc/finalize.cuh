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

// The scaler state machine and the update's scalars from the global sum of
// squares and overflow flag (one thread).
__device__ inline void finalize_state(double sumsq, unsigned any, int world, const Hparams& hp,
                                      DevState* st) {
  const double S = st->scale;
  const double D = hp.grad_divisor > 0.0 ? hp.grad_divisor : (double)world;
  const double inv = 1.0 / (S * D);
  st->steps += 1;
  st->need_fallback = 0;
  st->restore_params = 0;
  st->fast_path = 0;
  st->norm_sq_raw = sumsq;
  st->grad_norm = inv * sqrt(sumsq);
  st->overflow = any ? 1 : 0;
  if (any) {
    st->skipped = 1;
    st->skip = 1;
    st->clip_coef = 0.0;
    if (st->dynamic) {
      const double s2 = S * st->backoff_factor;
      st->scale = s2 < st->min_scale ? st->min_scale : s2;
    }
    st->counter = 0;
    return;
  }
  double c = 1.0;
  if (hp.max_grad_norm > 0.0) {
    c = hp.max_grad_norm / (st->grad_norm + 1e-6);
    if (c > 1.0) c = 1.0;
  }
  st->skipped = 0;
  st->skip = 0;
  st->clip_coef = c;
  st->predict_fallback = c < 1.0 ? 1 : 0;
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
    st->scale = S * st->growth_factor;
    st->counter = 0;
  }
}

// The speculative step's finalize (one thread): skip on overflow (and ask for
// the parameters back), ask for the two-pass kernels when clipping is active,
// else commit the single pass (flip the current state set).
__device__ inline void finalize_spec_state(double sumsq, unsigned any, int world, const Hparams& hp,
                                           DevState* st) {
  const double S = st->scale;
  const double D = hp.grad_divisor > 0.0 ? hp.grad_divisor : (double)world;
  const double inv = 1.0 / (S * D);
  st->need_fallback = 0;
  st->restore_params = 0;
  st->fast_path = 0;
  st->norm_sq_raw = sumsq;
  st->grad_norm = inv * sqrt(sumsq);
  st->overflow = any ? 1 : 0;
  if (any) {
    st->steps += 1;
    st->skipped = 1;
    st->skip = 1;
    st->clip_coef = 0.0;
    st->restore_params = 1;
    if (st->dynamic) {
      const double s2 = S * st->backoff_factor;
      st->scale = s2 < st->min_scale ? st->min_scale : s2;
    }
    st->counter = 0;
    return;
  }
  double c = 1.0;
  if (hp.max_grad_norm > 0.0) {
    c = hp.max_grad_norm / (st->grad_norm + 1e-6);
    if (c > 1.0) c = 1.0;
  }
  if (c < 1.0) {  // clipping active: the guarded two-pass kernels redo the step
    st->need_fallback = 1;
    st->skip = 1;
    st->predict_fallback = 1;
    return;
  }
  st->steps += 1;
  st->skipped = 0;
  st->skip = 1;  // the update already happened
  st->clip_coef = 1.0;
  double b1t, b2t;
  bias_powers(hp, st, b1t, b2t);
  st->t += 1;
  st->beta1_pow = b1t;
  st->beta2_pow = b2t;
  st->beta1_pow_of = hp.beta1;
  st->beta2_pow_of = hp.beta2;
  st->cur ^= 1;
  st->fast_path = 1;
  const AdamScalars a = derive_adam_scalars(hp, inv, 1.0, b1t, b2t);
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
    st->scale = S * st->growth_factor;
    st->counter = 0;
  }
}

// The speculative finalize when the single pass did not run (the last step
// clipped): go straight to the two-pass kernels.
__device__ inline void spec_predicted_state(DevState* st) {
  st->need_fallback = 1;
  st->restore_params = 0;
  st->fast_path = 0;
  st->skip = 1;
}

// Sum and OR of n block partials by one warp, in a fixed order (lane-strided,
// then a fixed shuffle tree), so the result is the same on every run. Reads
// through L2: other blocks wrote the partials during this kernel.
__device__ inline void warp_sum_partials(const double* part, const unsigned* ovf, int n,
                                         double& sum, unsigned& any) {
  const int lane = threadIdx.x & 31;
  double acc = 0.0;
  unsigned o = 0u;
  // Eight independent loads in flight per lane, then the adds in index order
  // (lane, lane + 32, ...): one L2 round trip per eight partials.
  constexpr int U = 8;
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
