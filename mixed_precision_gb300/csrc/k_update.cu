// K2 (finalize) and K3 (fused unscale / clip / AdamW / cast-out), plus the
// launch dispatch of K1.
#include "vec.cuh"

namespace zg {

const void* reduce_kernel_f32(int comm_dtype, int world, int stage);
const void* reduce_kernel_f16(int comm_dtype, int world, int stage);
const void* reduce_kernel_bf16(int comm_dtype, int world, int stage);

static const void* reduce_kernel(int grad_dtype, int comm_dtype, int world, int stage) {
  switch (grad_dtype) {
    case kF32: return reduce_kernel_f32(comm_dtype, world, stage);
    case kF16: return reduce_kernel_f16(comm_dtype, world, stage);
    case kBF16: return reduce_kernel_bf16(comm_dtype, world, stage);
    default: return nullptr;
  }
}

cudaError_t launch_reduce(const ReduceArgs& a, int grid, cudaStream_t s) {
  const void* f = reduce_kernel(a.grad_dtype, a.comm_dtype, a.world, a.stage);
  if (f == nullptr) return cudaErrorInvalidValue;
  void* args[] = {const_cast<ReduceArgs*>(&a)};
  return cudaLaunchKernel(f, dim3(grid), dim3(kThreads), args, 0, s);
}

int reduce_blocks_per_sm(int grad_dtype, int comm_dtype, int world, int stage) {
  const void* f = reduce_kernel(grad_dtype, comm_dtype, world, stage);
  int n = 0;
  if (f == nullptr || cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, f, kThreads, 0) != cudaSuccess)
    return 0;
  return n;
}

// ---------------------------------------------------------------------------
// K2: finalize. One block.
// "3.7 Megatron-LM, DeepSpeed & Parallelism in Practice", "ZeRO-Offload and
// ZeRO-Infinity": gradient_clipping, and fp16 loss_scale 0 (dynamic) with a
// loss_scale_window. "nano-deepspeed (Teaching Edition)", "2. Current Feature
// Range": FP16 dynamic loss scaling. The pages print no formula; the reading:
//   inv = 1 / (S * D), norm = inv * sqrt(sum r^2),
//   clip = min(1, max_norm / (norm + 1e-6)) (1 when max_norm <= 0);
//   overflow -> skip, S <- max(S * backoff, min_scale) (dynamic), counter <- 0;
//   clean    -> t += 1, counter += 1, S <- S * growth when counter == N.
// The block partials are summed in a fixed order (strided per thread, then a
// fixed shuffle tree), so the norm is the same on every run.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kFinalizeThreads)
    k_finalize(const double* __restrict__ part_sumsq, const unsigned* __restrict__ part_ovf,
               int n_part, int world, const Hparams hp, DevState* __restrict__ st) {
  __shared__ double s_red[kFinalizeThreads / 32];
  __shared__ unsigned s_or[kFinalizeThreads / 32];
  double acc = 0.0;
  unsigned ovf = 0u;
  for (int i = threadIdx.x; i < n_part; i += kFinalizeThreads) {
    acc += part_sumsq[i];
    ovf |= part_ovf[i];
  }
  const double sumsq = block_sum<kFinalizeThreads>(acc, s_red);
  const unsigned any = block_or<kFinalizeThreads>(ovf, s_or);
  if (threadIdx.x != 0) return;

  const double S = st->scale;
  const double D = hp.grad_divisor > 0.0 ? hp.grad_divisor : (double)world;
  const double inv = 1.0 / (S * D);
  st->steps += 1;
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
  st->t += 1;
  const double bc1 = 1.0 - pow(hp.beta1, (double)st->t);
  const double bc2 = 1.0 - pow(hp.beta2, (double)st->t);
  st->gscale = (float)(inv * c);
  st->decay = (float)(1.0 - hp.lr * hp.weight_decay);
  st->step_size = (float)(hp.lr / bc1);
  st->inv_sqrt_bc2 = (float)(1.0 / sqrt(bc2));
  st->beta1 = (float)hp.beta1;
  st->one_minus_beta1 = (float)(1.0 - hp.beta1);
  st->beta2 = (float)hp.beta2;
  st->one_minus_beta2 = (float)(1.0 - hp.beta2);
  st->eps = (float)hp.eps;
  st->counter += 1;
  if (st->dynamic && st->counter == st->growth_interval) {
    st->scale = S * st->growth_factor;
    st->counter = 0;
  }
}

cudaError_t launch_finalize(const double* part_sumsq, const unsigned* part_ovf, int n_part,
                            int world, const Hparams& hp, DevState* st, cudaStream_t s) {
  k_finalize<<<1, kFinalizeThreads, 0, s>>>(part_sumsq, part_ovf, n_part, world, hp, st);
  return cudaGetLastError();
}

__global__ void k_state_init(const ScalerCfg cfg, DevState* st) {
  DevState z = {};
  z.scale = cfg.init_scale;
  z.dynamic = cfg.dynamic;
  z.growth_interval = cfg.growth_interval;
  z.growth_factor = cfg.growth_factor;
  z.backoff_factor = cfg.backoff_factor;
  z.min_scale = cfg.min_scale;
  z.skip = 1;  // nothing to apply before the first finalize
  *st = z;
}

cudaError_t launch_state_init(const ScalerCfg& cfg, DevState* st, cudaStream_t s) {
  k_state_init<<<1, 1, 0, s>>>(cfg, st);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// K3: unscale + clip + AdamW + cast-out, one pass over every rank's shard.
// "nano-deepspeed (Teaching Edition)", "2. Current Feature Range": AdamW;
// "3.7 ...", "Initializing a DeepSpeed Engine": torch.optim.AdamW semantics
// (decoupled weight decay, bias correction). leetllm "Deep dive: Megatron",
// "Distributed optimizer": each rank updates its FP32 master slice and
// moments, then the all-gather rebuilds the BF16 parameter buffer -- here the
// cast result is written straight into the flat parameter buffer.
//   g = r * gscale;  p *= decay;  m = b1 m + (1-b1) g;  v = b2 v + (1-b2) g^2;
//   p -= step_size * m / (sqrt(v) * inv_sqrt_bc2 + eps);  param = RNE(p).
// Element math in fp32. A skipped step returns before touching memory.
// ---------------------------------------------------------------------------
template <typename CT, typename PT>
__global__ void __launch_bounds__(kThreads) k_adamw_cast(const __grid_constant__ UpdateArgs a) {
  const DevState* st = a.state;
  if (st->skip) return;
  const float gs = st->gscale, decay = st->decay, step = st->step_size;
  const float isb2 = st->inv_sqrt_bc2, eps = st->eps;
  const float b1 = st->beta1, omb1 = st->one_minus_beta1;
  const float b2 = st->beta2, omb2 = st->one_minus_beta2;

  auto adam = [&](float r, float& p, float& m, float& v) {
    const float g = r * gs;
    p = p * decay;
    m = b1 * m + omb1 * g;
    v = b2 * v + omb2 * (g * g);
    const float denom = sqrtf(v) * isb2 + eps;
    p = p - step * (m / denom);
  };

  for (int t = blockIdx.x; t < a.n_tiles; t += gridDim.x) {
    const Tile tl = a.tiles[t];
    const CT* red = a.stage == 1 ? static_cast<const CT*>(a.red.base[tl.rank]) + tl.flat
                                 : static_cast<const CT*>(a.red.base[0]) + tl.shard;
    float* mp = a.master + tl.shard;
    float* m1 = a.m + tl.shard;
    float* v1 = a.v + tl.shard;
    PT* pp = static_cast<PT*>(a.params_flat) + tl.flat;
    const int nvec = tl.len >> 3;
    for (int vi = threadIdx.x; vi < nvec; vi += kThreads) {
      const int64_t o = (int64_t)vi * 8;
      float r[8], p[8], m[8], v[8];
      load8(red + o, r);
      load8_f32(mp + o, p);
      load8_f32(m1 + o, m);
      load8_f32(v1 + o, v);
      Pack8<PT> out;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        adam(r[j], p[j], m[j], v[j]);
        out.e[j] = DT<PT>::from_f32(p[j]);
      }
      store8_f32(mp + o, p);
      store8_f32(m1 + o, m);
      store8_f32(v1 + o, v);
      store8_raw(pp + o, out);
    }
    const int rem = tl.len & 7;
    if (threadIdx.x < rem) {
      const int64_t i = (int64_t)nvec * 8 + threadIdx.x;
      float p = mp[i], m = m1[i], v = v1[i];
      adam(DT<CT>::to_f32(red[i]), p, m, v);
      mp[i] = p;
      m1[i] = m;
      v1[i] = v;
      pp[i] = DT<PT>::from_f32(p);
    }
  }
}

template <typename CT>
static const void* update_kernel_c(int param_dtype) {
  switch (param_dtype) {
    case kF16: return reinterpret_cast<const void*>(&k_adamw_cast<CT, __half>);
    case kBF16: return reinterpret_cast<const void*>(&k_adamw_cast<CT, __nv_bfloat16>);
    default: return nullptr;
  }
}

static const void* update_kernel(int comm_dtype, int param_dtype) {
  switch (comm_dtype) {
    case kF32: return update_kernel_c<float>(param_dtype);
    case kF16: return update_kernel_c<__half>(param_dtype);
    case kBF16: return update_kernel_c<__nv_bfloat16>(param_dtype);
    default: return nullptr;
  }
}

cudaError_t launch_update(const UpdateArgs& a, int grid, cudaStream_t s) {
  const void* f = update_kernel(a.comm_dtype, a.param_dtype);
  if (f == nullptr) return cudaErrorInvalidValue;
  void* args[] = {const_cast<UpdateArgs*>(&a)};
  return cudaLaunchKernel(f, dim3(grid), dim3(kThreads), args, 0, s);
}

int update_blocks_per_sm(int comm_dtype, int param_dtype) {
  const void* f = update_kernel(comm_dtype, param_dtype);
  int n = 0;
  if (f == nullptr || cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, f, kThreads, 0) != cudaSuccess)
    return 0;
  return n;
}

}  // namespace zg
