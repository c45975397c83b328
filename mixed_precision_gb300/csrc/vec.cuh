// Device helpers shared by the kernels: 8-element vector loads/stores of
// fp32 / fp16 / bf16 with streaming cache hints, dtype traits, and
// deterministic block reductions.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace zg {

// ---- streaming 16-byte accesses (each element is touched once per kernel) --

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ void st_stream(void* p, uint4 v) {
  __stcs(reinterpret_cast<uint4*>(p), v);
}

// ---- dtype traits -----------------------------------------------------------

template <typename T> struct DT;
template <> struct DT<float> {
  static constexpr int kBytes = 4;
  __device__ static float to_f32(float x) { return x; }
  __device__ static float from_f32(float x) { return x; }
  __device__ static bool finite_bits(float x) {
    return (__float_as_uint(x) & 0x7F800000u) != 0x7F800000u;
  }
};
template <> struct DT<__half> {
  static constexpr int kBytes = 2;
  __device__ static float to_f32(__half x) { return __half2float(x); }
  __device__ static __half from_f32(float x) { return __float2half_rn(x); }
  __device__ static bool finite_bits(__half x) {
    return (__half_as_ushort(x) & 0x7C00u) != 0x7C00u;
  }
};
template <> struct DT<__nv_bfloat16> {
  static constexpr int kBytes = 2;
  __device__ static float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
  __device__ static __nv_bfloat16 from_f32(float x) { return __float2bfloat16_rn(x); }
  __device__ static bool finite_bits(__nv_bfloat16 x) {
    return (__bfloat16_as_ushort(x) & 0x7F80u) != 0x7F80u;
  }
};

// 8 consecutive elements of T as fp32 (one 16-byte load for 2-byte types,
// two for fp32). p must be 16-byte aligned.
template <typename T>
__device__ __forceinline__ void load8(const T* p, float (&x)[8]) {
  if constexpr (sizeof(T) == 4) {
    uint4 a = ld_stream(p), b = ld_stream(p + 4);
    x[0] = __uint_as_float(a.x); x[1] = __uint_as_float(a.y);
    x[2] = __uint_as_float(a.z); x[3] = __uint_as_float(a.w);
    x[4] = __uint_as_float(b.x); x[5] = __uint_as_float(b.y);
    x[6] = __uint_as_float(b.z); x[7] = __uint_as_float(b.w);
  } else {
    uint4 a = ld_stream(p);
    const T* h = reinterpret_cast<const T*>(&a);
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = DT<T>::to_f32(h[j]);
  }
}

// 8 consecutive elements of T from shared memory as fp32 (16-byte aligned).
template <typename T>
__device__ __forceinline__ void load8_smem(const T* p, float (&x)[8]) {
  if constexpr (sizeof(T) == 4) {
    const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  } else {
    const uint4 a = *reinterpret_cast<const uint4*>(p);
    const T* h = reinterpret_cast<const T*>(&a);
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = DT<T>::to_f32(h[j]);
  }
}

// 4 consecutive elements of T from shared memory as fp32 (8 or 16 bytes, aligned).
template <typename T>
__device__ __forceinline__ void load4_smem(const T* p, float (&r)[4]) {
  if constexpr (sizeof(T) == 4) {
    const float4 x = *reinterpret_cast<const float4*>(p);
    r[0] = x.x; r[1] = x.y; r[2] = x.z; r[3] = x.w;
  } else {
    const uint2 x = *reinterpret_cast<const uint2*>(p);
    const T* h = reinterpret_cast<const T*>(&x);
#pragma unroll
    for (int j = 0; j < 4; ++j) r[j] = DT<T>::to_f32(h[j]);
  }
}

// 8 raw elements of T (no conversion).
template <typename T>
struct Pack8 {
  T e[8];
};

template <typename T>
__device__ __forceinline__ void store8_raw(T* p, const Pack8<T>& v) {
  if constexpr (sizeof(T) == 4) {
    const uint4* u = reinterpret_cast<const uint4*>(v.e);
    st_stream(p, u[0]);
    st_stream(p + 4, u[1]);
  } else {
    st_stream(p, *reinterpret_cast<const uint4*>(v.e));
  }
}

template <typename T>
__device__ __forceinline__ Pack8<T> load8_raw(const T* p) {
  Pack8<T> v;
  if constexpr (sizeof(T) == 4) {
    uint4* u = reinterpret_cast<uint4*>(v.e);
    u[0] = ld_stream(p);
    u[1] = ld_stream(p + 4);
  } else {
    *reinterpret_cast<uint4*>(v.e) = ld_stream(p);
  }
  return v;
}

__device__ __forceinline__ void load8_f32(const float* p, float (&x)[8]) {
  uint4 a = ld_stream(p), b = ld_stream(p + 4);
  x[0] = __uint_as_float(a.x); x[1] = __uint_as_float(a.y);
  x[2] = __uint_as_float(a.z); x[3] = __uint_as_float(a.w);
  x[4] = __uint_as_float(b.x); x[5] = __uint_as_float(b.y);
  x[6] = __uint_as_float(b.z); x[7] = __uint_as_float(b.w);
}

__device__ __forceinline__ void store8_f32(float* p, const float (&x)[8]) {
  st_stream(p, make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                          __float_as_uint(x[3])));
  st_stream(p + 4, make_uint4(__float_as_uint(x[4]), __float_as_uint(x[5]), __float_as_uint(x[6]),
                              __float_as_uint(x[7])));
}

__device__ __forceinline__ void store4_f32(float* p, const float (&x)[4]) {
  st_stream(p, make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                          __float_as_uint(x[3])));
}

// 4 elements of a 2-byte type as one 8-byte streaming store (8-byte aligned).
template <typename T>
__device__ __forceinline__ void store4_raw(T* p, const T (&e)[4]) {
  static_assert(sizeof(T) == 2, "4 x 2 bytes");
  uint2 u;
  T* h = reinterpret_cast<T*>(&u);
#pragma unroll
  for (int j = 0; j < 4; ++j) h[j] = e[j];
  __stcs(reinterpret_cast<uint2*>(p), u);
}

// ---- the element-wise AdamW update ----------------------------------------
// One fixed sequence of correctly rounded fp32 operations (explicit
// intrinsics, so no kernel's compiler contracts it differently): every
// update kernel produces the same bits for the same inputs and scalars.
//   g = r * gscale;  m = b1 m + (1-b1) g;  v = b2 v + (1-b2) g^2;
//   p -= lr_wd * p + step * m / (sqrt(v) * inv_sqrt_bc2 + eps)
struct AdamScalars {
  float gs, lr_wd, step, isb2, eps, b1, omb1, b2, omb2;

  __device__ static AdamScalars from(const DevState* st) {
    return AdamScalars{st->gscale, st->lr_wd, st->step_size, st->inv_sqrt_bc2, st->eps,
                       st->beta1, st->one_minus_beta1, st->beta2, st->one_minus_beta2};
  }

  // Zero operands are answered without calling sqrt or divide (sqrt(+0) =
  // +0; +-0 / denom = +-0, as denom >= eps > 0), which gives the same bits:
  // parameters whose gradient has been zero on every rank (MoE experts no
  // token reached) keep m = v = 0, and the correctly rounded sqrt and divide
  // are much slower on such operands than on ordinary ones.
  __device__ __forceinline__ void apply(float r, float& p, float& m, float& v) const {
    const float g = __fmul_rn(r, gs);
    // moments as interpolations m + (1-b1)(g - m) and v + (1-b2)(g^2 - v):
    // the implied beta is exactly 1 - (1-beta) in fp32, where b*x + (1-b)*y
    // with b and 1-b rounded separately would not sum to one (0.999f +
    // 0.001f exceeds 1 by 1.3e-8, a bias v's long memory accumulates)
    m = __fmaf_rn(omb1, __fsub_rn(g, m), m);
    v = __fmaf_rn(omb2, __fsub_rn(__fmul_rn(g, g), v), v);
    const bool vz = v == 0.0f, mz = m == 0.0f;  // v >= +0 always
    const float sv = __fsqrt_rn(vz ? 1.0f : v);
    const float denom = __fmaf_rn(vz ? 0.0f : sv, isb2, eps);
    const float q = mz ? m : __fdiv_rn(mz ? 1.0f : m, denom);
    // The step's whole change to p, decoupled decay included, formed at its
    // own scale (far below p's) and subtracted with one rounding: rounding p
    // twice per step (after the decay, then after the update) makes the fp32
    // state walk away from an exact update by up to half an ulp a step.
    p = __fsub_rn(p, __fmaf_rn(lr_wd, p, __fmul_rn(step, q)));
  }
};

// The per-step fp32 scalars of the update, derived in fp64 from the scale's
// inverse `inv` = 1/(S*D), the clip coefficient and the step count t of the
// update. The finalize kernel and the speculative pass both use this, so the
// two produce identical scalars.
// beta1^(t+1) and beta2^(t+1) for the step after the state's t. The state
// keeps beta^t as a running product, so this is one fp64 multiply each
// (GB300's fp64 pipe is narrow, and pow on one thread took most of the
// finalize's ~10 us); pow is used when the products are not valid for these
// betas (the first step, a restored t, betas changed between steps). The
// product differs from pow by at most about t rounding errors of 2^-53.
__device__ __forceinline__ void bias_powers(const Hparams& hp, const DevState* st, double& b1t,
                                            double& b2t) {
  if (hp.beta1 == st->beta1_pow_of && hp.beta2 == st->beta2_pow_of) {
    b1t = st->beta1_pow * hp.beta1;
    b2t = st->beta2_pow * hp.beta2;
  } else {
    b1t = pow(hp.beta1, (double)(st->t + 1));
    b2t = pow(hp.beta2, (double)(st->t + 1));
  }
}

// b1t = beta1^t and b2t = beta2^t for the step's t (bias_powers).
__device__ __forceinline__ AdamScalars derive_adam_scalars(const Hparams& hp, double inv, double c,
                                                          double b1t, double b2t) {
  const double bc1 = 1.0 - b1t;
  const double bc2 = 1.0 - b2t;
  AdamScalars s;
  s.gs = (float)(inv * c);
  s.lr_wd = (float)(hp.lr * hp.weight_decay);
  s.step = (float)(hp.lr / bc1);
  s.isb2 = (float)(1.0 / sqrt(bc2));
  s.eps = (float)hp.eps;
  s.b1 = (float)hp.beta1;
  s.omb1 = (float)(1.0 - hp.beta1);
  s.b2 = (float)hp.beta2;
  s.omb2 = (float)(1.0 - hp.beta2);
  return s;
}

// ---- deterministic block reductions (fixed shuffle tree, fixed warp order) --

template <int kBlock>
__device__ __forceinline__ double block_sum(double x, double* smem /* kBlock/32 */) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_down_sync(0xffffffffu, x, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) smem[warp] = x;
  __syncthreads();
  double r = 0.0;
  if (warp == 0) {
    r = lane < kBlock / 32 ? smem[lane] : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) r += __shfl_down_sync(0xffffffffu, r, o);
  }
  __syncthreads();
  return r;  // valid in thread 0
}

template <int kBlock>
__device__ __forceinline__ unsigned block_or(unsigned x, unsigned* smem) {
  x = __any_sync(0xffffffffu, x != 0u) ? 1u : 0u;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) smem[warp] = x;
  __syncthreads();
  unsigned r = 0u;
  if (warp == 0) {
    r = lane < kBlock / 32 ? smem[lane] : 0u;
    r = __any_sync(0xffffffffu, r != 0u) ? 1u : 0u;
  }
  __syncthreads();
  return r;
}

}  // namespace zg
