// K1: the reduce-scatter's arithmetic, fused with the overflow check and the
// per-block partial of the gradient norm.
//
// leetllm "Deep dive: Megatron", "Distributed optimizer: trade replicated
// state for collectives": the reduce-scatter combines the ranks' gradients
// and hands each rank its shard. "nano-deepspeed (Teaching Edition)",
// "9. Experimental Results": the reduction is communicated in a stated dtype
// (communication_data_type); "2. Current Feature Range": FP16 dynamic loss
// scaling, which needs the non-finite check.
//
// Per element i of a tile: r = RNE_comm(g_0[i] + g_1[i] + ... + g_{W-1}[i]),
// the adds in fp32 and in rank order. Stage 2 writes r once, into the
// rank-major scratch at the tile's shard offset (rank `tile.rank`'s
// reduce-scatter output). Stage 1 writes r into all W flat outputs (the
// all-reduce). Every thread accumulates sum(r^2) (fp32 over 8 elements, then
// fp64) and an "any non-finite r" flag; each block writes one fp64 partial and
// one flag. The grid is persistent (a multiple of the SM count) and walks the
// tile list with a fixed stride, so the partials are deterministic.
#pragma once

#include "vec.cuh"

namespace zg {

template <typename GT>
__device__ __forceinline__ void first8(const GT* p, float (&s)[8]) {
  if (p == nullptr) {
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j] = 0.0f;
  } else {
    load8(p, s);
  }
}

template <typename GT>
__device__ __forceinline__ void add8(const GT* p, float (&s)[8]) {
  float x[8];
  if (p == nullptr) {
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = 0.0f;
  } else {
    load8(p, x);
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) s[j] = __fadd_rn(s[j], x[j]);
}

template <typename GT>
__device__ __forceinline__ float load1(const GT* p, int64_t i) {
  return p == nullptr ? 0.0f : DT<GT>::to_f32(p[i]);
}

template <typename GT, typename CT, int WT, bool STAGE1>
__global__ void __launch_bounds__(kThreads) k_reduce_norm(const __grid_constant__ ReduceArgs a) {
  // Vectors in flight per thread: keep about eight 16-byte gradient loads
  // outstanding whatever W is.
  constexpr int U = (WT == 0 || WT >= 8) ? 1 : 8 / WT;
  __shared__ const GT* s_ptr[kMaxWorld];
  __shared__ CT* s_out[STAGE1 ? kMaxWorld : 1];
  __shared__ double s_red[kThreads / 32];
  __shared__ unsigned s_or[kThreads / 32];

  const int W = WT ? WT : a.world;
  double acc = 0.0;
  unsigned bad = 0u;

  for (int t = blockIdx.x; t < a.n_tiles; t += gridDim.x) {
    const Tile tl = a.tiles[t];
    __syncthreads();  // everyone is done with the previous tile's pointers
    for (int w = threadIdx.x; w < W; w += kThreads) {
      const GT* p;
      if (a.src.table_mode) {
        const void* q = a.src.table[(int64_t)w * a.src.n_params + tl.param];
        p = q ? static_cast<const GT*>(q) + tl.in_param : nullptr;
      } else {
        p = static_cast<const GT*>(a.src.base[w]) + tl.flat;
      }
      s_ptr[w] = p;
      if constexpr (STAGE1) s_out[w] = static_cast<CT*>(a.out.base[w]) + tl.flat;
    }
    __syncthreads();

    CT* out_shard = static_cast<CT*>(a.out.base[0]) + tl.shard;
    const int nvec = tl.len >> 3;
    for (int v0 = threadIdx.x; v0 < nvec; v0 += kThreads * U) {
      float s[U][8];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + u * kThreads;
        if (v < nvec) {
          const GT* p0 = s_ptr[0];
          first8(p0 ? p0 + (int64_t)v * 8 : nullptr, s[u]);
        }
      }
      for (int w = 1; w < W; ++w) {
        const GT* pw = s_ptr[w];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int v = v0 + u * kThreads;
          if (v < nvec) add8(pw ? pw + (int64_t)v * 8 : nullptr, s[u]);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + u * kThreads;
        if (v < nvec) {
          Pack8<CT> rc;
          float ss = 0.0f;
          bool fin = true;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            rc.e[j] = DT<CT>::from_f32(s[u][j]);
            const float rf = DT<CT>::to_f32(rc.e[j]);
            fin = fin && DT<CT>::finite_bits(rc.e[j]);
            ss = __fmaf_rn(rf, rf, ss);
          }
          if (!fin) bad = 1u;
          if (isfinite(ss)) {
            acc += (double)ss;
          } else {  // finite values whose squares overflow fp32 (or a non-finite r)
            double d = 0.0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const double rf = (double)DT<CT>::to_f32(rc.e[j]);
              d += rf * rf;
            }
            acc += d;
          }
          if constexpr (STAGE1) {
            for (int w = 0; w < W; ++w) store8_raw(s_out[w] + (int64_t)v * 8, rc);
          } else {
            store8_raw(out_shard + (int64_t)v * 8, rc);
          }
        }
      }
    }
    // Ragged tail of the tile (only a parameter's last tile has one).
    const int rem = tl.len & 7;
    if (threadIdx.x < rem) {
      const int64_t i = (int64_t)nvec * 8 + threadIdx.x;
      float sum = load1(s_ptr[0], i);
      for (int w = 1; w < W; ++w) sum = __fadd_rn(sum, load1(s_ptr[w], i));
      const CT rc = DT<CT>::from_f32(sum);
      const double rf = (double)DT<CT>::to_f32(rc);
      if (!DT<CT>::finite_bits(rc)) bad = 1u;
      acc += rf * rf;
      if constexpr (STAGE1) {
        for (int w = 0; w < W; ++w) s_out[w][i] = rc;
      } else {
        out_shard[i] = rc;
      }
    }
  }

  const double total = block_sum<kThreads>(acc, s_red);
  const unsigned any_bad = block_or<kThreads>(bad, s_or);
  if (threadIdx.x == 0) {
    a.part_sumsq[blockIdx.x] = total;
    a.part_ovf[blockIdx.x] = any_bad;
  }
}

template <typename GT, typename CT, bool S1>
const void* reduce_kernel_w(int world) {
  switch (world) {
    case 1: return reinterpret_cast<const void*>(&k_reduce_norm<GT, CT, 1, S1>);
    case 2: return reinterpret_cast<const void*>(&k_reduce_norm<GT, CT, 2, S1>);
    case 4: return reinterpret_cast<const void*>(&k_reduce_norm<GT, CT, 4, S1>);
    case 8: return reinterpret_cast<const void*>(&k_reduce_norm<GT, CT, 8, S1>);
    default: return reinterpret_cast<const void*>(&k_reduce_norm<GT, CT, 0, S1>);
  }
}

template <typename GT, typename CT>
const void* reduce_kernel_s(int world, int stage) {
  return stage == 1 ? reduce_kernel_w<GT, CT, true>(world) : reduce_kernel_w<GT, CT, false>(world);
}

// The kernel instance for (grad dtype GT, comm dtype, world, stage).
template <typename GT>
const void* reduce_kernel_for(int comm_dtype, int world, int stage) {
  switch (comm_dtype) {
    case kF32: return reduce_kernel_s<GT, float>(world, stage);
    case kF16: return reduce_kernel_s<GT, __half>(world, stage);
    case kBF16: return reduce_kernel_s<GT, __nv_bfloat16>(world, stage);
    default: return nullptr;
  }
}

}  // namespace zg
