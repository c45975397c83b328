// The local kernels of the sharded step (one process per GPU, this GPU holds
// one rank's shard). leetllm "Deep dive: Megatron", "Distributed optimizer:
// trade replicated state for collectives": the reduce-scatter hands each rank
// the sum of its slice of every bucket, the rank updates its fp32 master
// slice and moments, and the all-gather rebuilds the parameter buffer. The
// collectives themselves run in the caller's communication library; here are
// the pieces between them:
//   k_shard_norm     -- overflow flag and sum of squares of this rank's
//                       reduced slice (what the single-GPU reduce kernel fuses),
//                       as the pair {sum r^2, any non-finite ? 1 : 0} that the
//                       caller then sums over ranks (one 16-byte all-reduce);
//   k_dist_finalize  -- the finalize (norm, clip, loss-scale state machine)
//                       from that all-reduced pair, identical on every rank.
// The update is the single-GPU update kernel over this rank's tiles.
#include "finalize.cuh"
#include "k_reduce.cuh"
#include "vec.cuh"

namespace zg {

// Sum of squares and non-finite flag of the reduced values of this rank's
// tiles. Each block walks tiles grid-stride (fixed for a given grid, so the
// partials are deterministic), accumulating as the reduce kernel does: fp32
// squares over groups of 8, a compensated fp32 running sum, fp64 for huge
// groups. The last block to finish sums the block partials in index order
// and writes the pair.
template <typename CT>
__global__ void __launch_bounds__(kThreads)
    k_shard_norm(const Tile* __restrict__ tiles, int n_tiles, const CT* __restrict__ red,
                 int by_flat, double* part, unsigned* part_ovf, DevState* st,
                 double* __restrict__ pair) {
  if (st->error) return;
  __shared__ double s_red[kThreads / 32];
  __shared__ unsigned s_or[kThreads / 32];
  __shared__ bool s_last;
  float hi = 0.0f, lo = 0.0f;
  double big = 0.0;
  unsigned bad = 0u;
  for (int t = blockIdx.x; t < n_tiles; t += gridDim.x) {
    const Tile tl = tiles[t];
    const CT* r = red + (by_flat ? tl.flat : tl.shard);
    const int nvec = tl.len >> 3;
    for (int v = threadIdx.x; v < nvec; v += kThreads) {
      const Pack8<CT> bits = load8_raw(r + (int64_t)v * 8);
      float rf[8];
      float ss = 0.0f;
      bool fin = true;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        rf[j] = DT<CT>::to_f32(bits.e[j]);
        fin = fin && DT<CT>::finite_bits(bits.e[j]);
        ss = __fmaf_rn(rf[j], rf[j], ss);
      }
      if (!fin) bad = 1u;
      add_group(ss, hi, lo, big, rf);
    }
    const int rem = tl.len & 7;
    if (threadIdx.x < rem) {
      const CT x = r[(int64_t)nvec * 8 + threadIdx.x];
      const double d = (double)DT<CT>::to_f32(x);
      if (!DT<CT>::finite_bits(x)) bad = 1u;
      big += d * d;
    }
  }
  const double total = block_sum<kThreads>((double)hi + (double)lo + big, s_red);
  const unsigned any = block_or<kThreads>(bad, s_or);
  if (threadIdx.x == 0) {
    part[blockIdx.x] = total;
    part_ovf[blockIdx.x] = any;
    __threadfence();
    // wraps to 0 after the last block: no reset needed between launches
    s_last = atomicInc(&st->blocks_done, gridDim.x - 1) == gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last || threadIdx.x >= 32) return;
  __threadfence();
  double sum;
  unsigned ovf;
  warp_sum_partials(part, part_ovf, gridDim.x, sum, ovf);
  if (threadIdx.x == 0) {
    pair[0] = sum;
    pair[1] = ovf ? 1.0 : 0.0;
  }
}

// The finalize from the pair summed over every rank: pair[0] is the global
// sum of squares, pair[1] > 0 when any rank saw a non-finite value.
__global__ void k_dist_finalize(const double* __restrict__ pair, int world, const Hparams hp,
                                DevState* st) {
  if (st->error) return;
  finalize_state(pair[0], pair[1] != 0.0 ? 1u : 0u, world, hp, st);
}

// out[i] = fp32(g[i]) over a plain range (exact: every bf16 and fp16 value is
// an fp32 value). 16-byte vectors of 8 elements, then the tail.
template <typename GT>
__global__ void __launch_bounds__(kThreads)
    k_widen(const GT* __restrict__ g, float* __restrict__ out, int64_t n) {
  const int64_t nvec = n >> 3;
  for (int64_t v = (int64_t)blockIdx.x * kThreads + threadIdx.x; v < nvec;
       v += (int64_t)gridDim.x * kThreads) {
    float x[8];
    load8(g + v * 8, x);
    store8_f32(out + v * 8, x);
  }
  for (int64_t i = nvec * 8 + (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * kThreads)
    out[i] = DT<GT>::to_f32(g[i]);
}

cudaError_t launch_widen(const void* g, int grad_dtype, float* out, int64_t n, int grid,
                         cudaStream_t s) {
  if (grad_dtype == kF16)
    k_widen<__half><<<grid, kThreads, 0, s>>>(static_cast<const __half*>(g), out, n);
  else if (grad_dtype == kBF16)
    k_widen<__nv_bfloat16><<<grid, kThreads, 0, s>>>(static_cast<const __nv_bfloat16*>(g), out, n);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_shard_norm(const Tile* tiles, int n_tiles, const void* red, int comm_dtype,
                              int by_flat, double* part, unsigned* part_ovf, DevState* st,
                              double* pair, int grid, cudaStream_t s) {
  switch (comm_dtype) {
    case kF32:
      k_shard_norm<float><<<grid, kThreads, 0, s>>>(tiles, n_tiles, static_cast<const float*>(red),
                                                    by_flat, part, part_ovf, st, pair);
      break;
    case kF16:
      k_shard_norm<__half><<<grid, kThreads, 0, s>>>(tiles, n_tiles, static_cast<const __half*>(red),
                                                     by_flat, part, part_ovf, st, pair);
      break;
    case kBF16:
      k_shard_norm<__nv_bfloat16><<<grid, kThreads, 0, s>>>(
          tiles, n_tiles, static_cast<const __nv_bfloat16*>(red), by_flat, part, part_ovf, st, pair);
      break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_dist_finalize(const double* pair, int world, const Hparams& hp, DevState* st,
                                 cudaStream_t s) {
  k_dist_finalize<<<1, 1, 0, s>>>(pair, world, hp, st);
  return cudaGetLastError();
}

}  // namespace zg
