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
// a compensated fp32 running sum, fp64 for huge groups) and an "any non-finite
// r" flag; each block writes one fp64 partial and one flag. The grid (a
// multiple of the blocks the GPU holds at once, fixed at bind) walks the tile
// list with a fixed stride, so for a given grid the partials are
// deterministic. In the pipelined kernel,
// the last block to finish then runs the finalize (finalize.cuh).
#pragma once

#include "bulk.cuh"
#include "finalize.cuh"
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

// Rank w's gradient pointer for a tile (flat buffers, or the per-tensor table
// where NULL stands for an all-zero gradient).
template <typename GT>
__device__ __forceinline__ const GT* grad_ptr(const ReduceArgs& a, const Tile& tl, int w) {
  if (a.src.table_mode) {
    const void* q = a.src.table[(int64_t)w * a.src.n_params + tl.param];
    return q ? static_cast<const GT*>(q) + tl.in_param : nullptr;
  }
  return static_cast<const GT*>(a.src.base[w]) + tl.flat;
}

// Squares of one group of 8 reduced values, added to a compensated fp32
// running sum (hi, lo). A group whose fp32 sum is not below 2^100 (or not
// finite) goes to an fp64 accumulator instead, so the fp32 sum cannot
// overflow. GB300's fp64 pipe is narrow, so fp64 is kept off the common path.
template <int N>
__device__ __forceinline__ void add_group(float ss, float& hi, float& lo, double& big,
                                          const float (&rf)[N]) {
  if (ss < 0x1p100f) {  // false for +inf and NaN as well
    const float y = ss - lo;
    const float t = hi + y;
    lo = (t - hi) - y;
    hi = t;
  } else {
    double d = 0.0;
#pragma unroll
    for (int j = 0; j < N; ++j) d += (double)rf[j] * (double)rf[j];
    big += d;
  }
}

template <typename GT, typename CT, int WT, bool STAGE1>
__global__ void __launch_bounds__(kThreads, 4) k_reduce_norm(const __grid_constant__ ReduceArgs a) {
  griddep_wait();
  griddep_trigger();
  if (a.state->error || (a.guarded && !a.state->need_fallback)) return;
  // Vectors in flight per thread: keep up to eight 16-byte gradient loads
  // outstanding (at most four vectors, to stay within 64 registers).
  constexpr int U = (WT == 0 || WT >= 8) ? 1 : (8 / WT > 4 ? 4 : 8 / WT);
  __shared__ double s_red[kThreads / 32];
  __shared__ unsigned s_or[kThreads / 32];

  const int W = WT ? WT : a.world;
  float hi = 0.0f, lo = 0.0f;
  double big = 0.0;
  unsigned bad = 0u;

  for (int t = blockIdx.x; t < a.n_tiles; t += gridDim.x) {
    const Tile tl = a.tiles[t];
    CT* out_shard = static_cast<CT*>(a.out.base[0]) + tl.shard;
    const int nvec = tl.len >> 3;
    for (int v0 = threadIdx.x; v0 < nvec; v0 += kThreads * U) {
      float s[U][8];
      {
        const GT* p0 = grad_ptr<GT>(a, tl, 0);
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int v = v0 + u * kThreads;
          if (v < nvec) first8(p0 ? p0 + (int64_t)v * 8 : nullptr, s[u]);
        }
      }
#pragma unroll(WT ? WT : 1)
      for (int w = 1; w < W; ++w) {
        const GT* pw = grad_ptr<GT>(a, tl, w);
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
          float rf[8];
          float ss = 0.0f;
          bool fin = true;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            rc.e[j] = DT<CT>::from_f32(s[u][j]);
            rf[j] = DT<CT>::to_f32(rc.e[j]);
            fin = fin && DT<CT>::finite_bits(rc.e[j]);
            ss = __fmaf_rn(rf[j], rf[j], ss);
          }
          if (!fin) bad = 1u;
          add_group(ss, hi, lo, big, rf);
          if constexpr (STAGE1) {
            for (int w = 0; w < W; ++w)
              store8_raw(static_cast<CT*>(a.out.base[w]) + tl.flat + (int64_t)v * 8, rc);
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
      float sum = load1(grad_ptr<GT>(a, tl, 0), i);
      for (int w = 1; w < W; ++w) sum = __fadd_rn(sum, load1(grad_ptr<GT>(a, tl, w), i));
      const CT rc = DT<CT>::from_f32(sum);
      const double rf = (double)DT<CT>::to_f32(rc);
      if (!DT<CT>::finite_bits(rc)) bad = 1u;
      big += rf * rf;
      if constexpr (STAGE1) {
        for (int w = 0; w < W; ++w) static_cast<CT*>(a.out.base[w])[tl.flat + i] = rc;
      } else {
        out_shard[i] = rc;
      }
    }
  }

  const double total = block_sum<kThreads>((double)hi + (double)lo + big, s_red);
  const unsigned any_bad = block_or<kThreads>(bad, s_or);
  if (threadIdx.x == 0) {
    a.part_sumsq[blockIdx.x] = total;
    a.part_ovf[blockIdx.x] = any_bad;
  }
}

// ---------------------------------------------------------------------------
// K1, shared-memory pipeline (the default). Same arithmetic and outputs as
// k_reduce_norm. Each stage holds one chunk (a.chunk elements) of all W
// ranks' gradients (kRedStageBytes), copied in by cp.async.bulk, kRedStages
// stages deep; a NULL per-tensor gradient is not copied and reads as zeros;
// a chunk's last (len mod 8) elements come from global memory directly. One
// producer warp (lane 0) fills the stages with one
// cp.async.bulk per rank and chunk; NC consumer warps each reduce a fixed
// slice of every chunk and release the stage on its "empty" mbarrier. The
// block's norm partial is assembled without a block barrier: each consumer
// warp leaves its partial in a shared slot and the last warp to finish (a
// shared-memory counter) adds the slots in warp order, so the result is the
// same on every run. With fuse_finalize, that warp then counts its block in
// on a device counter, and the warp of the last block to do so sums all the
// partials and runs finalize_state. A warp whose bounded wait gives up
// records kErrWaitTimeout and leaves; the block then writes no partial (and
// the step's finalize does not run: the error is reported instead).
//
// TABLE (per-tensor pointers, NULL entries allowed): the pointer table is
// read once per tile, and a tile with NULL ranks is cut into longer chunks.
// Its live ranks' slices share the stage's W * C elements, one after the
// other in rank order, so a chunk is floor(W / live) * C elements (a tile
// whose ranks are mostly idle moves more bytes per pipeline round trip). The
// length depends on the tile alone, so the producer and the consumers cut
// every tile alike. The consumers take a chunk of k * C elements as k
// C-element stretches in order, with the warp slices of a C-element chunk,
// so every thread adds the same groups to its norm partial in the same order
// as in flat mode: the two modes give the same bits. A tile whose ranks are
// all NULL is stored as +0.0 without the sum and conversion work, its groups
// still passed to the norm sum as +0.0 (a zero addend can change the
// compensated sum's bits). The flat instance is the same code with those
// branches compiled out.
// ---------------------------------------------------------------------------
template <typename GT, typename CT, int WT, bool STAGE1, int NC, bool TABLE>
__device__ __forceinline__ void reduce_ws_body(const ReduceArgs& a) {
  griddep_wait();
  griddep_trigger();
  if (a.state->error || (a.guarded && !a.state->need_fallback)) return;
  constexpr int S = kRedStages;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t full[S];
  __shared__ __align__(8) uint64_t empty[S];
  __shared__ double s_part[NC];
  __shared__ unsigned s_flag[NC];
  __shared__ unsigned s_done;
  const int W = WT ? WT : a.world;
  const int C = a.chunk;
  const int kStage = W * C * (int)sizeof(GT);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NC);
    }
    s_done = 0u;
    mbar_init_fence();
  }
  __syncthreads();

  // table mode: the ranks whose gradient for a tile is NULL, and the tile's
  // chunk length
  auto null_mask = [&](const Tile& t) -> uint64_t {
    uint64_t mk = 0ull;
    for (int w = 0; w < W; ++w)
      if (grad_ptr<GT>(a, t, w) == nullptr) mk |= 1ull << w;
    return mk;
  };
  auto chunk_len = [&](uint64_t nulls) -> int {
    const int live = W - __popcll(nulls);
    return live >= W ? C : C * (W / max(live, 1));
  };

  if (warp == NC) {  // producer
    if (lane != 0) return;
    int pt = blockIdx.x, pc = 0;
    unsigned k = 0;
    bool ok = true;
    uint64_t nulls = 0ull;
    int tc = C;  // the current tile's chunk length
    while (pt < a.n_tiles) {
      const int s = (int)(k % S);
      if (k >= (unsigned)S && !mbar_wait(&empty[s], ((k / S) - 1) & 1u)) {
        ok = false;
        break;
      }
      const Tile tl = a.tiles[pt];
      if constexpr (TABLE) {
        if (pc == 0) {
          nulls = null_mask(tl);
          tc = chunk_len(nulls);
        }
      }
      const int clen = min(tc, tl.len - pc);
      const int nb = clen & ~7;
      GT* base = reinterpret_cast<GT*>(smem + s * kStage);
      if constexpr (TABLE) {
        const uint32_t bytes = (uint32_t)((W - __popcll(nulls)) * nb) * (uint32_t)sizeof(GT);
        if (bytes > 0) {
          mbar_arrive_expect_tx(&full[s], bytes);
          GT* dst = base;
          for (int w = 0; w < W; ++w) {
            if ((nulls >> w) & 1ull) continue;
            bulk_g2s(dst, grad_ptr<GT>(a, tl, w) + pc, nb * (int)sizeof(GT), &full[s]);
            dst += tc;
          }
        } else {
          mbar_arrive(&full[s]);
        }
      } else {
        uint32_t bytes = 0;
        for (int w = 0; w < W; ++w)
          if (nb > 0 && grad_ptr<GT>(a, tl, w) != nullptr) bytes += nb * (uint32_t)sizeof(GT);
        if (bytes > 0) {
          mbar_arrive_expect_tx(&full[s], bytes);
          for (int w = 0; w < W; ++w) {
            const GT* g = grad_ptr<GT>(a, tl, w);
            if (g != nullptr) bulk_g2s(base + w * C, g + pc, nb * (int)sizeof(GT), &full[s]);
          }
        } else {
          mbar_arrive(&full[s]);
        }
      }
      ++k;
      pc += tc;
      if (pc >= tl.len) {
        pc = 0;
        pt += gridDim.x;
      }
    }
    if (!ok) {
      atomicOr(a.error, kErrWaitTimeout);
      for (unsigned j = k > (unsigned)S ? k - S : 0u; j < k; ++j) mbar_wait(&full[j % S], (j / S) & 1u);
    }
    return;
  }

  // consumers: warp `warp` owns elements [warp*per, (warp+1)*per) of every chunk
  const int per = ((C / NC) + 7) & ~7;
  float hi = 0.0f, lo = 0.0f;
  double big = 0.0;
  unsigned bad = 0u;
  int ct = blockIdx.x, cc = 0;
  unsigned k = 0;
  uint64_t nulls = 0ull;
  int tc = C;
  while (ct < a.n_tiles) {
    const int s = (int)(k % S);
    const Tile tl = a.tiles[ct];
    if constexpr (TABLE) {
      if (cc == 0) {
        nulls = null_mask(tl);
        tc = chunk_len(nulls);
      }
    }
    const int clen = min(tc, tl.len - cc);
    const int nb = clen & ~7;
    if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (k / S) & 1u))) {
      if (lane == 0) atomicOr(a.error, kErrWaitTimeout);
      return;
    }
    const GT* base = reinterpret_cast<const GT*>(smem + s * kStage);
    if constexpr (TABLE) {
      if (__popcll(nulls) == W) {
        // Every rank's gradient is NULL: each reduced value is +0.0. The
        // same groups still go through add_group, with the +0.0 sum the
        // general path would compute, so the norm partial keeps its bits.
        Pack8<CT> rc;
        float rf[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          rc.e[j] = DT<CT>::from_f32(0.0f);
          rf[j] = 0.0f;
        }
        for (int v0 = 0; v0 < nb; v0 += C) {
          const int e_end = min(nb, v0 + (warp + 1) * per);
          for (int e = v0 + warp * per + 8 * lane; e < e_end; e += 256) {
            add_group(0.0f, hi, lo, big, rf);
            if constexpr (STAGE1) {
              for (int w = 0; w < W; ++w)
                store8_raw(static_cast<CT*>(a.out.base[w]) + tl.flat + cc + e, rc);
            } else {
              store8_raw(static_cast<CT*>(a.out.base[0]) + tl.shard + cc + e, rc);
            }
          }
        }
      } else {
        for (int v0 = 0; v0 < nb; v0 += C) {
          const int e_end = min(nb, v0 + (warp + 1) * per);
          for (int e = v0 + warp * per + 8 * lane; e < e_end; e += 256) {
            float acc[8];
            const GT* src = base;  // the next live rank's slice; a NULL rank adds +0.0
            if (!(nulls & 1ull)) {
              load8_smem(src + e, acc);
              src += tc;
            } else {
#pragma unroll
              for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
            }
#pragma unroll(WT ? WT : 1)
            for (int w = 1; w < W; ++w) {
              float x[8];
              if (!((nulls >> w) & 1ull)) {
                load8_smem(src + e, x);
                src += tc;
              } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) x[j] = 0.0f;
              }
#pragma unroll
              for (int j = 0; j < 8; ++j) acc[j] = __fadd_rn(acc[j], x[j]);
            }
            // from here as in flat mode
            Pack8<CT> rc;
            float rf[8];
            float ss = 0.0f;
            bool fin = true;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              rc.e[j] = DT<CT>::from_f32(acc[j]);
              rf[j] = DT<CT>::to_f32(rc.e[j]);
              fin = fin && DT<CT>::finite_bits(rc.e[j]);
              ss = __fmaf_rn(rf[j], rf[j], ss);
            }
            if (!fin) bad = 1u;
            add_group(ss, hi, lo, big, rf);
            if constexpr (STAGE1) {
              for (int w = 0; w < W; ++w)
                store8_raw(static_cast<CT*>(a.out.base[w]) + tl.flat + cc + e, rc);
            } else {
              store8_raw(static_cast<CT*>(a.out.base[0]) + tl.shard + cc + e, rc);
            }
          }
        }
      }
    } else {
      const int e_end = min(nb, (warp + 1) * per);
      for (int e = warp * per + 8 * lane; e < e_end; e += 256) {
        float acc[8];
        if (grad_ptr<GT>(a, tl, 0) != nullptr) {
          load8_smem(base + e, acc);
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
        }
#pragma unroll(WT ? WT : 1)
        for (int w = 1; w < W; ++w) {
          float x[8];
          if (grad_ptr<GT>(a, tl, w) != nullptr) {
            load8_smem(base + w * C + e, x);
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) x[j] = 0.0f;
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[j] = __fadd_rn(acc[j], x[j]);
        }
        Pack8<CT> rc;
        float rf[8];
        float ss = 0.0f;
        bool fin = true;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          rc.e[j] = DT<CT>::from_f32(acc[j]);
          rf[j] = DT<CT>::to_f32(rc.e[j]);
          fin = fin && DT<CT>::finite_bits(rc.e[j]);
          ss = __fmaf_rn(rf[j], rf[j], ss);
        }
        if (!fin) bad = 1u;
        add_group(ss, hi, lo, big, rf);
        if constexpr (STAGE1) {
          for (int w = 0; w < W; ++w)
            store8_raw(static_cast<CT*>(a.out.base[w]) + tl.flat + cc + e, rc);
        } else {
          store8_raw(static_cast<CT*>(a.out.base[0]) + tl.shard + cc + e, rc);
        }
      }
    }
    if (warp == 0 && lane < clen - nb) {
      const int64_t i = (int64_t)cc + nb + lane;
      float sum = load1(grad_ptr<GT>(a, tl, 0), i);
      for (int w = 1; w < W; ++w) sum = __fadd_rn(sum, load1(grad_ptr<GT>(a, tl, w), i));
      const CT rc = DT<CT>::from_f32(sum);
      const double rf = (double)DT<CT>::to_f32(rc);
      if (!DT<CT>::finite_bits(rc)) bad = 1u;
      big += rf * rf;
      if constexpr (STAGE1) {
        for (int w = 0; w < W; ++w) static_cast<CT*>(a.out.base[w])[tl.flat + i] = rc;
      } else {
        static_cast<CT*>(a.out.base[0])[tl.shard + i] = rc;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    ++k;
    cc += tc;
    if (cc >= tl.len) {
      cc = 0;
      ct += gridDim.x;
    }
  }
  const bool last = publish_block_partial<NC>((double)hi + (double)lo + big, bad, s_part, s_flag,
                                              &s_done, a.part_sumsq, a.part_ovf,
                                              a.fuse_finalize ? &a.state_rw->blocks_done : nullptr);
  // The last block to finish (every other block has written its partial and
  // is past its reads of the state) finishes the step: the global sums and
  // finalize_state, by the warp that counted it in.
  if (last) {
    __threadfence();
    double sumsq;
    unsigned ovf;
    warp_sum_partials(a.part_sumsq, a.part_ovf, gridDim.x, sumsq, ovf);
    if (lane == 0) finalize_state(sumsq, ovf, a.world, a.hp, a.state_rw);
  }
}

// Resident blocks per SM that the default stages allow (three stages of 24 KB
// where the W ranks' gradients take at most 4 bytes per element, else of
// 32 KB): the table instance's register budget is sized for that many.
template <typename GT, int WT>
constexpr int red_min_blocks() {
  return (WT > 0 && WT * (int)sizeof(GT) <= 4) ? 3 : 2;
}

template <typename GT, typename CT, int WT, bool STAGE1, int NC>
__global__ void __launch_bounds__((NC + 1) * 32)
    k_reduce_norm_ws(const __grid_constant__ ReduceArgs a) {
  reduce_ws_body<GT, CT, WT, STAGE1, NC, false>(a);
}

// Flat buffers, W known only at run time (W not 1, 2, 4 or 8): two resident
// blocks of 32 KB stages, the registers budgeted for that (without the
// bound ptxas spilled these instances).
template <typename GT, typename CT, bool STAGE1, int NC>
__global__ void __launch_bounds__((NC + 1) * 32, 2)
    k_reduce_norm_ws_anyw(const __grid_constant__ ReduceArgs a) {
  reduce_ws_body<GT, CT, 0, STAGE1, NC, false>(a);
}

template <typename GT, typename CT, int WT, bool STAGE1, int NC>
__global__ void __launch_bounds__((NC + 1) * 32, red_min_blocks<GT, WT>())
    k_reduce_norm_ws_table(const __grid_constant__ ReduceArgs a) {
  reduce_ws_body<GT, CT, WT, STAGE1, NC, true>(a);
}

// variant 0: register-staged; 1: pipelined over flat buffers; 2: pipelined
// over a per-tensor pointer table (NULL entries allowed).
template <typename GT, typename CT, int WT, bool S1>
const void* reduce_kernel_v(int variant) {
  if (variant == 2)
    return reinterpret_cast<const void*>(&k_reduce_norm_ws_table<GT, CT, WT, S1, kRedConsumers>);
  if (variant == 1) {
    if constexpr (WT == 0)
      return reinterpret_cast<const void*>(&k_reduce_norm_ws_anyw<GT, CT, S1, kRedConsumers>);
    else
      return reinterpret_cast<const void*>(&k_reduce_norm_ws<GT, CT, WT, S1, kRedConsumers>);
  }
  return reinterpret_cast<const void*>(&k_reduce_norm<GT, CT, WT, S1>);
}

template <typename GT, typename CT, bool S1>
const void* reduce_kernel_w(int world, int variant) {
  switch (world) {
    case 1: return reduce_kernel_v<GT, CT, 1, S1>(variant);
    case 2: return reduce_kernel_v<GT, CT, 2, S1>(variant);
    case 4: return reduce_kernel_v<GT, CT, 4, S1>(variant);
    case 8: return reduce_kernel_v<GT, CT, 8, S1>(variant);
    default: return reduce_kernel_v<GT, CT, 0, S1>(variant);
  }
}

template <typename GT, typename CT>
const void* reduce_kernel_s(int world, int stage, int variant) {
  return stage == 1 ? reduce_kernel_w<GT, CT, true>(world, variant)
                    : reduce_kernel_w<GT, CT, false>(world, variant);
}

// The kernel instance for (grad dtype GT, comm dtype, world, stage, variant).
template <typename GT>
const void* reduce_kernel_for(int comm_dtype, int world, int stage, int variant) {
  switch (comm_dtype) {
    case kF32: return reduce_kernel_s<GT, float>(world, stage, variant);
    case kF16: return reduce_kernel_s<GT, __half>(world, stage, variant);
    case kBF16: return reduce_kernel_s<GT, __nv_bfloat16>(world, stage, variant);
    default: return nullptr;
  }
}

}  // namespace zg
