// The speculative single-pass step.
//
// The two-pass step reads every gradient twice over (the reduce writes the
// reduced gradient, the update reads it back) because clipping and the
// overflow skip need the global norm before any update. When clipping turns
// out inactive and nothing overflows, the clip coefficient is exactly 1, so
// the update could have run in the same pass as the reduce. This pass does
// exactly that, speculatively:
//   - reduce the W ranks' gradients (same rounding as the reduce kernel),
//     accumulate the norm partials and the overflow flag;
//   - apply AdamW with clip 1 to the CURRENT state set and write the result
//     to the OTHER set (the current one stays intact), and the cast
//     parameters in place.
// The last block to finish then runs finalize_spec_state (finalize.cuh): it
// commits (flips DevState::cur), skips (overflow: the parameters are recast
// from the untouched master), or asks for the ordinary two-pass step
// (clipping active), whose kernels run guarded on that flag.
// A committed step is bit-identical to the two-pass step: same reduced
// values, same scalars (derive_adam_scalars with clip 1), same update.
// While the last finalized step clipped, the pass returns at once (the
// finalize's one-bit predictor) and costs one near-empty launch.
// Bytes per element when it commits: 2W (grads) + 24 (state) + 2 (params).
#pragma once

#include <type_traits>

#include "k_reduce.cuh"

namespace zg {

// Rank w's gradient pointer for a tile: its flat buffer, or its per-tensor
// pointer from the table, where NULL stands for an all-zero gradient (never
// read; its values count as +0, as in the reduce kernel).
template <typename GT>
__device__ __forceinline__ const GT* spec_grad_ptr(const GradSrc& src, const Tile& tl, int w) {
  if (src.table_mode) {
    const void* q = src.table[(int64_t)w * src.n_params + tl.param];
    return q ? static_cast<const GT*>(q) + tl.in_param : nullptr;
  }
  return static_cast<const GT*>(src.base[w]) + tl.flat;
}

constexpr int kSpecStages = kSpecStagesHost;

// S1: stage 1 (ZeRO-1), where the pass also writes every rank's copy of the
// reduced gradient into the W all-reduce outputs (a.out), as the two-pass
// reduce does.
template <typename GT, typename CT, typename PT, int WT, int NC, bool S1>
__device__ __forceinline__ void spec_body(const SpecArgs& a) {
  constexpr int S = kSpecStages;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t full[S];
  __shared__ __align__(8) uint64_t empty[S];
  __shared__ double s_part[NC];
  __shared__ unsigned s_flag[NC];
  __shared__ unsigned s_done;
  __shared__ AdamScalars s_sc;
  const int W = WT ? WT : a.world;
  const int C = a.chunk;
  const int kGrad = W * C * (int)sizeof(GT);
  const int kStage = kGrad + 12 * C;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  griddep_wait();
  griddep_trigger();
  const DevState* st = a.state;
  if (st->error) return;
  if (st->predict_fallback) {  // predicted to clip: the two-pass kernels run instead
    if (a.fuse_finalize && blockIdx.x == 0 && threadIdx.x == 0) spec_predicted_state(a.state_rw);
    return;
  }
  const int cs = st->cur;
  const float* src_master = a.master[cs];
  const float* src_m = a.m[cs];
  const float* src_v = a.v[cs];
  float* dst_master = a.master[cs ^ 1];
  float* dst_m = a.m[cs ^ 1];
  float* dst_v = a.v[cs ^ 1];

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NC);
    }
    s_done = 0u;
    const double D = a.hp.grad_divisor > 0.0 ? a.hp.grad_divisor : (double)a.world;
    const double inv = 1.0 / (st->scale * D);
    double b1t, b2t;  // the same powers the finalize will commit with
    bias_powers(a.hp, st, b1t, b2t);
    s_sc = derive_adam_scalars(a.hp, inv, 1.0, b1t, b2t);
    mbar_init_fence();
  }
  __syncthreads();

  if (warp == NC) {  // producer
    if (lane != 0) return;
    int pt = blockIdx.x, pc = 0;
    unsigned k = 0;
    bool ok = true;
    while (pt < a.n_tiles) {
      const int s = (int)(k % S);
      if (k >= (unsigned)S && !mbar_wait(&empty[s], ((k / S) - 1) & 1u)) {
        ok = false;
        break;
      }
      const Tile tl = a.tiles[pt];
      const int clen = min(C, tl.len - pc);
      const int nb = clen & ~7;
      unsigned char* base = smem + s * kStage;
      if (nb > 0) {
        int live = 0;  // ranks with a gradient to copy (table mode: non-NULL)
        for (int w = 0; w < W; ++w) live += spec_grad_ptr<GT>(a.src, tl, w) != nullptr;
        mbar_arrive_expect_tx(&full[s], (uint32_t)nb * (uint32_t)(live * (int)sizeof(GT) + 12));
        for (int w = 0; w < W; ++w) {
          const GT* g = spec_grad_ptr<GT>(a.src, tl, w);
          if (g != nullptr)
            bulk_g2s(base + w * C * (int)sizeof(GT), g + pc, nb * (int)sizeof(GT), &full[s]);
        }
        const int64_t so = tl.shard + pc;
        bulk_g2s(base + kGrad, src_master + so, nb * 4, &full[s]);
        bulk_g2s(base + kGrad + C * 4, src_m + so, nb * 4, &full[s]);
        bulk_g2s(base + kGrad + C * 8, src_v + so, nb * 4, &full[s]);
      } else {
        mbar_arrive(&full[s]);
      }
      ++k;
      pc += C;
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

  const AdamScalars sc = s_sc;
  const int per = ((C / NC) + 7) & ~7;
  float hi = 0.0f, lo = 0.0f;
  double big = 0.0;
  unsigned bad = 0u;
  int ct = blockIdx.x, cc = 0;
  unsigned k = 0;
  Tile tl = a.tiles[ct < a.n_tiles ? ct : 0];
  // Ranks whose gradient for the current tile is NULL (table mode only).
  auto null_mask = [&](const Tile& t) -> uint64_t {
    if (!a.src.table_mode) return 0ull;
    uint64_t mk = 0ull;
    for (int w = 0; w < W; ++w)
      if (spec_grad_ptr<GT>(a.src, t, w) == nullptr) mk |= 1ull << w;
    return mk;
  };
  uint64_t nulls = ct < a.n_tiles ? null_mask(tl) : 0ull;
  while (ct < a.n_tiles) {
    const int s = (int)(k % S);
    const int clen = min(C, tl.len - cc);
    const int nb = clen & ~7;
    if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (k / S) & 1u))) {
      if (lane == 0) atomicOr(a.error, kErrWaitTimeout);
      return;
    }
    const unsigned char* base = smem + s * kStage;
    const GT* sg = reinterpret_cast<const GT*>(base);
    const float* sp = reinterpret_cast<const float*>(base + kGrad);
    const float* sm = reinterpret_cast<const float*>(base + kGrad + C * 4);
    const float* sv = reinterpret_cast<const float*>(base + kGrad + C * 8);
    const int64_t so = tl.shard + cc;
    PT* pp = static_cast<PT*>(a.params) + (a.stage == 3 ? tl.shard : tl.flat) + cc;
    // Each lane takes two runs of 4 elements per 256-element span of its
    // warp's slice: [4 lane, 4 lane + 4) and 128 further on. Every shared
    // load (8 or 16 bytes per lane) and global store then covers contiguous
    // bytes across the warp: no bank conflicts, fully coalesced stores.
    const int w1 = min(nb, (warp + 1) * per);
    // The warp's slice of the stage. Instantiated twice: without NULL-rank
    // tests (flat buffers, or a tile every rank has a gradient for) and with
    // them, so the common case carries no per-rank branch.
    auto slice = [&](auto with_nulls) {
      constexpr bool kNulls = decltype(with_nulls)::value;
      for (int base = warp * per; base < w1; base += 256) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int e = base + 128 * h + 4 * lane;
          if (e >= w1) continue;
          float acc[4];
          if (kNulls && (nulls & 1ull)) {
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[j] = 0.0f;
          } else {
            load4_smem(sg + e, acc);
          }
#pragma unroll(WT ? WT : 1)
          for (int w = 1; w < W; ++w) {
            float x[4];
            if (kNulls && ((nulls >> w) & 1ull)) {
#pragma unroll
              for (int j = 0; j < 4; ++j) x[j] = 0.0f;
            } else {
              load4_smem(sg + w * C + e, x);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[j] = __fadd_rn(acc[j], x[j]);
          }
          float rf[4], p[4], m[4], v[4];
          float ss = 0.0f;
          bool fin = true;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const CT rc = DT<CT>::from_f32(acc[j]);
            rf[j] = DT<CT>::to_f32(rc);
            fin = fin && DT<CT>::finite_bits(rc);
            ss = __fmaf_rn(rf[j], rf[j], ss);
          }
          if (!fin) bad = 1u;
          add_group(ss, hi, lo, big, rf);
          if constexpr (S1) {  // every rank's copy of the reduced gradient
            if constexpr (sizeof(CT) == 4) {  // fp32: the reduced value is rf itself
              for (int w = 0; w < W; ++w)
                store4_f32(static_cast<float*>(a.out.base[w]) + tl.flat + cc + e, rf);
            } else {
              CT rq[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) rq[j] = DT<CT>::from_f32(rf[j]);
              for (int w = 0; w < W; ++w)
                store4_raw(static_cast<CT*>(a.out.base[w]) + tl.flat + cc + e, rq);
            }
          }
          load4_smem(sp + e, p);
          load4_smem(sm + e, m);
          load4_smem(sv + e, v);
          PT q[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            sc.apply(rf[j], p[j], m[j], v[j]);
            q[j] = DT<PT>::from_f32(p[j]);
          }
          store4_f32(dst_master + so + e, p);
          store4_f32(dst_m + so + e, m);
          store4_f32(dst_v + so + e, v);
          store4_raw(pp + e, q);
        }
      }
    };
    if (nulls == 0ull) {
      slice(std::false_type{});
    } else {
      slice(std::true_type{});
    }
    if (warp == 0 && lane < clen - nb) {  // ragged tail, from global memory
      const int e = nb + lane;
      const GT* g0 = spec_grad_ptr<GT>(a.src, tl, 0);
      float sum = g0 ? load1(g0, (int64_t)cc + e) : 0.0f;
      for (int w = 1; w < W; ++w) {
        const GT* gw = spec_grad_ptr<GT>(a.src, tl, w);
        sum = __fadd_rn(sum, gw ? load1(gw, (int64_t)cc + e) : 0.0f);
      }
      const CT rc = DT<CT>::from_f32(sum);
      const float rf = DT<CT>::to_f32(rc);
      if (!DT<CT>::finite_bits(rc)) bad = 1u;
      big += (double)rf * (double)rf;
      if constexpr (S1)
        for (int w = 0; w < W; ++w) static_cast<CT*>(a.out.base[w])[tl.flat + cc + e] = rc;
      float p = src_master[so + e], m = src_m[so + e], v = src_v[so + e];
      sc.apply(rf, p, m, v);
      dst_master[so + e] = p;
      dst_m[so + e] = m;
      dst_v[so + e] = v;
      pp[e] = DT<PT>::from_f32(p);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    ++k;
    cc += C;
    if (cc >= tl.len) {
      cc = 0;
      ct += gridDim.x;
      if (ct < a.n_tiles) {
        tl = a.tiles[ct];
        nulls = null_mask(tl);
      }
    }
  }
  const bool last = publish_block_partial<NC>((double)hi + (double)lo + big, bad, s_part, s_flag,
                                              &s_done, a.part_sumsq, a.part_ovf,
                                              a.fuse_finalize ? &a.state_rw->blocks_done : nullptr);
  // The last block to finish runs the speculative finalize (commit, skip or
  // fallback); every other block is past its reads of the state by then.
  if (last) {
    __threadfence();
    double sumsq;
    unsigned ovf;
    warp_sum_partials(a.part_sumsq, a.part_ovf, gridDim.x, sumsq, ovf);
    if (lane == 0) finalize_spec_state(sumsq, ovf, a.world, a.hp, a.state_rw);
  }
}

template <typename GT, typename CT, typename PT, int WT, int NC>
__global__ void __launch_bounds__((NC + 1) * 32) k_spec_step(const __grid_constant__ SpecArgs a) {
  spec_body<GT, CT, PT, WT, NC, false>(a);
}

// Stage 1: the all-reduce stores need registers of their own; two resident
// blocks (what the 96 KB of stages allow) get the budget for them.
template <typename GT, typename CT, typename PT, int WT, int NC>
__global__ void __launch_bounds__((NC + 1) * 32, 2) k_spec_step_s1(const __grid_constant__ SpecArgs a) {
  spec_body<GT, CT, PT, WT, NC, true>(a);
}

template <typename GT, typename CT, typename PT, int WT, bool S1>
const void* spec_kernel_one() {
  if constexpr (S1)
    return reinterpret_cast<const void*>(&k_spec_step_s1<GT, CT, PT, WT, kRedConsumers>);
  else
    return reinterpret_cast<const void*>(&k_spec_step<GT, CT, PT, WT, kRedConsumers>);
}

template <typename GT, typename CT, typename PT, bool S1>
const void* spec_kernel_w(int world) {
  switch (world) {
    case 2: return spec_kernel_one<GT, CT, PT, 2, S1>();
    case 4: return spec_kernel_one<GT, CT, PT, 4, S1>();
    case 8: return spec_kernel_one<GT, CT, PT, 8, S1>();
    default: return spec_kernel_one<GT, CT, PT, 0, S1>();
  }
}

template <typename GT, typename CT, bool S1>
const void* spec_kernel_p(int param_dtype, int world) {
  return param_dtype == kF16 ? spec_kernel_w<GT, CT, __half, S1>(world)
                             : spec_kernel_w<GT, CT, __nv_bfloat16, S1>(world);
}

// The kernel instance for (grad dtype GT, comm dtype, param dtype, world;
// S1: stage 1).
template <typename GT, bool S1>
const void* spec_kernel_for(int comm_dtype, int param_dtype, int world) {
  switch (comm_dtype) {
    case kF32: return spec_kernel_p<GT, float, S1>(param_dtype, world);
    case kF16: return spec_kernel_p<GT, __half, S1>(param_dtype, world);
    case kBF16: return spec_kernel_p<GT, __nv_bfloat16, S1>(param_dtype, world);
    default: return nullptr;
  }
}

}  // namespace zg
