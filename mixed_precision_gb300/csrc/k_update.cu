// K2 (the one-block finalize, for the paths that do not fuse it into K1), K3
// (fused unscale / clip / AdamW / cast-out), the launch dispatch of K1, and
// the speculative pass's launch.
#include <cstdlib>

#include "bulk.cuh"
#include "finalize.cuh"
#include "vec.cuh"

namespace zg {

// Launches of the step kernels: with programmatic dependent launch (the
// default; ZERO_PDL=0 in the environment turns it off) a kernel's blocks may
// be scheduled while the kernel ahead of it finishes; each kernel waits for
// that kernel's completion before touching memory (griddep_wait), so results
// are those of plain stream order.
static bool pdl_on() {
  static const bool on = [] {
    const char* v = std::getenv("ZERO_PDL");
    return v == nullptr || std::atoi(v) != 0;
  }();
  return on;
}

cudaError_t launch_step_kernel(const void* f, int grid, int threads, void** args, int smem,
                               cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (pdl_on()) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelExC(&cfg, f, args);
}

const void* reduce_kernel_f32(int comm_dtype, int world, int stage, int variant);
const void* reduce_kernel_f16(int comm_dtype, int world, int stage, int variant);
const void* reduce_kernel_bf16(int comm_dtype, int world, int stage, int variant);

static const void* reduce_kernel(int grad_dtype, int comm_dtype, int world, int stage, int variant) {
  switch (grad_dtype) {
    case kF32: return reduce_kernel_f32(comm_dtype, world, stage, variant);
    case kF16: return reduce_kernel_f16(comm_dtype, world, stage, variant);
    case kBF16: return reduce_kernel_bf16(comm_dtype, world, stage, variant);
    default: return nullptr;
  }
}

// Elements per stage of the pipelined reduce: the W ranks' slices of one chunk
// fill about kRedStageBytes; a multiple of 128 elements, at least 128.
int reduce_chunk(int world, int grad_dtype, int stage_bytes) {
  const int g = grad_dtype == kF32 ? 4 : 2;
  int c = stage_bytes / (world * g);
  c &= ~127;
  return c < 128 ? 128 : c;
}

static int reduce_threads(int variant) { return variant != 0 ? (kRedConsumers + 1) * 32 : kThreads; }

static int reduce_smem(int world, int grad_dtype, int variant, int chunk) {
  if (variant == 0) return 0;
  const int g = grad_dtype == kF32 ? 4 : 2;
  return kRedStages * world * chunk * g;
}

cudaError_t launch_reduce(const ReduceArgs& a, int grid, int variant, cudaStream_t s) {
  // the pipelined kernel has an instance of its own for per-tensor pointers
  if (variant == 1 && a.src.table_mode) variant = 2;
  const void* f = reduce_kernel(a.grad_dtype, a.comm_dtype, a.world, a.stage, variant);
  if (f == nullptr) return cudaErrorInvalidValue;
  void* args[] = {const_cast<ReduceArgs*>(&a)};
  return launch_step_kernel(f, grid, reduce_threads(variant), args,
                            reduce_smem(a.world, a.grad_dtype, variant, a.chunk), s);
}

int reduce_blocks_per_sm(int grad_dtype, int comm_dtype, int world, int stage, int variant,
                         int chunk) {
  const void* f = reduce_kernel(grad_dtype, comm_dtype, world, stage, variant);
  if (f == nullptr) return 0;
  const int smem = reduce_smem(world, grad_dtype, variant, chunk);
  if (smem > 0 && cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
                      cudaSuccess)
    return 0;
  if (variant == 1) {  // the per-tensor pointer instance launches with the same shared memory
    const void* ft = reduce_kernel(grad_dtype, comm_dtype, world, stage, 2);
    if (ft == nullptr ||
        cudaFuncSetAttribute(ft, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return 0;
  }
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, f, reduce_threads(variant), smem) !=
      cudaSuccess)
    return 0;
  return n;
}

// ---------------------------------------------------------------------------
// K2: finalize. One block: the global sums, then finalize_state (finalize.cuh,
// which cites the passages and states the reading). Used where the reduce
// kernel cannot finish the step itself (per-tensor launches, the
// register-staged reduce, an empty model); otherwise the reduce kernel's last
// block does this work. The block partials are summed in a fixed order
// (strided per thread, then a fixed shuffle tree): the same norm on every run.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kFinalizeThreads)
    k_finalize(const double* __restrict__ part_sumsq, const unsigned* __restrict__ part_ovf,
               int n_part, int world, const Hparams hp, DevState* __restrict__ st, int guarded) {
  if (st->error || (guarded && !st->need_fallback)) return;
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

  finalize_state(sumsq, any, world, hp, st);
}

cudaError_t launch_finalize(const double* part_sumsq, const unsigned* part_ovf, int n_part,
                            int world, const Hparams& hp, DevState* st, int guarded, cudaStream_t s) {
  k_finalize<<<1, kFinalizeThreads, 0, s>>>(part_sumsq, part_ovf, n_part, world, hp, st, guarded);
  return cudaGetLastError();
}

__global__ void k_state_init(const ScalerCfg cfg, DevState* st, int* hint) {
  DevState z = {};
  z.hint = hint;
  if (hint != nullptr) *reinterpret_cast<volatile int*>(hint) = 0;
  z.scale = cfg.init_scale;
  z.dynamic = cfg.dynamic;
  z.growth_interval = cfg.growth_interval;
  z.growth_factor = cfg.growth_factor;
  z.backoff_factor = cfg.backoff_factor;
  z.min_scale = cfg.min_scale;
  z.skip = 1;  // nothing to apply before the first finalize
  z.beta1_pow = z.beta2_pow = 1.0;  // beta^0
  z.beta1_pow_of = z.beta2_pow_of = __longlong_as_double(0x7FF8000000000000ll);  // NaN: use pow
  *st = z;
}

cudaError_t launch_state_init(const ScalerCfg& cfg, DevState* st, int* hint, cudaStream_t s) {
  k_state_init<<<1, 1, 0, s>>>(cfg, st, hint);
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
//   g = r * gscale;  m = b1 m + (1-b1) g;  v = b2 v + (1-b2) g^2;
//   p -= lr_wd * p + step_size * m / (sqrt(v) * inv_sqrt_bc2 + eps);  param = RNE(p).
// Element math in fp32. A skipped step returns before touching memory.
// ---------------------------------------------------------------------------
template <typename CT, typename PT>
__global__ void __launch_bounds__(kThreads) k_adamw_cast(const __grid_constant__ UpdateArgs a) {
  griddep_wait();
  griddep_trigger();
  const DevState* st = a.state;
  if (st->skip || st->error) return;
  const AdamScalars sc = AdamScalars::from(st);
  auto adam = [&](float r, float& p, float& m, float& v) { sc.apply(r, p, m, v); };
  const int cs = st->cur;
  float* const s_master = a.master[cs];
  float* const s_m = a.m[cs];
  float* const s_v = a.v[cs];

  for (int t = blockIdx.x; t < a.n_tiles; t += gridDim.x) {
    const Tile tl = a.tiles[t];
    const CT* red = a.stage == 1 ? static_cast<const CT*>(a.red.base[tl.rank]) + tl.flat
                                 : static_cast<const CT*>(a.red.base[0]) + tl.shard;
    float* mp = s_master + tl.shard;
    float* m1 = s_m + tl.shard;
    float* v1 = s_v + tl.shard;
    // stage 3 keeps the parameters sharded (rank-major, like master)
    PT* pp = static_cast<PT*>(a.params_flat) + (a.stage == 3 ? tl.shard : tl.flat);
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
struct UpdStage {
  __host__ __device__ static constexpr int bytes(int C) { return C * (12 + (int)sizeof(CT)); }
};

// ---------------------------------------------------------------------------
// K3, shared-memory pipeline (the default). The same arithmetic as
// k_adamw_cast; the four input streams of each chunk of C elements (master,
// m, v, reduced gradient: 14 bytes per element) arrive in a shared-memory
// stage by cp.async.bulk, S stages deep, completed on the stage's "full"
// mbarrier. One thread moving them in four bulk requests replaces seven
// 16-byte loads per thread, which kept the load/store queues full; a chunk's
// last (len mod 8) elements are not bulk-copied (16-byte rule) and come from
// global memory directly. One producer warp (its lane 0) issues the bulk
// copies of each chunk into the next free stage and leaves the chunk's
// offsets in a descriptor beside it; NC consumer warps each update a fixed
// slice of every chunk and release the stage by arriving on its "empty"
// mbarrier. No block-wide barrier in the loop: consumer warps never wait for
// one another, only for data. The table instance (the step from per-tensor
// pointers) checks each tile's W pointers; where all are NULL the reduced
// gradient is +0.0 (what the reduce stored), so it is not copied in.
//
// Tile scheduling. With a.tile_next (the default), the producer takes its
// next tile from a device counter (atomicInc, one tile ahead of the one it
// is copying), so a grid of the blocks the GPU holds at once works through
// the tiles in order, lowest first, and no block waits behind a long tile.
// The counter wraps at n_tiles + gridDim.x - 1: every producer stops after
// its first fetch past the end, so after the launch's last fetch the counter
// is 0 again, ready for the next launch. Without a.tile_next, block b takes
// tiles b, b + grid, ... The producer ends the work with a descriptor of
// length -1.
//
// Bounded, warp-uniform waits: a consumer warp that times out records
// kErrWaitTimeout and leaves; the producer then times out on the stage that
// warp never releases, records the error, waits (bounded) for its copies in
// flight and leaves (the counter is then not back at 0: the layout's steps
// stay frozen until zero_state_init resets the device state).
// ---------------------------------------------------------------------------
struct ChunkDesc {
  int64_t so;    // shard offset of the chunk (master, m, v)
  int64_t po;    // parameter offset (flat; stage 3: shard)
  int64_t ro;    // reduced-gradient offset (stage 1: flat; else shard)
  int32_t rb;    // reduced-gradient buffer (stage 1: the tile's rank; else 0);
                 // -1 (table instance): every rank's gradient is NULL, take +0.0
  int32_t clen;  // elements in the chunk; -1: no more work
};

template <typename CT, typename PT, int C, int S, int NC, bool TABLE>
__device__ __forceinline__ void update_ws_body(const UpdateArgs& a) {
  constexpr int kPerWarp = C / NC;
  static_assert(kPerWarp % 128 == 0, "a warp's slice must be whole 4-element groups per lane");
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t full[S];
  __shared__ __align__(8) uint64_t empty[S];
  __shared__ ChunkDesc desc[S];
  constexpr int kStage = UpdStage<CT>::bytes(C);

  griddep_wait();
  griddep_trigger();
  const DevState* st = a.state;
  if (a.restore && st->restore_params && !st->error) {
    // The speculative step overflowed: its single pass wrote the parameters,
    // the state stays as it was, so the parameters are recast from the
    // current master (every block, tiles b, b + grid, ...).
    const float* mp = a.master[st->cur];
    for (int t = blockIdx.x; t < a.n_tiles; t += gridDim.x) {
      const Tile tl = a.tiles[t];
      const float* src = mp + tl.shard;
      PT* dst = static_cast<PT*>(a.params_flat) + (a.stage == 3 ? tl.shard : tl.flat);
      const int ng = tl.len >> 3;
      for (int g = threadIdx.x; g < ng; g += blockDim.x) {
        float x[8];
        load8_f32(src + (int64_t)g * 8, x);
        Pack8<PT> q;
#pragma unroll
        for (int j = 0; j < 8; ++j) q.e[j] = DT<PT>::from_f32(x[j]);
        store8_raw(dst + (int64_t)g * 8, q);
      }
      for (int i = ng * 8 + threadIdx.x; i < tl.len; i += blockDim.x) dst[i] = DT<PT>::from_f32(src[i]);
    }
    return;
  }
  if (st->skip || st->error) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cs = st->cur;
  float* const s_master = a.master[cs];
  float* const s_m = a.m[cs];
  float* const s_v = a.v[cs];
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NC);
    }
    mbar_init_fence();
  }
  __syncthreads();

  if (warp == NC) {  // producer
    if (lane != 0) return;
    const int n_tiles = a.n_tiles;
    const unsigned wrap = (unsigned)n_tiles + gridDim.x - 1u;
    // the tile after `t` for this block (-1: none left)
    auto next_tile = [&](int t) -> int {
      if (a.tile_next != nullptr) {
        const unsigned x = atomicInc(a.tile_next, wrap);
        return x < (unsigned)n_tiles ? (int)x : -1;
      }
      const int x = t < 0 ? (int)blockIdx.x : t + (int)gridDim.x;
      return x < n_tiles ? x : -1;
    };
    int pt = next_tile(-1);
    Tile tl = a.tiles[pt >= 0 ? pt : 0];
    // The next tile is claimed one tile ahead, and its descriptor is loaded
    // after the first chunk of the current tile is issued: neither the
    // counter's round trip nor the descriptor load stalls a tile boundary.
    int pn = pt >= 0 ? next_tile(pt) : -1;
    Tile tn = tl;
    bool tn_loaded = false;
    int pc = 0;
    unsigned k = 0;
    bool ok = true;
    bool zero_tile = false;  // table mode: every rank's gradient for the tile is NULL
    while (true) {
      const int s = (int)(k % S);
      if (k >= (unsigned)S && !mbar_wait(&empty[s], ((k / S) - 1) & 1u)) {
        ok = false;
        break;
      }
      ChunkDesc& d = desc[s];
      if (pt < 0) {  // no more work: the consumers stop at this stage
        d.clen = -1;
        mbar_arrive(&full[s]);
        break;
      }
      if constexpr (TABLE) {
        if (pc == 0) {
          zero_tile = true;
          for (int w = 0; w < a.world; ++w)
            if (a.table[(int64_t)w * a.n_params + tl.param] != nullptr) zero_tile = false;
        }
      }
      const int clen = min(C, tl.len - pc);
      const int nb = clen & ~7;
      d.so = tl.shard + pc;
      d.po = (a.stage == 3 ? tl.shard : tl.flat) + pc;
      d.ro = (a.stage == 1 ? tl.flat : tl.shard) + pc;
      d.rb = a.stage == 1 ? tl.rank : 0;
      if (TABLE && zero_tile) d.rb = -1;  // the consumers take +0.0 for the gradient
      d.clen = clen;
      unsigned char* base = smem + s * kStage;
      if (nb > 0) {
        const bool grad = !(TABLE && zero_tile);
        mbar_arrive_expect_tx(&full[s], (uint32_t)nb * (12u + (grad ? (uint32_t)sizeof(CT) : 0u)));
        bulk_g2s(base, s_master + d.so, nb * 4, &full[s]);
        bulk_g2s(base + C * 4, s_m + d.so, nb * 4, &full[s]);
        bulk_g2s(base + C * 8, s_v + d.so, nb * 4, &full[s]);
        if (grad)
          bulk_g2s(base + C * 12, static_cast<const CT*>(a.red.base[d.rb]) + d.ro,
                   nb * (int)sizeof(CT), &full[s]);
      } else {
        mbar_arrive(&full[s]);
      }
      ++k;
      pc += C;
      if (!tn_loaded && pn >= 0) {
        tn = a.tiles[pn];
        tn_loaded = true;
      }
      if (pc >= tl.len) {
        pc = 0;
        pt = pn;
        if (pt >= 0) {
          tl = tn;
          tn_loaded = false;
          pn = next_tile(pt);
        }
      }
    }
    if (!ok) {
      atomicOr(a.error, kErrWaitTimeout);
      for (unsigned j = k > (unsigned)S ? k - S : 0u; j < k; ++j) mbar_wait(&full[j % S], (j / S) & 1u);
    }
    return;
  }

  const AdamScalars sc = AdamScalars::from(st);
  auto adam = [&](float r, float& p, float& m, float& v) { sc.apply(r, p, m, v); };

  unsigned k = 0;
  while (true) {
    const int s = (int)(k % S);
    if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (k / S) & 1u))) {
      if (lane == 0) atomicOr(a.error, kErrWaitTimeout);
      return;
    }
    const ChunkDesc d = desc[s];
    if (d.clen < 0) break;
    const int nb = d.clen & ~7;
    const unsigned char* base = smem + s * kStage;
    const float* sp = reinterpret_cast<const float*>(base);
    const float* sm = reinterpret_cast<const float*>(base + C * 4);
    const float* sv = reinterpret_cast<const float*>(base + C * 8);
    const CT* sr = reinterpret_cast<const CT*>(base + C * 12);
    const int64_t so = d.so;
    PT* pp = static_cast<PT*>(a.params_flat) + d.po;
    const int e_end = min(nb, (warp + 1) * kPerWarp);
#pragma unroll 2
    for (int e = warp * kPerWarp + 4 * lane; e < e_end; e += 128) {
      float4 p = *reinterpret_cast<const float4*>(sp + e);
      float4 m = *reinterpret_cast<const float4*>(sm + e);
      float4 v = *reinterpret_cast<const float4*>(sv + e);
      float r[4];
      if constexpr (TABLE) {
        if (d.rb >= 0) {
          load4_smem(sr + e, r);
        } else {
          r[0] = r[1] = r[2] = r[3] = 0.0f;
        }
      } else {
        load4_smem(sr + e, r);
      }
      adam(r[0], p.x, m.x, v.x);
      adam(r[1], p.y, m.y, v.y);
      adam(r[2], p.z, m.z, v.z);
      adam(r[3], p.w, m.w, v.w);
      __stcs(reinterpret_cast<float4*>(s_master + so + e), p);
      __stcs(reinterpret_cast<float4*>(s_m + so + e), m);
      __stcs(reinterpret_cast<float4*>(s_v + so + e), v);
      PT q[4] = {DT<PT>::from_f32(p.x), DT<PT>::from_f32(p.y), DT<PT>::from_f32(p.z),
                 DT<PT>::from_f32(p.w)};
      __stcs(reinterpret_cast<uint2*>(pp + e), *reinterpret_cast<const uint2*>(q));
    }
    if (warp == 0 && lane < d.clen - nb) {
      const int e = nb + lane;
      float p = s_master[so + e], m = s_m[so + e], v = s_v[so + e];
      float r = 0.0f;
      if (!TABLE || d.rb >= 0) r = DT<CT>::to_f32(static_cast<const CT*>(a.red.base[d.rb])[d.ro + e]);
      adam(r, p, m, v);
      s_master[so + e] = p;
      s_m[so + e] = m;
      s_v[so + e] = v;
      pp[e] = DT<PT>::from_f32(p);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    ++k;
  }
}

template <typename CT, typename PT, int C, int S, int NC>
__global__ void __launch_bounds__((NC + 1) * 32)
    k_adamw_cast_ws(const __grid_constant__ UpdateArgs a) {
  update_ws_body<CT, PT, C, S, NC, false>(a);
}

// The step from per-tensor gradient pointers (UpdateArgs::table).
template <typename CT, typename PT, int C, int S, int NC>
__global__ void __launch_bounds__((NC + 1) * 32)
    k_adamw_cast_ws_table(const __grid_constant__ UpdateArgs a) {
  update_ws_body<CT, PT, C, S, NC, true>(a);
}

constexpr int kWsChunk = 2048;
constexpr int kWsStages = 4;
constexpr int kWsConsumers = 8;

// variant 0: register-staged; 1: pipelined; 2: pipelined, per-tensor pointers
template <typename CT, typename PT>
static const void* update_kernel_cp(int variant) {
  if (variant == 2)
    return reinterpret_cast<const void*>(
        &k_adamw_cast_ws_table<CT, PT, kWsChunk, kWsStages, kWsConsumers>);
  if (variant == 1)
    return reinterpret_cast<const void*>(
        &k_adamw_cast_ws<CT, PT, kWsChunk, kWsStages, kWsConsumers>);
  return reinterpret_cast<const void*>(&k_adamw_cast<CT, PT>);
}

template <typename CT>
static const void* update_kernel_c(int param_dtype, int variant) {
  switch (param_dtype) {
    case kF16: return update_kernel_cp<CT, __half>(variant);
    case kBF16: return update_kernel_cp<CT, __nv_bfloat16>(variant);
    default: return nullptr;
  }
}

static const void* update_kernel(int comm_dtype, int param_dtype, int variant) {
  switch (comm_dtype) {
    case kF32: return update_kernel_c<float>(param_dtype, variant);
    case kF16: return update_kernel_c<__half>(param_dtype, variant);
    case kBF16: return update_kernel_c<__nv_bfloat16>(param_dtype, variant);
    default: return nullptr;
  }
}

static int update_smem(int comm_dtype, int variant) {
  const int cb = comm_dtype == kF32 ? 4 : 2;
  return variant != 0 ? kWsStages * kWsChunk * (12 + cb) : 0;
}

static int update_threads(int variant) { return variant != 0 ? (kWsConsumers + 1) * 32 : kThreads; }

cudaError_t launch_update(const UpdateArgs& a, int grid, int variant, cudaStream_t s) {
  if (variant == 1 && a.table != nullptr) variant = 2;
  const void* f = update_kernel(a.comm_dtype, a.param_dtype, variant);
  if (f == nullptr) return cudaErrorInvalidValue;
  void* args[] = {const_cast<UpdateArgs*>(&a)};
  return launch_step_kernel(f, grid, update_threads(variant), args,
                            update_smem(a.comm_dtype, variant), s);
}

int update_blocks_per_sm(int comm_dtype, int param_dtype, int variant) {
  const void* f = update_kernel(comm_dtype, param_dtype, variant);
  if (f == nullptr) return 0;
  const int smem = update_smem(comm_dtype, variant);
  if (smem > 0 && cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
                      cudaSuccess)
    return 0;
  if (variant == 1) {  // the per-tensor pointer instance launches with the same shared memory
    const void* ft = update_kernel(comm_dtype, param_dtype, 2);
    if (ft == nullptr ||
        cudaFuncSetAttribute(ft, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return 0;
  }
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, f, update_threads(variant), smem) !=
      cudaSuccess)
    return 0;
  return n;
}

}  // namespace zg

namespace zg {

// ---------------------------------------------------------------------------
// The speculative step's launch (k_spec.cuh). Its last block runs the
// speculative finalize (finalize_spec_state): commit, skip or fallback.
// ---------------------------------------------------------------------------
const void* spec_kernel_f32(int comm_dtype, int param_dtype, int world);
const void* spec_kernel_f16(int comm_dtype, int param_dtype, int world);
const void* spec_kernel_bf16(int comm_dtype, int param_dtype, int world);
const void* spec_kernel_s1_f32(int comm_dtype, int param_dtype, int world);
const void* spec_kernel_s1_f16(int comm_dtype, int param_dtype, int world);
const void* spec_kernel_s1_bf16(int comm_dtype, int param_dtype, int world);

// stage1: the instance that also writes the W all-reduce outputs
static const void* spec_kernel(int grad_dtype, int comm_dtype, int param_dtype, int world,
                               bool stage1) {
  switch (grad_dtype) {
    case kF32:
      return stage1 ? spec_kernel_s1_f32(comm_dtype, param_dtype, world)
                    : spec_kernel_f32(comm_dtype, param_dtype, world);
    case kF16:
      return stage1 ? spec_kernel_s1_f16(comm_dtype, param_dtype, world)
                    : spec_kernel_f16(comm_dtype, param_dtype, world);
    case kBF16:
      return stage1 ? spec_kernel_s1_bf16(comm_dtype, param_dtype, world)
                    : spec_kernel_bf16(comm_dtype, param_dtype, world);
    default: return nullptr;
  }
}

// Elements per stage: the W ranks' gradient slices plus 12 bytes of state per
// element fill about `stage_bytes`; a multiple of 128 elements, at least 128.
int spec_chunk(int world, int grad_dtype, int stage_bytes) {
  const int g = grad_dtype == kF32 ? 4 : 2;
  int c = stage_bytes / (world * g + 12);
  c &= ~127;
  return c < 128 ? 128 : c;
}

static int spec_smem(int world, int grad_dtype, int chunk) {
  const int g = grad_dtype == kF32 ? 4 : 2;
  return kSpecStagesHost * chunk * (world * g + 12);
}

cudaError_t launch_spec(const SpecArgs* args, int grad_dtype, int comm_dtype, int param_dtype, int world,
                        int grid, cudaStream_t s) {
  const void* f = spec_kernel(grad_dtype, comm_dtype, param_dtype, world, args->stage == 1);
  if (f == nullptr) return cudaErrorInvalidValue;
  void* a[] = {const_cast<SpecArgs*>(args)};
  return launch_step_kernel(f, grid, (kRedConsumers + 1) * 32, a,
                            spec_smem(world, grad_dtype, args->chunk), s);
}

int spec_blocks_per_sm(int grad_dtype, int comm_dtype, int param_dtype, int world, int chunk,
                       bool stage1) {
  const void* f = spec_kernel(grad_dtype, comm_dtype, param_dtype, world, stage1);
  if (f == nullptr) return 0;
  const int smem = spec_smem(world, grad_dtype, chunk);
  if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, f, (kRedConsumers + 1) * 32, smem) !=
      cudaSuccess)
    return 0;
  return n;
}

}  // namespace zg
