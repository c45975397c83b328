// Host side of the C ABI declared in include/zero.h: layout construction,
// argument validation, the library's small device block, and the launch
// sequence of one step. No compute happens here; every step of the path runs
// in the kernels (k_reduce*.cu, k_update.cu, k_copy.cu).
#include "zero.h"

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <memory>
#include <new>
#include <string>
#include <vector>

#include <cuda_runtime.h>

#include "internal.h"

#ifndef ZERO_NO_NVTX
#include <nvtx3/nvToolsExt.h>
#endif

using namespace zg;

namespace {

// NVTX ranges around every entry point and kernel launch, so a timeline tool
// (nsys --trace cuda,nvtx) shows the step's phases by name. Without a tool
// attached each range costs a few nanoseconds. Built out with -DZERO_NO_NVTX.
struct Range {
#ifndef ZERO_NO_NVTX
  explicit Range(const char* name) { nvtxRangePushA(name); }
  ~Range() { nvtxRangePop(); }
#else
  explicit Range(const char*) {}
#endif
  Range(const Range&) = delete;
  Range& operator=(const Range&) = delete;
};


thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(ZERO_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

#define ZERO_CUDA(call)                              \
  do {                                               \
    cudaError_t e_ = (call);                         \
    if (e_ != cudaSuccess) return cuda_fail(e_, #call); \
  } while (0)

int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int dtype_bytes(int d) { return d == ZERO_F32 ? 4 : 2; }
bool valid_dtype(int d) { return d == ZERO_F32 || d == ZERO_F16 || d == ZERO_BF16; }

constexpr int kMaxPartials = 8192;  // upper bound on the reduce and single-pass grids
constexpr int kMaxPerTensorGrid = 1024;  // per-tensor launches: blocks per launch at most

void* default_alloc(size_t n, void*) {
  void* p = nullptr;
  return cudaMalloc(&p, n) == cudaSuccess ? p : nullptr;
}
void default_free(void* p, void*) { cudaFree(p); }

}  // namespace

int zg::zero_internal_fail(int code, const char* msg) { return fail(code, "%s", msg); }

struct zero_layout {
  zero_config cfg{};
  int comm_dtype = 0;
  std::vector<int64_t> numel, offset;
  std::vector<int> bucket_of;
  std::vector<int64_t> bstart, blen;
  int64_t n_real = 0, np = 0;
  std::vector<Tile> tiles;
  // the same tiles grouped by parameter (per-tensor launches): parameter p's
  // tiles are tiles_pt[pt_begin[p] .. pt_begin[p+1])
  std::vector<int> bucket_tile_begin;  // bucket b's tiles: [begin[b], begin[b+1])
  std::vector<Tile> tiles_pt;
  std::vector<int> pt_begin;
  int64_t pt_partials = 0;  // sum over parameters of min(tiles, kMaxPerTensorGrid)

  zero_alloc_fn alloc = default_alloc;
  zero_free_fn free_fn = default_free;
  void* alloc_ctx = nullptr;

  // bound state (caller-owned buffers)
  bool bound = false;
  bool initialized = false;
  int device = -1;
  float* master = nullptr;
  float* m = nullptr;
  float* v = nullptr;
  // optional second state set for the speculative step (DevState::cur picks)
  float* master2 = nullptr;
  float* m2 = nullptr;
  float* v2 = nullptr;
  void* params = nullptr;
  void* scratch = nullptr;

  // library-owned device block
  void* dblock = nullptr;
  size_t dblock_bytes = 0;
  Tile* d_tiles = nullptr;
  double* d_part = nullptr;
  unsigned* d_ovf = nullptr;
  DevState* d_state = nullptr;
  const void** d_table = nullptr;  // W * n_params grad pointers (table mode)
  Tile* d_tiles_pt = nullptr;
  int64_t* d_pm_delta = nullptr;  // per parameter: parameter-major start - flat offset
  double* d_part_pt = nullptr;
  unsigned* d_ovf_pt = nullptr;
  void* d_gather = nullptr;        // replica pointer table for K4 (grown on demand)
  size_t gather_cap = 0;

  int grid_reduce = 0, grid_update = 0, grid_copy = 0;
  // the speculative step's guarded update and parameter restore: no-ops on
  // committed steps, so their grids stay small (each block still starts)
  int grid_update_guarded = 0, grid_copy_guarded = 0;
  int grid_spec = 0;  // speculative single pass (set by zero_state_bind_alternate)
  int chunk_reduce = 0;  // the pipelined reduce's elements per stage (set at bind)
  int chunk_spec = 0;  // its elements per pipeline stage
  // 1 (default): shared-memory pipelines fed by cp.async.bulk; 0: the
  // register-staged kernels, kept as the comparison baseline (environment
  // ZERO_REDUCE_VARIANT / ZERO_UPDATE_VARIANT = 0 at bind selects them)
  int reduce_variant = 1, update_variant = 1;
  // The pipelined update's tile schedule. The step's own update: 0 (default)
  // = block b takes tiles b, b + grid, ... with one block per tile; 1 =
  // a device counter hands out tiles to a grid of the resident blocks
  // (environment ZERO_UPDATE_SCHED=dynamic at bind). The speculative step's
  // guarded update always takes the counter: as a no-op (committed steps) it
  // then costs one wave of resident blocks, not one block per tile.
  int update_sched = 0;
  cudaEvent_t events[4] = {nullptr, nullptr, nullptr, nullptr};
  bool timing = false;

  // zero_step_host: host-to-device copies split over several copy streams
  static constexpr int kCopyStreams = 4;
  int n_copy_streams = kCopyStreams;
  bool copy_ready = false;
  cudaStream_t copy_stream[kCopyStreams] = {};
  cudaEvent_t copy_start = nullptr;
  cudaEvent_t copy_done[kCopyStreams] = {};
  // The device gradient buffer sets zero_step_host has copied into (keyed by
  // all W pointers), each with an event after the last reduce
  // kernel that read it: a new copy into a set waits only for that kernel, so
  // a caller alternating two sets keeps the host link busy.
  static constexpr int kHostSets = 4;
  struct HostSet {
    std::vector<const void*> key;
    cudaEvent_t k1 = nullptr;
    bool recorded = false;
    unsigned long long used = 0;
  };
  HostSet host_sets[kHostSets];
  unsigned long long host_calls = 0;
  cudaEvent_t k1_done = nullptr;  // set only while zero_step_host runs its step: recorded after K1
  bool k1_recorded = false;

  // Sharded mode (zero_dist_set_rank): this process holds rank `local_rank`'s
  // shard only; -1 = every simulated rank in this process (the default).
  int local_rank = -1;
  int sms = 0;

  // The speculative step's clip prediction, written by every finalize into a
  // mapped pinned host word (allocated by zero_state_bind_alternate). When
  // the latest written prediction says the last finalized step clipped, the
  // next speculative call launches the two-pass kernels directly instead of
  // an empty single pass and guarded kernels (the same step either way).
  // ZERO_SPEC_HINT=0 at bind_alternate leaves every decision to the device.
  int* hint_host = nullptr;
  int* hint_dev = nullptr;
  bool use_hint = true;

  int world() const { return cfg.world; }
  int n_params() const { return (int)numel.size(); }
  bool sharded() const { return local_rank >= 0; }
  // elements of the bound master/m/v (and scratch) buffers, and of params
  int64_t state_elems() const { return sharded() ? np / cfg.world : np; }
  int64_t param_elems() const { return sharded() && cfg.stage == 3 ? np / cfg.world : np; }
};

namespace {

int check_layout(const zero_layout_t* L) {
  if (L == nullptr) return fail(ZERO_ERR_INVALID, "layout is NULL");
  return ZERO_OK;
}

int check_ready(const zero_layout_t* L, bool need_init) {
  if (int rc = check_layout(L)) return rc;
  if (!L->bound) return fail(ZERO_ERR_STATE, "zero_state_bind has not been called");
  if (need_init && !L->initialized) return fail(ZERO_ERR_STATE, "zero_state_init has not been called");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev != L->device)
    return fail(ZERO_ERR_STATE, "current device %d is not the bound device %d", dev, L->device);
  return ZERO_OK;
}

// The two state sets the kernels choose from (the second defaults to the first).
void state_sets(const zero_layout* L, float* master[2], float* m[2], float* v[2]) {
  master[0] = L->master;
  m[0] = L->m;
  v[0] = L->v;
  master[1] = L->master2 ? L->master2 : L->master;
  m[1] = L->m2 ? L->m2 : L->m;
  v[1] = L->v2 ? L->v2 : L->v;
}

// The flat bucketed layout and the tile list (see zero_layout_create).
void build_layout(zero_layout* L) {
  const int W = L->cfg.world;
  const int64_t cap = L->cfg.bucket_bytes / dtype_bytes(L->cfg.grad_dtype);
  const int64_t unit = (int64_t)W * kShardUnit;
  const int P = L->n_params();
  L->offset.assign(P, 0);
  L->bucket_of.assign(P, 0);
  int64_t cursor = 0, bucket_begin = 0;
  int first_in_bucket = 0;
  auto close_bucket = [&](int64_t end) {
    L->bstart.push_back(bucket_begin);
    L->blen.push_back(align_up(end - bucket_begin, unit));
    bucket_begin += L->blen.back();
  };
  for (int p = 0; p < P; ++p) {
    int64_t at = align_up(cursor, kParamAlign);
    const bool holds_one = p > first_in_bucket;
    if (holds_one && at + L->numel[p] - bucket_begin > cap) {
      close_bucket(cursor);
      first_in_bucket = p;
      at = bucket_begin;
    }
    L->offset[p] = at;
    L->bucket_of[p] = (int)L->bstart.size();
    cursor = at + L->numel[p];
  }
  close_bucket(cursor);
  L->np = bucket_begin;

  // Tiles in flat order: bucket, then rank slice, then parameter runs.
  const int64_t shard_total = L->np / W;
  int64_t shard_prefix = 0;  // sum of len/W over the buckets before b
  int p_lo = 0;
  for (size_t b = 0; b < L->bstart.size(); ++b) {
    L->bucket_tile_begin.push_back((int)L->tiles.size());
    const int64_t slice = L->blen[b] / W;
    int p_hi = p_lo;
    while (p_hi < P && L->bucket_of[p_hi] == (int)b) ++p_hi;
    for (int r = 0; r < W; ++r) {
      const int64_t lo = L->bstart[b] + r * slice, hi = lo + slice;
      const int64_t shard_base = r * shard_total + shard_prefix;
      for (int p = p_lo; p < p_hi; ++p) {
        const int64_t a = std::max(lo, L->offset[p]);
        const int64_t e = std::min(hi, L->offset[p] + L->numel[p]);
        for (int64_t x = a; x < e; x += kTileElems) {
          Tile t{};
          t.flat = x;
          t.shard = shard_base + (x - lo);
          t.in_param = x - L->offset[p];
          t.len = (int32_t)std::min<int64_t>(kTileElems, e - x);
          t.param = p;
          t.rank = r;
          L->tiles.push_back(t);
        }
      }
    }
    shard_prefix += slice;
    p_lo = p_hi;
  }

  L->bucket_tile_begin.push_back((int)L->tiles.size());
  L->tiles_pt = L->tiles;
  std::stable_sort(L->tiles_pt.begin(), L->tiles_pt.end(),
                   [](const Tile& a, const Tile& b) { return a.param < b.param; });
  L->pt_begin.assign(P + 1, 0);
  for (const Tile& t : L->tiles_pt) L->pt_begin[t.param + 1] += 1;
  for (int p = 0; p < P; ++p) L->pt_begin[p + 1] += L->pt_begin[p];
  L->pt_partials = 0;
  for (int p = 0; p < P; ++p)
    L->pt_partials += std::min(L->pt_begin[p + 1] - L->pt_begin[p], kMaxPerTensorGrid);
}

// Sizes of the library's device block, in allocation order.
struct BlockPlan {
  size_t tiles, part, ovf, state, table, tiles_pt, part_pt, ovf_pt, pm_delta, total;
};

BlockPlan plan_block(const zero_layout* L) {
  BlockPlan b{};
  b.tiles = align_up((int64_t)L->tiles.size() * sizeof(Tile), 256);
  b.part = align_up(kMaxPartials * sizeof(double), 256);
  b.ovf = align_up(kMaxPartials * sizeof(unsigned), 256);
  b.state = align_up(sizeof(DevState), 256);
  b.table = align_up((int64_t)L->cfg.world * (int64_t)L->numel.size() * sizeof(void*), 256);
  b.tiles_pt = b.tiles;
  b.part_pt = align_up(std::max<int64_t>(1, L->pt_partials) * sizeof(double), 256);
  b.ovf_pt = align_up(std::max<int64_t>(1, L->pt_partials) * sizeof(unsigned), 256);
  b.pm_delta = align_up((int64_t)L->numel.size() * sizeof(int64_t), 256);
  b.total = b.tiles + b.part + b.ovf + b.state + b.table + b.tiles_pt + b.part_pt + b.ovf_pt +
            b.pm_delta;
  return b;
}

// The two-pass step: reduce (its last block runs the finalize, or the
// finalize kernel follows), then the update. `guarded` (the speculative
// step's fallback): each kernel runs only if the speculative finalize asked.
int launch_step(zero_layout* L, const GradSrc& src, void* const* allreduce_out,
                const zero_hparams* hp, cudaStream_t s, int guarded = 0) {
  const int W = L->world();
  const int n_tiles = (int)L->tiles.size();
  ReduceArgs ra{};
  ra.tiles = L->d_tiles;
  ra.n_tiles = n_tiles;
  ra.world = W;
  ra.stage = L->cfg.stage;
  ra.grad_dtype = L->cfg.grad_dtype;
  ra.comm_dtype = L->comm_dtype;
  ra.src = src;
  if (L->cfg.stage == 1) {
    for (int w = 0; w < W; ++w) ra.out.base[w] = allreduce_out[w];
  } else {
    ra.out.base[0] = L->scratch;
  }
  ra.part_sumsq = L->d_part;
  ra.part_ovf = L->d_ovf;
  ra.chunk = L->chunk_reduce;
  ra.error = &L->d_state->error;
  ra.state = L->d_state;
  ra.guarded = guarded;
  Hparams h{hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay, hp->max_grad_norm,
            hp->grad_divisor};
  // The pipelined reduce finishes the step in its last block when one launch
  // covers every tile; otherwise (register-staged reduce, empty model) the
  // finalize kernel follows.
  const bool fused = n_tiles > 0 && L->reduce_variant == 1;
  ra.fuse_finalize = fused ? 1 : 0;
  ra.hp = h;
  ra.state_rw = L->d_state;
  int n_part = 0;
  if (L->timing) ZERO_CUDA(cudaEventRecord(L->events[0], s));
  if (n_tiles > 0) {
    Range r(guarded ? "K1 reduce+norm (guarded)" : "K1 reduce+norm");
    cudaError_t e = launch_reduce(ra, L->grid_reduce, L->reduce_variant, s);
    if (e != cudaSuccess) return cuda_fail(e, "reduce kernel launch");
    n_part = L->grid_reduce;
  }
  if (L->k1_done != nullptr) {
    ZERO_CUDA(cudaEventRecord(L->k1_done, s));
    L->k1_recorded = true;
  }
  if (L->timing) ZERO_CUDA(cudaEventRecord(L->events[1], s));
  cudaError_t e = cudaSuccess;
  if (!fused) {
    Range r(guarded ? "K2 finalize (guarded)" : "K2 finalize");
    e = launch_finalize(L->d_part, L->d_ovf, n_part, W, h, L->d_state, guarded, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "finalize kernel launch");
  if (L->timing) ZERO_CUDA(cudaEventRecord(L->events[2], s));
  if (n_tiles > 0) {
    UpdateArgs ua{};
    ua.tiles = L->d_tiles;
    ua.n_tiles = n_tiles;
    ua.stage = L->cfg.stage;
    ua.comm_dtype = L->comm_dtype;
    ua.param_dtype = L->cfg.param_dtype;
    ua.red = ra.out;
    state_sets(L, ua.master, ua.m, ua.v);
    ua.params_flat = L->params;
    ua.state = L->d_state;
    ua.error = &L->d_state->error;
    const bool counter = L->update_variant == 1 && (guarded || L->update_sched);
    ua.tile_next = counter ? &L->d_state->tiles_next : nullptr;
    ua.restore = guarded && L->update_variant == 1 ? 1 : 0;  // the parameter restore rides along
    if (src.table_mode) {
      ua.table = src.table;
      ua.n_params = src.n_params;
      ua.world = W;
    }
    Range r("K3 unscale+clip+AdamW+cast");
    e = launch_update(ua, guarded ? L->grid_update_guarded : L->grid_update, L->update_variant, s);
    if (e != cudaSuccess) return cuda_fail(e, "update kernel launch");
  }
  if (L->timing) ZERO_CUDA(cudaEventRecord(L->events[3], s));
  return ZERO_OK;
}

// The speculative step: the single pass and its finalize; then the two-pass
// kernels guarded on DevState::need_fallback (they return at once unless
// clipping turned out active): the reduce, and the update (skipped unless the
// fallback finalize cleared DevState::skip), which instead recasts the
// parameters after an overflow (DevState::restore_params).
int launch_step_spec(zero_layout* L, const GradSrc& src, void* const* allreduce_out,
                     const zero_hparams* hp, cudaStream_t s) {
  const int n_tiles = (int)L->tiles.size();
  if (n_tiles == 0) return launch_step(L, src, allreduce_out, hp, s);
  // The latest finalize predicted clipping: the two-pass kernels, unguarded.
  // Not while the stream is being captured: a graph keeps the device-guarded
  // sequence, which decides on every replay.
  if (L->use_hint && L->hint_host != nullptr && *reinterpret_cast<volatile int*>(L->hint_host) != 0) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    ZERO_CUDA(cudaStreamIsCapturing(s, &cs));
    if (cs == cudaStreamCaptureStatusNone) {
      Range r_hint("speculative step: predicted clipping, two-pass kernels");
      return launch_step(L, src, allreduce_out, hp, s);
    }
  }
  SpecArgs sa{};
  sa.tiles = L->d_tiles;
  sa.n_tiles = n_tiles;
  sa.world = L->world();
  sa.stage = L->cfg.stage;
  sa.src = src;
  if (L->cfg.stage == 1)
    for (int w = 0; w < L->world(); ++w) sa.out.base[w] = allreduce_out[w];
  state_sets(L, sa.master, sa.m, sa.v);
  sa.params = L->params;
  sa.state = L->d_state;
  sa.hp = Hparams{hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay, hp->max_grad_norm,
                  hp->grad_divisor};
  sa.part_sumsq = L->d_part;
  sa.part_ovf = L->d_ovf;
  sa.chunk = L->chunk_spec;
  sa.fuse_finalize = 1;  // the single pass's last block runs the speculative finalize
  sa.state_rw = L->d_state;
  sa.error = &L->d_state->error;
  if (L->timing) ZERO_CUDA(cudaEventRecord(L->events[0], s));
  Range r_all("speculative step");
  cudaError_t e = launch_spec(&sa, L->cfg.grad_dtype, L->comm_dtype, L->cfg.param_dtype, L->world(),
                              L->grid_spec, s);
  if (e != cudaSuccess) return cuda_fail(e, "speculative kernel launch");
  if (L->timing) ZERO_CUDA(cudaEventRecord(L->events[1], s));
  if (L->timing) ZERO_CUDA(cudaEventRecord(L->events[2], s));
  const bool timing = L->timing;
  L->timing = false;
  Range r_fb("guarded two-pass fallback and restore");
  int rc = launch_step(L, src, allreduce_out, hp, s, /*guarded=*/1);
  L->timing = timing;
  if (rc != ZERO_OK) return rc;
  // The parameter restore after an overflow: inside the guarded update (the
  // pipelined kernel), else a guarded launch of its own.
  if (L->update_variant != 1) {
    e = launch_recast(L->d_tiles, n_tiles, sa.master, L->params, L->cfg.param_dtype,
                      L->cfg.stage == 3, L->d_state, /*guarded=*/1, L->grid_copy_guarded, s);
    if (e != cudaSuccess) return cuda_fail(e, "parameter restore launch");
  }
  if (L->timing) ZERO_CUDA(cudaEventRecord(L->events[3], s));
  return ZERO_OK;
}

// The step launched tensor by tensor (the hook-style baseline): per
// parameter, the reduce kernel over that parameter's tiles with its own slice
// of the partials; the finalize over all of them; per parameter, the update.
int launch_step_per_tensor(zero_layout* L, const GradSrc& src, void* const* allreduce_out,
                           const zero_hparams* hp, cudaStream_t s) {
  const int W = L->world();
  const int P = L->n_params();
  ReduceArgs ra{};
  ra.world = W;
  ra.stage = L->cfg.stage;
  ra.grad_dtype = L->cfg.grad_dtype;
  ra.comm_dtype = L->comm_dtype;
  ra.src = src;
  if (L->cfg.stage == 1) {
    for (int w = 0; w < W; ++w) ra.out.base[w] = allreduce_out[w];
  } else {
    ra.out.base[0] = L->scratch;
  }
  ra.chunk = L->chunk_reduce;
  ra.error = &L->d_state->error;
  ra.state = L->d_state;
  ra.guarded = 0;
  if (L->timing) ZERO_CUDA(cudaEventRecord(L->events[0], s));
  int64_t part_at = 0;
  for (int p = 0; p < P; ++p) {
    const int n = L->pt_begin[p + 1] - L->pt_begin[p];
    if (n == 0) continue;
    const int grid = std::min({n, kMaxPerTensorGrid, L->grid_reduce});
    ra.tiles = L->d_tiles_pt + L->pt_begin[p];
    ra.n_tiles = n;
    ra.part_sumsq = L->d_part_pt + part_at;
    ra.part_ovf = L->d_ovf_pt + part_at;
    cudaError_t e = launch_reduce(ra, grid, L->reduce_variant, s);
    if (e != cudaSuccess) return cuda_fail(e, "reduce kernel launch");
    part_at += grid;
  }
  if (L->timing) ZERO_CUDA(cudaEventRecord(L->events[1], s));
  Hparams h{hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay, hp->max_grad_norm,
            hp->grad_divisor};
  cudaError_t e = launch_finalize(L->d_part_pt, L->d_ovf_pt, (int)part_at, W, h, L->d_state, 0, s);
  if (e != cudaSuccess) return cuda_fail(e, "finalize kernel launch");
  if (L->timing) ZERO_CUDA(cudaEventRecord(L->events[2], s));
  UpdateArgs ua{};
  ua.stage = L->cfg.stage;
  ua.comm_dtype = L->comm_dtype;
  ua.param_dtype = L->cfg.param_dtype;
  ua.red = ra.out;
  state_sets(L, ua.master, ua.m, ua.v);
  ua.params_flat = L->params;
  ua.state = L->d_state;
  ua.error = &L->d_state->error;
  ua.tile_next = L->update_sched ? &L->d_state->tiles_next : nullptr;
  for (int p = 0; p < P; ++p) {
    const int n = L->pt_begin[p + 1] - L->pt_begin[p];
    if (n == 0) continue;
    ua.tiles = L->d_tiles_pt + L->pt_begin[p];
    ua.n_tiles = n;
    e = launch_update(ua, std::min(n, L->grid_update), L->update_variant, s);
    if (e != cudaSuccess) return cuda_fail(e, "update kernel launch");
  }
  if (L->timing) ZERO_CUDA(cudaEventRecord(L->events[3], s));
  return ZERO_OK;
}

// The per-tensor entry points copy the caller's host pointer array to the
// device on the stream, and the host-gradient entry point copies on streams
// of its own ordered by events of earlier calls. A graph would keep copies
// of host memory the caller may since have changed or freed, so a capturing
// stream is refused before anything is enqueued.
static int check_not_capturing(cudaStream_t s, const char* what) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  ZERO_CUDA(cudaStreamIsCapturing(s, &cs));
  if (cs != cudaStreamCaptureStatusNone)
    return fail(ZERO_ERR_INVALID,
                "%s copies from host memory on its own and cannot be captured into a graph; "
                "capture zero_step or zero_step_speculative over device buffers instead",
                what);
  return ZERO_OK;
}

// Entry points that step or copy every simulated rank's data in one process
// have no meaning for a layout that holds one rank's shard.
int check_not_sharded(const zero_layout* L, const char* what) {
  if (L->sharded())
    return fail(ZERO_ERR_STATE, "%s runs every rank in one process; this layout holds rank %d's "
                "shard only (zero_dist_set_rank): use the zero_dist_* calls", what, L->local_rank);
  return ZERO_OK;
}

int check_hparams(const zero_hparams* hp) {
  if (hp == nullptr) return fail(ZERO_ERR_INVALID, "hparams is NULL");
  if (!(hp->lr >= 0.0) || !(hp->beta1 >= 0.0 && hp->beta1 < 1.0) ||
      !(hp->beta2 >= 0.0 && hp->beta2 < 1.0) || !(hp->eps > 0.0) || !(hp->weight_decay >= 0.0))
    return fail(ZERO_ERR_INVALID, "hparams out of range (lr>=0, 0<=beta<1, eps>0, wd>=0)");
  if (hp->max_grad_norm != hp->max_grad_norm || hp->grad_divisor != hp->grad_divisor)
    return fail(ZERO_ERR_INVALID, "hparams contain NaN");
  return ZERO_OK;
}

int check_allreduce(const zero_layout* L, void* const* allreduce_out) {
  if (L->cfg.stage != 1) {
    if (allreduce_out != nullptr) return fail(ZERO_ERR_INVALID, "stages 2/3 take no allreduce_out");
    return ZERO_OK;
  }
  if (allreduce_out == nullptr) return fail(ZERO_ERR_INVALID, "stage 1 needs allreduce_out");
  for (int w = 0; w < L->world(); ++w) {
    if (allreduce_out[w] == nullptr || !aligned16(allreduce_out[w]))
      return fail(ZERO_ERR_INVALID, "allreduce_out[%d] is NULL or not 16-byte aligned", w);
  }
  return ZERO_OK;
}

}  // namespace

// No C++ exception crosses the C ABI: the entry points that allocate host
// memory run their bodies through this.
template <typename F>
int guarded(F&& body) {
  try {
    return body();
  } catch (const std::bad_alloc&) {
    return fail(ZERO_ERR_OOM, "host allocation failed");
  } catch (...) {
    return fail(ZERO_ERR_INVALID, "unexpected host error");
  }
}

extern "C" {

const char* zero_last_error(void) { return g_last_error.c_str(); }

int zero_set_step_events(zero_layout_t* L, void* const* events) {
  if (int rc = check_layout(L)) return rc;
  if (events == nullptr) {
    L->timing = false;
    return ZERO_OK;
  }
  for (int k = 0; k < 4; ++k) {
    if (events[k] == nullptr) return fail(ZERO_ERR_INVALID, "events[%d] is NULL", k);
  }
  for (int k = 0; k < 4; ++k) L->events[k] = static_cast<cudaEvent_t>(events[k]);
  L->timing = true;
  return ZERO_OK;
}

static int layout_create(const int64_t* const* shapes, const int* ndims, int n_params,
                         const zero_config* cfg, zero_layout_t** out) {
  if (out == nullptr || cfg == nullptr) return fail(ZERO_ERR_INVALID, "NULL argument");
  *out = nullptr;
  if (n_params <= 0) return fail(ZERO_ERR_INVALID, "n_params must be positive");
  if (shapes == nullptr || ndims == nullptr) return fail(ZERO_ERR_INVALID, "shapes/ndims NULL");
  if (cfg->world < 1 || cfg->world > ZERO_MAX_WORLD)
    return fail(ZERO_ERR_INVALID, "world %d outside 1..%d", cfg->world, ZERO_MAX_WORLD);
  if (cfg->stage < 1 || cfg->stage > 3) return fail(ZERO_ERR_INVALID, "stage must be 1, 2 or 3");
  if (cfg->bucket_bytes <= 0) return fail(ZERO_ERR_INVALID, "bucket_bytes must be positive");
  if (!valid_dtype(cfg->grad_dtype)) return fail(ZERO_ERR_INVALID, "bad grad_dtype");
  if (cfg->param_dtype != ZERO_F16 && cfg->param_dtype != ZERO_BF16)
    return fail(ZERO_ERR_INVALID, "param_dtype must be ZERO_F16 or ZERO_BF16");
  const int comm = cfg->comm_dtype < 0 ? cfg->grad_dtype : cfg->comm_dtype;
  if (!valid_dtype(comm)) return fail(ZERO_ERR_INVALID, "bad comm_dtype");
  if (cfg->bucket_bytes / dtype_bytes(cfg->grad_dtype) < 1)
    return fail(ZERO_ERR_INVALID, "bucket_bytes smaller than one gradient element");

  std::unique_ptr<zero_layout> L(new zero_layout());
  L->cfg = *cfg;
  L->comm_dtype = comm;
  L->numel.resize(n_params);
  for (int p = 0; p < n_params; ++p) {
    if (ndims[p] < 0 || ndims[p] > 8 || (ndims[p] > 0 && shapes[p] == nullptr))
      return fail(ZERO_ERR_INVALID, "parameter %d: bad ndims/shape", p);
    int64_t n = 1;
    for (int d = 0; d < ndims[p]; ++d) {
      const int64_t k = shapes[p][d];
      if (k < 0 || (k > 0 && n > ZERO_MAX_ELEMS / k))
        return fail(ZERO_ERR_INVALID, "parameter %d: negative or oversized dimension", p);
      n *= k;
    }
    if (n > ZERO_MAX_ELEMS - L->n_real)
      return fail(ZERO_ERR_INVALID, "more than %lld elements in all", (long long)ZERO_MAX_ELEMS);
    L->numel[p] = n;
    L->n_real += n;
  }
  build_layout(L.get());
  if (L->tiles.size() > (size_t)INT32_MAX) return fail(ZERO_ERR_INVALID, "model too large for the tile table");
  *out = L.release();
  return ZERO_OK;
}

int zero_layout_create(const int64_t* const* shapes, const int* ndims, int n_params,
                       const zero_config* cfg, zero_layout_t** out) {
  return guarded([&] { return layout_create(shapes, ndims, n_params, cfg, out); });
}

int zero_layout_destroy(zero_layout_t* L) {
  if (L == nullptr) return ZERO_OK;
  if (L->copy_ready) {
    for (int i = 0; i < L->n_copy_streams; ++i) {
      cudaStreamDestroy(L->copy_stream[i]);
      cudaEventDestroy(L->copy_done[i]);
    }
    cudaEventDestroy(L->copy_start);
    for (auto& hs : L->host_sets) cudaEventDestroy(hs.k1);
  }
  if (L->dblock) L->free_fn(L->dblock, L->alloc_ctx);
  if (L->d_gather) L->free_fn(L->d_gather, L->alloc_ctx);
  if (L->hint_host) cudaFreeHost(L->hint_host);
  delete L;
  return ZERO_OK;
}

int zero_layout_set_allocator(zero_layout_t* L, zero_alloc_fn alloc, zero_free_fn free_fn,
                              void* ctx) {
  if (int rc = check_layout(L)) return rc;
  if ((alloc == nullptr) != (free_fn == nullptr))
    return fail(ZERO_ERR_INVALID, "alloc and free must both be set or both be NULL");
  if (L->dblock != nullptr) return fail(ZERO_ERR_STATE, "allocator must be set before bind");
  L->alloc = alloc ? alloc : default_alloc;
  L->free_fn = free_fn ? free_fn : default_free;
  L->alloc_ctx = ctx;
  return ZERO_OK;
}

int zero_layout_query(const zero_layout_t* L, zero_layout_info* o) {
  if (int rc = check_layout(L)) return rc;
  if (o == nullptr) return fail(ZERO_ERR_INVALID, "out is NULL");
  const int W = L->world();
  const double G = dtype_bytes(L->cfg.grad_dtype), P = dtype_bytes(L->cfg.param_dtype);
  const int C = dtype_bytes(L->comm_dtype);
  std::memset(o, 0, sizeof(*o));
  o->n_params = L->n_params();
  o->n_real = L->n_real;
  o->n_padded = L->np;
  o->shard_elems = L->np / W;
  o->n_buckets = (int64_t)L->bstart.size();
  o->n_tiles = (int64_t)L->tiles.size();
  o->grad_bytes = L->np * (int64_t)G;
  o->state_bytes = L->state_elems() * 4;
  o->params_bytes = L->param_elems() * (int64_t)P;
  o->scratch_bytes = L->cfg.stage != 1 ? L->state_elems() * C : 0;
  o->allreduce_bytes = L->cfg.stage == 1 ? L->np * C : 0;
  o->device_bytes_owned = (int64_t)plan_block(L).total;
  o->ledger_bytes_per_param = L->cfg.stage == 1   ? P + G + 12.0 / W
                              : L->cfg.stage == 2 ? P + G / W + 12.0 / W
                                                  : (P + G + 12.0) / W;
  o->step_bytes_per_elem = W * G + 24.0 + P;
  o->state_blob_used = (int64_t)sizeof(DevState);
  return ZERO_OK;
}

int zero_param_offset(const zero_layout_t* L, int param, int64_t* off) {
  if (int rc = check_layout(L)) return rc;
  if (off == nullptr || param < 0 || param >= L->n_params())
    return fail(ZERO_ERR_INVALID, "param index out of range");
  *off = L->offset[param];
  return ZERO_OK;
}

int zero_bucket_range(const zero_layout_t* L, int bucket, int64_t* start, int64_t* len) {
  if (int rc = check_layout(L)) return rc;
  if (start == nullptr || len == nullptr || bucket < 0 || bucket >= (int)L->bstart.size())
    return fail(ZERO_ERR_INVALID, "bucket index out of range");
  *start = L->bstart[bucket];
  *len = L->blen[bucket];
  return ZERO_OK;
}

int zero_shard_range(const zero_layout_t* L, int bucket, int rank, int64_t* flat_begin,
                     int64_t* shard_offset, int64_t* len) {
  if (int rc = check_layout(L)) return rc;
  if (flat_begin == nullptr || shard_offset == nullptr || len == nullptr || bucket < 0 ||
      bucket >= (int)L->bstart.size() || rank < 0 || rank >= L->world())
    return fail(ZERO_ERR_INVALID, "bucket or rank out of range");
  const int W = L->world();
  int64_t prefix = 0;
  for (int b = 0; b < bucket; ++b) prefix += L->blen[b] / W;
  const int64_t slice = L->blen[bucket] / W;
  *flat_begin = L->bstart[bucket] + rank * slice;
  *shard_offset = rank * (L->np / W) + prefix;
  *len = slice;
  return ZERO_OK;
}

// Grid sizes of the streaming kernels, as multiples of the blocks that fit on
// the GPU at once. Every kernel walks its tiles grid-stride, so any grid is
// correct; launching several times the resident blocks, so that blocks
// finish and new ones start throughout the pass, moved more bytes per second
// than a grid of exactly the resident blocks (measured on GB300: the update
// 2.65 -> 2.42 ms at 32x and 2.37 ms at one block per tile, the reduce
// 0.570 -> 0.547 ms, the single pass 2.84 -> 2.60 ms on the 596M-element
// workload). The update's gain grew with the grid up to one block per tile
// (blocks start in index order, so the tiles in flight are consecutive); the
// reduce and the single pass keep one norm partial per block and stop at 4x
// and 13-26x.
// The environment variable `name`, read at bind, overrides the default
// (1..2048).
constexpr int kReduceGridMult = 4;
constexpr int kCopyGridMult = 128;
constexpr int kGuardedGridMult = 32;
// The single pass: 26x up to W = 4, 13x above (at W = 8 its consumers do
// more work per byte and 26x was 1.6 % slower than 13x; at W = 2 and 4, 26x
// was 0.6-0.9 % faster).
static int spec_grid_mult_default(int world) { return world <= 4 ? 26 : 13; }
static int grid_mult(const char* name, int dflt) {
  const char* v = std::getenv(name);
  const int m = v ? std::atoi(v) : dflt;
  return m < 1 ? 1 : (m > 2048 ? 2048 : m);
}

static int state_bind(zero_layout_t* L, void* master, void* m, void* v, void* params_flat,
                      void* scratch) {
  if (int rc = check_layout(L)) return rc;
  if (master == nullptr || m == nullptr || v == nullptr || params_flat == nullptr)
    return fail(ZERO_ERR_INVALID, "master/m/v/params_flat must not be NULL");
  if (!aligned16(master) || !aligned16(m) || !aligned16(v) || !aligned16(params_flat))
    return fail(ZERO_ERR_INVALID, "state buffers must be 16-byte aligned");
  if (L->cfg.stage != 1 && (scratch == nullptr || !aligned16(scratch)))
    return fail(ZERO_ERR_INVALID, "stages 2/3 need a 16-byte aligned scratch buffer");

  if (L->dblock == nullptr) {
    const BlockPlan b = plan_block(L);
    void* blk = L->alloc(b.total, L->alloc_ctx);
    if (blk == nullptr) return fail(ZERO_ERR_OOM, "device allocation of %zu bytes failed", b.total);
    char* c = static_cast<char*>(blk);
    L->dblock = blk;
    L->dblock_bytes = b.total;
    L->d_tiles = reinterpret_cast<Tile*>(c);
    c += b.tiles;
    L->d_part = reinterpret_cast<double*>(c);
    c += b.part;
    L->d_ovf = reinterpret_cast<unsigned*>(c);
    c += b.ovf;
    L->d_state = reinterpret_cast<DevState*>(c);
    c += b.state;
    L->d_table = reinterpret_cast<const void**>(c);
    c += b.table;
    L->d_tiles_pt = reinterpret_cast<Tile*>(c);
    c += b.tiles_pt;
    L->d_part_pt = reinterpret_cast<double*>(c);
    c += b.part_pt;
    L->d_ovf_pt = reinterpret_cast<unsigned*>(c);
    c += b.ovf_pt;
    L->d_pm_delta = reinterpret_cast<int64_t*>(c);
    {
      std::vector<int64_t> delta(L->n_params());
      int64_t pm = 0;
      for (int p = 0; p < L->n_params(); ++p) {
        delta[p] = pm - L->offset[p];
        pm += L->numel[p];
      }
      cudaError_t e = cudaMemcpy(L->d_pm_delta, delta.data(), delta.size() * sizeof(int64_t),
                                 cudaMemcpyHostToDevice);
      if (e != cudaSuccess) return cuda_fail(e, "upload of the parameter-major offsets");
    }
    if (!L->tiles.empty()) {
      cudaError_t e = cudaMemcpy(L->d_tiles, L->tiles.data(), L->tiles.size() * sizeof(Tile),
                                 cudaMemcpyHostToDevice);
      if (e == cudaSuccess)
        e = cudaMemcpy(L->d_tiles_pt, L->tiles_pt.data(), L->tiles_pt.size() * sizeof(Tile),
                       cudaMemcpyHostToDevice);
      if (e != cudaSuccess) return cuda_fail(e, "upload of the tile tables");
    }
    int dev = 0, sms = 0;
    ZERO_CUDA(cudaGetDevice(&dev));
    ZERO_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    L->device = dev;
    L->sms = sms;
    const int n_tiles = (int)L->tiles.size();
    if (const char* v = std::getenv("ZERO_REDUCE_VARIANT")) L->reduce_variant = std::atoi(v) == 0 ? 0 : 1;
    if (const char* v = std::getenv("ZERO_UPDATE_VARIANT")) L->update_variant = std::atoi(v) == 0 ? 0 : 1;
    // Launch-shape knobs of the pipelined reduce, read here like the variants:
    // ZERO_REDUCE_STAGE_BYTES (bytes per stage, 3 stages) and
    // ZERO_REDUCE_BLOCKS_PER_SM (a cap on resident blocks).
    // The default stage is 32 KB, but 24 KB where the W ranks' gradients take
    // at most 4 bytes per element (W = 2 in 2-byte dtypes): measured with the
    // grid multiple, K1 0.546 -> 0.534 ms on the 596M-element bf16 W = 2
    // workload; at W = 8 (fp16) 24 KB was 3.6 % slower.
    const int red_elem_bytes = L->world() * dtype_bytes(L->cfg.grad_dtype);
    int red_stage_bytes = red_elem_bytes <= 4 ? 24576 : kRedStageBytes, red_bps_cap = 0;
    if (const char* v = std::getenv("ZERO_REDUCE_STAGE_BYTES")) {
      const int b = std::atoi(v);
      if (b >= 4096 && b <= 73728) red_stage_bytes = b;
    }
    if (const char* v = std::getenv("ZERO_REDUCE_BLOCKS_PER_SM")) red_bps_cap = std::atoi(v);
    L->chunk_reduce = reduce_chunk(L->world(), L->cfg.grad_dtype, red_stage_bytes);
    int bps_r = reduce_blocks_per_sm(L->cfg.grad_dtype, L->comm_dtype, L->world(), L->cfg.stage,
                                     L->reduce_variant, L->chunk_reduce);
    if (red_bps_cap > 0 && bps_r > red_bps_cap) bps_r = red_bps_cap;
    const int bps_u = update_blocks_per_sm(L->comm_dtype, L->cfg.param_dtype, L->update_variant);
    if (bps_r <= 0 || bps_u <= 0)
      return fail(ZERO_ERR_CUDA, "kernel occupancy query failed (no sm_103a image for this GPU?)");
    L->grid_reduce =
        std::max(1, std::min({n_tiles, sms * bps_r * grid_mult("ZERO_REDUCE_GRID_MULT", kReduceGridMult), kMaxPartials}));
    // The update: with the device tile counter (the default), a grid of the
    // resident blocks times ZERO_UPDATE_GRID_MULT (default 1), the guarded
    // update of the speculative step included; with the static schedule
    // (ZERO_UPDATE_SCHED=static, register-staged variant too), one block per
    // tile unless ZERO_UPDATE_GRID_MULT asks for a multiple of the resident
    // blocks, and the guarded update at ZERO_GUARDED_GRID_MULT.
    if (const char* v = std::getenv("ZERO_UPDATE_SCHED")) L->update_sched = std::strcmp(v, "dynamic") == 0;
    if (L->update_variant == 0) L->update_sched = 0;
    const int gm = grid_mult("ZERO_GUARDED_GRID_MULT", kGuardedGridMult);
    const int resident_u = std::max(1, std::min(n_tiles, sms * bps_u));
    if (L->update_sched) {
      L->grid_update = std::max(1, std::min(n_tiles, sms * bps_u * grid_mult("ZERO_UPDATE_GRID_MULT", 1)));
    } else {
      L->grid_update = std::getenv("ZERO_UPDATE_GRID_MULT") == nullptr
                           ? std::max(1, n_tiles)
                           : std::max(1, std::min(n_tiles, sms * bps_u * grid_mult("ZERO_UPDATE_GRID_MULT", 1)));
    }
    // the guarded update: the counter and one wave of resident blocks (the
    // register-staged variant has no counter: ZERO_GUARDED_GRID_MULT waves)
    L->grid_update_guarded =
        L->update_variant == 1 ? resident_u : std::max(1, std::min(n_tiles, sms * bps_u * gm));
    L->grid_copy = std::max(1, std::min(n_tiles, sms * 4 * grid_mult("ZERO_COPY_GRID_MULT", kCopyGridMult)));
    // the guarded parameter restore is a no-op on every step that did not
    // overflow: one wave of resident blocks unless ZERO_GUARDED_GRID_MULT asks
    L->grid_copy_guarded = std::max(
        1, std::min(n_tiles, std::getenv("ZERO_GUARDED_GRID_MULT") ? sms * 4 * gm : sms * kMaxBlocksPerSm));
  }
  L->master = static_cast<float*>(master);
  L->m = static_cast<float*>(m);
  L->v = static_cast<float*>(v);
  L->params = params_flat;
  L->scratch = scratch;
  L->master2 = L->m2 = L->v2 = nullptr;
  L->grid_spec = 0;
  L->bound = true;
  L->initialized = false;
  return ZERO_OK;
}

int zero_state_bind(zero_layout_t* L, void* master, void* m, void* v, void* params_flat,
                    void* scratch) {
  return guarded([&] { return state_bind(L, master, m, v, params_flat, scratch); });
}

int zero_state_bind_alternate(zero_layout_t* L, void* master2, void* m2, void* v2) {
  if (int rc = check_ready(L, false)) return rc;
  if (int rc = check_not_sharded(L, "zero_state_bind_alternate")) return rc;
  if (master2 == nullptr || m2 == nullptr || v2 == nullptr)
    return fail(ZERO_ERR_INVALID, "master2/m2/v2 must not be NULL");
  if (!aligned16(master2) || !aligned16(m2) || !aligned16(v2))
    return fail(ZERO_ERR_INVALID, "alternate state buffers must be 16-byte aligned");
  const void* mine[4] = {L->master, L->m, L->v, L->params};
  for (const void* q : {master2, m2, v2})
    for (const void* o : mine)
      if (q == o) return fail(ZERO_ERR_INVALID, "alternate state buffers must differ from the bound ones");
  // Tuning knobs read at bind, like the kernel variants: ZERO_SPEC_STAGE_BYTES
  // (bytes per pipeline stage, 3 stages) and ZERO_SPEC_BLOCKS_PER_SM (a cap
  // on resident blocks, below what the occupancy allows).
  int stage_bytes = kSpecStageBytesHost, bps_cap = 0;
  if (const char* v = std::getenv("ZERO_SPEC_STAGE_BYTES")) {
    const int b = std::atoi(v);
    if (b >= 4096 && b <= 73728) stage_bytes = b;
  }
  if (const char* v = std::getenv("ZERO_SPEC_BLOCKS_PER_SM")) bps_cap = std::atoi(v);
  const int chunk = spec_chunk(L->world(), L->cfg.grad_dtype, stage_bytes);
  int bps = spec_blocks_per_sm(L->cfg.grad_dtype, L->comm_dtype, L->cfg.param_dtype, L->world(), chunk,
                               L->cfg.stage == 1);
  if (bps <= 0) return fail(ZERO_ERR_CUDA, "speculative kernel occupancy query failed");
  if (bps_cap > 0) bps = std::min(bps, bps_cap);
  L->chunk_spec = chunk;
  int sms = 0;
  ZERO_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, L->device));
  L->grid_spec = std::max(
      1, std::min({(int)L->tiles.size(), sms * bps * grid_mult("ZERO_SPEC_GRID_MULT", spec_grid_mult_default(L->world())), kMaxPartials}));
  if (L->hint_host == nullptr) {
    // Without mapped pinned memory the step still runs, every decision on
    // the device: the word is an optimisation only.
    void* h = nullptr;
    void* d = nullptr;
    if (cudaHostAlloc(&h, sizeof(int), cudaHostAllocMapped) == cudaSuccess &&
        cudaHostGetDevicePointer(&d, h, 0) == cudaSuccess) {
      L->hint_host = static_cast<int*>(h);
      *L->hint_host = 0;
      L->hint_dev = static_cast<int*>(d);
    } else {
      if (h != nullptr) cudaFreeHost(h);
      (void)cudaGetLastError();  // clear the failure: it is not the caller's
    }
  }
  if (const char* v = std::getenv("ZERO_SPEC_HINT")) L->use_hint = std::atoi(v) != 0;
  L->master2 = static_cast<float*>(master2);
  L->m2 = static_cast<float*>(m2);
  L->v2 = static_cast<float*>(v2);
  L->initialized = false;
  return ZERO_OK;
}

int zero_state_init(zero_layout_t* L, const float* master_init_flat, const zero_scaler_cfg* cfg,
                    void* stream) {
  if (int rc = check_ready(L, false)) return rc;
  if (master_init_flat == nullptr || !aligned16(master_init_flat) || cfg == nullptr)
    return fail(ZERO_ERR_INVALID, "master_init_flat (16-byte aligned) and cfg are required");
  if (!(cfg->init_scale > 0.0) || cfg->growth_interval <= 0 || !(cfg->growth_factor >= 1.0) ||
      !(cfg->backoff_factor > 0.0 && cfg->backoff_factor <= 1.0) || !(cfg->min_scale > 0.0))
    return fail(ZERO_ERR_INVALID, "scaler config out of range");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t nbytes = (size_t)L->state_elems() * 4;
  ZERO_CUDA(cudaMemsetAsync(L->master, 0, nbytes, s));
  ZERO_CUDA(cudaMemsetAsync(L->m, 0, nbytes, s));
  ZERO_CUDA(cudaMemsetAsync(L->v, 0, nbytes, s));
  ZERO_CUDA(cudaMemsetAsync(L->params, 0,
                            (size_t)L->param_elems() * dtype_bytes(L->cfg.param_dtype), s));
  ScalerCfg sc{cfg->init_scale, cfg->dynamic ? 1 : 0, cfg->growth_interval, cfg->growth_factor,
               cfg->backoff_factor, cfg->min_scale};
  cudaError_t e = launch_state_init(sc, L->d_state, L->master2 ? L->hint_dev : nullptr, s);
  if (e != cudaSuccess) return cuda_fail(e, "state init launch");
  if (!L->tiles.empty()) {
    e = launch_init_from_flat(L->d_tiles, (int)L->tiles.size(), master_init_flat, L->master,
                              L->params, L->cfg.param_dtype, L->cfg.stage == 3, L->grid_copy, s);
    if (e != cudaSuccess) return cuda_fail(e, "init kernel launch");
  }
  L->initialized = true;
  return ZERO_OK;
}

int zero_step(zero_layout_t* L, const void* const* grads, void* const* allreduce_out,
              const zero_hparams* hp, void* stream) {
  Range r_entry("zero_step");
  if (int rc = check_ready(L, true)) return rc;
  if (int rc = check_not_sharded(L, "zero_step")) return rc;
  if (int rc = check_hparams(hp)) return rc;
  if (int rc = check_allreduce(L, allreduce_out)) return rc;
  if (grads == nullptr) return fail(ZERO_ERR_INVALID, "grads is NULL");
  GradSrc src{};
  for (int w = 0; w < L->world(); ++w) {
    if (grads[w] == nullptr || !aligned16(grads[w]))
      return fail(ZERO_ERR_INVALID, "grads[%d] is NULL or not 16-byte aligned", w);
    src.base[w] = grads[w];
  }
  return launch_step(L, src, allreduce_out, hp, static_cast<cudaStream_t>(stream));
}

int zero_step_speculative_allreduce(zero_layout_t* L, const void* const* grads,
                                    void* const* allreduce_out, const zero_hparams* hp,
                                    void* stream) {
  if (int rc = check_ready(L, true)) return rc;
  if (int rc = check_not_sharded(L, "zero_step_speculative")) return rc;
  if (int rc = check_hparams(hp)) return rc;
  if (L->master2 == nullptr) return fail(ZERO_ERR_STATE, "zero_state_bind_alternate has not been called");
  if (int rc = check_allreduce(L, allreduce_out)) return rc;
  if (grads == nullptr) return fail(ZERO_ERR_INVALID, "grads is NULL");
  GradSrc src{};
  for (int w = 0; w < L->world(); ++w) {
    if (grads[w] == nullptr || !aligned16(grads[w]))
      return fail(ZERO_ERR_INVALID, "grads[%d] is NULL or not 16-byte aligned", w);
    src.base[w] = grads[w];
  }
  if (L->cfg.stage == 1) {
    // The single pass writes the outputs before the step's decision; a
    // fallback then reduces the gradients again, so they must still hold
    // every rank's own values: no output may overlap a gradient buffer.
    const uintptr_t gb = (uintptr_t)L->np * dtype_bytes(L->cfg.grad_dtype);
    const uintptr_t ob = (uintptr_t)L->np * dtype_bytes(L->comm_dtype);
    for (int w = 0; w < L->world(); ++w)
      for (int v = 0; v < L->world(); ++v) {
        const uintptr_t o = reinterpret_cast<uintptr_t>(allreduce_out[w]);
        const uintptr_t g = reinterpret_cast<uintptr_t>(grads[v]);
        if (o < g + gb && g < o + ob)
          return fail(ZERO_ERR_INVALID, "allreduce_out[%d] overlaps grads[%d]: the speculative "
                      "step reduces the gradients again when it falls back", w, v);
      }
  }
  return launch_step_spec(L, src, allreduce_out, hp, static_cast<cudaStream_t>(stream));
}

int zero_step_speculative(zero_layout_t* L, const void* const* grads, const zero_hparams* hp,
                          void* stream) {
  return zero_step_speculative_allreduce(L, grads, nullptr, hp, stream);
}

int zero_step_speculative_tensors(zero_layout_t* L, const void* const* grad_ptrs,
                                  const zero_hparams* hp, void* stream) {
  Range r_entry("zero_step_speculative_tensors");
  if (int rc = check_ready(L, true)) return rc;
  if (int rc = check_not_sharded(L, "zero_step_speculative_tensors")) return rc;
  if (int rc = check_hparams(hp)) return rc;
  if (L->master2 == nullptr) return fail(ZERO_ERR_STATE, "zero_state_bind_alternate has not been called");
  if (L->cfg.stage == 1)
    return fail(ZERO_ERR_INVALID, "stage 1 writes the all-reduce outputs: use "
                "zero_step_speculative_allreduce with flat gradients");
  if (grad_ptrs == nullptr) return fail(ZERO_ERR_INVALID, "grad_ptrs is NULL");
  const int64_t n = (int64_t)L->world() * L->n_params();
  for (int64_t i = 0; i < n; ++i) {
    if (grad_ptrs[i] != nullptr && !aligned16(grad_ptrs[i]))
      return fail(ZERO_ERR_INVALID, "grad_ptrs[%lld] is not 16-byte aligned", (long long)i);
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (int rc = check_not_capturing(s, "zero_step_speculative_tensors")) return rc;
  // The host array is staged by the runtime before this call returns.
  ZERO_CUDA(cudaMemcpyAsync(L->d_table, grad_ptrs, (size_t)n * sizeof(void*),
                            cudaMemcpyHostToDevice, s));
  GradSrc src{};
  src.table = L->d_table;
  src.n_params = L->n_params();
  src.table_mode = 1;
  return launch_step_spec(L, src, nullptr, hp, s);
}

int zero_step_per_tensor_launch(zero_layout_t* L, const void* const* grads,
                                void* const* allreduce_out, const zero_hparams* hp, void* stream) {
  Range r_entry("zero_step_per_tensor_launch");
  if (int rc = check_ready(L, true)) return rc;
  if (int rc = check_not_sharded(L, "zero_step_per_tensor_launch")) return rc;
  if (int rc = check_hparams(hp)) return rc;
  if (int rc = check_allreduce(L, allreduce_out)) return rc;
  if (grads == nullptr) return fail(ZERO_ERR_INVALID, "grads is NULL");
  GradSrc src{};
  for (int w = 0; w < L->world(); ++w) {
    if (grads[w] == nullptr || !aligned16(grads[w]))
      return fail(ZERO_ERR_INVALID, "grads[%d] is NULL or not 16-byte aligned", w);
    src.base[w] = grads[w];
  }
  return launch_step_per_tensor(L, src, allreduce_out, hp, static_cast<cudaStream_t>(stream));
}

int zero_step_tensors(zero_layout_t* L, const void* const* grad_ptrs, void* const* allreduce_out,
                      const zero_hparams* hp, void* stream) {
  Range r_entry("zero_step_tensors");
  if (int rc = check_ready(L, true)) return rc;
  if (int rc = check_not_sharded(L, "zero_step_tensors")) return rc;
  if (int rc = check_hparams(hp)) return rc;
  if (int rc = check_allreduce(L, allreduce_out)) return rc;
  if (grad_ptrs == nullptr) return fail(ZERO_ERR_INVALID, "grad_ptrs is NULL");
  const int64_t n = (int64_t)L->world() * L->n_params();
  for (int64_t i = 0; i < n; ++i) {
    if (grad_ptrs[i] != nullptr && !aligned16(grad_ptrs[i]))
      return fail(ZERO_ERR_INVALID, "grad_ptrs[%lld] is not 16-byte aligned", (long long)i);
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (int rc = check_not_capturing(s, "zero_step_tensors")) return rc;
  // The host array is staged by the runtime before this call returns.
  ZERO_CUDA(cudaMemcpyAsync(L->d_table, grad_ptrs, (size_t)n * sizeof(void*),
                            cudaMemcpyHostToDevice, s));
  GradSrc src{};
  src.table = L->d_table;
  src.n_params = L->n_params();
  src.table_mode = 1;
  return launch_step(L, src, allreduce_out, hp, s);
}

static int step_host(zero_layout_t* L, const void* const* host_grads, void* const* dev_grads,
                     void* const* allreduce_out, const zero_hparams* hp, void* stream) {
  Range r_entry("zero_step_host");
  if (int rc = check_ready(L, true)) return rc;
  if (int rc = check_not_sharded(L, "zero_step_host")) return rc;
  if (host_grads == nullptr || dev_grads == nullptr)
    return fail(ZERO_ERR_INVALID, "host_grads/dev_grads is NULL");
  const size_t bytes = (size_t)L->np * dtype_bytes(L->cfg.grad_dtype);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int w = 0; w < L->world(); ++w) {
    if (host_grads[w] == nullptr || dev_grads[w] == nullptr || !aligned16(dev_grads[w]))
      return fail(ZERO_ERR_INVALID, "host_grads[%d]/dev_grads[%d] NULL or misaligned", w, w);
  }
  if (int rc = check_hparams(hp)) return rc;
  if (int rc = check_allreduce(L, allreduce_out)) return rc;
  if (int rc = check_not_capturing(s, "zero_step_host")) return rc;
  if (!L->copy_ready) {
    if (const char* v = std::getenv("ZERO_H2D_STREAMS")) {
      const int n = std::atoi(v);
      L->n_copy_streams = n >= 1 && n <= zero_layout::kCopyStreams ? n : zero_layout::kCopyStreams;
    }
    ZERO_CUDA(cudaEventCreateWithFlags(&L->copy_start, cudaEventDisableTiming));
    for (auto& hs : L->host_sets) ZERO_CUDA(cudaEventCreateWithFlags(&hs.k1, cudaEventDisableTiming));
    for (int i = 0; i < L->n_copy_streams; ++i) {
      ZERO_CUDA(cudaStreamCreateWithFlags(&L->copy_stream[i], cudaStreamNonBlocking));
      ZERO_CUDA(cudaEventCreateWithFlags(&L->copy_done[i], cudaEventDisableTiming));
    }
    L->copy_ready = true;
  }
  // The copies start once nothing can still read this set of dev_grads:
  // after the last reduce kernel that read it (stages 2/3: the update kernel
  // never reads the gradients, so the copies overlap it, and with two sets in
  // turn they overlap the other set's reduce too), else after everything
  // already on `stream`. They run as pieces of at most 128 MB spread over the
  // copy streams, and `stream` waits for all of them before the step.
  const std::vector<const void*> key(dev_grads, dev_grads + L->world());
  zero_layout::HostSet* hs = nullptr;
  for (auto& h : L->host_sets)
    if (h.key == key) hs = &h;
  if (hs == nullptr) {  // a new set: take a free slot, else the least recently used
    hs = &L->host_sets[0];
    for (auto& h : L->host_sets)
      if (h.used < hs->used) hs = &h;
    hs->key = key;
    hs->recorded = false;
  }
  hs->used = ++L->host_calls;
  Range r_copy("host-to-device gradient copies");
  const size_t piece = size_t(128) << 20;
  const int n = L->n_copy_streams;
  cudaEvent_t after = L->copy_start;
  if (L->cfg.stage != 1 && hs->recorded) {
    after = hs->k1;
  } else {
    ZERO_CUDA(cudaEventRecord(L->copy_start, s));
  }
  for (int i = 0; i < n; ++i) ZERO_CUDA(cudaStreamWaitEvent(L->copy_stream[i], after, 0));
  int next = 0;
  for (int w = 0; w < L->world(); ++w) {
    for (size_t off = 0; off < bytes; off += piece) {
      const size_t len = std::min(piece, bytes - off);
      ZERO_CUDA(cudaMemcpyAsync(static_cast<char*>(dev_grads[w]) + off,
                                static_cast<const char*>(host_grads[w]) + off, len,
                                cudaMemcpyHostToDevice, L->copy_stream[next]));
      next = (next + 1) % n;
    }
  }
  for (int i = 0; i < n; ++i) {
    ZERO_CUDA(cudaEventRecord(L->copy_done[i], L->copy_stream[i]));
    ZERO_CUDA(cudaStreamWaitEvent(s, L->copy_done[i], 0));
  }
  L->k1_done = hs->k1;
  L->k1_recorded = false;
  const int rc = zero_step(L, dev_grads, allreduce_out, hp, stream);
  hs->recorded = L->k1_recorded;
  L->k1_done = nullptr;
  return rc;
}

int zero_step_host(zero_layout_t* L, const void* const* host_grads, void* const* dev_grads,
                   void* const* allreduce_out, const zero_hparams* hp, void* stream) {
  return guarded([&] { return step_host(L, host_grads, dev_grads, allreduce_out, hp, stream); });
}

int zero_accumulate(zero_layout_t* L, const void* const* micro, int micro_dtype, float* const* main,
                    int first, void* stream) {
  Range r_entry("zero_accumulate");
  if (int rc = check_ready(L, false)) return rc;
  if (int rc = check_not_sharded(L, "zero_accumulate")) return rc;
  if (micro == nullptr || main == nullptr) return fail(ZERO_ERR_INVALID, "micro/main is NULL");
  if (!valid_dtype(micro_dtype)) return fail(ZERO_ERR_INVALID, "bad micro_dtype");
  AccArgs a{};
  for (int w = 0; w < L->world(); ++w) {
    if (micro[w] == nullptr || main[w] == nullptr || !aligned16(micro[w]) || !aligned16(main[w]))
      return fail(ZERO_ERR_INVALID, "micro[%d]/main[%d] NULL or not 16-byte aligned", w, w);
    a.micro[w] = micro[w];
    a.main[w] = main[w];
  }
  a.world = L->world();
  a.micro_dtype = micro_dtype;
  a.first = first ? 1 : 0;
  a.tiles = L->d_tiles;
  a.n_tiles = (int)L->tiles.size();
  if (a.n_tiles == 0) return ZERO_OK;
  cudaError_t e = launch_accumulate(a, L->grid_copy, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "accumulate kernel launch");
  return ZERO_OK;
}

static_assert(sizeof(DevState) <= ZERO_STATE_BLOB_BYTES, "state blob too small");

int zero_loss_scale_state_async(zero_layout_t* L, void* blob, void* stream) {
  if (int rc = check_ready(L, true)) return rc;
  if (blob == nullptr) return fail(ZERO_ERR_INVALID, "blob is NULL");
  ZERO_CUDA(cudaMemcpyAsync(blob, L->d_state, sizeof(DevState), cudaMemcpyDeviceToHost,
                            static_cast<cudaStream_t>(stream)));
  return ZERO_OK;
}

int zero_state_blob_decode(const void* blob, zero_scaler_state* out) {
  if (blob == nullptr || out == nullptr) return fail(ZERO_ERR_INVALID, "blob/out is NULL");
  DevState h;
  std::memcpy(&h, blob, sizeof(h));
  out->scale = h.scale;
  out->counter = h.counter;
  out->t = h.t;
  out->overflow = h.overflow;
  out->skipped = h.skipped;
  out->grad_norm = h.grad_norm;
  out->clip_coef = h.clip_coef;
  out->norm_sq_raw = h.norm_sq_raw;
  out->steps = h.steps;
  out->state_set = h.cur;
  out->fast_path = h.fast_path;
  if (h.error != 0)
    return fail(ZERO_ERR_TIMEOUT, "a kernel's bounded wait gave up (device error word %u)", h.error);
  return ZERO_OK;
}

int zero_loss_scale_state(zero_layout_t* L, void* stream, zero_scaler_state* out) {
  if (int rc = check_ready(L, true)) return rc;
  if (out == nullptr) return fail(ZERO_ERR_INVALID, "out is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DevState h{};
  ZERO_CUDA(cudaMemcpyAsync(&h, L->d_state, sizeof(DevState), cudaMemcpyDeviceToHost, s));
  ZERO_CUDA(cudaStreamSynchronize(s));
  return zero_state_blob_decode(&h, out);
}

int zero_gather_params(zero_layout_t* L, void* const* dst, int n_replicas, void* stream) {
  if (int rc = check_ready(L, true)) return rc;
  if (int rc = check_not_sharded(L, "zero_gather_params")) return rc;
  if (dst == nullptr || n_replicas < 1) return fail(ZERO_ERR_INVALID, "dst NULL or n_replicas < 1");
  const int64_t n = (int64_t)n_replicas * L->n_params();
  for (int64_t i = 0; i < n; ++i) {
    if (dst[i] == nullptr && L->numel[i % L->n_params()] > 0)
      return fail(ZERO_ERR_INVALID, "dst[%lld] is NULL", (long long)i);
    if ((reinterpret_cast<uintptr_t>(dst[i]) & 1u) != 0)
      return fail(ZERO_ERR_INVALID, "dst[%lld] is not 2-byte aligned", (long long)i);
  }
  const size_t need = (size_t)n * sizeof(void*);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (need > L->gather_cap) {
    ZERO_CUDA(cudaStreamSynchronize(s));  // the old table may still be read
    if (L->d_gather) L->free_fn(L->d_gather, L->alloc_ctx);
    L->d_gather = L->alloc(need, L->alloc_ctx);
    L->gather_cap = L->d_gather ? need : 0;
    if (L->d_gather == nullptr) return fail(ZERO_ERR_OOM, "device allocation for the dst table");
  }
  ZERO_CUDA(cudaMemcpyAsync(L->d_gather, dst, need, cudaMemcpyHostToDevice, s));
  if (L->tiles.empty()) return ZERO_OK;
  Range r("K4 gather params");
  cudaError_t e = launch_gather(L->d_tiles, (int)L->tiles.size(), L->params,
                                static_cast<void* const*>(L->d_gather), L->n_params(), n_replicas,
                                dtype_bytes(L->cfg.param_dtype), L->cfg.stage == 3, L->grid_copy, s);
  if (e != cudaSuccess) return cuda_fail(e, "gather kernel launch");
  return ZERO_OK;
}

int zero_gather_bucket(zero_layout_t* L, int bucket, void* dst, void* stream) {
  Range r_entry("zero_gather_bucket");
  if (int rc = check_ready(L, true)) return rc;
  if (int rc = check_not_sharded(L, "zero_gather_bucket")) return rc;
  if (L->cfg.stage != 3)
    return fail(ZERO_ERR_STATE, "zero_gather_bucket is for stage 3 (parameters sharded)");
  if (bucket < 0 || bucket >= (int)L->bstart.size()) return fail(ZERO_ERR_INVALID, "bucket out of range");
  if (dst == nullptr || !aligned16(dst)) return fail(ZERO_ERR_INVALID, "dst NULL or not 16-byte aligned");
  const int t0 = L->bucket_tile_begin[bucket], t1 = L->bucket_tile_begin[bucket + 1];
  if (t1 == t0) return ZERO_OK;
  cudaError_t e = launch_gather_bucket(L->d_tiles + t0, t1 - t0, L->params, dst,
                                       std::min(t1 - t0, L->grid_copy), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "bucket gather launch");
  return ZERO_OK;
}

static int state_copy(zero_layout_t* L, float* a, float* b, float* c, int dir, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* flat[3] = {a, b, c};
  float* sm[2];
  float* sv1[2];
  float* sv2[2];
  state_sets(L, sm, sv1, sv2);
  float* const* shard[3] = {sm, sv1, sv2};
  for (int k = 0; k < 3; ++k) {
    if (flat[k] == nullptr) continue;
    if (!aligned16(flat[k])) return fail(ZERO_ERR_INVALID, "state buffer not 16-byte aligned");
    if (dir == 0) ZERO_CUDA(cudaMemsetAsync(flat[k], 0, (size_t)L->np * 4, s));
    if (L->tiles.empty()) continue;
    cudaError_t e = launch_state_copy(L->d_tiles, (int)L->tiles.size(), shard[k], flat[k], dir,
                                      L->d_state, L->grid_copy, s);
    if (e != cudaSuccess) return cuda_fail(e, "state copy launch");
  }
  return ZERO_OK;
}

static int state_pm_copy(zero_layout_t* L, float* a, float* b, float* c, int dir, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* pm[3] = {a, b, c};
  float* sm[2];
  float* sv1[2];
  float* sv2[2];
  state_sets(L, sm, sv1, sv2);
  float* const* shard[3] = {sm, sv1, sv2};
  for (int k = 0; k < 3; ++k) {
    if (pm[k] == nullptr) continue;
    if (!aligned16(pm[k])) return fail(ZERO_ERR_INVALID, "state buffer not 16-byte aligned");
    // a sharded layout exports its own elements only: the rest reads as zero
    if (dir == 0 && L->sharded()) ZERO_CUDA(cudaMemsetAsync(pm[k], 0, (size_t)L->n_real * 4, s));
    if (L->tiles.empty()) continue;
    cudaError_t e = launch_state_pm(L->d_tiles, (int)L->tiles.size(), L->d_pm_delta, shard[k], pm[k],
                                    dir, L->d_state, L->grid_copy, s);
    if (e != cudaSuccess) return cuda_fail(e, "state copy launch");
  }
  return ZERO_OK;
}

int zero_state_export_params(zero_layout_t* L, float* master_pm, float* m_pm, float* v_pm,
                             void* stream) {
  if (int rc = check_ready(L, true)) return rc;
  return state_pm_copy(L, master_pm, m_pm, v_pm, 0, stream);
}

int zero_state_import_params(zero_layout_t* L, const float* master_pm, const float* m_pm,
                             const float* v_pm, void* stream) {
  if (int rc = check_ready(L, true)) return rc;
  if (master_pm == nullptr) return fail(ZERO_ERR_INVALID, "master_pm is required");
  if (int rc = state_pm_copy(L, const_cast<float*>(master_pm), const_cast<float*>(m_pm),
                             const_cast<float*>(v_pm), 1, stream))
    return rc;
  if (L->tiles.empty()) return ZERO_OK;
  float* sm[2];
  float* sv1[2];
  float* sv2[2];
  state_sets(L, sm, sv1, sv2);
  cudaError_t e = launch_recast(L->d_tiles, (int)L->tiles.size(), sm, L->params,
                                L->cfg.param_dtype, L->cfg.stage == 3, L->d_state, 0, L->grid_copy,
                                static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "recast launch");
  return ZERO_OK;
}

int zero_scaler_restore(zero_layout_t* L, const zero_scaler_state* st, void* stream) {
  if (int rc = check_ready(L, true)) return rc;
  if (st == nullptr || !(st->scale > 0.0) || st->counter < 0 || st->t < 0)
    return fail(ZERO_ERR_INVALID, "scaler state NULL or out of range");
  cudaError_t e = launch_scaler_restore(L->d_state, st->scale, st->counter, st->t,
                                        static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "scaler restore launch");
  return ZERO_OK;
}

int zero_selftest_layout_timeout(zero_layout_t* L, uint32_t spin_limit, void* stream) {
  if (int rc = check_ready(L, true)) return rc;
  if (spin_limit < 1 || spin_limit > kSpinLimit)
    return fail(ZERO_ERR_INVALID, "spin_limit outside 1..2^22");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_selftest_wait(spin_limit, &L->d_state->error, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "self-test");
  // the layout's own error word decides, as for any step
  zero_scaler_state out;
  return zero_loss_scale_state(L, stream, &out);
}

int zero_state_export(zero_layout_t* L, float* master_flat, float* m_flat, float* v_flat,
                      void* stream) {
  if (int rc = check_ready(L, true)) return rc;
  return state_copy(L, master_flat, m_flat, v_flat, 0, stream);
}

int zero_state_import(zero_layout_t* L, const float* master_flat, const float* m_flat,
                      const float* v_flat, void* stream) {
  if (int rc = check_ready(L, true)) return rc;
  return state_copy(L, const_cast<float*>(master_flat), const_cast<float*>(m_flat),
                    const_cast<float*>(v_flat), 1, stream);
}

// ---------------------------------------------------------------------------
// Sharded mode: one process per GPU, this layout holds one rank's shard.
// leetllm "Deep dive: Megatron", "Distributed optimizer: trade replicated
// state for collectives": reduce-scatter of each bucket, local fp32 update of
// the rank's master slice and moments, all-gather of the parameters. The
// caller's communication library runs the collectives between these calls.
// ---------------------------------------------------------------------------

static int dist_set_rank(zero_layout_t* L, int rank) {
  if (int rc = check_layout(L)) return rc;
  if (rank < 0 || rank >= L->world())
    return fail(ZERO_ERR_INVALID, "rank %d outside 0..%d", rank, L->world() - 1);
  if (L->sharded()) return fail(ZERO_ERR_STATE, "zero_dist_set_rank was already called");
  if (L->dblock != nullptr) return fail(ZERO_ERR_STATE, "zero_dist_set_rank must come before zero_state_bind");
  if (L->comm_dtype != L->cfg.grad_dtype && L->comm_dtype != ZERO_F32)
    return fail(ZERO_ERR_INVALID, "the sharded step needs comm_dtype == grad_dtype or ZERO_F32 "
                "(the collectives reduce in the communication dtype; widening to fp32 is exact)");
  // This rank's tiles, in the same order, with shard offsets relative to the
  // start of its own slice of the rank-major buffers.
  const int64_t base = (int64_t)rank * (L->np / L->world());
  std::vector<Tile> mine;
  std::vector<int> begin;
  for (size_t b = 0; b + 1 < L->bucket_tile_begin.size(); ++b) {
    begin.push_back((int)mine.size());
    for (int t = L->bucket_tile_begin[b]; t < L->bucket_tile_begin[b + 1]; ++t) {
      Tile x = L->tiles[t];
      if (x.rank != rank) continue;
      x.shard -= base;
      mine.push_back(x);
    }
  }
  begin.push_back((int)mine.size());
  L->tiles.swap(mine);
  L->bucket_tile_begin.swap(begin);
  L->tiles_pt = L->tiles;
  std::stable_sort(L->tiles_pt.begin(), L->tiles_pt.end(),
                   [](const Tile& a, const Tile& b) { return a.param < b.param; });
  const int P = L->n_params();
  L->pt_begin.assign(P + 1, 0);
  for (const Tile& t : L->tiles_pt) L->pt_begin[t.param + 1] += 1;
  for (int p = 0; p < P; ++p) L->pt_begin[p + 1] += L->pt_begin[p];
  L->pt_partials = 0;
  for (int p = 0; p < P; ++p)
    L->pt_partials += std::min(L->pt_begin[p + 1] - L->pt_begin[p], kMaxPerTensorGrid);
  L->local_rank = rank;
  return ZERO_OK;
}

int zero_dist_set_rank(zero_layout_t* L, int rank) {
  return guarded([&] { return dist_set_rank(L, rank); });
}

static int check_dist(zero_layout_t* L, const void* allreduced) {
  if (int rc = check_ready(L, true)) return rc;
  if (!L->sharded()) return fail(ZERO_ERR_STATE, "zero_dist_set_rank has not been called");
  if (L->cfg.stage == 1) {
    if (allreduced == nullptr || !aligned16(allreduced))
      return fail(ZERO_ERR_INVALID, "stage 1 needs the all-reduced gradient (16-byte aligned)");
  } else if (allreduced != nullptr) {
    return fail(ZERO_ERR_INVALID, "stages 2/3 read the bound scratch: allreduced must be NULL");
  }
  return ZERO_OK;
}

int zero_dist_widen(zero_layout_t* L, const void* grads, float* out, void* stream) {
  Range r_entry("zero_dist_widen");
  if (int rc = check_ready(L, false)) return rc;
  if (!L->sharded()) return fail(ZERO_ERR_STATE, "zero_dist_set_rank has not been called");
  if (L->cfg.grad_dtype == ZERO_F32 || L->comm_dtype != ZERO_F32)
    return fail(ZERO_ERR_INVALID, "zero_dist_widen is for 16-bit gradients and an fp32 comm_dtype");
  if (grads == nullptr || out == nullptr || !aligned16(grads) || !aligned16(out))
    return fail(ZERO_ERR_INVALID, "grads/out NULL or not 16-byte aligned");
  if (L->np == 0) return ZERO_OK;
  const int grid = (int)std::max<int64_t>(
      1, std::min<int64_t>((L->np / 8 + kThreads - 1) / kThreads, (int64_t)L->sms * kMaxBlocksPerSm * 4));
  cudaError_t e = launch_widen(grads, L->cfg.grad_dtype, out, L->np, grid,
                               static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "widen launch");
  return ZERO_OK;
}

int zero_dist_shard_norm(zero_layout_t* L, const void* allreduced, double* norm_pair, void* stream) {
  Range r_entry("zero_dist_shard_norm");
  if (int rc = check_dist(L, allreduced)) return rc;
  if (norm_pair == nullptr || (reinterpret_cast<uintptr_t>(norm_pair) & 7u) != 0)
    return fail(ZERO_ERR_INVALID, "norm_pair is NULL or not 8-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int n_tiles = (int)L->tiles.size();
  if (n_tiles == 0) {  // this rank owns no real element
    ZERO_CUDA(cudaMemsetAsync(norm_pair, 0, 2 * sizeof(double), s));
    return ZERO_OK;
  }
  const bool s1 = L->cfg.stage == 1;
  const int grid = std::max(1, std::min({n_tiles, L->sms * kMaxBlocksPerSm * 2, kMaxPartials}));
  cudaError_t e = launch_shard_norm(L->d_tiles, n_tiles, s1 ? allreduced : L->scratch, L->comm_dtype,
                                    s1 ? 1 : 0, L->d_part, L->d_ovf, L->d_state, norm_pair, grid, s);
  if (e != cudaSuccess) return cuda_fail(e, "shard norm launch");
  return ZERO_OK;
}

int zero_dist_finalize(zero_layout_t* L, const double* norm_pair, const zero_hparams* hp,
                       void* stream) {
  Range r_entry("zero_dist_finalize");
  if (int rc = check_ready(L, true)) return rc;
  if (!L->sharded()) return fail(ZERO_ERR_STATE, "zero_dist_set_rank has not been called");
  if (int rc = check_hparams(hp)) return rc;
  if (norm_pair == nullptr || (reinterpret_cast<uintptr_t>(norm_pair) & 7u) != 0)
    return fail(ZERO_ERR_INVALID, "norm_pair is NULL or not 8-byte aligned");
  Hparams h{hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay, hp->max_grad_norm,
            hp->grad_divisor};
  cudaError_t e = launch_dist_finalize(norm_pair, L->world(), h, L->d_state,
                                       static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "finalize launch");
  return ZERO_OK;
}

int zero_dist_update_buckets(zero_layout_t* L, const void* allreduced, int first_bucket,
                             int n_buckets, void* stream) {
  Range r_entry("zero_dist_update_buckets");
  if (int rc = check_dist(L, allreduced)) return rc;
  const int nb = (int)L->bucket_tile_begin.size() - 1;
  if (first_bucket < 0 || n_buckets < 0 || first_bucket + n_buckets > nb)
    return fail(ZERO_ERR_INVALID, "buckets [%d, %d) outside the layout's %d", first_bucket,
                first_bucket + n_buckets, nb);
  const int t0 = L->bucket_tile_begin[first_bucket];
  const int n_tiles = L->bucket_tile_begin[first_bucket + n_buckets] - t0;
  if (n_tiles == 0) return ZERO_OK;  // this rank owns no real element there
  UpdateArgs ua{};
  ua.tiles = L->d_tiles + t0;
  ua.n_tiles = n_tiles;
  ua.stage = L->cfg.stage;
  ua.comm_dtype = L->comm_dtype;
  ua.param_dtype = L->cfg.param_dtype;
  if (L->cfg.stage == 1)
    ua.red.base[L->local_rank] = const_cast<void*>(allreduced);  // read at each tile's flat offset
  else
    ua.red.base[0] = L->scratch;
  state_sets(L, ua.master, ua.m, ua.v);
  ua.params_flat = L->params;
  ua.state = L->d_state;
  ua.error = &L->d_state->error;
  // the counter wraps back to 0 at the end of every launch, whatever its tiles
  ua.tile_next = L->update_sched ? &L->d_state->tiles_next : nullptr;
  Range r("K3 unscale+clip+AdamW+cast (this rank)");
  cudaError_t e = launch_update(ua, std::min(n_tiles, L->grid_update), L->update_variant,
                                static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "update kernel launch");
  return ZERO_OK;
}

int zero_dist_update(zero_layout_t* L, const void* allreduced, void* stream) {
  if (int rc = check_dist(L, allreduced)) return rc;
  return zero_dist_update_buckets(L, allreduced, 0, (int)L->bucket_tile_begin.size() - 1, stream);
}

}  // extern "C"
