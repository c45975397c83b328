// Internal interface between the host side (api.cpp) and the kernels (*.cu).
// Not part of the public ABI (include/zero.h is).
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

namespace zg {

constexpr int kMaxWorld = 64;         // == ZERO_MAX_WORLD
constexpr int64_t kParamAlign = 64;   // every parameter starts on a multiple of this
constexpr int64_t kShardUnit = 128;   // buckets are padded to a multiple of W * this
constexpr int kTileElems = 8192;      // longest work unit (multiple of kParamAlign)
constexpr int kThreads = 256;         // threads per block of the streaming kernels
constexpr int kMaxBlocksPerSm = 8;    // 2048 threads / kThreads
constexpr int kFinalizeThreads = 256;
constexpr uint32_t kSpinLimit = 1u << 22;  // mbarrier try_wait retries before giving up
constexpr unsigned kErrWaitTimeout = 1u;  // DevState::error bit: a bounded wait gave up

enum Dtype : int { kF32 = 0, kF16 = 1, kBF16 = 2 };

// One work unit: a run of REAL elements (never padding) of one parameter
// inside one rank's slice of one bucket, at most kTileElems long. Its start
// is a multiple of 64 elements in both coordinate systems, so every 16-byte
// vector access inside it is aligned when the buffers are.
struct Tile {
  int64_t flat;      // offset in the flat layout (grads, params, all-reduce outputs)
  int64_t shard;     // offset in the rank-major shard buffers (master, m, v, scratch)
  int64_t in_param;  // offset inside its parameter (per-tensor pointers)
  int32_t len;       // elements, 1..kTileElems
  int32_t param;     // parameter index
  int32_t rank;      // owning rank
  int32_t reserved;
};

// Device-resident scalars: the loss-scale state machine, the last step's
// report, and the per-step values the update kernel reads.
struct DevState {
  double scale;
  long long counter;
  long long t;
  long long steps;
  long long growth_interval;
  double growth_factor, backoff_factor, min_scale;
  int dynamic;
  int overflow;
  int skipped;
  int skip;  // read by the update kernel: 1 = leave everything untouched
  double grad_norm, clip_coef, norm_sq_raw;
  // per-step values for the update kernel (fp32, derived in fp64)
  float gscale;        // clip / (S * D)
  float lr_wd;         // lr * wd (decoupled decay: p <- p - lr_wd * p)
  float step_size;     // lr / (1 - beta1^t)
  float inv_sqrt_bc2;  // 1 / sqrt(1 - beta2^t)
  float beta1, one_minus_beta1, beta2, one_minus_beta2, eps;
  unsigned error;  // bit 0: a kernel's bounded wait gave up (reported as ZERO_ERR_TIMEOUT);
                   // while set, every kernel of the step returns at once
  int cur;             // which bound state set holds the current master/m/v (0 or 1)
  int need_fallback;   // speculative step: the two-pass step must run
  int restore_params;  // speculative step overflowed: recast params from the master
  int fast_path;       // last step was committed by the speculative single pass
  int predict_fallback;  // the last finalized step clipped: the next speculative
                         // step skips its single pass and runs the two-pass kernels
  unsigned blocks_done;  // blocks of the running reduce / speculative pass that have
                         // written their partial (wraps to 0 after the last one)
  double beta1_pow, beta2_pow;        // beta1^t and beta2^t as running products ...
  double beta1_pow_of, beta2_pow_of;  // ... of these betas (NaN: not valid, use pow)
  unsigned tiles_next;  // the update kernel's tile counter (0 between launches)
  int* hint;  // device address of a mapped pinned host word, or null: every
              // finalize copies predict_fallback there, so the host can read
              // the latest prediction without synchronising
};

struct Hparams {  // mirror of zero_hparams
  double lr, beta1, beta2, eps, weight_decay, max_grad_norm, grad_divisor;
};

struct ScalerCfg {
  double init_scale;
  int dynamic;
  long long growth_interval;
  double growth_factor, backoff_factor, min_scale;
};

// Where the reduce kernel reads rank w's gradient for a tile.
struct GradSrc {
  const void* base[kMaxWorld];  // flat mode: rank w's flat buffer
  const void* const* table;     // table mode: device array [W * n_params] (entries may be null)
  int n_params;
  int table_mode;
};

// Reduced-gradient buffers: stage 2 -> base[0] is the rank-major scratch;
// stage 1 -> base[w] is rank w's flat all-reduce output.
struct RedBufs {
  void* base[kMaxWorld];
};

struct ReduceArgs {
  const Tile* tiles;
  int n_tiles;
  int world;
  int stage;
  int grad_dtype, comm_dtype;
  GradSrc src;
  RedBufs out;
  double* part_sumsq;   // [grid]
  unsigned* part_ovf;   // [grid]
  int chunk;            // shared-memory pipeline: elements per stage
  unsigned* error;      // DevState::error
  const DevState* state;
  int guarded;          // 1: run only if state->need_fallback (the speculative step's fallback)
  int fuse_finalize;    // 1: the last block to finish runs the finalize (one launch covers
                        //    every partial); 0: a separate finalize kernel follows
  Hparams hp;           // for the fused finalize
  DevState* state_rw;   // the same state, written by the fused finalize
};

struct UpdateArgs {
  const Tile* tiles;
  int n_tiles;
  int stage;
  int comm_dtype, param_dtype;
  RedBufs red;
  float* master[2];  // the two state sets; DevState::cur picks the current one
  float* m[2];
  float* v[2];
  void* params_flat;
  const DevState* state;
  unsigned* error;  // &state->error
  unsigned* tile_next;  // the pipelined kernel's tile counter (&state->tiles_next), or
                        // nullptr: block b takes tiles b, b + grid, ...
  int restore;  // 1 (the speculative step's guarded update): when the state asks
                // for the parameters back after an overflow, recast them from
                // the current master instead (pipelined kernel only)
  // The step's per-tensor gradient pointers (device array [world * n_params],
  // NULL = all-zero gradient), or nullptr for flat buffers. With a table the
  // pipelined kernel's table instance runs: a tile whose ranks are all NULL
  // has a reduced gradient of +0.0 (the reduce stored exactly that), so it
  // is not read back.
  const void* const* table;
  int n_params;
  int world;
};

// Kernel launchers. Each returns the launch's cudaError_t.
// Kernel variants: 0 = register-staged loads; 1 = shared-memory stages filled
// by cp.async.bulk from a producer warp, consumed by 8 consumer warps.
constexpr int kRedStages = 3;
constexpr int kRedStageBytes = 32768;
constexpr int kRedConsumers = 8;  // consumer warps of the warp-specialised reduce
// elements per stage of the pipelined variant (stage_bytes: kRedStageBytes by default)
int reduce_chunk(int world, int grad_dtype, int stage_bytes);
cudaError_t launch_reduce(const ReduceArgs& a, int grid, int variant, cudaStream_t s);
int reduce_blocks_per_sm(int grad_dtype, int comm_dtype, int world, int stage, int variant,
                         int chunk);
cudaError_t launch_finalize(const double* part_sumsq, const unsigned* part_ovf, int n_part,
                            int world, const Hparams& hp, DevState* st, int guarded, cudaStream_t s);
cudaError_t launch_update(const UpdateArgs& a, int grid, int variant, cudaStream_t s);
int update_blocks_per_sm(int comm_dtype, int param_dtype, int variant);
cudaError_t launch_state_init(const ScalerCfg& cfg, DevState* st, int* hint, cudaStream_t s);
cudaError_t launch_init_from_flat(const Tile* tiles, int n_tiles, const float* master_flat,
                                  float* master, void* params_flat, int param_dtype,
                                  int params_by_shard, int grid, cudaStream_t s);
// dir 0: rank-major -> flat (export); 1: flat -> rank-major (import).
// shard_buf: the two state sets' buffers; st->cur picks one.
cudaError_t launch_state_copy(const Tile* tiles, int n_tiles, float* const* shard_buf, float* flat_buf,
                              int dir, const DevState* st, int grid, cudaStream_t s);
struct AccArgs {
  const void* micro[kMaxWorld];
  float* main[kMaxWorld];
  int world;
  int micro_dtype;
  int first;
  const Tile* tiles;
  int n_tiles;
};
cudaError_t launch_accumulate(const AccArgs& a, int grid, cudaStream_t s);
// The bounded-wait self-test; err (optional): a device error word to OR the
// timeout into.
cudaError_t launch_selftest_wait(uint32_t limit, unsigned* err, cudaStream_t s);

// The speculative single-pass step (k_spec.cuh).
struct SpecArgs {  // arguments of k_spec_step
  const Tile* tiles;
  int n_tiles;
  int world;
  int stage;  // 1, 2 or 3 (3: parameters sharded)
  GradSrc src;
  RedBufs out;  // stage 1: the W all-reduce outputs (flat layout), written every step
  float* master[2];
  float* m[2];
  float* v[2];
  void* params;
  const DevState* state;
  Hparams hp;
  double* part_sumsq;
  unsigned* part_ovf;
  int chunk;
  int fuse_finalize;   // 1: the last block to finish runs the speculative finalize
  DevState* state_rw;  // the same state, written by it
  unsigned* error;
};

constexpr int kSpecStagesHost = 3;        // == kSpecStages
constexpr int kSpecStageBytesHost = 32768;  // default bytes per pipeline stage
int spec_chunk(int world, int grad_dtype, int stage_bytes);
cudaError_t launch_spec(const SpecArgs* args, int grad_dtype, int comm_dtype, int param_dtype, int world,
                        int grid, cudaStream_t s);
int spec_blocks_per_sm(int grad_dtype, int comm_dtype, int param_dtype, int world, int chunk,
                       bool stage1);

// Record a failure message for zero_last_error() and return `code` (for entry
// points defined outside api.cpp).
int zero_internal_fail(int code, const char* msg);

cudaError_t launch_state_pm(const Tile* tiles, int n_tiles, const int64_t* pm_delta,
                            float* const* shard_buf, float* pm_buf, int dir, const DevState* st,
                            int grid, cudaStream_t s);
// params <- RNE(current master); with `guarded`, only if st->restore_params.
cudaError_t launch_recast(const Tile* tiles, int n_tiles, float* const* master, void* params,
                          int param_dtype, int params_by_shard, const DevState* st, int guarded,
                          int grid, cudaStream_t s);
cudaError_t launch_gather_bucket(const Tile* tiles, int n_tiles, const void* shards, void* dst,
                                 int grid, cudaStream_t s);
cudaError_t launch_scaler_restore(DevState* st, double scale, long long counter, long long t,
                                  cudaStream_t s);
// The sharded step's local kernels (k_dist.cu): the sum of squares and
// non-finite flag of this rank's reduced values as the pair {sum, 1.0 | 0.0}
// (by_flat: read red at each tile's flat offset, else at its shard offset),
// and the finalize from that pair summed over ranks.
cudaError_t launch_shard_norm(const Tile* tiles, int n_tiles, const void* red, int comm_dtype,
                              int by_flat, double* part, unsigned* part_ovf, DevState* st,
                              double* pair, int grid, cudaStream_t s);
cudaError_t launch_dist_finalize(const double* pair, int world, const Hparams& hp, DevState* st,
                                 cudaStream_t s);
// out[i] = fp32(g[i]), i < n (16-bit gradients widened for an fp32 collective).
cudaError_t launch_widen(const void* g, int grad_dtype, float* out, int64_t n, int grid,
                         cudaStream_t s);
cudaError_t launch_gather(const Tile* tiles, int n_tiles, const void* params_flat,
                          void* const* dst_table, int n_params, int n_replicas, int elem_bytes,
                          int src_by_shard, int grid, cudaStream_t s);

}  // namespace zg
