/*
 * zero.h -- C ABI of the GB300 ZeRO-1/2 gradient-and-optimizer step.
 *
 * One process, one GPU. W data-parallel ranks are simulated: each rank's full
 * low-precision gradient set is a separate buffer in HBM. One step
 *   reduce-scatters those W buffers (each rank's shard of every bucket is the
 *   sum over the W ranks), checks the reduced values for inf/NaN, forms the
 *   global gradient norm and clip coefficient, advances the loss-scale state
 *   machine, applies AdamW to each rank's fp32 master/m/v shard and casts the
 *   updated parameters back into one flat low-precision buffer (the
 *   all-gather).
 *
 * Sources (page title, section):
 *   [DO]  leetllm "Deep dive: Megatron", "Distributed optimizer: trade
 *         replicated state for collectives" -- reduce-scatter, local fp32
 *         update, all-gather; equal contiguous shards; contiguous bucketed
 *         buffers; reduction scaled to the loss normalisation; byte ledger.
 *   [ND]  "nano-deepspeed (Teaching Edition)", "2. Current Feature Range" --
 *         ZeRO stages 1/2, AdamW only, FP16 dynamic loss scaling and the bf16
 *         path, stage 2 as packed all-reduce plus local scatter-back;
 *         "9. Experimental Results" -- communication_data_type, runs checked
 *         for non-finite values.
 *   [MD]  "3.7 Megatron-LM, DeepSpeed & Parallelism in Practice",
 *         "ZeRO-Offload and ZeRO-Infinity" -- fp16 loss_scale 0 (dynamic),
 *         loss_scale_window, gradient_clipping, bucket sizes;
 *         "Initializing a DeepSpeed Engine" -- backward()/step() with
 *         torch.optim.AdamW; "DeepSpeed config for this run" -- 500 MB buckets.
 *   [NM]  "nanoMegatron", "Comparison with production frameworks" and
 *         "Benchmarks" -- flat-buffer bucketed reduction versus per-parameter
 *         hooks.
 *
 * Conventions for every call:
 *   - Return value: ZERO_OK (0) or a zero_status code. No C++ exception
 *     crosses this boundary. zero_last_error() gives a message for the last
 *     failing call on the calling thread.
 *   - "device pointer": memory on the current CUDA device, owned by the
 *     caller (for instance a torch tensor's data_ptr()). The library never
 *     frees caller memory. All device pointers must be 16-byte aligned.
 *   - "stream": a cudaStream_t passed as void*; NULL is the legacy default
 *     stream. Calls that take a stream only enqueue work on it and return
 *     without waiting, unless stated otherwise.
 *   - A layout is used from one host thread and one stream at a time.
 *   - Arguments are validated on the host before anything is enqueued; an
 *     invalid call changes no state.
 *   - zero_step and zero_step_speculative enqueue kernels only (no
 *     allocation, no host synchronisation, no events unless
 *     zero_set_step_events is active), and every decision of the step is
 *     taken on the device, so both can be captured into a CUDA graph and
 *     replayed on new gradients written into the captured buffers. The
 *     hyper-parameters are captured by value. zero_step_host and the
 *     per-tensor step calls copy from host memory and are not capturable:
 *     on a capturing stream they return ZERO_ERR_INVALID and enqueue
 *     nothing.
 */
#ifndef ZERO_GB300_H
#define ZERO_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ZERO_ABI_VERSION 1
#define ZERO_MAX_WORLD 64
/* Most elements of all parameters together (2^36: more than one GPU holds). */
#define ZERO_MAX_ELEMS (((long long)1) << 36)

typedef enum {
  ZERO_OK = 0,
  ZERO_ERR_INVALID = 1, /* bad argument: null, size, alignment, dtype, stage, world */
  ZERO_ERR_CUDA = 2,    /* a CUDA runtime call failed; the message names it */
  ZERO_ERR_OOM = 3,     /* the library's own small device allocation, or a host allocation, failed */
  ZERO_ERR_TIMEOUT = 4, /* reserved: a bounded device wait gave up */
  ZERO_ERR_STATE = 5    /* call out of order (e.g. step before bind/init) */
} zero_status;

typedef enum { ZERO_F32 = 0, ZERO_F16 = 1, ZERO_BF16 = 2 } zero_dtype;

typedef struct zero_layout zero_layout_t; /* opaque, host-owned */

/* Layout configuration. [ND] stages 1/2; [MD] bucket sizes in bytes; [MD]
 * "ZeRO Stages Recap" and [NM] "What's in the box" for stage 3.
 *   world        W simulated data-parallel ranks, 1..ZERO_MAX_WORLD.
 *   stage        1: every rank receives the whole reduced gradient (all-reduce)
 *                   and updates only its optimizer shard (ZeRO-1);
 *                2: every rank receives only its reduced shard (ZeRO-2);
 *                3: as 2, and the low-precision parameters stay sharded too:
 *                   the bound params buffer is RANK-MAJOR like master/m/v,
 *                   and zero_gather_bucket all-gathers a bucket before use.
 *   bucket_bytes bucket capacity in bytes of gradient dtype (> 0).
 *   grad_dtype   dtype of the W input gradient buffers.
 *   param_dtype  dtype of the cast-out parameters (ZERO_F16 or ZERO_BF16).
 *   comm_dtype   dtype the reduced gradient is rounded to once after the fp32
 *                sum ([ND] communication_data_type); -1 = grad_dtype. */
typedef struct {
  int32_t world;
  int32_t stage;
  int64_t bucket_bytes;
  int32_t grad_dtype;
  int32_t param_dtype;
  int32_t comm_dtype;
  int32_t reserved;
} zero_config;

/* What zero_layout_query reports. Element counts unless noted. */
typedef struct {
  int64_t n_params;
  int64_t n_real;          /* N: sum of the parameters' element counts */
  int64_t n_padded;        /* Np: length of the flat layout */
  int64_t shard_elems;     /* Np / W: one rank's shard (all buckets) */
  int64_t n_buckets;
  int64_t n_tiles;         /* work units the kernels iterate over */
  int64_t grad_bytes;      /* bytes of ONE rank's flat gradient buffer (Np * size(grad)) */
  int64_t state_bytes;     /* bytes of ONE of master/m/v (Np * 4, all ranks' shards;
                              after zero_dist_set_rank: Np/W * 4, this rank's) */
  int64_t params_bytes;    /* bytes of the parameter buffer (Np * size(param); after
                              zero_dist_set_rank in stage 3: Np/W * size(param)) */
  int64_t scratch_bytes;   /* stages 2/3: reduced shards (Np * size(comm); after
                              zero_dist_set_rank: Np/W * size(comm)); stage 1: 0 */
  int64_t allreduce_bytes; /* stage 1: bytes of ONE rank's all-reduce output; stage 2: 0 */
  int64_t device_bytes_owned; /* device bytes the library allocates at bind */
  double ledger_bytes_per_param; /* [DO] per-rank persistent bytes per parameter:
                                    stage 1: P + G + 12/W; stage 2: P + G/W + 12/W;
                                    stage 3: (P + G + 12)/W
                                    (P, G = param and grad dtype sizes) */
  double step_bytes_per_elem;    /* roofline bytes per real element of one step:
                                    2W grad reads + 24 master/m/v + P param write */
  int64_t state_blob_used;       /* bytes of the state blob that
                                    zero_loss_scale_state_async copies (<= ZERO_STATE_BLOB_BYTES) */
} zero_layout_info;

/* Loss-scaler configuration. [MD] fp16 loss_scale 0 = dynamic with
 * loss_scale_window N; [ND] the bf16 path uses no loss scaling.
 *   init_scale       starting S (> 0).
 *   dynamic          1: halve on overflow, grow after growth_interval clean
 *                    steps; 0: S stays init_scale (overflow still skips).
 *   growth_interval  N (> 0).
 *   growth_factor    > 1 (2.0); backoff_factor in (0,1) (0.5); min_scale > 0 (1.0). */
typedef struct {
  double init_scale;
  int32_t dynamic;
  int32_t reserved;
  int64_t growth_interval;
  double growth_factor;
  double backoff_factor;
  double min_scale;
} zero_scaler_cfg;

/* Per-step hyper-parameters ([ND] AdamW; [MD] gradient_clipping).
 *   max_grad_norm <= 0 turns clipping off.
 *   grad_divisor  D in g = r * clip / (S * D); <= 0 means W (replica mean,
 *                 [DO] sharded-SGD example); 1 is the plain sum. Weighting by
 *                 token counts is the caller's job ([DO] failure case). */
typedef struct {
  double lr;
  double beta1;
  double beta2;
  double eps;
  double weight_decay;
  double max_grad_norm;
  double grad_divisor;
} zero_hparams;

/* Scaler state and the last step's report, read back by zero_loss_scale_state. */
typedef struct {
  double scale;        /* S for the next step */
  int64_t counter;     /* clean steps since the last overflow or growth */
  int64_t t;           /* Adam step count: applied steps only */
  int32_t overflow;    /* last step saw a non-finite reduced gradient */
  int32_t skipped;     /* last step was skipped (== overflow) */
  double grad_norm;    /* last step: norm of the unscaled, divided gradient */
  double clip_coef;    /* last step: clip coefficient (0 if skipped) */
  double norm_sq_raw;  /* last step: sum of squares of the reduced (scaled) values */
  int64_t steps;       /* zero_step calls since zero_state_init */
  int32_t state_set;   /* which bound state set holds the current master/m/v:
                          0 = the zero_state_bind buffers, 1 = the alternate set */
  int32_t fast_path;   /* last step was a committed speculative single pass */
} zero_scaler_state;

/* ------------------------------------------------------------------------ */
/* Layout ([DO] contiguous bucketed buffers, equal contiguous shards).        */
/* ------------------------------------------------------------------------ */

/* Build the flat bucketed layout of n_params parameters.
 *   shapes[p]  host array of ndims[p] dimensions (each >= 0); ndims[p] in
 *              0..8 (0 = scalar, one element).
 * Rules: parameters keep their order; each starts at a multiple of 64
 * elements; a new bucket opens when the next parameter would take the
 * bucket's span past bucket_bytes / size(grad) elements and the bucket
 * already holds a parameter (a parameter is never split); each bucket is
 * padded to a multiple of W*128 elements; rank r owns
 * [start + r*len/W, start + (r+1)*len/W) of every bucket.
 * *out receives a host object freed by zero_layout_destroy. Host only.
 * ZERO_ERR_INVALID when the parameters hold more than ZERO_MAX_ELEMS
 * elements in all; ZERO_ERR_OOM when host memory runs out (*out stays NULL
 * in both cases). */
int zero_layout_create(const int64_t* const* shapes, const int* ndims, int n_params,
                       const zero_config* cfg, zero_layout_t** out);

/* Free a layout and the device memory it allocated (synchronises the device
 * memory free). NULL is accepted. */
int zero_layout_destroy(zero_layout_t* layout);

int zero_layout_query(const zero_layout_t* layout, zero_layout_info* out);

/* Element offset of parameter `param` in the flat layout (host only). */
int zero_param_offset(const zero_layout_t* layout, int param, int64_t* elem_offset);

/* Bucket `bucket`: flat start and padded length (host only). */
int zero_bucket_range(const zero_layout_t* layout, int bucket, int64_t* start, int64_t* len);

/* Rank `rank`'s slice of bucket `bucket`: flat begin, its offset inside the
 * rank-major shard buffers (master/m/v/scratch), and its length. */
int zero_shard_range(const zero_layout_t* layout, int bucket, int rank, int64_t* flat_begin,
                     int64_t* shard_offset, int64_t* len);

/* ------------------------------------------------------------------------ */
/* State                                                                     */
/* ------------------------------------------------------------------------ */

/* Bind caller-owned device buffers and allocate the library's small device
 * block (work tables, norm partials, scalars: device_bytes_owned bytes).
 *   master, m, v  fp32, Np elements each, RANK-MAJOR: rank r's shard is
 *                 [r*Np/W, (r+1)*Np/W), holding its slice of bucket 0, then
 *                 bucket 1, ... (zero_shard_range gives each slice).
 *   params_flat   param_dtype, Np elements, flat layout (the gathered view);
 *                 stage 3: rank-major parameter shards instead.
 *   scratch       stages 2/3: comm_dtype, Np elements, rank-major (each rank's
 *                 reduce-scatter output); stage 1: ignored (may be NULL).
 * Rebinding replaces the pointers (and reuses the device block). Synchronous. */
int zero_state_bind(zero_layout_t* layout, void* master, void* m, void* v, void* params_flat,
                    void* scratch);

/* Bind a second master/m/v set (fp32, Np elements each, rank-major like the
 * first, all distinct from the bound buffers) for zero_step_speculative,
 * which writes its result into whichever set is not current and then makes
 * that set current. zero_scaler_state.state_set tells which set holds the
 * current state; every other call (steps, export/import, gathers) follows it.
 * Any stage. Call after zero_state_bind and before zero_state_init
 * (the layout counts as not initialised afterwards; init makes set 0
 * current). Rebinding with zero_state_bind drops the alternate set.
 * Synchronous (queries the kernel's occupancy). */
int zero_state_bind_alternate(zero_layout_t* layout, void* master2, void* m2, void* v2);

/* Initialise the bound state: master <- master_init_flat (device fp32, Np,
 * flat layout; padding ignored), m = v = 0, params_flat <- RNE(master) with
 * padding zero, scaler <- cfg, t = 0. Enqueued on `stream`. */
int zero_state_init(zero_layout_t* layout, const float* master_init_flat,
                    const zero_scaler_cfg* cfg, void* stream);

/* ------------------------------------------------------------------------ */
/* The step ([DO] ownership trace; [MD] backward()/step(); [ND] FP16 dynamic   */
/* loss scaling).                                                            */
/* ------------------------------------------------------------------------ */

/* One ZeRO-1/2 step over W flat-layout gradient buffers.
 *   grads          host array of W device pointers; grads[w] holds rank w's
 *                  gradients in the flat layout (Np elements of grad_dtype;
 *                  padding is never read). Read only.
 *   allreduce_out  stage 1: host array of W device pointers, Np elements of
 *                  comm_dtype each, flat layout; receives the reduced
 *                  gradient for every rank (may alias grads when
 *                  comm_dtype == grad_dtype; padding is not written).
 *                  stage 2: must be NULL.
 *   hp             host struct, copied at the call.
 * Enqueues two kernels on `stream` (three with the register-staged reduce):
 *   reduce + overflow/norm partials, whose last block to finish runs the
 *   finalize (norm, clip, scaler, t); then the fused unscale/clip/AdamW/
 *   cast-out (returns at once on a skipped step). After a kernel's bounded
 *   wait gives up (reported as ZERO_ERR_TIMEOUT by the next state read),
 *   every kernel of every step entry point returns at once: master, m, v,
 *   the parameters and the scaler stay as they were until zero_state_init
 *   initialises the state again.
 * Reduced value r = RNE_comm(g_0 + ... + g_{W-1}) (fp32 adds in rank order);
 * overflow = any non-finite r over real elements; on overflow the update is
 * skipped, S is multiplied by backoff (dynamic mode, floored at min_scale)
 * and the clean counter resets; otherwise t += 1, g = r * clip / (S * D),
 * decoupled-decay AdamW with bias correction, master/m/v stored fp32,
 * params_flat <- RNE_param(master), and S grows after N clean steps. */
int zero_step(zero_layout_t* layout, const void* const* grads, void* const* allreduce_out,
              const zero_hparams* hp, void* stream);

/* Same step, gradients given per tensor instead of flat ([NM] per-parameter
 * gradients of the hook-based prior art).
 *   grad_ptrs  host array of W * n_params device pointers, rank-major
 *              (grad_ptrs[w * n_params + p]); each points at parameter p's
 *              numel elements of grad_dtype, 16-byte aligned; NULL means an
 *              all-zero gradient (not read at all).
 * The results are those of zero_step on flat buffers holding the same
 * values, bit for bit (norm included). The pointer table is read once per
 * tile; where some ranks' pointers are NULL, the other ranks' slices of a
 * tile move in longer chunks, and a tile whose ranks are all NULL is stored
 * as zeros without being summed and is not read back by the update.
 * The table is copied to the device on `stream` before the call returns, so
 * the call cannot be captured into a CUDA graph: on a capturing stream it
 * returns ZERO_ERR_INVALID and enqueues nothing.
 * Everything else as zero_step. */
int zero_step_tensors(zero_layout_t* layout, const void* const* grad_ptrs,
                      void* const* allreduce_out, const zero_hparams* hp, void* stream);

/* The same step launched tensor by tensor: one reduce launch per parameter,
 * the finalize, then one update launch per parameter (2P + 1 launches). This
 * is the per-parameter, hook-driven form of the prior art ([NM] "Benchmarks":
 * about 2k collective calls per backward, bound by launch cost), kept as the
 * baseline the flat two-launch step is measured against. Arguments,
 * arithmetic and results are those of zero_step; only the norm's summation
 * order differs. */
int zero_step_per_tensor_launch(zero_layout_t* layout, const void* const* grads,
                                void* const* allreduce_out, const zero_hparams* hp, void* stream);

/* The same step in one pass over memory when it can be: the reduce, the norm
 * partials and the AdamW update with clip coefficient 1 run in one kernel,
 * which reads the current state set and writes the other one (and the
 * parameters) without knowing the global norm yet. Its last block to finish
 * runs the finalize, which then
 *   - commits (no overflow, clip coefficient exactly 1): the other set
 *     becomes current; results are bit-identical to zero_step;
 *   - skips (overflow, [ND] FP16 dynamic loss scaling): state unchanged, the
 *     parameters are recast from the current master (so they are unchanged
 *     too), scale backs off;
 *   - falls back (clipping active, [MD] gradient_clipping): the ordinary
 *     reduce / finalize / update kernels run, results those of zero_step.
 * The decision is taken on the device; every branch's kernels are enqueued
 * and those not taken return at once, so the call never synchronises.
 * While the last finalized step clipped, the single pass is predicted to
 * fall back. Every finalize writes that prediction into a mapped pinned host
 * word (allocated by zero_state_bind_alternate); when the latest value
 * written says "clipped", the call launches the reduce / finalize / update
 * kernels directly, unguarded, and costs what zero_step costs. The word may
 * lag the GPU by the steps still queued: it only chooses which kernels run,
 * and both choices compute the same step. While the stream is being
 * captured, the word is not read (the graph keeps the device-guarded
 * sequence, whose single pass then returns at once when predicted).
 * ZERO_SPEC_HINT=0 in the environment at bind_alternate turns the word off.
 * Only the step on which clipping switches on pays for both passes.
 * The commit decision uses the single pass's own norm, summed in another
 * grouping than zero_step's (both within the parity tolerance of the exact
 * norm); only a norm within that rounding of the clip threshold could make
 * the two calls decide differently.
 * A committed step moves W*size(grad) + 24 + size(param) bytes per element,
 * the whole step's ledger; the reduced gradients are never stored, so the
 * scratch buffer's contents are unspecified afterwards.
 *   grads  flat gradients as for zero_step. Stages 2 and 3 (stage 1 through
 *          zero_step_speculative_allreduce); needs
 *          zero_state_bind_alternate. Errors as zero_step. */
int zero_step_speculative(zero_layout_t* layout, const void* const* grads, const zero_hparams* hp,
                          void* stream);

/* The speculative step in any stage. allreduce_out as zero_step's: stage 1
 * (ZeRO-1) takes W device pointers, Np elements of comm_dtype each, flat
 * layout, and the single pass writes every rank's copy of the reduced
 * gradient there on every step (committed, skipped or falling back), the
 * values zero_step writes; stages 2 and 3 take NULL and behave as
 * zero_step_speculative. Unlike zero_step's, the outputs must not overlap
 * the gradient buffers (ZERO_ERR_INVALID): a step that falls back reduces
 * the gradients again after the single pass has written the outputs. A
 * committed stage-1 step moves W*size(grad) + 24 + size(param) +
 * W*size(comm) bytes per element. Errors as zero_step. */
int zero_step_speculative_allreduce(zero_layout_t* layout, const void* const* grads,
                                    void* const* allreduce_out, const zero_hparams* hp,
                                    void* stream);

/* The speculative step with gradients given per tensor, as zero_step_tensors
 * takes them: grad_ptrs is a host array of W * n_params device pointers
 * (grad_ptrs[w * n_params + p]), 16-byte aligned, NULL for an all-zero
 * gradient, which is never read. Results are those of zero_step_speculative
 * on flat buffers holding zeros there, bit for bit. Stages 2 and 3 (stage 1
 * is refused: its all-reduce outputs are written from flat gradients). The
 * table is copied to the device on `stream` before the call returns, so it
 * is not capturable into a CUDA graph (ZERO_ERR_INVALID on a capturing
 * stream, nothing enqueued). Errors as zero_step_tensors. */
int zero_step_speculative_tensors(zero_layout_t* layout, const void* const* grad_ptrs,
                                  const zero_hparams* hp, void* stream);

/* Same step from HOST gradients: copies host_grads[w] (Np elements of
 * grad_dtype each, flat layout; pinned memory gives asynchronous copies) into
 * the device buffers dev_grads[w], then runs zero_step on dev_grads.
 * The copies run as pieces of at most 128 MB on copy streams the layout owns
 * (created on the first call); `stream` waits for them before the step. They
 * start after the last zero_step_host reduce kernel that read the same
 * dev_grads set has finished (stages 2/3) -- so they overlap that step's
 * update kernel -- or after all work queued on `stream` (stage 1, whose
 * all-reduce outputs may alias the gradients, and a set's first call). The
 * library remembers the last four sets (identified by their W pointers): a
 * caller that alternates two disjoint sets lets each step's copies overlap the
 * previous step's reduce as well, so the host link never waits for the GPU.
 * dev_grads must not be written by anything else between calls, and two sets
 * must not overlap in memory. */
int zero_step_host(zero_layout_t* layout, const void* const* host_grads, void* const* dev_grads,
                   void* const* allreduce_out, const zero_hparams* hp, void* stream);

/* Asynchronous form of zero_loss_scale_state: enqueues a copy of the
 * library's device state block (ZERO_STATE_BLOB_BYTES bytes) into `blob` on
 * `stream` and returns at once. `blob` should be pinned host memory (pageable
 * memory makes the copy synchronous). After the stream has reached that
 * point, zero_state_blob_decode turns the blob into a zero_scaler_state. */
#define ZERO_STATE_BLOB_BYTES 256
int zero_loss_scale_state_async(zero_layout_t* layout, void* blob, void* stream);
/* Host only. Returns ZERO_ERR_TIMEOUT if the blob records a kernel whose
 * bounded wait gave up. */
int zero_state_blob_decode(const void* blob, zero_scaler_state* out);

/* Read the scaler state and the last step's report. Enqueues a device-to-host
 * copy on `stream` and WAITS for it (synchronises the stream). */
int zero_loss_scale_state(zero_layout_t* layout, void* stream, zero_scaler_state* out);

/* Copy the flat parameters out to per-tensor storage ([DO] the all-gather
 * rebuilds the parameter buffer for the next forward).
 *   dst  host array of n_replicas * n_params device pointers
 *        (dst[k * n_params + p]: replica k's parameter p, numel elements of
 *        param_dtype). Enqueued on `stream`. */
int zero_gather_params(zero_layout_t* layout, void* const* dst, int n_replicas, void* stream);

/* Stage 3: all-gather bucket `bucket` of the sharded parameters into `dst`,
 * a device buffer in the FLAT layout (Np elements of param_dtype, or at least
 * up to the bucket's end); only that bucket's real elements are written.
 * Enqueued on `stream` -- issue the next bucket's gather on a second stream
 * to prefetch it while the current one is in use. ZERO_ERR_STATE for stages
 * 1/2 (their parameters are always gathered). */
int zero_gather_bucket(zero_layout_t* layout, int bucket, void* dst, void* stream);

/* Copy the rank-major fp32 state out to / in from flat-layout device buffers
 * (Np elements each; padding of the flat buffers is written as 0 on export
 * and ignored on import). Any of the three pointers may be NULL to skip it.
 * Enqueued on `stream`. */
int zero_state_export(zero_layout_t* layout, float* master_flat, float* m_flat, float* v_flat,
                      void* stream);
int zero_state_import(zero_layout_t* layout, const float* master_flat, const float* m_flat,
                      const float* v_flat, void* stream);

/* Optional timing hook. events: host array of 4 cudaEvent_t (as void*),
 * created by the caller; every later step records events[0] before the
 * reduce kernel, events[1] after it, events[2] after the finalize kernel and
 * events[3] after the update kernel, on the step's stream. NULL turns the
 * hook off. The events must outlive their use. No counterpart on the pages:
 * it exists so a benchmark can time each kernel with CUDA events. */
int zero_set_step_events(zero_layout_t* layout, void* const* events);

/* Reduce + overflow check + squared norm of W flat gradient buffers, using no
 * device memory of its own. The pages have no counterpart: this exists for
 * callers that cannot allocate -- code that must not call cudaMalloc while a
 * graph is being captured elsewhere in the process, embeddings whose device
 * memory is all handed out at start-up, hosts that forbid a library from
 * growing its footprint later. It computes what the step's first kernel
 * computes over the plain range [0, n) (no layout, no padding mask):
 *   r[i] = RNE_comm(g_0[i] + ... + g_{W-1}[i])  (fp32 adds in rank order),
 *   *norm_sq_out = sum of r[i]^2 (fp64 result), *overflow_out = any r non-finite.
 *   grads         host array of `world` device pointers (1..64), n elements of
 *                 grad_dtype each, 16-byte aligned. Read only.
 *   comm_dtype    dtype of r; -1 = grad_dtype.
 *   reduced_out   device, n elements of comm_dtype (16-byte aligned), or NULL
 *                 to skip writing r.
 *   norm_sq_out   device double; overflow_out: device int32.
 * Scratch: a fixed array inside the library (about 768 KB on every GPU that
 * loads it, held until the process exits) for one partial per 65,536
 * elements; n above 2^32 is rejected with ZERO_ERR_INVALID. Each CUDA
 * context holds its own copy of the array, so the first call made in each
 * context looks up that copy's device address (cudaGetSymbolAddress) and
 * caches it under the context's unique ID: the device's primary context, a
 * context the caller made current through the driver API, and the new
 * primary context after cudaDeviceReset are looked up separately. Make the
 * first call in each context before any stream capture. Every call shares
 * the one array: calls whose work overlaps on the GPU (different streams, no
 * ordering between them) race and give wrong results. Allocates nothing: no
 * cudaMalloc, cudaFree or allocating library call. Enqueued on `stream`. */
int zero_reduce_norm_noalloc(const void* const* grads, int world, int64_t n, int grad_dtype,
                             int comm_dtype, void* reduced_out, double* norm_sq_out,
                             int32_t* overflow_out, void* stream);

/* Self-test of the bounded-wait path every pipelined kernel relies on. One
 * block arms an mbarrier for 16 bytes that never arrive, waits on it with at
 * most `spin_limit` retries (1..2^22), records the timeout in a device error
 * word as the kernels do, and returns. Returns ZERO_ERR_TIMEOUT when the wait
 * gave up (the expected outcome), ZERO_OK if it did not, ZERO_ERR_CUDA on a
 * CUDA failure. Synchronises `stream`; the context stays usable. No
 * counterpart on the pages: it tests failure detection without a GPU fault. */
int zero_selftest_wait_timeout(uint32_t spin_limit, void* stream);

/* The same self-test bound to a layout: the wait's timeout is OR-ed into the
 * layout's device error word, exactly as a step kernel records one. Requires
 * zero_state_init. Synchronises `stream` and returns what the next state
 * read reports: ZERO_ERR_TIMEOUT when the wait gave up (the expected
 * outcome). From then on the layout's step kernels return at once, until
 * zero_state_init. */
int zero_selftest_layout_timeout(zero_layout_t* layout, uint32_t spin_limit, void* stream);

/* ------------------------------------------------------------------------ */
/* Gradient accumulation into fp32 main-gradient buffers ([DO] "BF16 model   */
/* parameters and FP32 main gradients"; [MD] "Initializing a DeepSpeed       */
/* Engine": backward/step fire the reduction only on boundary micro-steps).  */
/* ------------------------------------------------------------------------ */

/* main[w][i] = (first ? 0 : main[w][i]) + fp32(micro[w][i]) for every real
 * element i of the layout (padding untouched), for w = 0..W-1.
 *   micro  host array of W device pointers, flat layout, layout's grad_dtype
 *          or any ZERO_* dtype given by micro_dtype; read only.
 *   main   host array of W device pointers, flat layout, fp32.
 *   first  nonzero on the first micro-step of an accumulation window.
 * The boundary step then runs zero_step on a layout whose grad_dtype is
 * ZERO_F32 over `main`. Enqueued on `stream`. */
int zero_accumulate(zero_layout_t* layout, const void* const* micro, int micro_dtype,
                    float* const* main, int first, void* stream);

/* ------------------------------------------------------------------------ */
/* Checkpoints that survive a change of W or bucket size (leetllm "Deep     */
/* dive: Megatron", "Checkpoints, resharding, and recovery": optimizer      */
/* moments and iteration counters are saved; a parameter-shaped             */
/* representation (fully_reshardable) permits resharding).                  */
/* ------------------------------------------------------------------------ */

/* fp32 master/m/v in PARAMETER-MAJOR order: parameter 0's elements, then
 * parameter 1's, ... (n_real elements, no padding), independent of W, stage
 * and bucket size. Any pointer may be NULL to skip that buffer. Device
 * pointers, 16-byte aligned. Enqueued on `stream`. */
int zero_state_export_params(zero_layout_t* layout, float* master_pm, float* m_pm, float* v_pm,
                             void* stream);

/* The inverse: loads master/m/v from parameter-major buffers into this
 * layout's rank-major shards (any W, stage or bucket size over the same
 * parameter list) and recasts the flat parameters from the loaded master. A
 * NULL m_pm / v_pm leaves that state untouched. Enqueued on `stream`. */
int zero_state_import_params(zero_layout_t* layout, const float* master_pm, const float* m_pm,
                             const float* v_pm, void* stream);

/* Restore the scaler's scale, clean-step counter and Adam step t (from a
 * saved zero_scaler_state); the other fields of `st` are ignored. Enqueued
 * on `stream`. */
int zero_scaler_restore(zero_layout_t* layout, const zero_scaler_state* st, void* stream);

/* ------------------------------------------------------------------------ */
/* Sharded step: one process per GPU ([DO] "Distributed optimizer: trade      */
/* replicated state for collectives": reduce-scatter of each bucket, local   */
/* FP32 update of the rank's master slice and moments, all-gather of the     */
/* parameters). The caller's communication library (NCCL, through its own    */
/* bindings) runs the collectives between these calls; the library computes  */
/* everything between them. The layout's world is the number of GPUs.        */
/* ------------------------------------------------------------------------ */

/* Make this layout rank `rank`'s (0..W-1) of a W-GPU job. Call after
 * zero_layout_create and before zero_state_bind; the layout then holds only
 * this rank's shard, and the buffers bound later are:
 *   master, m, v, scratch  Np/W elements: this rank's slice of bucket 0, then
 *                          bucket 1, ... (bucket b's slice starts at
 *                          shard_offset - rank*Np/W of zero_shard_range);
 *   params_flat            stages 1/2: Np elements, flat layout (the step
 *                          writes this rank's slices; the caller's all-gather
 *                          of each bucket fills the rest); stage 3: Np/W
 *                          elements, this rank's slices.
 * zero_state_init then initialises this rank's slices only (master_init_flat
 * is still the whole flat buffer): all-gather the parameters once after it.
 * Requires comm_dtype == grad_dtype, or ZERO_F32 with 16-bit gradients (the
 * collectives reduce in the communication dtype; zero_dist_widen gives the
 * fp32 copy to reduce). ZERO_ERR_STATE if called twice or after bind; every entry point
 * that steps all W ranks in one process (zero_step*, accumulation, gathers)
 * then returns ZERO_ERR_STATE. zero_state_export / import and
 * zero_state_export_params / import_params move this rank's elements only:
 * an export writes them and zero-fills the rest of the destination (so the
 * ranks' exports, summed as 32-bit integers, give the whole buffer, -0.0
 * included); an import reads them from a whole buffer, which may come from a
 * job of any W, stage or bucket size. Host only. */
int zero_dist_set_rank(zero_layout_t* layout, int rank);

/* With an fp32 comm_dtype and 16-bit gradients ([ND] "9. Experimental
 * Results": communication_data_type): out[i] = fp32(grads[i]) for the whole
 * flat buffer, i < Np (exact), the buffer this rank then reduce-scatters (or,
 * stage 1, all-reduces) in fp32. grads: device, Np elements of grad_dtype;
 * out: device, Np floats; both 16-byte aligned. */
int zero_dist_widen(zero_layout_t* layout, const void* grads, float* out, void* stream);

/* This rank's share of the global norm and overflow check: enqueues a kernel
 * that writes norm_pair[0] = sum of r^2 over this rank's real elements (fp64
 * partials, a fixed order for a given device) and norm_pair[1] = 1.0 if any
 * of them is non-finite, else 0.0. The caller then sums the pair over ranks
 * (one 16-byte all-reduce) and passes the result to zero_dist_finalize.
 *   allreduced  stages 2/3: NULL (the bound scratch holds this rank's
 *               reduce-scatter output); stage 1: device, Np elements of
 *               comm_dtype, flat layout, this rank's all-reduced gradient.
 *   norm_pair   device, 2 doubles, 8-byte aligned. */
int zero_dist_shard_norm(zero_layout_t* layout, const void* allreduced, double* norm_pair,
                         void* stream);

/* The finalize from the all-reduced pair (device, 2 doubles: global sum of
 * squares, > 0 when any rank overflowed): norm, clip coefficient, loss-scale
 * state machine and t, exactly as zero_step's finalize with world W. Every
 * rank gets the same pair, so every rank takes the same decision. */
int zero_dist_finalize(zero_layout_t* layout, const double* norm_pair, const zero_hparams* hp,
                       void* stream);

/* Unscale + clip + AdamW on this rank's fp32 slice and cast-out of its
 * parameters (stages 1/2: into params_flat at flat offsets; stage 3: into
 * its own slices). Returns at once on the device after an overflow (the step
 * is skipped). allreduced as for zero_dist_shard_norm. Then the caller
 * all-gathers each bucket of params_flat (stages 1/2). */
int zero_dist_update(zero_layout_t* layout, const void* allreduced, void* stream);

/* zero_dist_update restricted to buckets [first_bucket, first_bucket +
 * n_buckets): this rank's tiles of those buckets only. Updating bucket by
 * bucket lets the caller start each bucket's all-gather while the next
 * bucket is being updated ([DO] "Distributed optimizer": the parameters come
 * back bucket by bucket). The union of the ranges over a step must be every
 * bucket once, after zero_dist_finalize. ZERO_ERR_INVALID for a range
 * outside the layout's buckets; an empty range enqueues nothing. */
int zero_dist_update_buckets(zero_layout_t* layout, const void* allreduced, int first_bucket,
                             int n_buckets, void* stream);

/* Message for the last failing call on this thread ("" if none). The pointer
 * stays valid until the next failing call on this thread. */
const char* zero_last_error(void);

/* Replace the allocator used for the library's own device block (default:
 * cudaMalloc / cudaFree). alloc returns NULL on failure -> ZERO_ERR_OOM. */
typedef void* (*zero_alloc_fn)(size_t bytes, void* ctx);
typedef void (*zero_free_fn)(void* ptr, void* ctx);
int zero_layout_set_allocator(zero_layout_t* layout, zero_alloc_fn alloc, zero_free_fn free_fn,
                              void* ctx);

#ifdef __cplusplus
}
#endif
#endif /* ZERO_GB300_H */
