/*
 * Oracle for the ZeRO-1/2 gradient-and-optimizer step: plain, slow host code.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark load this library. The product path (the CUDA library
 * under mixed_precision_gb300/) shares no code with it and never calls it.
 *
 * Storage is fp32 for master weights and Adam moments; every element-wise
 * formula is evaluated in fp64 and rounded once to fp32 on store. Low-precision
 * values are decoded and encoded with this file's own bit-level IEEE-754 code
 * (round to nearest, ties to even). The gradient reduction is, by definition,
 * a rank-ordered fp32 sum, so it is evaluated in fp32 here as well.
 *
 * Sources (page title, then section):
 *  - "Deep dive: Megatron" (leetllm), section "Distributed optimizer: trade
 *    replicated state for collectives": reduce-scatter of gradients, local
 *    update of the fp32 master shard and moments, all-gather of the bf16
 *    parameters; equal contiguous shards; the byte ledger; reduction scaled to
 *    the loss normalisation.
 *  - "nano-deepspeed (Teaching Edition)", section "2. Current Feature Range":
 *    AdamW only, FP16 dynamic loss scaling, the bf16 path, stage-2 packed
 *    all-reduce then local scatter-back (ZeRO-1 semantics here).
 *  - "3.7 Megatron-LM, DeepSpeed & Parallelism in Practice", sections
 *    "ZeRO-Offload and ZeRO-Infinity" (loss_scale 0 = dynamic,
 *    loss_scale_window, gradient_clipping 1.0, reduce_bucket_size) and
 *    "DeepSpeed config for this run" (500 MB buckets).
 * The pages print no AdamW, clipping or loss-scaler equations; the readings
 * used are stated at each function.
 */
#ifndef ZERO_ORACLE_H
#define ZERO_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2 };

typedef struct {
  double lr, beta1, beta2, eps, weight_decay;
  double max_grad_norm; /* <= 0 turns clipping off */
  double grad_divisor;  /* <= 0 means "world size" (replica mean) */
} orc_hparams;

typedef struct {
  double scale;           /* current loss scale S */
  int64_t counter;        /* clean steps since the last overflow or growth */
  int64_t t;              /* Adam step count (applied steps only) */
  int32_t dynamic;        /* 1: fp16 dynamic scaling; 0: static scale */
  int32_t _pad;
  int64_t growth_interval;/* N clean steps before the scale grows */
  double growth_factor, backoff_factor, min_scale;
} orc_scaler;

typedef struct {
  int32_t overflow, skipped;
  double norm_sq_raw;     /* sum of squares of the reduced, still-scaled gradient */
  double grad_norm;       /* unscaled, divided gradient norm */
  double clip_coef;
  double gscale;          /* factor applied to each reduced value: clip / (S * D) */
  double bc1, bc2;        /* 1 - beta^t for the step just applied */
} orc_info;

/* ---- layout (flat bucketed buffer, per-bucket W-way shards) ---- */
int orc_layout(const int64_t* numel, int n_params, int world, int64_t bucket_bytes,
               int grad_bytes, int64_t* param_offset, int* param_bucket,
               int64_t* bucket_start, int64_t* bucket_len, int* n_buckets, int64_t* np_total);

/* ---- bit-level conversions ---- */
void orc_encode(const float* x, int64_t n, int dtype, void* out);
void orc_decode(const void* in, int64_t n, int dtype, float* out);

/* ---- individual steps, exported so tests can check each one ---- */
void orc_reduce(const void* const* grads, int world, int grad_dtype, int64_t begin, int64_t end,
                const uint8_t* real_mask, int comm_dtype, void* out);
void orc_overflow_sumsq(const void* reduced, int comm_dtype, int64_t n, const uint8_t* real_mask,
                        int32_t* overflow, double* sumsq);
void orc_finalize(double norm_sq_raw, int32_t overflow, int world, const orc_hparams* hp,
                  orc_scaler* scaler, orc_info* info);
void orc_adamw(const void* reduced, int comm_dtype, int64_t n, const orc_hparams* hp,
               const orc_info* info, float* master, float* m, float* v);

/* ---- gradient accumulation into fp32 main gradients ---- */
void orc_accumulate(const void* micro, int micro_dtype, float* main_grad, int64_t n,
                    const uint8_t* real_mask, int first);

/* ---- composed steps ---- */
int orc_ddp_step(int world, int64_t n, int grad_dtype, int comm_dtype, int param_dtype,
                 const void* const* grads, float* master, float* m, float* v, void* params,
                 const orc_hparams* hp, orc_scaler* scaler, orc_info* info);

int orc_zero_step(const int64_t* numel, int n_params, int world, int stage, int64_t bucket_bytes,
                  int grad_dtype, int comm_dtype, int param_dtype,
                  const void* const* grads, void* const* allreduce_out,
                  float* master_shards, float* m_shards, float* v_shards, void* params_flat,
                  const orc_hparams* hp, orc_scaler* scaler, orc_info* info);

#ifdef __cplusplus
}
#endif
#endif
