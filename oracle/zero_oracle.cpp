/*
 * Oracle for the ZeRO-1/2 gradient-and-optimizer step (see zero_oracle.h).
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
 * benchmark's CPU-baseline leg, never by the product path. Deliberately plain:
 * one element at a time, no blocking, no threads, no vector tricks.
 *
 * Built with -ffp-contract=off so that no multiply-add is fused behind the
 * reader's back, and the results are the same on x86-64 and aarch64 hosts.
 */
#include "zero_oracle.h"

#include <cmath>
#include <cstring>
#include <vector>

namespace {

/* ------------------------------------------------------------------------ */
/* IEEE-754 binary formats, written out from the standard's definition.      */
/* ------------------------------------------------------------------------ */

struct Fmt {
  int exp_bits;
  int man_bits;
};
const Fmt kF16 = {5, 10};
const Fmt kBF16 = {8, 7};

int bias_of(Fmt f) { return (1 << (f.exp_bits - 1)) - 1; }

/* bits -> exact value (as double, which holds every binary16/bfloat16 value). */
double decode_fmt(uint32_t bits, Fmt f) {
  const uint32_t exp_all = (1u << f.exp_bits) - 1;
  const uint32_t sign = (bits >> (f.exp_bits + f.man_bits)) & 1u;
  const uint32_t e = (bits >> f.man_bits) & exp_all;
  const uint32_t m = bits & ((1u << f.man_bits) - 1);
  const int bias = bias_of(f);
  double mag;
  if (e == exp_all) {
    mag = m ? NAN : INFINITY;
  } else if (e == 0) { /* zero or subnormal: m * 2^(1 - bias - man_bits) */
    mag = std::ldexp((double)m, 1 - bias - f.man_bits);
  } else { /* normal: (1.m) * 2^(e - bias) */
    mag = std::ldexp((double)(m | (1u << f.man_bits)), (int)e - bias - f.man_bits);
  }
  return sign ? -mag : mag;
}

/* value -> bits, rounding to nearest with ties to even. The value is rounded
 * to an integer multiple of the format's quantum at its binade (the subnormal
 * quantum below the smallest normal); a result at or above 2^(emax+1)
 * becomes infinity. NaN maps to a quiet NaN with the input's sign. */
uint32_t encode_fmt(double x, Fmt f) {
  const uint32_t exp_all = (1u << f.exp_bits) - 1;
  const uint32_t sign = std::signbit(x) ? (1u << (f.exp_bits + f.man_bits)) : 0u;
  const int bias = bias_of(f);
  const int emin = 1 - bias; /* exponent of the smallest normal */
  const int emax = bias;     /* exponent of the largest finite binade */
  if (std::isnan(x)) return sign | (exp_all << f.man_bits) | (1u << (f.man_bits - 1));
  const double a = std::fabs(x);
  if (std::isinf(a)) return sign | (exp_all << f.man_bits);
  if (a == 0.0) return sign;
  int e;
  std::frexp(a, &e); /* a = frac * 2^e, frac in [0.5, 1) */
  e -= 1;            /* a = 1.x * 2^e */
  const int quantum_exp = (e < emin ? emin : e) - f.man_bits;
  const double n = std::nearbyint(std::ldexp(a, -quantum_exp)); /* ties-to-even integer */
  if (n == 0.0) return sign;
  const double r = std::ldexp(n, quantum_exp);
  if (r >= std::ldexp(1.0, emax + 1)) return sign | (exp_all << f.man_bits);
  int re;
  std::frexp(r, &re);
  re -= 1;
  if (re < emin) { /* subnormal result */
    const uint32_t mant = (uint32_t)std::ldexp(r, f.man_bits - emin);
    return sign | mant;
  }
  const uint32_t field = (uint32_t)(re + bias);
  const uint32_t mant = (uint32_t)std::ldexp(r, f.man_bits - re) - (1u << f.man_bits);
  return sign | (field << f.man_bits) | mant;
}

int elem_bytes(int dtype) { return dtype == ORC_F32 ? 4 : 2; }

/* Read element i of a buffer of the given dtype as an fp32 value (exact). */
float load_f32(const void* buf, int64_t i, int dtype) {
  if (dtype == ORC_F32) return static_cast<const float*>(buf)[i];
  const uint16_t bits = static_cast<const uint16_t*>(buf)[i];
  return (float)decode_fmt(bits, dtype == ORC_F16 ? kF16 : kBF16);
}

/* Round an fp32 value to the dtype and store it as element i. */
void store_rne(void* buf, int64_t i, int dtype, float x) {
  if (dtype == ORC_F32) {
    static_cast<float*>(buf)[i] = x;
    return;
  }
  static_cast<uint16_t*>(buf)[i] = (uint16_t)encode_fmt((double)x, dtype == ORC_F16 ? kF16 : kBF16);
}

int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

/* Alignment of every parameter's offset in the flat buffer, and the unit the
 * padded bucket length is a multiple of (times the world size). Reading: the
 * pages fix no alignment; 64 elements keeps every parameter start on a 128-byte
 * line for 2-byte types. */
const int64_t kParamAlign = 64;
const int64_t kShardUnit = 128;

} /* namespace */

extern "C" {

/* ------------------------------------------------------------------------ */
/* a1. Flat bucketed layout.                                                 */
/* "Deep dive: Megatron", "Distributed optimizer": parameter and gradient    */
/* buffers are contiguous and communicated bucket by bucket; each rank owns  */
/* an equal contiguous shard (the SGD example there needs a buffer divisible */
/* by the group size). "3.7 ...", "DeepSpeed config for this run": bucket    */
/* sizes in bytes (reduce_bucket_size).                                      */
/* Reading: parameters keep their given order; a parameter is never split;   */
/* a new bucket opens when the next parameter would take the bucket's span   */
/* past bucket_bytes / grad_bytes elements and the bucket already holds one; */
/* each bucket is padded to a multiple of world * 128 elements and rank r    */
/* owns [start + r*len/W, start + (r+1)*len/W) of every bucket.              */
/* ------------------------------------------------------------------------ */
int orc_layout(const int64_t* numel, int n_params, int world, int64_t bucket_bytes,
               int grad_bytes, int64_t* param_offset, int* param_bucket,
               int64_t* bucket_start, int64_t* bucket_len, int* n_buckets, int64_t* np_total) {
  if (n_params <= 0 || world <= 0 || bucket_bytes <= 0 || grad_bytes <= 0) return 1;
  const int64_t cap = bucket_bytes / grad_bytes;
  const int64_t unit = (int64_t)world * kShardUnit;
  int nb = 0;
  int64_t pos = 0;
  int64_t b0 = 0;
  bool open_has_param = false;
  for (int p = 0; p < n_params; ++p) {
    if (numel[p] < 0) return 1;
    int64_t off = align_up(pos, kParamAlign);
    if (open_has_param && off + numel[p] - b0 > cap) {
      bucket_start[nb] = b0;
      bucket_len[nb] = align_up(pos - b0, unit);
      pos = b0 + bucket_len[nb];
      ++nb;
      b0 = pos;
      off = pos;
    }
    param_offset[p] = off;
    param_bucket[p] = nb;
    pos = off + numel[p];
    open_has_param = true;
  }
  bucket_start[nb] = b0;
  bucket_len[nb] = align_up(pos - b0, unit);
  pos = b0 + bucket_len[nb];
  ++nb;
  *n_buckets = nb;
  *np_total = pos;
  return 0;
}

void orc_encode(const float* x, int64_t n, int dtype, void* out) {
  for (int64_t i = 0; i < n; ++i) store_rne(out, i, dtype, x[i]);
}

void orc_decode(const void* in, int64_t n, int dtype, float* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = load_f32(in, i, dtype);
}

/* ------------------------------------------------------------------------ */
/* a2. Reduce (the reduce-scatter's arithmetic) over elements [begin, end).  */
/* "Deep dive: Megatron", "Distributed optimizer": the reduce-scatter sums   */
/* the ranks' gradients. "nano-deepspeed", "9. Experimental Results": the    */
/* communication runs in a stated data type (communication_data_type).      */
/* Reading: s = g_0 + g_1 + ... + g_{W-1}, left to right, each add rounded   */
/* to fp32; then one rounding to the communication dtype. Padding elements   */
/* (real_mask[i] == 0) are not read and come out as +0.                      */
/* Output element k holds element begin + k.                                 */
/* ------------------------------------------------------------------------ */
void orc_reduce(const void* const* grads, int world, int grad_dtype, int64_t begin, int64_t end,
                const uint8_t* real_mask, int comm_dtype, void* out) {
  for (int64_t i = begin; i < end; ++i) {
    float s = 0.0f;
    if (real_mask == nullptr || real_mask[i]) {
      s = load_f32(grads[0], i, grad_dtype);
      for (int w = 1; w < world; ++w) s = s + load_f32(grads[w], i, grad_dtype);
    }
    store_rne(out, i - begin, comm_dtype, s);
  }
}

/* ------------------------------------------------------------------------ */
/* a3 + a4 (partial). Overflow flag and sum of squares of reduced values.    */
/* "nano-deepspeed", "2. Current Feature Range" (FP16 dynamic loss scaling)  */
/* and "9. Experimental Results" (runs checked for non-finite values).       */
/* Reading: the check is on the reduced, communication-dtype values, so an   */
/* fp16 sum that rounds to infinity counts; padding is excluded.             */
/* The sum of squares is taken in fp64, element by element, in index order.  */
/* ------------------------------------------------------------------------ */
void orc_overflow_sumsq(const void* reduced, int comm_dtype, int64_t n, const uint8_t* real_mask,
                        int32_t* overflow, double* sumsq) {
  int32_t ovf = 0;
  double acc = 0.0;
  for (int64_t i = 0; i < n; ++i) {
    if (real_mask != nullptr && !real_mask[i]) continue;
    const double r = (double)load_f32(reduced, i, comm_dtype);
    if (!std::isfinite(r)) ovf = 1;
    acc += r * r;
  }
  *overflow = ovf;
  *sumsq = acc;
}

/* ------------------------------------------------------------------------ */
/* a4 + a5. Global norm, clip coefficient, loss-scale state machine.         */
/* "3.7 ...", "ZeRO-Offload and ZeRO-Infinity": gradient_clipping 1.0,       */
/* loss_scale 0 (dynamic) with loss_scale_window. No formula is printed;     */
/* readings:                                                                 */
/*  - inv = 1 / (S * D); D = grad_divisor, or the world size when <= 0.      */
/*  - norm = inv * sqrt(sum r^2)  (L2 norm of the unscaled, divided grads).  */
/*  - clip: c = min(1, max_norm / (norm + 1e-6)), c = 1 when max_norm <= 0.  */
/*  - overflow: skip the update (t unchanged), S <- max(S * backoff, min),   */
/*    counter <- 0 (dynamic mode only changes S).                            */
/*  - clean step: t <- t + 1, the update is applied, counter <- counter + 1; */
/*    when counter reaches N (dynamic mode) S <- S * growth, counter <- 0.   */
/* ------------------------------------------------------------------------ */
void orc_finalize(double norm_sq_raw, int32_t overflow, int world, const orc_hparams* hp,
                  orc_scaler* sc, orc_info* info) {
  const double divisor = hp->grad_divisor > 0.0 ? hp->grad_divisor : (double)world;
  const double inv = 1.0 / (sc->scale * divisor);
  info->overflow = overflow ? 1 : 0;
  info->norm_sq_raw = norm_sq_raw;
  info->grad_norm = inv * std::sqrt(norm_sq_raw);
  if (overflow) {
    info->skipped = 1;
    info->clip_coef = 0.0;
    info->gscale = 0.0;
    info->bc1 = 0.0;
    info->bc2 = 0.0;
    if (sc->dynamic) {
      double s = sc->scale * sc->backoff_factor;
      sc->scale = s < sc->min_scale ? sc->min_scale : s;
    }
    sc->counter = 0;
    return;
  }
  double c = 1.0;
  if (hp->max_grad_norm > 0.0) {
    c = hp->max_grad_norm / (info->grad_norm + 1e-6);
    if (c > 1.0) c = 1.0;
  }
  info->skipped = 0;
  info->clip_coef = c;
  info->gscale = inv * c;
  sc->t += 1;
  info->bc1 = 1.0 - std::pow(hp->beta1, (double)sc->t);
  info->bc2 = 1.0 - std::pow(hp->beta2, (double)sc->t);
  sc->counter += 1;
  if (sc->dynamic && sc->counter == sc->growth_interval) {
    sc->scale = sc->scale * sc->growth_factor;
    sc->counter = 0;
  }
}

/* ------------------------------------------------------------------------ */
/* a6. Unscale + clip + AdamW on n elements (one shard).                     */
/* "nano-deepspeed", "2. Current Feature Range": AdamW is the optimizer;     */
/* "3.7 ...", "Initializing a DeepSpeed Engine": torch.optim.AdamW.          */
/* Reading: decoupled weight decay as in torch.optim.AdamW, no amsgrad:      */
/*   g = r * clip / (S * D)                                                  */
/*   p = p * (1 - lr * wd)                                                   */
/*   m = b1 * m + (1 - b1) * g                                               */
/*   v = b2 * v + (1 - b2) * g^2                                             */
/*   p = p - (lr / (1 - b1^t)) * m / (sqrt(v) / sqrt(1 - b2^t) + eps)        */
/* Element math in fp64; master, m and v are stored back as fp32.            */
/* A skipped step leaves everything untouched.                               */
/* ------------------------------------------------------------------------ */
void orc_adamw(const void* reduced, int comm_dtype, int64_t n, const orc_hparams* hp,
               const orc_info* info, float* master, float* m, float* v) {
  if (info->skipped) return;
  const double b1 = hp->beta1, b2 = hp->beta2;
  const double step_size = hp->lr / info->bc1;
  const double sqrt_bc2 = std::sqrt(info->bc2);
  for (int64_t i = 0; i < n; ++i) {
    const double g = (double)load_f32(reduced, i, comm_dtype) * info->gscale;
    double p = (double)master[i];
    double mi = (double)m[i];
    double vi = (double)v[i];
    p = p * (1.0 - hp->lr * hp->weight_decay);
    mi = b1 * mi + (1.0 - b1) * g;
    vi = b2 * vi + (1.0 - b2) * g * g;
    const double denom = std::sqrt(vi) / sqrt_bc2 + hp->eps;
    p = p - step_size * mi / denom;
    master[i] = (float)p;
    m[i] = (float)mi;
    v[i] = (float)vi;
  }
}

/* ------------------------------------------------------------------------ */
/* Gradient accumulation into fp32 main gradients.                           */
/* "Deep dive: Megatron", "Distributed optimizer": BF16 parameters with FP32 */
/* main gradients (the 18-byte ledger). "3.7 ...", "Initializing a DeepSpeed */
/* Engine": backward and step are accumulation-aware and reduce only on the  */
/* boundary micro-step. Reading: main = (first ? +0 : main) + fp32(micro),   */
/* one fp32 add per micro-step, in micro-step order; padding untouched.      */
/* ------------------------------------------------------------------------ */
void orc_accumulate(const void* micro, int micro_dtype, float* main_grad, int64_t n,
                    const uint8_t* real_mask, int first) {
  for (int64_t i = 0; i < n; ++i) {
    if (real_mask != nullptr && !real_mask[i]) continue;
    const float base = first ? 0.0f : main_grad[i];
    main_grad[i] = base + load_f32(micro, i, micro_dtype);
  }
}

/* ------------------------------------------------------------------------ */
/* Unpartitioned (DDP) step over the whole model, no padding, no shards.     */
/* "nanoMegatron", "What's in the box": DDP keeps the full model on every    */
/* GPU and all-reduces gradients. Every rank then runs the same update, so   */
/* one copy of the state stands for all of them.                             */
/* grads: world pointers to n elements (parameters concatenated in order).   */
/* ------------------------------------------------------------------------ */
int orc_ddp_step(int world, int64_t n, int grad_dtype, int comm_dtype, int param_dtype,
                 const void* const* grads, float* master, float* m, float* v, void* params,
                 const orc_hparams* hp, orc_scaler* scaler, orc_info* info) {
  if (world <= 0 || n < 0) return 1;
  std::vector<uint8_t> reduced((size_t)n * elem_bytes(comm_dtype) + 4);
  orc_reduce(grads, world, grad_dtype, 0, n, nullptr, comm_dtype, reduced.data());
  int32_t ovf = 0;
  double sumsq = 0.0;
  orc_overflow_sumsq(reduced.data(), comm_dtype, n, nullptr, &ovf, &sumsq);
  orc_finalize(sumsq, ovf, world, hp, scaler, info);
  orc_adamw(reduced.data(), comm_dtype, n, hp, info, master, m, v);
  if (!info->skipped)
    for (int64_t i = 0; i < n; ++i) store_rne(params, i, param_dtype, master[i]);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Partitioned ZeRO-1/2 step, written rank by rank.                          */
/* "Deep dive: Megatron", "Distributed optimizer": backward fills a gradient */
/* buffer on each rank; the reduce-scatter gives each rank its shard; each   */
/* rank updates its fp32 master shard and moments; the all-gather rebuilds   */
/* the low-precision parameter buffer. "nano-deepspeed", "2. Current Feature */
/* Range": stage 2 done as a packed all-reduce then a local scatter-back --  */
/* here stage 1: every rank receives the whole reduced gradient             */
/* (allreduce_out[w], flat layout) and still updates only its shard.         */
/*                                                                          */
/* grads[w]: rank w's gradients in the flat layout (np_total elements; the   */
/*   padding is never read).                                                 */
/* master/m/v_shards: rank-major, rank r's shard at [r*np/W, (r+1)*np/W),    */
/*   holding its slice of bucket 0, then of bucket 1, and so on.             */
/* params_flat: the gathered low-precision parameters, flat layout; padding  */
/*   is written as zero.                                                     */
/* ------------------------------------------------------------------------ */
int orc_zero_step(const int64_t* numel, int n_params, int world, int stage, int64_t bucket_bytes,
                  int grad_dtype, int comm_dtype, int param_dtype,
                  const void* const* grads, void* const* allreduce_out,
                  float* master_shards, float* m_shards, float* v_shards, void* params_flat,
                  const orc_hparams* hp, orc_scaler* scaler, orc_info* info) {
  if (stage != 1 && stage != 2) return 1;
  std::vector<int64_t> poff(n_params);
  std::vector<int> pbucket(n_params);
  std::vector<int64_t> bstart(n_params + 1), blen(n_params + 1);
  int nb = 0;
  int64_t np = 0;
  if (orc_layout(numel, n_params, world, bucket_bytes, elem_bytes(grad_dtype), poff.data(),
                 pbucket.data(), bstart.data(), blen.data(), &nb, &np))
    return 1;
  std::vector<uint8_t> real(np, 0);
  for (int p = 0; p < n_params; ++p)
    for (int64_t k = 0; k < numel[p]; ++k) real[poff[p] + k] = 1;

  const int cb = elem_bytes(comm_dtype);
  const int64_t shard_total = np / world; /* every bucket gives each rank len/W */

  /* Each rank's reduce-scatter output: its slice of every bucket, in order. */
  std::vector<std::vector<uint8_t>> shard_grad(world, std::vector<uint8_t>(shard_total * cb + 4));
  for (int r = 0; r < world; ++r) {
    int64_t at = 0;
    for (int b = 0; b < nb; ++b) {
      const int64_t slice = blen[b] / world;
      const int64_t lo = bstart[b] + r * slice;
      orc_reduce(grads, world, grad_dtype, lo, lo + slice, real.data(), comm_dtype,
                 shard_grad[r].data() + at * cb);
      at += slice;
    }
  }
  /* Stage 1: the all-reduce hands the full reduced gradient to every rank. */
  if (stage == 1) {
    for (int w = 0; w < world; ++w) {
      std::vector<uint8_t> full(np * cb + 4);
      orc_reduce(grads, world, grad_dtype, 0, np, real.data(), comm_dtype, full.data());
      std::memcpy(allreduce_out[w], full.data(), (size_t)(np * cb));
    }
  }

  /* Each rank: overflow flag and squared norm of its own shard; then the     */
  /* all-reduce of both (sum in rank order, logical OR).                      */
  double sumsq = 0.0;
  int32_t ovf = 0;
  for (int r = 0; r < world; ++r) {
    std::vector<uint8_t> shard_real(shard_total);
    int64_t at = 0;
    for (int b = 0; b < nb; ++b) {
      const int64_t slice = blen[b] / world;
      const int64_t lo = bstart[b] + r * slice;
      for (int64_t k = 0; k < slice; ++k) shard_real[at + k] = real[lo + k];
      at += slice;
    }
    int32_t o = 0;
    double s = 0.0;
    /* Stage 1 reads its shard out of its own all-reduced copy. */
    if (stage == 1) {
      std::vector<uint8_t> mine(shard_total * cb + 4);
      int64_t at2 = 0;
      for (int b = 0; b < nb; ++b) {
        const int64_t slice = blen[b] / world;
        const int64_t lo = bstart[b] + r * slice;
        std::memcpy(mine.data() + at2 * cb, static_cast<const uint8_t*>(allreduce_out[r]) + lo * cb,
                    (size_t)(slice * cb));
        at2 += slice;
      }
      shard_grad[r] = mine;
    }
    orc_overflow_sumsq(shard_grad[r].data(), comm_dtype, shard_total, shard_real.data(), &o, &s);
    sumsq += s;
    ovf |= o;
  }

  orc_finalize(sumsq, ovf, world, hp, scaler, info);
  if (info->skipped) return 0;

  /* Each rank updates its shard, then the all-gather writes every rank's     */
  /* updated parameters into the flat low-precision buffer.                   */
  for (int r = 0; r < world; ++r) {
    float* ms = master_shards + r * shard_total;
    float* mm = m_shards + r * shard_total;
    float* vv = v_shards + r * shard_total;
    orc_adamw(shard_grad[r].data(), comm_dtype, shard_total, hp, info, ms, mm, vv);
    int64_t at = 0;
    for (int b = 0; b < nb; ++b) {
      const int64_t slice = blen[b] / world;
      const int64_t lo = bstart[b] + r * slice;
      for (int64_t k = 0; k < slice; ++k) {
        const float val = real[lo + k] ? ms[at + k] : 0.0f;
        store_rne(params_flat, lo + k, param_dtype, val);
      }
      at += slice;
    }
  }
  return 0;
}

} /* extern "C" */
