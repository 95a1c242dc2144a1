/* Oracle for the ZeRO shard step: a plain, slow, single-threaded CPU statement of what
 * the step computes. TEST INFRASTRUCTURE ONLY: it exists so that tests and the bench's
 * CPU-baseline leg can check the GPU library against an independent implementation.
 * The product library never links, loads or calls it, and it shares no code with the
 * product.
 *
 * Sources (the three web pages on ZeRO, cited by page and section):
 *   - "ZeRO" method entry (codewithpapers.app/method/zero), description paragraph:
 *     model states are partitioned across data-parallel processes instead of replicated.
 *   - ZeRO explainer (papermap.vercel.app), "The 16 Bytes per Parameter Audit" and
 *     Chapter 02 "The Three Stages" (memory per parameter; what each stage shards;
 *     all-gather before forward, reduce-scatter after backward), and the stage table
 *     after Chapter 05.
 * The pages print no formula for the optimizer step. The step is the textbook
 * mixed-precision AdamW (fp16 gradients summed in fp32 in rank order, unscaled by the
 * loss scale, inf/nan skip, global-norm clipping, fp32 master weights and moments,
 * fp16 cast), with each reading stated where it is used in oracle.c.
 *
 * Compile with -ffp-contract=off: every float operation below is a single IEEE
 * operation rounded to nearest even.
 */
#ifndef ZERO_ORACLE_H
#define ZERO_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  float lr, beta1, beta2, eps, weight_decay;
} oracle_hparams;

/* Every scalar the per-element update uses, plus the step's bookkeeping. */
typedef struct {
  int32_t overflow;   /* any non-finite summed gradient among the real elements   */
  int32_t skipped;    /* step not applied (== overflow)                           */
  int64_t step;       /* step counter after this call (t+1, or t when skipped)    */
  double ss;          /* exact sum of squares of the summed (scaled) gradients,   */
                      /* rounded once to double                                   */
  double norm;        /* sqrt(ss) / loss_scale, +inf on overflow                  */
  double clip_coef;   /* min(1, clip / (norm + 1e-6)); 1 when clip <= 0           */
  float s;            /* clip_coef / loss_scale rounded to fp32                   */
  float omb1, omb2;   /* 1 - beta1, 1 - beta2 rounded to fp32                     */
  float bc1, bc2;     /* 1 - beta^t' rounded to fp32                              */
  float decay;        /* 1 - lr * weight_decay rounded to fp32                    */
  float lr, beta1, beta2, eps;
} oracle_scalars;

/* Partition: Np = ceil(N / (Nd*align)) * Nd * align, S = Np / Nd. Returns 0, or -1 on
 * N < 1, Nd < 1 or align < 1. */
int oracle_partition(int64_t n, int32_t nd, int32_t align, int64_t* padded, int64_t* shard);

/* Per-rank model-state bytes for stage 0 (plain data parallel), 1, 2 or 3 under the
 * 2 + 2 + 12 bytes-per-parameter audit, counting the padded shard. -1 on bad input. */
int64_t oracle_memory_bytes(int64_t n, int32_t nd, int32_t align, int32_t stage);

/* fp16 <-> fp32 from the IEEE 754 binary16 definition. */
float oracle_f16_to_f32(uint16_t h);
uint16_t oracle_f32_to_f16(float x);
void oracle_f32_to_f16_array(const float* x, uint16_t* out, int64_t n);
void oracle_f16_to_f32_array(const uint16_t* h, float* out, int64_t n);

/* Reduce: gsum[i] = (((0 + c_0[i]) + c_1[i]) + ... + c_{nd-1}[i]) in fp32 for
 * i < n_valid, and 0 for n_valid <= i < n (padding). */
void oracle_reduce(int32_t nd, const uint16_t* const* contrib, int64_t n, int64_t n_valid,
                   float* gsum);

/* Statistics of gsum[0 .. n): count of non-finite values, and the exact sum of
 * (gsum[i] * 2^24)^2 over the finite values as an unsigned 128-bit integer split into
 * (lo, hi) 64-bit halves. Returns -1 if the sum would not fit in 128 bits. */
int oracle_stats(const float* gsum, int64_t n, int64_t* nonfinite, uint64_t* ss_lo,
                 uint64_t* ss_hi);

/* Scalars of one step from the span's statistics and the step counter t before it. */
void oracle_scalars_from_stats(int64_t nonfinite, uint64_t ss_lo, uint64_t ss_hi,
                               float loss_scale, float clip, const oracle_hparams* hp,
                               int64_t t, oracle_scalars* out);

/* AdamW update and fp16 cast of n elements given the step's scalars. Does nothing when
 * sc->skipped. */
void oracle_adam(int64_t n, const float* gsum, float* master, float* exp_avg,
                 float* exp_avg_sq, uint16_t* param16, const oracle_scalars* sc);

/* The whole shard step over one span of n elements whose first n_valid are real
 * parameters: reduce, statistics, scalars, update. gsum_work holds n floats. */
void oracle_step(int32_t nd, const uint16_t* const* contrib, int64_t n, int64_t n_valid,
                 float* master, float* exp_avg, float* exp_avg_sq, uint16_t* param16,
                 float* gsum_work, float loss_scale, float clip, const oracle_hparams* hp,
                 int64_t t, oracle_scalars* out);

/* Dynamic loss scaling after a step (mixed-precision practice; the pages name mixed
 * precision but no scaler): on overflow the scale is multiplied by backoff and the count
 * of good steps restarts; otherwise the count grows, and when it reaches interval the
 * scale is multiplied by growth (unless that product is not finite) and the count
 * restarts. fp32 multiplies. */
void oracle_scaler_update(float* scale, int32_t* good_steps, int32_t overflow, float growth,
                          float backoff, int32_t interval);

/* ZeRO-3 parameter gather: dst[l][j] = flat[off[l] + j] for j < off[l+1] - off[l], where
 * flat is the concatenation of the nd shards of shard_len elements each. */
void oracle_gather(int32_t nd, int64_t shard_len, const uint16_t* const* shards,
                   int32_t n_layers, const int64_t* layer_offsets, uint16_t* const* dst);

/* Which shard, and which element of it, holds flat index i. */
void oracle_gather_source(int64_t shard_len, int64_t i, int32_t* rank, int64_t* offset);

#ifdef __cplusplus
}
#endif
#endif
