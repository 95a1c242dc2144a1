/* Oracle for the ZeRO shard step. TEST INFRASTRUCTURE ONLY (see oracle.h): plain,
 * slow, single-threaded C that states what the step computes, for the tests and the
 * bench's CPU baseline. Nothing in the product library uses it.
 *
 * Build: cc -O2 -ffp-contract=off -fno-fast-math -shared -fPIC oracle.c -lm
 */
#include "oracle.h"

#include <math.h>
#include <stddef.h>

typedef unsigned __int128 u128;

/* ---------------------------------------------------------------------------------
 * Partition. ZeRO partitions the model states across the Nd data-parallel ranks
 * instead of replicating them ("ZeRO" method entry, description; ZeRO explainer,
 * "The 16 Bytes per Parameter Audit": "partition it"). The flat buffer of N
 * parameters is padded to a multiple of Nd * align so that each of the Nd equal
 * shards starts on an aligned element; shard r is [r*S, (r+1)*S).
 */
int oracle_partition(int64_t n, int32_t nd, int32_t align, int64_t* padded, int64_t* shard) {
  if (n < 1 || nd < 1 || align < 1) return -1;
  int64_t unit = (int64_t)nd * (int64_t)align;
  int64_t units = n / unit;
  if (units * unit < n) units += 1; /* ceiling */
  *padded = units * unit;
  *shard = *padded / nd;
  return 0;
}

/* ---------------------------------------------------------------------------------
 * Memory accounting. ZeRO explainer, "The 16 Bytes per Parameter Audit" and Chapter 02
 * "Memory per parameter": fp16 weight 2 B, fp32 master 4 B, Adam momentum and variance
 * 8 B, and the gradient. The audit's own sum is garbled (it names 2+4+8 and then
 * "2+4" more, and the chapter says 16-20 B). The reading taken: 16 B = 2 (fp16 weight)
 * + 2 (fp16 gradient) + 12 (K = fp32 master, momentum, variance); the fp32 gradient
 * copy is a transient workspace, not model state. This is the split under which the
 * stage table's ~4x and ~8x reductions hold as Nd grows.
 * Stages (Chapter 02 "What each stage shards" and the stage table):
 *   0 plain data parallel: everything replicated      -> 16 N
 *   1 optimizer states partitioned                    -> 4 N + 12 S
 *   2 + gradients partitioned                         -> 2 N + 14 S
 *   3 + parameters partitioned                        -> 16 S
 * with S the padded shard length.
 */
int64_t oracle_memory_bytes(int64_t n, int32_t nd, int32_t align, int32_t stage) {
  int64_t np, s;
  if (oracle_partition(n, nd, align, &np, &s) != 0) return -1;
  switch (stage) {
    case 0: return 16 * n;
    case 1: return 4 * n + 12 * s;
    case 2: return 2 * n + 14 * s;
    case 3: return 16 * s;
    default: return -1;
  }
}

/* ---------------------------------------------------------------------------------
 * fp16 <-> fp32, from the IEEE 754 binary16 layout: 1 sign bit, 5 exponent bits (bias
 * 15), 10 fraction bits.
 */
float oracle_f16_to_f32(uint16_t h) {
  int sign = (h >> 15) & 1;
  int exp = (h >> 10) & 0x1f;
  int frac = h & 0x3ff;
  float v;
  if (exp == 0) {
    v = ldexpf((float)frac, -24); /* subnormal: frac * 2^-24 (exact) */
  } else if (exp == 31) {
    v = frac == 0 ? INFINITY : NAN;
  } else {
    v = ldexpf((float)(1024 + frac), exp - 25); /* (1.frac) * 2^(exp-15) */
  }
  return sign ? -v : v;
}

/* Round to nearest, ties to even. Values at or above 65520 (halfway between the largest
 * finite fp16, 65504, and 65536) round to infinity. */
uint16_t oracle_f32_to_f16(float x) {
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  if (isnan(x)) return sign | 0x7e00;
  float a = fabsf(x);
  if (a >= 65520.0f) return sign | 0x7c00;
  if (a < 0x1p-14f) {
    /* subnormal range: the result is q * 2^-24 with q an integer in [0, 1024]. */
    float q = rintf(a * 0x1p24f); /* exact scaling, then nearest-even to an integer */
    return sign | (uint16_t)q;    /* q == 1024 encodes 2^-14, the smallest normal */
  }
  int e2;
  frexpf(a, &e2); /* a = f * 2^e2, f in [0.5, 1) */
  int e = e2 - 1; /* a in [2^e, 2^(e+1)), e in [-14, 15] */
  float q = rintf(ldexpf(a, 10 - e)); /* 11-bit significand, nearest-even */
  if (q == 2048.0f) {
    q = 1024.0f;
    e += 1;
  }
  return sign | (uint16_t)((e + 15) << 10) | (uint16_t)((int)q - 1024);
}

void oracle_f32_to_f16_array(const float* x, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_f16(x[i]);
}

void oracle_f16_to_f32_array(const uint16_t* h, float* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_f16_to_f32(h[i]);
}

/* A table of all 65536 conversions, filled from oracle_f16_to_f32, so that the large
 * reductions below run at a usable speed. */
static float g_f16_table[65536];
static int g_f16_table_ready = 0;

static void ensure_table(void) {
  if (g_f16_table_ready) return;
  for (int i = 0; i < 65536; ++i) g_f16_table[i] = oracle_f16_to_f32((uint16_t)i);
  g_f16_table_ready = 1;
}

/* ---------------------------------------------------------------------------------
 * Reduce: the arithmetic of the reduce-scatter ("reduce-scatter after backward",
 * ZeRO explainer, Chapter 02 "What each stage shards", ZeRO-3 item, and the stage
 * table). Each of the Nd ranks holds an fp16 gradient for the whole flat buffer; the
 * owner of a partition receives their sum. The sum is taken in fp32, in rank order
 * 0..Nd-1, starting from +0, one IEEE add per rank. It is a sum, not a mean: the loss
 * scale passed to the step unscales it, and a caller who wants a mean passes Nd times
 * the loss scale. Padding elements (flat index >= N) are not parameters; they sum to 0.
 */
void oracle_reduce(int32_t nd, const uint16_t* const* contrib, int64_t n, int64_t n_valid,
                   float* gsum) {
  ensure_table();
  for (int64_t i = 0; i < n; ++i) {
    float acc = 0.0f;
    if (i < n_valid) {
      for (int32_t r = 0; r < nd; ++r) acc = acc + g_f16_table[contrib[r][i]];
    }
    gsum[i] = acc;
  }
}

/* ---------------------------------------------------------------------------------
 * Overflow flag and sum of squares. Mixed precision (ZeRO explainer, "The mixed-
 * precision era": Adam + FP16) needs an inf/nan check on the gradients, and global-norm
 * clipping needs sum_i gsum[i]^2 over the span.
 *
 * The sum of squares is taken exactly. Every fp16 value is an integer multiple of 2^-24
 * (the smallest subnormal), and so is every fp32 sum of such values (a value below 1 is
 * exact in fp32, and above 1 the fp32 ulp is itself a multiple of 2^-24). So
 * k = gsum * 2^24 is an exact integer, |k| < Nd * 65504 * 2^24 * (1 + 2^-20), and k^2 is
 * an exact integer that the 128-bit sum holds while n * Nd^2 < 2^47. The result is
 * rounded to double once, afterwards, so it does not depend on the order of summation.
 */
int oracle_stats(const float* gsum, int64_t n, int64_t* nonfinite, uint64_t* ss_lo,
                 uint64_t* ss_hi) {
  int64_t bad = 0;
  u128 acc = 0;
  int overflow128 = 0;
  for (int64_t i = 0; i < n; ++i) {
    float g = gsum[i];
    if (!isfinite(g)) {
      bad += 1;
      continue;
    }
    int64_t k = (int64_t)(g * 0x1p24f); /* exact integer; the cast does not round */
    uint64_t a = (uint64_t)(k < 0 ? -k : k);
    u128 sq = (u128)a * (u128)a;
    u128 next = acc + sq;
    if (next < acc) overflow128 = 1;
    acc = next;
  }
  *nonfinite = bad;
  *ss_lo = (uint64_t)acc;
  *ss_hi = (uint64_t)(acc >> 64);
  return overflow128 ? -1 : 0;
}

/* ---------------------------------------------------------------------------------
 * Scalars of the step. The pages name mixed-precision Adam without its formulas, so
 * these are the textbook ones (Adam with bias correction, weight decay decoupled as in
 * AdamW and applied before the Adam term, and global-norm clipping with the same
 * coefficient as torch.nn.utils.clip_grad_norm_), computed in double from the fp32
 * hyperparameters and rounded once to fp32:
 *   norm  = sqrt(ss) / loss_scale       (norm of the unscaled summed gradient)
 *   coef  = clip / (norm + 1e-6) when clip > 0 and that is below 1, else 1
 *   s     = coef / loss_scale           (one factor: unscale and clip)
 *   bc1   = 1 - beta1^t', bc2 = 1 - beta2^t', with t' = t + 1
 *   decay = 1 - lr * weight_decay
 * On overflow the step is skipped: nothing is written and t stays.
 */
void oracle_scalars_from_stats(int64_t nonfinite, uint64_t ss_lo, uint64_t ss_hi,
                               float loss_scale, float clip, const oracle_hparams* hp,
                               int64_t t, oracle_scalars* out) {
  u128 acc = ((u128)ss_hi << 64) | (u128)ss_lo;
  out->lr = hp->lr;
  out->beta1 = hp->beta1;
  out->beta2 = hp->beta2;
  out->eps = hp->eps;
  out->ss = (double)acc * 0x1p-48; /* (k * 2^-24)^2 = k^2 * 2^-48; scaling is exact */
  out->overflow = nonfinite > 0;
  out->skipped = out->overflow;
  if (out->overflow) {
    out->norm = INFINITY;
    out->clip_coef = 1.0;
    out->step = t;
  } else {
    out->norm = sqrt(out->ss) / (double)loss_scale;
    double coef = 1.0;
    if (clip > 0.0f) {
      double c = (double)clip / (out->norm + 1e-6);
      if (c < 1.0) coef = c;
    }
    out->clip_coef = coef;
    out->step = t + 1;
  }
  double tp = (double)(t + 1);
  out->s = (float)(out->clip_coef / (double)loss_scale);
  out->omb1 = (float)(1.0 - (double)hp->beta1);
  out->omb2 = (float)(1.0 - (double)hp->beta2);
  out->bc1 = (float)(1.0 - pow((double)hp->beta1, tp));
  out->bc2 = (float)(1.0 - pow((double)hp->beta2, tp));
  out->decay = (float)(1.0 - (double)hp->lr * (double)hp->weight_decay);
}

/* ---------------------------------------------------------------------------------
 * The AdamW update of one partition (ZeRO explainer, Chapter 02 "Memory per parameter":
 * fp32 master weight, Adam momentum and variance are the optimizer state each rank
 * keeps for its own partition; the fp16 weight is what it hands back). Per element, in
 * fp32, one IEEE operation at a time:
 *   g  = gsum * s
 *   m  = beta1 * m + (1 - beta1) * g
 *   v  = beta2 * v + (1 - beta2) * (g * g)
 *   mh = m / bc1,  vh = v / bc2
 *   u  = mh / (sqrt(vh) + eps)
 *   p  = master * decay - lr * u
 *   master = p,  param16 = fp16(p)
 */
void oracle_adam(int64_t n, const float* gsum, float* master, float* exp_avg,
                 float* exp_avg_sq, uint16_t* param16, const oracle_scalars* sc) {
  if (sc->skipped) return;
  for (int64_t i = 0; i < n; ++i) {
    float g = gsum[i] * sc->s;
    float m = sc->beta1 * exp_avg[i] + sc->omb1 * g;
    float v = sc->beta2 * exp_avg_sq[i] + sc->omb2 * (g * g);
    float mh = m / sc->bc1;
    float vh = v / sc->bc2;
    float u = mh / (sqrtf(vh) + sc->eps);
    float p = master[i] * sc->decay;
    p = p - sc->lr * u;
    exp_avg[i] = m;
    exp_avg_sq[i] = v;
    master[i] = p;
    param16[i] = oracle_f32_to_f16(p);
  }
}

void oracle_step(int32_t nd, const uint16_t* const* contrib, int64_t n, int64_t n_valid,
                 float* master, float* exp_avg, float* exp_avg_sq, uint16_t* param16,
                 float* gsum_work, float loss_scale, float clip, const oracle_hparams* hp,
                 int64_t t, oracle_scalars* out) {
  int64_t bad;
  uint64_t lo, hi;
  if (n_valid > n) n_valid = n;
  if (n_valid < 0) n_valid = 0;
  oracle_reduce(nd, contrib, n, n_valid, gsum_work);
  oracle_stats(gsum_work, n_valid, &bad, &lo, &hi);
  oracle_scalars_from_stats(bad, lo, hi, loss_scale, clip, hp, t, out);
  oracle_adam(n_valid, gsum_work, master, exp_avg, exp_avg_sq, param16, out);
}

/* ---------------------------------------------------------------------------------
 * Dynamic loss scale. The pages say only "mixed precision"; the scaler is the usual
 * companion of a skipped overflow step: back off on overflow, grow after a run of good
 * steps.
 */
void oracle_scaler_update(float* scale, int32_t* good_steps, int32_t overflow, float growth,
                          float backoff, int32_t interval) {
  if (overflow) {
    *scale = *scale * backoff;
    *good_steps = 0;
    return;
  }
  int32_t good = *good_steps + 1;
  if (good >= interval) {
    float grown = *scale * growth;
    if (isfinite(grown)) *scale = grown;
    good = 0;
  }
  *good_steps = good;
}

/* ---------------------------------------------------------------------------------
 * ZeRO-3 parameter gather: the arithmetic of the all-gather before forward (ZeRO
 * explainer, Chapter 02, ZeRO-3 item). The fp16 shards concatenate to the flat buffer;
 * layer l is the slice [off[l], off[l+1]) of it, copied to its own contiguous buffer.
 */
void oracle_gather_source(int64_t shard_len, int64_t i, int32_t* rank, int64_t* offset) {
  *rank = (int32_t)(i / shard_len);
  *offset = i - (int64_t)(*rank) * shard_len;
}

void oracle_gather(int32_t nd, int64_t shard_len, const uint16_t* const* shards,
                   int32_t n_layers, const int64_t* layer_offsets, uint16_t* const* dst) {
  (void)nd;
  for (int32_t l = 0; l < n_layers; ++l) {
    int64_t len = layer_offsets[l + 1] - layer_offsets[l];
    for (int64_t j = 0; j < len; ++j) {
      int32_t r;
      int64_t off;
      oracle_gather_source(shard_len, layer_offsets[l] + j, &r, &off);
      dst[l][j] = shards[r][off];
    }
  }
}
