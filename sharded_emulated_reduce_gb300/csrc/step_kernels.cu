// Kernels of the ZeRO shard step on sm_103a: the rank-order reduce with the overflow flag
// and the exact sum of squares, the finalize of the step's scalars, and the fused
// unscale + clip + AdamW + fp16-cast update.
//
// The step is two passes over the span because clipping and the overflow skip need
// the global norm and flag before any state is written:
//   reduce:  reads the nd fp16 contributions (2*nd B/param), writes the fp32 sum to the
//            workspace (4 B/param), and leaves one 128-bit sum of squares and one
//            non-finite count per CTA; the last CTA to finish combines them.
//   update:  reads the sum and the fp32 master/m/v (16 B/param), writes master/m/v and
//            the fp16 parameter (14 B/param).
// For more than 8 ranks the reduce (k_reduce_bulk) stages the contribution streams through
// a shared-memory ring with the TMA engine's 1-D bulk copies, a producer warp claiming
// tiles and 8 consumer warps summing them; for 8 ranks or fewer (k_reduce) it is a
// persistent grid-stride loop over groups of 8 elements, one 16-byte vector per rank per
// thread, coalesced across the warp. The update streams tiles through shared memory with
// bulk copies too (see k_update).
//
// The combine's scalars that depend only on the step counter (the bias corrections'
// double-precision powers, slow on this part) are prepared one step ahead in a tagged
// slot: by a spare CTA of the reduce when the span needs less than one wave, otherwise
// by k_next_scalars, which the host runs on a second stream beside the update.
//
// Exactness: each summed gradient gsum is an integer multiple of 2^-24 (fp16 values
// are, and an fp32 sum of them stays one), so k = gsum * 2^24 is an exact integer and
// the sum of k^2 is carried exactly in 128 bits. The norm therefore does not depend on
// the grid, the CTA order or the warp shuffle order, and it is rounded once.
// Every fp32 operation of the update is an explicit round-to-nearest intrinsic (no
// contraction), so the result is the same bits as a sequential IEEE evaluation.
#include <cuda_fp16.h>
#include <math.h>

#include <atomic>

#include "bounds.h"
#include "bulk_async.h"
#include "grid_sync.h"
#include "internal.h"

namespace zero {
namespace {

struct U128 {
  unsigned long long lo, hi;
};

__device__ __forceinline__ void add128(U128& a, unsigned long long lo, unsigned long long hi) {
  const unsigned long long l = a.lo + lo;
  a.hi += hi + (l < lo ? 1ull : 0ull);
  a.lo = l;
}

__device__ __forceinline__ bool is_finite(float x) {
  return (__float_as_uint(x) & 0x7f800000u) != 0x7f800000u;
}

// (gsum * 2^24)^2 added to a 128-bit accumulator; the caller masks non-finite values.
__device__ __forceinline__ void add_square(U128& a, float g) {
  const long long k = __float2ll_rn(__fmul_rn(g, 16777216.0f));
  const unsigned long long u = (unsigned long long)(k < 0 ? -k : k);
  add128(a, u * u, __umul64hi(u, u));
}

// acc0 += fp16 low half of w, acc1 += fp16 high half, each one fp32 add rounded to
// nearest (sm_100+ mixed-precision add: the fp16 operand is widened exactly).
__device__ __forceinline__ void add_f16x2(float& acc0, float& acc1, unsigned w) {
  asm("{\n\t.reg .f16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "add.rn.f32.f16 %0, l, %0;\n\tadd.rn.f32.f16 %1, h, %1;\n\t}"
      : "+f"(acc0), "+f"(acc1)
      : "r"(w));
}

__device__ __forceinline__ void add_vec(float (&s)[8], const uint4& w) {
  add_f16x2(s[0], s[1], w.x);
  add_f16x2(s[2], s[3], w.y);
  add_f16x2(s[4], s[5], w.z);
  add_f16x2(s[6], s[7], w.w);
}

// Correctly rounded conversion of an unsigned 128-bit integer to double.
__device__ double u128_to_double(U128 a) {
  if (a.hi == 0) return __ull2double_rn(a.lo);
  const int lz = __clzll((long long)a.hi);
  const int shift = 64 - lz;  // 1..64 bits below the top 64
  unsigned long long top, sticky;
  if (shift == 64) {
    top = a.hi;
    sticky = a.lo;
  } else {
    top = (a.hi << lz) | (a.lo >> shift);
    sticky = a.lo << lz;
  }
  // bit 0 of top lies below the 53-bit significand's rounding bit, so or-ing the
  // dropped bits into it preserves round-to-nearest-even
  top |= (sticky != 0) ? 1ull : 0ull;
  // times 2^shift (1..64): an exact scaling by a power of two, as one multiply
  return __dmul_rn(__ull2double_rn(top), __longlong_as_double((long long)(1023 + shift) << 52));
}

// The scalars that depend only on t and the hyperparameters: double arithmetic, each
// operation rounded to nearest, then one rounding to fp32. The two powers dominate the
// cost (double precision is slow on this part).
__device__ __forceinline__ DevPre pre_scalars(long long t, const HostHParams& hp) {
  DevPre p;
  const double tp = (double)(t + 1);
  p.omb1 = __double2float_rn(__dadd_rn(1.0, -(double)hp.beta1));
  p.omb2 = __double2float_rn(__dadd_rn(1.0, -(double)hp.beta2));
  p.bc1 = __double2float_rn(__dadd_rn(1.0, -pow((double)hp.beta1, tp)));
  p.bc2 = __double2float_rn(__dadd_rn(1.0, -pow((double)hp.beta2, tp)));
  p.decay = __double2float_rn(__dadd_rn(1.0, -__dmul_rn((double)hp.lr, (double)hp.weight_decay)));
  p.lr = hp.lr;
  p.beta1 = hp.beta1;
  p.beta2 = hp.beta2;
  p.weight_decay = hp.weight_decay;
  p.valid = kPreValid;
  p.t = t;
  return p;
}

// The same, as a call (kept out of line where it would crowd a hot kernel's registers).
__device__ __noinline__ DevPre pre_scalars_call(long long t, const HostHParams& hp) {
  return pre_scalars(t, hp);
}

// The same with the two powers computed side by side, by lanes 0 and 1 of the calling
// warp, in about half the time of one after the other (every lane calls it; the result
// is valid in lane 0).
__device__ __noinline__ DevPre pre_scalars_warp(long long t, const HostHParams& hp) {
  const int lane = threadIdx.x & 31;
  const double tp = (double)(t + 1);
  const double pw = pow(lane == 1 ? (double)hp.beta2 : (double)hp.beta1, tp);
  const double pw2 = __shfl_sync(0xffffffffu, pw, 1);
  DevPre p;
  p.omb1 = __double2float_rn(__dadd_rn(1.0, -(double)hp.beta1));
  p.omb2 = __double2float_rn(__dadd_rn(1.0, -(double)hp.beta2));
  p.bc1 = __double2float_rn(__dadd_rn(1.0, -pw));
  p.bc2 = __double2float_rn(__dadd_rn(1.0, -pw2));
  p.decay = __double2float_rn(__dadd_rn(1.0, -__dmul_rn((double)hp.lr, (double)hp.weight_decay)));
  p.lr = hp.lr;
  p.beta1 = hp.beta1;
  p.beta2 = hp.beta2;
  p.weight_decay = hp.weight_decay;
  p.valid = kPreValid;
  p.t = t;
  return p;
}

static_assert(sizeof(DevPre) == 48, "a slot is three 16-byte vectors");

// Slot `p` read through L2 in one round trip (three independent 16-byte loads).
__device__ __forceinline__ DevPre load_pre(const DevPre* p) {
  const int4* q = reinterpret_cast<const int4*>(p);
  const int4 w0 = __ldcg(q), w1 = __ldcg(q + 1), w2 = __ldcg(q + 2);
  DevPre r;
  int4* o = reinterpret_cast<int4*>(&r);
  o[0] = w0;
  o[1] = w1;
  o[2] = w2;
  return r;
}

// Whether a slot holds the t-only scalars of step counter t under hp.
__device__ __forceinline__ bool pre_matches(const DevPre& p, long long t, const HostHParams& hp) {
  return p.valid == kPreValid && p.t == t && p.lr == hp.lr && p.beta1 == hp.beta1 &&
         p.beta2 == hp.beta2 && p.weight_decay == hp.weight_decay;
}

// The t-only scalars of step counter t into slot t & 1, unless the slot holds them
// already; every lane of the calling warp calls it (the two powers run side by side).
__device__ __forceinline__ void fill_pre_slot(DevScratch* st, long long t, const HostHParams& hp) {
  DevPre* slot = &st->pre[t & 1];
  if (__shfl_sync(0xffffffffu, pre_matches(load_pre(slot), t, hp) ? 1 : 0, 0)) return;
  const DevPre p = pre_scalars_warp(t, hp);
  if ((threadIdx.x & 31) == 0) *slot = p;
}

// The t-only scalars for step counter t: from slot t & 1 when its tag matches, otherwise
// computed here, inline with INLINE (the full-wave reduce, whose code generation is tuned
// with it) or as a call.
template <bool INLINE>
__device__ __forceinline__ DevPre t_scalars(const DevScratch* st, long long t,
                                            const HostHParams& hp) {
  DevPre pre = load_pre(&st->pre[t & 1]);
  if (pre_matches(pre, t, hp)) {
    // the slot's values
  } else if constexpr (INLINE) {
    pre = pre_scalars(t, hp);
  } else {
    pre = pre_scalars_call(t, hp);
  }
  return pre;
}

// x / L, rounded to nearest, for the fp32 loss scale L > 0. When L is a power of two
// (as loss scales are in practice) this is the multiplication by the exact double 1 / L:
// both round the same real number once, so the result is the same double, and a double
// division is a long dependent sequence on this part.
__device__ __forceinline__ double div_by_loss_scale(double x, float L) {
  const unsigned b = __float_as_uint(L);
  const unsigned e = (b >> 23) & 0xffu;
  if ((b & 0x007fffffu) == 0u && e != 0u && e != 0xffu) {
    const long long inv = (long long)(1023 + 127 - (int)e) << 52;  // 2^(127 - e)
    return __dmul_rn(x, __longlong_as_double(inv));
  }
  return __ddiv_rn(x, (double)L);
}

// The step's scalars from its statistics (one thread), writing nothing: t and `scaler`
// are the step counter and loss scaler before the step, *next the scaler after it.
// Double arithmetic, each operation rounded to nearest, then one rounding to fp32. With
// REPORT false only what the update reads is exact: the sum of squares and the norm (a
// square root, and a long dependent chain of double operations on this part) are then
// computed only when clipping needs them, and are 0 otherwise.
template <bool REPORT = true>
__device__ __forceinline__ DevScalars make_scalars(long long t, DevScaler scaler, long long bad,
                                                   U128 ss, float loss_scale_arg, float clip,
                                                   const HostHParams& hp, const DevPre& pre,
                                                   DevScaler* next) {
  DevScalars sc;
  // with the dynamic scaler on, the gradients carry the device-resident scale
  const bool dynamic = scaler.interval > 0;
  const float loss_scale = dynamic ? scaler.scale : loss_scale_arg;
  sc.loss_scale = loss_scale;
  sc.pad2 = 0.0f;
  sc.pad = 0;
  sc.status = 0;
  sc.overflow = bad > 0 ? 1 : 0;
  sc.skipped = sc.overflow;
  const bool norm_needed = REPORT || (!sc.overflow && clip > 0.0f);
  sc.ss = norm_needed ? __dmul_rn(u128_to_double(ss), 0x1p-48) : 0.0;
  if (sc.overflow) {
    sc.norm = __longlong_as_double(0x7ff0000000000000ll);  // +inf
    sc.clip_coef = 1.0;
    sc.step = t;
  } else {
    sc.norm = norm_needed ? div_by_loss_scale(__dsqrt_rn(sc.ss), loss_scale) : 0.0;
    double coef = 1.0;
    if (clip > 0.0f) {
      const double c = __ddiv_rn((double)clip, __dadd_rn(sc.norm, 1e-6));
      if (c < 1.0) coef = c;
    }
    sc.clip_coef = coef;
    sc.step = t + 1;
  }
  sc.s = __double2float_rn(div_by_loss_scale(sc.clip_coef, loss_scale));
  sc.omb1 = pre.omb1;
  sc.omb2 = pre.omb2;
  sc.bc1 = pre.bc1;
  sc.bc2 = pre.bc2;
  sc.decay = pre.decay;
  sc.lr = hp.lr;
  sc.beta1 = hp.beta1;
  sc.beta2 = hp.beta2;
  sc.eps = hp.eps;
  if (dynamic) {
    // back off on overflow; grow after `interval` consecutive applied steps
    if (sc.overflow) {
      scaler.scale = __fmul_rn(scaler.scale, scaler.backoff);
      scaler.good_steps = 0;
    } else {
      int good = scaler.good_steps + 1;
      if (good >= scaler.interval) {
        const float grown = __fmul_rn(scaler.scale, scaler.growth);
        if (is_finite(grown)) scaler.scale = grown;
        good = 0;
      }
      scaler.good_steps = good;
    }
  }
  *next = scaler;
  return sc;
}

// The step's scalars from its statistics, committed to the scratch (one thread): the
// scalars, the step counter (advanced on an applied step) and the dynamic scaler.
template <bool INLINE>
__device__ void compute_scalars(DevScratch* st, long long bad, U128 ss, float loss_scale_arg,
                                float clip, const HostHParams& hp) {
  const long long t = st->step;
  const DevPre pre = t_scalars<INLINE>(st, t, hp);
  const DevScaler scaler = st->scaler;
  DevScaler next;
  const DevScalars sc = make_scalars(t, scaler, bad, ss, loss_scale_arg, clip, hp, pre, &next);
  st->sc = sc;
  if (!sc.skipped) st->step = t + 1;
  if (scaler.interval > 0) st->scaler = next;
}

__device__ __forceinline__ void bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void bar_arrive(int id, int n) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Sum (acc, bad) over a CTA of NT threads; the result is valid in thread 0.
template <int NT>
__device__ void block_reduce(U128& acc, long long& bad) {
  static_assert(NT % 32 == 0, "whole warps");
  __shared__ unsigned long long s_lo[NT / 32], s_hi[NT / 32];
  __shared__ long long s_bad[NT / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long lo = __shfl_xor_sync(0xffffffffu, acc.lo, o);
    const unsigned long long hi = __shfl_xor_sync(0xffffffffu, acc.hi, o);
    bad += __shfl_xor_sync(0xffffffffu, bad, o);
    add128(acc, lo, hi);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();  // the shared arrays may still be read by a previous call
  if (lane == 0) {
    s_lo[warp] = acc.lo;
    s_hi[warp] = acc.hi;
    s_bad[warp] = bad;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    U128 t{0, 0};
    long long b = 0;
    for (int w = 0; w < NT / 32; ++w) {
      add128(t, s_lo[w], s_hi[w]);
      b += s_bad[w];
    }
    acc = t;
    bad = b;
  }
}

template <int CAP>
struct ReduceArgs {
  const void* g[CAP];  // rank k's contribution for the span
  float* gsum;
  long long n_vec;     // groups of 8 elements in the span
  long long n_valid;   // real parameters in the span
  DevScratch* st;
  float loss_scale, clip;
  HostHParams hp;
  int nd;
  int finalize;
};

// Sum the contributions of group v in rank order. ND > 0 fixes the rank count at
// compile time; ND == 0 reads it from the arguments. Up to 8 ranks all loads are issued
// at once; beyond that they are issued 8 ranks at a time, which keeps the register count
// (and so the number of resident warps) at the level that saturates HBM.
// Group v (8 elements, 16 bytes) of rank r's contribution, streamed (evict-first).
template <int CAP>
__device__ __forceinline__ uint4 load_contribution(const ReduceArgs<CAP>& a, int r, long long v) {
  const uint4* p = reinterpret_cast<const uint4*>(a.g[r]) + v;
  if (!ZERO_IN_BOUNDS(kSiteReduceLoad, p, 16, a.g[r], (size_t)a.n_vec * 16))
    return make_uint4(0u, 0u, 0u, 0u);
  return __ldcs(p);
}

// Group v's fp32 sums into the workspace.
template <int CAP>
__device__ __forceinline__ void store_sums(const ReduceArgs<CAP>& a, long long v,
                                           const float (&s)[8]) {
  float4* o = reinterpret_cast<float4*>(a.gsum) + 2 * v;
  if (!ZERO_IN_BOUNDS(kSiteReduceStore, o, 32, a.gsum, (size_t)a.n_vec * 32)) return;
  o[0] = make_float4(s[0], s[1], s[2], s[3]);
  o[1] = make_float4(s[4], s[5], s[6], s[7]);
}

template <int ND, int CAP>
__device__ __forceinline__ void sum_group(const ReduceArgs<CAP>& a, long long v, float (&s)[8]) {
  if constexpr (ND > 0 && ND <= 8) {
    uint4 w[ND];
#pragma unroll
    for (int r = 0; r < ND; ++r) w[r] = load_contribution(a, r, v);
#pragma unroll
    for (int r = 0; r < ND; ++r) add_vec(s, w[r]);
  } else {
    const int nd = ND > 0 ? ND : a.nd;
#pragma unroll 1
    for (int r0 = 0; r0 < nd; r0 += 8) {
      uint4 w[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (r0 + j < nd) w[j] = load_contribution(a, r0 + j, v);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (r0 + j < nd) add_vec(s, w[j]);
    }
  }
}

// With PRE, CTA 0 has no reduce work: it computes the t-only scalars of the next step
// (counter t + 1) into slot (t + 1) & 1 unless that slot holds them already, and takes
// no part in the combine, which then finds this step's in slot t & 1. The other CTAs
// reduce; the last of them to finish combines their partials.
template <int ND, int CAP, bool PRE>
__global__ void __launch_bounds__(kThreads, (ND >= 32) ? 5 : 0)
    k_reduce(const __grid_constant__ ReduceArgs<CAP> a) {
  DevScratch* st = a.st;
  if constexpr (PRE) {
    if (blockIdx.x == 0) {
      if (threadIdx.x < 32) fill_pre_slot(st, st->step + 1, a.hp);
      return;
    }
  }
  U128 acc{0, 0};
  long long bad = 0;
  const unsigned nred = gridDim.x - (PRE ? 1u : 0u);  // reducing CTAs
  const unsigned b = blockIdx.x - (PRE ? 1u : 0u);
  const long long stride = (long long)nred * kThreads;
  for (long long v = (long long)b * kThreads + threadIdx.x; v < a.n_vec; v += stride) {
    float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    sum_group<ND, CAP>(a, v, s);
    const long long base = v * 8;
    if (base + 8 <= a.n_valid) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const bool fin = is_finite(s[j]);
        bad += fin ? 0 : 1;
        add_square(acc, fin ? s[j] : 0.0f);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (base + j >= a.n_valid) s[j] = 0.0f;  // padding: not a parameter
        const bool fin = is_finite(s[j]);
        bad += fin ? 0 : 1;
        add_square(acc, fin ? s[j] : 0.0f);
      }
    }
    store_sums(a, v, s);
  }

  // CTA partial, then the last CTA to arrive combines all partials (no waiting).
  block_reduce<kThreads>(acc, bad);
  __shared__ int s_last;
  if (threadIdx.x == 0) {
    st->partials[b].lo = acc.lo;
    st->partials[b].hi = acc.hi;
    st->partials[b].bad = bad;
    __threadfence();
    const unsigned prev = atomicAdd(&st->ticket, 1u);
    s_last = prev == nred - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  U128 tot{0, 0};
  long long tb = 0;
  for (int i = threadIdx.x; i < (int)nred; i += kThreads) {
    const DevPartial* p = &st->partials[i];
    add128(tot, __ldcg(&p->lo), __ldcg(&p->hi));
    tb += __ldcg(&p->bad);
  }
  block_reduce<kThreads>(tot, tb);
  if (threadIdx.x == 0) {
    st->stats[0] = tb;
    st->stats[1] = (long long)(tot.lo & 0xffffffffull);
    st->stats[2] = (long long)(tot.lo >> 32);
    st->stats[3] = (long long)(tot.hi & 0xffffffffull);
    st->stats[4] = (long long)(tot.hi >> 32);
    st->stats[5] = st->stats[6] = st->stats[7] = 0;
    if (a.finalize) compute_scalars<!PRE>(st, tb, tot, a.loss_scale, a.clip, a.hp);
    st->ticket = 0;
  }
}

// ---- the bulk-load reduce --------------------------------------------------------------
// The same rank-order sums, statistics and last-CTA combine as k_reduce, with the Nd
// contribution streams staged through shared memory by TMA bulk copies instead of register
// loads. A register-load reduce keeps only its resident warps' loads in flight (about
// 160 KB per SM at Nd = 64, at 61% occupancy); the bulk copies keep five 32 KiB stages in
// flight per SM whatever the registers and occupancy, which is what a pure bulk-copy read
// needs to reach its rate on this part.
//
// One CTA per SM: a producer warp and CONS consumer threads. A tile is TG groups of 8
// elements (TG = CONS when Nd is at least kRanks = 2048 / CONS). Its ranks are taken RC at a
// time (RC = min(Nd, kRanks)), each chunk of RC ranks one 32 KiB stage of a kRbStages-stage
// ring: RC bulk loads of the tile's slice of RC consecutive ranks, rank-major in the stage.
// The producer claims tiles one at a time from the plan's counter, when it needs the next
// one (so CTAs on slower SMs take fewer and no CTA holds a tile it has not started), waits
// until a stage is empty, records the tile in it and issues the loads; after the last tile
// it posts an end mark. Each consumer thread owns groups tid + CONS * j of the tile and
// adds the chunks' ranks in order, so the sums are the same rank-order fp32 additions as
// k_reduce's. The consumers' work per byte (the exact sum of squares per element) is
// latency-bound at few warps, so 8 ranks, whose sums are a fifth of the traffic, use 512
// consumers; more ranks use 256. Every wait is bounded; a CTA whose wait expired publishes a
// non-finite count (the step is then skipped) and a failure flag that the combine turns
// into kStatusReduceWait.
constexpr int kRbStages = 6;
constexpr uint32_t kRbStageBytes = 32768;
constexpr int32_t kStatusReduceWait = 3;

constexpr long long kRbFailBad = 1ll << 40;  // non-finite count a failed CTA publishes
constexpr size_t kRbSmem = (size_t)kRbStages * kRbStageBytes + 2 * kRbStages * sizeof(uint64_t);

// CONS consumer threads take one group each from every rank of a stage: a 32 KiB stage
// then holds kRanks = 2048 / CONS ranks of a tile of CONS groups.
template <int CONS>
struct RbCfg {
  static constexpr int kRanks = 2048 / CONS;
  static constexpr int kThreads = CONS + 32;  // + the producer warp
};

template <int RC, int CONS>
struct RbGeom {
  static constexpr int R = RbCfg<CONS>::kRanks;
  static constexpr int G = (RC >= R) ? 1 : R / RC;           // groups per consumer per tile
  static constexpr long long TG = (long long)CONS * G;       // groups per tile
  static_assert(RC * TG * 16 <= kRbStageBytes, "a chunk fits its stage");
};

// Sum (acc, bad) over the CONS consumer threads (named barrier 1); thread 0 holds the
// result.
template <int CONS>
__device__ void rb_block_reduce(U128& acc, long long& bad) {
  constexpr int W = CONS / 32;
  __shared__ unsigned long long s_lo[W], s_hi[W];
  __shared__ long long s_bad[W];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long lo = __shfl_xor_sync(0xffffffffu, acc.lo, o);
    const unsigned long long hi = __shfl_xor_sync(0xffffffffu, acc.hi, o);
    bad += __shfl_xor_sync(0xffffffffu, bad, o);
    add128(acc, lo, hi);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  bar_sync(1, CONS);  // the shared arrays may still be read by a previous call
  if (lane == 0) {
    s_lo[warp] = acc.lo;
    s_hi[warp] = acc.hi;
    s_bad[warp] = bad;
  }
  bar_sync(1, CONS);
  if (threadIdx.x == 0) {
    U128 t{0, 0};
    long long b = 0;
    for (int w = 0; w < W; ++w) {
      add128(t, s_lo[w], s_hi[w]);
      b += s_bad[w];
    }
    acc = t;
    bad = b;
  }
}

__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(b)) : "memory");
}

// ND > 0: the rank count at compile time (RC = min(ND, kRanks) ranks per stage); ND == 0:
// the count from the arguments, kRanks ranks per stage (the last chunk may hold fewer).
template <int ND, int CAP, bool PRE, int CONS>
__global__ void __launch_bounds__(RbCfg<CONS>::kThreads, 1)
    k_reduce_bulk(const __grid_constant__ ReduceArgs<CAP> a, unsigned long long* next_tile) {
  constexpr int kRbConsumers = CONS;
  constexpr int RC = (ND > 0 && ND < RbCfg<CONS>::kRanks) ? ND : RbCfg<CONS>::kRanks;
  using Geo = RbGeom<RC, CONS>;
  constexpr int G = Geo::G;
  constexpr long long TG = Geo::TG;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)kRbStages * kRbStageBytes);
  uint64_t* empty = full + kRbStages;
  __shared__ long long s_tile[kRbStages];  // the stage's tile, or -1: no more tiles
  __shared__ int s_chunk[kRbStages];       // which chunk of the tile's ranks
  __shared__ int s_fail;
  DevScratch* st = a.st;
  const int tid = threadIdx.x;
  if constexpr (PRE) {
    if (blockIdx.x == 0) {  // no reduce work: the next step's t-only scalars
      if (tid < 32) fill_pre_slot(st, st->step + 1, a.hp);
      return;
    }
  }
  const int nd = ND > 0 ? ND : a.nd;
  const int nchunks = (nd + RC - 1) / RC;
  const long long tiles = (a.n_vec + TG - 1) / TG;
  const unsigned nred = gridDim.x - (PRE ? 1u : 0u);
  const unsigned b = blockIdx.x - (PRE ? 1u : 0u);
  if (tid == 0) {
    for (int s = 0; s < kRbStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kRbConsumers / 32);
    }
    mbar_fence_init();
    s_fail = 0;
  }
  __syncthreads();

  if (tid >= kRbConsumers) {  // the producer warp
    if (tid == kRbConsumers) {
      long long q = 0;  // stages issued
      bool ok = true;
      auto take_stage = [&](int* s_out) {  // the next stage, once its consumers are done
        const int s = (int)(q % kRbStages);
        if (q >= kRbStages &&
            !mbar_wait(&empty[s], (uint32_t)(((q / kRbStages) - 1) & 1))) {
          ok = false;
          return false;
        }
        *s_out = s;
        return true;
      };
      for (;;) {
        const long long t = (long long)atomicAdd(next_tile, 1ull);
        if (t >= tiles) break;
        const long long v0 = t * TG;
        const long long nv = a.n_vec - v0 < TG ? a.n_vec - v0 : TG;
        const uint32_t bytes = (uint32_t)(nv * 16);
        for (int k = 0; k < nchunks && ok; ++k) {
          int s;
          if (!take_stage(&s)) break;
          const int r0 = k * RC;
          const int nr = nd - r0 < RC ? nd - r0 : RC;
          s_tile[s] = t;
          s_chunk[s] = k;
          mbar_expect_tx(&full[s], bytes * (uint32_t)nr);
          unsigned char* dst = smem + (size_t)s * kRbStageBytes;
          for (int j = 0; j < nr; ++j) {
            const unsigned char* src =
                reinterpret_cast<const unsigned char*>(a.g[r0 + j]) + v0 * 16;
            if (ZERO_IN_BOUNDS(kSiteBulkReduceLoad, src, bytes, a.g[r0 + j],
                               (size_t)a.n_vec * 16))
              bulk_load(dst + (size_t)j * TG * 16, src, bytes, &full[s]);
          }
          ++q;
        }
        if (!ok) break;
      }
      int s;
      if (ok && take_stage(&s)) {  // the end mark
        s_tile[s] = -1;
        mbar_arrive(&full[s]);
        ++q;
      }
      if (!ok) {
        atomicExch(&s_fail, 1);
        // let the loads of the last kRbStages issued stages land before the CTA ends
        for (long long k = q > kRbStages ? q - kRbStages : 0; k < q; ++k)
          mbar_wait(&full[(int)(k % kRbStages)], (uint32_t)((k / kRbStages) & 1));
      }
    }
    return;
  }

  // the consumers
  U128 acc{0, 0};
  long long bad = 0;
  float s[G][8];
  long long q = 0;  // stages consumed
  const int lane = tid & 31;
  for (;;) {
    const int si = (int)(q % kRbStages);
    if (!mbar_wait(&full[si], (uint32_t)((q / kRbStages) & 1))) {
      atomicExch(&s_fail, 1);
      break;
    }
    const long long t = s_tile[si];
    if (t < 0) break;
    const int k = s_chunk[si];
    if (k == 0) {
#pragma unroll
      for (int j = 0; j < G; ++j)
#pragma unroll
        for (int e = 0; e < 8; ++e) s[j][e] = 0.0f;
    }
    const int r0 = k * RC;
    const int nr = nd - r0 < RC ? nd - r0 : RC;
    const long long v0 = t * TG;
    const long long nv = a.n_vec - v0 < TG ? a.n_vec - v0 : TG;
    const uint4* w = reinterpret_cast<const uint4*>(smem + (size_t)si * kRbStageBytes);
#pragma unroll
    for (int j = 0; j < G; ++j) {
      const long long g = tid + (long long)kRbConsumers * j;
      if (g < nv) {
        if (ND > 0 && RC == nr) {
#pragma unroll
          for (int r = 0; r < RC; ++r) add_vec(s[j], w[r * TG + g]);
        } else {
          for (int r = 0; r < nr; ++r) add_vec(s[j], w[r * TG + g]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[si]);
    ++q;
    if (k == nchunks - 1) {  // the tile's sums are complete
#pragma unroll
      for (int j = 0; j < G; ++j) {
        const long long g = tid + (long long)kRbConsumers * j;
        if (g >= nv) continue;
        const long long v = v0 + g;
        const long long base = v * 8;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (base + e >= a.n_valid) s[j][e] = 0.0f;  // padding: not a parameter
          const bool fin = is_finite(s[j][e]);
          bad += fin ? 0 : 1;
          add_square(acc, fin ? s[j][e] : 0.0f);
        }
        store_sums(a, v, s[j]);
      }
    }
  }

  // CTA partial, then the last CTA to arrive combines all partials (no waiting)
  rb_block_reduce<CONS>(acc, bad);
  __shared__ int s_last;
  if (tid == 0) {
    const int failed = s_fail;
    st->partials[b].lo = acc.lo;
    st->partials[b].hi = acc.hi;
    st->partials[b].bad = bad + (failed ? kRbFailBad : 0);
    st->partials[b].pad = failed;
    __threadfence();
    const unsigned prev = atomicAdd(&st->ticket, 1u);
    s_last = prev == nred - 1;
  }
  bar_sync(1, kRbConsumers);
  if (!s_last) return;
  __threadfence();
  U128 tot{0, 0};
  long long tb = 0;
  long long tf = 0;
  for (int i = tid; i < (int)nred; i += kRbConsumers) {
    const DevPartial* p = &st->partials[i];
    add128(tot, __ldcg(&p->lo), __ldcg(&p->hi));
    tb += __ldcg(&p->bad);
    tf += __ldcg(&p->pad);
  }
  bad = tb;
  rb_block_reduce<CONS>(tot, bad);
  // the failure flags, summed the same way (their 128-bit part unused)
  U128 dummy{0, 0};
  rb_block_reduce<CONS>(dummy, tf);
  if (tid == 0) {
    st->stats[0] = bad;
    st->stats[1] = (long long)(tot.lo & 0xffffffffull);
    st->stats[2] = (long long)(tot.lo >> 32);
    st->stats[3] = (long long)(tot.hi & 0xffffffffull);
    st->stats[4] = (long long)(tot.hi >> 32);
    st->stats[5] = tf;  // CTAs whose bounded wait expired (0 on a healthy GPU)
    st->stats[6] = st->stats[7] = 0;
    if (a.finalize) {
      compute_scalars<!PRE>(st, bad, tot, a.loss_scale, a.clip, a.hp);
      if (tf != 0) st->sc.status = kStatusReduceWait;
    }
    *next_tile = 0;  // every producer has made its last claim
    st->ticket = 0;
  }
}

// Scalars from the exchange buffer, after the caller's all-reduce (one thread).
__global__ void k_finalize(DevScratch* st, float loss_scale, float clip, HostHParams hp) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  const long long bad = st->stats[0];
  U128 ss{0, 0};
  for (int i = 0; i < 4; ++i) {
    const unsigned long long l = (unsigned long long)st->stats[1 + i];
    switch (i) {
      case 0: add128(ss, l, 0ull); break;
      case 1: add128(ss, l << 32, l >> 32); break;
      case 2: add128(ss, 0ull, l); break;
      default: add128(ss, 0ull, l << 32); break;
    }
  }
  compute_scalars<false>(st, bad, ss, loss_scale, clip, hp);
  if (st->stats[5] != 0) st->sc.status = kStatusReduceWait;  // a reduce CTA's wait expired
}

// The t-only scalars for the counter now in the scratch (the next step's), off the
// step's critical path: launched on a second stream while the update runs.
__global__ void k_next_scalars(DevScratch* st, HostHParams hp) {
  if (blockIdx.x != 0 || threadIdx.x >= 32) return;
  fill_pre_slot(st, st->step, hp);
}

struct UpdateArgs {
  const float* gsum;
  float *master, *m, *v;
  uint16_t* p16;
  long long n_valid;
  DevScratch* st;
};

struct Sc {
  float s, b1, b2, omb1, omb2, bc1, bc2, eps, decay, lr;
};

__device__ __forceinline__ float adam_elem(float gs, float p0, float& m, float& v, const Sc& c) {
  const float g = __fmul_rn(gs, c.s);
  m = __fadd_rn(__fmul_rn(c.b1, m), __fmul_rn(c.omb1, g));
  v = __fadd_rn(__fmul_rn(c.b2, v), __fmul_rn(c.omb2, __fmul_rn(g, g)));
  const float mh = __fdiv_rn(m, c.bc1);
  const float vh = __fdiv_rn(v, c.bc2);
  const float u = __fdiv_rn(mh, __fadd_rn(__fsqrt_rn(vh), c.eps));
  const float p = __fmul_rn(p0, c.decay);
  return __fsub_rn(p, __fmul_rn(c.lr, u));
}

__device__ __forceinline__ unsigned pack_h2(float a, float b) {
  const __half2 h = __halves2half2(__float2half_rn(a), __float2half_rn(b));
  return *reinterpret_cast<const unsigned*>(&h);
}

// ---- the update kernel -------------------------------------------------------------------
// One CTA of 512 threads per SM walks tiles of kUpdTile parameters. For each tile the TMA
// engine brings the fp32 sum and master/m/v into a 3-stage shared-memory ring; the threads
// update 4 parameters each into a double-buffered output area, and one thread sends the
// new master/m/v and fp16 parameters back with bulk stores and refills the freed stage.
// Loads for the next tiles stay in flight while the division-heavy arithmetic runs, so
// the kernel streams at the HBM copy rate. Parameters past the last multiple of 8 (at most
// 7, at the end of the real ones) are updated one by one after the tiles.
constexpr int kUpdTile = 2048;
constexpr int kUpdStages = 3;
constexpr int kUpdThreads = 512;
constexpr size_t kUpdIn = (size_t)kUpdStages * 4 * kUpdTile * sizeof(float);
constexpr size_t kUpdOutF = (size_t)2 * 3 * kUpdTile * sizeof(float);
constexpr size_t kUpdOutH = (size_t)2 * kUpdTile * sizeof(uint16_t);
constexpr size_t kUpdSmem = kUpdIn + kUpdOutF + kUpdOutH + kUpdStages * sizeof(uint64_t);
static_assert(kUpdThreads * 4 == kUpdTile, "each thread updates 4 parameters per tile");
constexpr int32_t kStatusUpdateWait = 2;  // a bulk load did not arrive in time

__global__ void __launch_bounds__(kUpdThreads, 1) k_update(const __grid_constant__ UpdateArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  float* in = reinterpret_cast<float*>(smem);
  float* outf = reinterpret_cast<float*>(smem + kUpdIn);
  uint16_t* outh = reinterpret_cast<uint16_t*>(smem + kUpdIn + kUpdOutF);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kUpdIn + kUpdOutF + kUpdOutH);
  DevScratch* st = a.st;
  const DevScalars* scp = &st->sc;
  if (scp->skipped) return;  // overflow: the state keeps its bits
  Sc c;
  c.s = scp->s;
  c.b1 = scp->beta1;
  c.b2 = scp->beta2;
  c.omb1 = scp->omb1;
  c.omb2 = scp->omb2;
  c.bc1 = scp->bc1;
  c.bc2 = scp->bc2;
  c.eps = scp->eps;
  c.decay = scp->decay;
  c.lr = scp->lr;

  const long long n8 = a.n_valid & ~7ll;  // tiles cover whole groups of 8 (16-byte rule)
  const long long ntiles = (n8 + kUpdTile - 1) / kUpdTile;
  const int tid = threadIdx.x;
  auto tile_of = [&](long long k) { return (long long)blockIdx.x + k * gridDim.x; };
  auto tile_len = [&](long long t) {
    const long long left = n8 - t * kUpdTile;
    return left < kUpdTile ? left : (long long)kUpdTile;
  };
  auto issue = [&](long long k, int s) {  // one thread: load tile k into stage s
    const long long t = tile_of(k);
    const long long base = t * kUpdTile;
    const uint32_t bytes = (uint32_t)(tile_len(t) * sizeof(float));
    float* d = in + (size_t)s * 4 * kUpdTile;
    mbar_expect_tx(&full[s], 4 * bytes);
    const size_t ext = (size_t)a.n_valid * sizeof(float);
    if (ZERO_IN_BOUNDS(kSiteUpdateLoad, a.gsum + base, bytes, a.gsum, ext))
      bulk_load(d, a.gsum + base, bytes, &full[s]);
    if (ZERO_IN_BOUNDS(kSiteUpdateLoad, a.master + base, bytes, a.master, ext))
      bulk_load(d + kUpdTile, a.master + base, bytes, &full[s]);
    if (ZERO_IN_BOUNDS(kSiteUpdateLoad, a.m + base, bytes, a.m, ext))
      bulk_load(d + 2 * kUpdTile, a.m + base, bytes, &full[s]);
    if (ZERO_IN_BOUNDS(kSiteUpdateLoad, a.v + base, bytes, a.v, ext))
      bulk_load(d + 3 * kUpdTile, a.v + base, bytes, &full[s]);
  };

  if (tid == 0) {
    for (int s = 0; s < kUpdStages; ++s) mbar_init(&full[s], 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (tid == 0)
    for (int s = 0; s < kUpdStages; ++s)
      if (tile_of(s) < ntiles) issue(s, s);

  bool ok = true;
  long long k = 0;
  for (; tile_of(k) < ntiles; ++k) {
    const int s = (int)(k % kUpdStages);
    const int ob = (int)(k & 1);
    const long long t = tile_of(k);
    const long long base = t * kUpdTile;
    const long long cnt = tile_len(t);
    const bool arrived = mbar_wait(&full[s], (uint32_t)((k / kUpdStages) & 1));
    if (tid == 0) bulk_wait_read_all_but_one();  // tile k-2's stores have read buffer ob
    if (!__syncthreads_and(arrived)) {
      ok = false;
      break;
    }
    const int j = tid * 4;
    if (j < cnt) {
      const float* d = in + (size_t)s * 4 * kUpdTile;
      const float4 g = *reinterpret_cast<const float4*>(d + j);
      const float4 p = *reinterpret_cast<const float4*>(d + kUpdTile + j);
      float4 m = *reinterpret_cast<const float4*>(d + 2 * kUpdTile + j);
      float4 v = *reinterpret_cast<const float4*>(d + 3 * kUpdTile + j);
      float4 q;
      q.x = adam_elem(g.x, p.x, m.x, v.x, c);
      q.y = adam_elem(g.y, p.y, m.y, v.y, c);
      q.z = adam_elem(g.z, p.z, m.z, v.z, c);
      q.w = adam_elem(g.w, p.w, m.w, v.w, c);
      float* o = outf + (size_t)ob * 3 * kUpdTile;
      *reinterpret_cast<float4*>(o + j) = q;
      *reinterpret_cast<float4*>(o + kUpdTile + j) = m;
      *reinterpret_cast<float4*>(o + 2 * kUpdTile + j) = v;
      *reinterpret_cast<uint2*>(outh + (size_t)ob * kUpdTile + j) =
          make_uint2(pack_h2(q.x, q.y), pack_h2(q.z, q.w));
    }
    fence_to_async_proxy();  // shared-memory writes become visible to the bulk stores
    __syncthreads();         // every thread is done with stage s and buffer ob
    if (tid == 0) {
      const float* o = outf + (size_t)ob * 3 * kUpdTile;
      const uint32_t bytes = (uint32_t)(cnt * sizeof(float));
      const size_t ext = (size_t)a.n_valid * sizeof(float);
      const uint32_t hbytes = (uint32_t)(cnt * sizeof(uint16_t));
      if (ZERO_IN_BOUNDS(kSiteUpdateStore, a.master + base, bytes, a.master, ext))
        bulk_store(a.master + base, o, bytes);
      if (ZERO_IN_BOUNDS(kSiteUpdateStore, a.m + base, bytes, a.m, ext))
        bulk_store(a.m + base, o + kUpdTile, bytes);
      if (ZERO_IN_BOUNDS(kSiteUpdateStore, a.v + base, bytes, a.v, ext))
        bulk_store(a.v + base, o + 2 * kUpdTile, bytes);
      if (ZERO_IN_BOUNDS(kSiteUpdateStore, a.p16 + base, hbytes, a.p16,
                         (size_t)a.n_valid * sizeof(uint16_t)))
        bulk_store(a.p16 + base, outh + (size_t)ob * kUpdTile, hbytes);
      bulk_commit();
      if (tile_of(k + kUpdStages) < ntiles) issue(k + kUpdStages, s);
    }
  }
  if (!ok) {
    if (tid == 0) atomicExch(&st->sc.status, kStatusUpdateWait);
    // let the loads already issued land before this CTA's shared memory is released
    for (long long q = k; q < k + kUpdStages && tile_of(q) < ntiles; ++q)
      mbar_wait(&full[(int)(q % kUpdStages)], (uint32_t)((q / kUpdStages) & 1));
  }
  if (tid == 0) bulk_wait_all();
  const long long rem = a.n_valid - n8;
  if (ok && rem != 0 && blockIdx.x == gridDim.x - 1 && tid == 0) {
    for (long long i = n8; i < a.n_valid; ++i) {
      float m = a.m[i], v = a.v[i];
      const float p = adam_elem(a.gsum[i], a.master[i], m, v, c);
      a.master[i] = p;
      a.m[i] = m;
      a.v[i] = v;
      const __half h = __float2half_rn(p);
      a.p16[i] = *reinterpret_cast<const uint16_t*>(&h);
    }
  }
}

// ---- the fused step for small spans -------------------------------------------------
// A span of at most kWideVecs groups of 8 per SM runs as one cooperative launch (all
// CTAs resident at once), one 512-thread CTA per SM, each owning a contiguous slice:
//   1. the CTA sums its slice of the contributions in rank order into shared memory and
//      adds its 128-bit sum of squares (as four 32-bit limbs) and non-finite count to the
//      launch's counting sums (grid_sync.h);
//   2. warp 0 of every CTA waits until those count every CTA (the grid-wide barrier;
//      bounded: it gives up after about kWaitNs and records kStatusStepWait) and reads
//      the exact totals in the same round trip, so every CTA derives the same scalars;
//   3. unless the step is skipped, the CTA updates its slice from the sums it kept.
// The fp32 sums never go to HBM and the step is one launch. A slice of at most
// kSmallVecs groups also has its master/m/v brought into shared memory by bulk loads
// issued once the CTA has added its statistics, so they arrive while the CTAs wait and
// derive the scalars (DRAM is otherwise idle then); a longer slice reads them from global
// memory in the update. A 17th warp of CTA 0 prepares the next step's t-only
// scalars, then takes the totals from warp 0 (named barrier 2) and commits the step's
// statistics, scalars, step counter and scaler to the scratch while the CTAs update: so
// the update waits for the norm's square root and divisions only when clipping is on
// (the scale the update applies depends on the norm only then). The CTAs' own
// synchronisation uses named barrier 1 over the 512 working threads only.
constexpr int kSmallThreads = 512;
constexpr int kSmallVecs = 1024;  // groups of 8 per CTA whose state is prefetched
constexpr int kWideVecs = 3072;   // groups of 8 per CTA at most (96 KiB of fp32 sums)
constexpr size_t kSmallSlice = (size_t)kSmallVecs * 8 * sizeof(float);  // one fp32 array
// shared memory: sums, master, m, v (kSmallSlice each) and an mbarrier; a slice longer
// than kSmallVecs groups keeps only its sums there (up to kWideVecs groups) and reads
// its state from global memory in the update
constexpr size_t kSmallSmem = 4 * kSmallSlice + 16;
static_assert((size_t)kWideVecs * 8 * sizeof(float) <= 4 * kSmallSlice, "sums fit");
constexpr unsigned kBarrierPolls = 1u << 24;

template <int CAP>
struct SmallArgs {
  ReduceArgs<CAP> r;  // contributions, span sizes, scratch, loss scale, clip, hparams
  float *master, *m, *v;
  uint16_t* p16;
  long long vecs_per_cta;
};

// Sum (acc, bad) over the CTA's kSmallThreads working threads (named barrier 1); the
// result is valid in thread 0.
__device__ void small_block_reduce(U128& acc, long long& bad) {
  constexpr int W = kSmallThreads / 32;
  __shared__ unsigned long long s_lo[W], s_hi[W];
  __shared__ long long s_bad[W];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long lo = __shfl_xor_sync(0xffffffffu, acc.lo, o);
    const unsigned long long hi = __shfl_xor_sync(0xffffffffu, acc.hi, o);
    bad += __shfl_xor_sync(0xffffffffu, bad, o);
    add128(acc, lo, hi);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    s_lo[warp] = acc.lo;
    s_hi[warp] = acc.hi;
    s_bad[warp] = bad;
  }
  bar_sync(1, kSmallThreads);
  if (threadIdx.x == 0) {
    U128 t{0, 0};
    long long b = 0;
    for (int w = 0; w < W; ++w) {
      add128(t, s_lo[w], s_hi[w]);
      b += s_bad[w];
    }
    acc = t;
    bad = b;
  }
}

// The step's statistics, scalars, step counter and loss scaler committed to the scratch
// (one thread of CTA 0, once every CTA has added its statistics): every scalar field
// but the status word, which a CTA whose barrier expired may set.
template <int CAP>
__device__ __noinline__ void commit_small(DevScratch* st, long long t, DevScaler scaler,
                                          DevPre pre, long long tb, U128 tot,
                                          const ReduceArgs<CAP>& r) {
  if (!pre_matches(pre, t, r.hp)) pre = pre_scalars_call(t, r.hp);
  DevScaler next;
  const DevScalars sc = make_scalars(t, scaler, tb, tot, r.loss_scale, r.clip, r.hp, pre, &next);
  st->stats[0] = tb;
  st->stats[1] = (long long)(tot.lo & 0xffffffffull);
  st->stats[2] = (long long)(tot.lo >> 32);
  st->stats[3] = (long long)(tot.hi & 0xffffffffull);
  st->stats[4] = (long long)(tot.hi >> 32);
  st->stats[5] = st->stats[6] = st->stats[7] = 0;
  DevScalars* d = &st->sc;
  d->overflow = sc.overflow;
  d->skipped = sc.skipped;
  d->pad = sc.pad;
  d->step = sc.step;
  d->ss = sc.ss;
  d->norm = sc.norm;
  d->clip_coef = sc.clip_coef;
  d->s = sc.s;
  d->omb1 = sc.omb1;
  d->omb2 = sc.omb2;
  d->bc1 = sc.bc1;
  d->bc2 = sc.bc2;
  d->decay = sc.decay;
  d->lr = sc.lr;
  d->beta1 = sc.beta1;
  d->beta2 = sc.beta2;
  d->eps = sc.eps;
  d->loss_scale = sc.loss_scale;
  d->pad2 = sc.pad2;
  if (!sc.skipped) st->step = t + 1;
  if (scaler.interval > 0) st->scaler = next;
}

template <int ND, int CAP>
__global__ void __launch_bounds__(kSmallThreads + 32, 1)
    k_step_small(const __grid_constant__ SmallArgs<CAP> a) {
  extern __shared__ __align__(128) unsigned char smem[];
  float* sums = reinterpret_cast<float*>(smem);
  float* s_master = reinterpret_cast<float*>(smem + kSmallSlice);
  float* s_m = reinterpret_cast<float*>(smem + 2 * kSmallSlice);
  float* s_v = reinterpret_cast<float*>(smem + 3 * kSmallSlice);
  uint64_t* state_bar = reinterpret_cast<uint64_t*>(smem + 4 * kSmallSlice);
  __shared__ DevScalars s_sc;
  __shared__ long long s_t;
  __shared__ DevScaler s_scaler;
  __shared__ DevPre s_pre;
  __shared__ int s_ok;
  __shared__ U128 s_tot;
  __shared__ long long s_tb;
  __shared__ unsigned long long s_k;  // this launch's number (its counting sums: set s_k & 1)
  DevScratch* st = a.r.st;
  const int tid = threadIdx.x;
  if (tid >= kSmallThreads) {  // the 17th warp
    if (blockIdx.x == 0) {
      // the next step's t-only scalars (for the counter after an applied step), off the
      // critical path: the two powers take about half as long as the rest of the step
      fill_pre_slot(st, st->step + 1, a.r.hp);
      // warp 0 has waited for the counting sums (s_ok) and, if they completed, has the totals
      __syncwarp();
      bar_sync(2, 64);
      if (tid == kSmallThreads && s_ok) commit_small(st, s_t, s_scaler, s_pre, s_tb, s_tot, a.r);
    }
    return;
  }
  // this CTA's slice: groups [v0, v1), real parameters [e0, e1), whole quads up to eq
  const long long v0 = (long long)blockIdx.x * a.vecs_per_cta;
  long long v1 = v0 + a.vecs_per_cta;
  if (v1 > a.r.n_vec) v1 = a.r.n_vec;
  const long long e0 = v0 * 8;
  long long e1 = v1 * 8;
  if (e1 > a.r.n_valid) e1 = a.r.n_valid;
  const long long eq = e1 > e0 ? e0 + (((e1 - e0) >> 2) << 2) : e0;
  const bool prefetch = a.vecs_per_cta <= kSmallVecs;  // the same for every CTA
  const uint32_t state_bytes =
      prefetch ? (uint32_t)((eq - e0) * sizeof(float)) : 0u;  // 16-byte multiple
  if (tid == 0) {
    s_t = st->step;  // before this CTA arrives at the barrier, so before any commit
    s_scaler = st->scaler;
    // this step's t-only scalars, read while the CTA reduces (slot t & 1; this launch
    // writes only slot (t + 1) & 1)
    s_pre = load_pre(&st->pre[s_t & 1]);
    // read before this CTA adds to the counting sums (their address depends on it), so
    // before CTA 0 advances it once every CTA has added
    s_k = st->small_launch;
    if (blockIdx.x == 0) {
      st->sc.status = 0;
      // the next launch's counting sums start from zero (the previous launch, which used
      // them, has ended)
      unsigned long long* next = st->small_sums[(s_k + 1) & 1];
#pragma unroll
      for (int j = 0; j < kSmallWords; ++j) next[j * kSumStride] = 0;
    }
    if (state_bytes > 0) {
      mbar_init(state_bar, 1);
      mbar_fence_init();
    }
  }
  // the slice's state is brought in by bulk loads issued once this CTA has added its
  // statistics (so that they compete neither with the reduce's loads nor with the
  // counting sums' atomics); it arrives while the CTAs wait and derive the scalars
  auto issue_state_loads = [&]() {
    if (tid == 0 && state_bytes > 0) {
      mbar_expect_tx(state_bar, 3 * state_bytes);
      const size_t ext = (size_t)a.r.n_valid * sizeof(float);
      if (ZERO_IN_BOUNDS(kSiteSmallState, a.master + e0, state_bytes, a.master, ext))
        bulk_load(s_master, a.master + e0, state_bytes, state_bar);
      if (ZERO_IN_BOUNDS(kSiteSmallState, a.m + e0, state_bytes, a.m, ext))
        bulk_load(s_m, a.m + e0, state_bytes, state_bar);
      if (ZERO_IN_BOUNDS(kSiteSmallState, a.v + e0, state_bytes, a.v, ext))
        bulk_load(s_v, a.v + e0, state_bytes, state_bar);
    }
  };

  // every exit of thread 0 from here on first lets the state loads land (bounded)
  auto drain = [&]() { if (tid == 0 && state_bytes > 0) mbar_wait(state_bar, 0u); };

  // 1. rank-order sums of this CTA's slice into shared memory, and its statistics
  U128 acc{0, 0};
  long long bad = 0;
  auto finish = [&](long long v, float (&s)[8]) {  // statistics, then the sums to smem
    const long long base = v * 8;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (base + j >= a.r.n_valid) s[j] = 0.0f;  // padding: not a parameter
      const bool fin = is_finite(s[j]);
      bad += fin ? 0 : 1;
      add_square(acc, fin ? s[j] : 0.0f);
    }
    float4* o = reinterpret_cast<float4*>(sums) + 2 * (v - v0);
    o[0] = make_float4(s[0], s[1], s[2], s[3]);
    o[1] = make_float4(s[4], s[5], s[6], s[7]);
  };
  for (long long v = v0 + tid; v < v1; v += kSmallThreads) {
    float s0[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    sum_group<ND, CAP>(a.r, v, s0);
    finish(v, s0);
  }
  small_block_reduce(acc, bad);

  // 2. the CTAs' statistics summed by the counting sums, which are also the grid barrier
  //    (bounded: the wait gives up after about kWaitNs and records kStatusStepWait); every
  //    CTA gets the same exact totals and derives the same scalars for its update
  unsigned long long* counting = st->small_sums[s_k & 1];
  if (tid == 0) {
    const unsigned long long v[kSmallWords] = {acc.lo & 0xffffffffull, acc.lo >> 32,
                                               acc.hi & 0xffffffffull, acc.hi >> 32,
                                               (unsigned long long)bad};
    sum_arrive<kSmallWords>(counting, kSumStride, v);
    issue_state_loads();
  }
  if (tid < 32) {
    unsigned long long w = 0;
    const bool met = sum_wait<kSmallWords>(counting, kSumStride, gridDim.x, kBarrierPolls, &w);
    // met: every CTA has added its partial; lane j holds the sum of word j
    const unsigned long long l0 = __shfl_sync(0xffffffffu, w, 0);
    const unsigned long long l1 = __shfl_sync(0xffffffffu, w, 1);
    const unsigned long long l2 = __shfl_sync(0xffffffffu, w, 2);
    const unsigned long long l3 = __shfl_sync(0xffffffffu, w, 3);
    const long long tb = (long long)__shfl_sync(0xffffffffu, w, 4);
    U128 tot{l0, 0};  // l0 + l1 2^32 + l2 2^64 + l3 2^96 (each limb sum < 2^48)
    add128(tot, l1 << 32, l1 >> 32);
    add128(tot, 0, l2);
    add128(tot, 0, l3 << 32);
    if (tid == 0) s_ok = met ? 1 : 0;
    if (blockIdx.x == 0) {  // the totals to the 17th warp, which commits the step
      if (tid == 0) {
        st->small_launch = s_k + 1;
        s_tot = tot;
        s_tb = tb;
      }
      __syncwarp();
      bar_arrive(2, 64);
    }
    if (met && tid == 0) {  // what the update needs, with the norm only if clipping uses it
      DevPre pre = s_pre;
      if (!pre_matches(pre, s_t, a.r.hp)) pre = pre_scalars_call(s_t, a.r.hp);
      DevScaler next;
      s_sc = make_scalars<false>(s_t, s_scaler, tb, tot, a.r.loss_scale, a.r.clip, a.r.hp, pre,
                                 &next);
    }
  }
  bar_sync(1, kSmallThreads);
  if (!s_ok) {
    if (tid == 0) atomicExch(&st->sc.status, kStatusStepWait);
    drain();
    return;
  }

  // 3. the update of this CTA's slice from the sums and state it holds
  if (s_sc.skipped) {  // overflow: the state keeps its bits
    drain();
    return;
  }
  if (state_bytes > 0 && !mbar_wait(state_bar, 0u)) {
    if (tid == 0) atomicExch(&st->sc.status, kStatusUpdateWait);
    drain();
    return;
  }
  Sc c;
  c.s = s_sc.s;
  c.b1 = s_sc.beta1;
  c.b2 = s_sc.beta2;
  c.omb1 = s_sc.omb1;
  c.omb2 = s_sc.omb2;
  c.bc1 = s_sc.bc1;
  c.bc2 = s_sc.bc2;
  c.eps = s_sc.eps;
  c.decay = s_sc.decay;
  c.lr = s_sc.lr;
  if (e1 <= e0) return;
  float* __restrict__ master = a.master;
  float* __restrict__ mm = a.m;
  float* __restrict__ vv = a.v;
  const long long nq = (eq - e0) >> 2;  // whole quads of parameters
  const float4* g4 = reinterpret_cast<const float4*>(sums);
  // one loop per state source (shared memory or global), so the loop itself has no branch
  auto update = [&](auto load_state) {
    for (long long q = tid; q < nq; q += kSmallThreads) {
      const long long i = e0 + 4 * q;
      // master, m, v and the fp16 parameters share the index: one range test covers them
      if (!ZERO_IN_BOUNDS(kSiteSmallStore, master + i, 16, master,
                          (size_t)a.r.n_valid * sizeof(float)))
        continue;
      const float4 g = g4[q];
      float4 p, m, v;
      load_state(q, i, p, m, v);
      float4 r;
      r.x = adam_elem(g.x, p.x, m.x, v.x, c);
      r.y = adam_elem(g.y, p.y, m.y, v.y, c);
      r.z = adam_elem(g.z, p.z, m.z, v.z, c);
      r.w = adam_elem(g.w, p.w, m.w, v.w, c);
      *reinterpret_cast<float4*>(master + i) = r;
      *reinterpret_cast<float4*>(mm + i) = m;
      *reinterpret_cast<float4*>(vv + i) = v;
      *reinterpret_cast<uint2*>(a.p16 + i) = make_uint2(pack_h2(r.x, r.y), pack_h2(r.z, r.w));
    }
  };
  if (prefetch) {
    update([&](long long q, long long, float4& p, float4& m, float4& v) {
      p = reinterpret_cast<const float4*>(s_master)[q];
      m = reinterpret_cast<const float4*>(s_m)[q];
      v = reinterpret_cast<const float4*>(s_v)[q];
    });
  } else {
    update([&](long long, long long i, float4& p, float4& m, float4& v) {
      p = *reinterpret_cast<const float4*>(master + i);
      m = *reinterpret_cast<const float4*>(mm + i);
      v = *reinterpret_cast<const float4*>(vv + i);
    });
  }
  if (tid < e1 - eq) {  // at most 3 parameters, at the end of the real ones
    const long long i = eq + tid;
    float m = mm[i], v = vv[i];
    const float p = adam_elem(sums[i - e0], master[i], m, v, c);
    master[i] = p;
    mm[i] = m;
    vv[i] = v;
    const __half h = __float2half_rn(p);
    a.p16[i] = *reinterpret_cast<const uint16_t*>(&h);
  }
}

constexpr int kMaxDevices = 64;

// Per-device values below are computed once; several host threads may race to compute
// the same value, so they are relaxed atomics.

// SM count of the current device, looked up once per device.
int sm_count(int* dev_out) {
  static std::atomic<int> sms[kMaxDevices];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev_out) *dev_out = dev;
  int n = 0;
  if (dev >= 0 && dev < kMaxDevices) {
    n = sms[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
  }
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (dev >= 0 && dev < kMaxDevices) sms[dev].store(n, std::memory_order_relaxed);
  return n;
}

// Persistent grid for `kernel`: SMs x resident CTAs per SM, capped by the CTAs the work
// needs. `per_sm` is the caller's per-device cache for this kernel (one static table per
// launcher instantiation, because kernels of the same signature differ in occupancy).
template <typename K>
int occupancy_grid(K kernel, long long work_items, std::atomic<int> (&per_sm)[kMaxDevices],
                   int* resident = nullptr) {
  int dev = 0;
  const int sms = sm_count(&dev);
  int occ = 0;
  if (dev >= 0 && dev < kMaxDevices) occ = per_sm[dev].load(std::memory_order_relaxed);
  if (occ <= 0) {
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, kThreads, 0);
    if (occ < 1) occ = 1;
    if (dev >= 0 && dev < kMaxDevices) per_sm[dev].store(occ, std::memory_order_relaxed);
  }
  long long g = (long long)sms * occ;
  if (resident) *resident = (int)(g < 0x7fffffff ? g : 0x7fffffff);
  const long long need = (work_items + kThreads - 1) / kThreads;
  if (g > need) g = need;
  if (g < 1) g = 1;
  return (int)g;
}

template <int ND, int CAP>
cudaError_t go_reduce(const ReduceLaunch& p, cudaStream_t s, int* spare_cta) {
  ReduceArgs<CAP> a;
  for (int r = 0; r < CAP; ++r) a.g[r] = r < p.nd ? p.grads[r] : nullptr;
  a.gsum = p.gsum;
  a.n_vec = p.n_span / 8;
  a.n_valid = p.n_valid;
  a.st = p.scratch;
  a.loss_scale = p.loss_scale;
  a.clip = p.clip;
  a.hp = p.hp;
  a.nd = p.nd;
  a.finalize = p.finalize ? 1 : 0;
  static std::atomic<int> occ_cache[kMaxDevices];  // this instantiation's occupancy
  // One wave of reducing CTAs. When the span needs less than a wave, a spare CTA slot
  // computes the next step's t-only scalars, which takes their double-precision powers
  // off the serial combine; a full wave keeps every slot for the reduce (one CTA fewer
  // would cost more than the powers) and computes them in the combine.
  int resident = 0;
  int grid = occupancy_grid(k_reduce<ND, CAP, false>, a.n_vec, occ_cache, &resident);
  if (p.grid > 0 && p.grid < grid) grid = p.grid;
  if (grid > kMaxPartialBlocks) grid = kMaxPartialBlocks;
  if (spare_cta) *spare_cta = grid < resident ? 1 : 0;
  if (grid < resident)
    k_reduce<ND, CAP, true><<<grid + 1, kThreads, 0, s>>>(a);
  else
    k_reduce<ND, CAP, false><<<grid, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

template <int ND, int CAP, int CONS>
cudaError_t go_reduce_bulk(const ReduceLaunch& p, cudaStream_t s, int* spare_cta) {
  ReduceArgs<CAP> a;
  for (int r = 0; r < CAP; ++r) a.g[r] = r < p.nd ? p.grads[r] : nullptr;
  a.gsum = p.gsum;
  a.n_vec = p.n_span / 8;
  a.n_valid = p.n_valid;
  a.st = p.scratch;
  a.loss_scale = p.loss_scale;
  a.clip = p.clip;
  a.hp = p.hp;
  a.nd = p.nd;
  a.finalize = p.finalize ? 1 : 0;
  static std::atomic<bool> attr_set[kMaxDevices];
  int dev = 0;
  const int sms = sm_count(&dev);
  if (dev < 0 || dev >= kMaxDevices || !attr_set[dev].load(std::memory_order_relaxed)) {
    cudaError_t e = cudaFuncSetAttribute(k_reduce_bulk<ND, CAP, false, CONS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRbSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k_reduce_bulk<ND, CAP, true, CONS>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRbSmem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices) attr_set[dev].store(true, std::memory_order_relaxed);
  }
  constexpr int RC = (ND > 0 && ND < RbCfg<CONS>::kRanks) ? ND : RbCfg<CONS>::kRanks;
  const long long tiles = (a.n_vec + RbGeom<RC, CONS>::TG - 1) / RbGeom<RC, CONS>::TG;
  // one CTA per SM, at most one per tile; a grid below one wave gets one more CTA that
  // computes the next step's t-only scalars while the others reduce
  long long grid = sms;
  if (p.grid > 0 && p.grid < grid) grid = p.grid;
  if (grid > tiles) grid = tiles;
  if (grid > kMaxPartialBlocks) grid = kMaxPartialBlocks;
  if (grid < 1) grid = 1;
  const bool pre = grid < sms;
  if (spare_cta) *spare_cta = pre ? 1 : 0;
  unsigned long long* next_tile = &p.scratch->reduce_next;
  constexpr int kThreads = RbCfg<CONS>::kThreads;
  if (pre)
    k_reduce_bulk<ND, CAP, true, CONS><<<(unsigned)grid + 1, kThreads, kRbSmem, s>>>(a, next_tile);
  else
    k_reduce_bulk<ND, CAP, false, CONS><<<(unsigned)grid, kThreads, kRbSmem, s>>>(a, next_tile);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_reduce(const ReduceLaunch& p, cudaStream_t s, int* spare_cta) {
  // 8 ranks: the bulk-load reduce with 512 consumers (4 ranks per stage); more: with 256
  // (8 ranks per stage); fewer: the register-load reduce
  switch (p.nd) {
    case 1: return go_reduce<1, 16>(p, s, spare_cta);
    case 2: return go_reduce<2, 16>(p, s, spare_cta);
    case 4: return go_reduce<4, 16>(p, s, spare_cta);
    case 8: return go_reduce_bulk<8, 16, 512>(p, s, spare_cta);
    case 16: return go_reduce_bulk<16, 16, 256>(p, s, spare_cta);
    case 32: return go_reduce_bulk<32, 64, 256>(p, s, spare_cta);
    case 64: return go_reduce_bulk<64, 64, 256>(p, s, spare_cta);
    default:
      if (p.nd < 8) return go_reduce<0, 16>(p, s, spare_cta);
      if (p.nd <= 64) return go_reduce_bulk<0, 64, 256>(p, s, spare_cta);
      return go_reduce_bulk<0, ZERO_MAX_ND, 256>(p, s, spare_cta);
  }
}

namespace {

// The fused kernel's shared-memory limit, raised once per instantiation and device.
template <int ND, int CAP>
cudaError_t prepare_small() {
  static std::atomic<bool> done[kMaxDevices];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < kMaxDevices && done[dev].load(std::memory_order_relaxed))
    return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(
      k_step_small<ND, CAP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmallSmem);
  if (e == cudaSuccess && dev >= 0 && dev < kMaxDevices)
    done[dev].store(true, std::memory_order_relaxed);
  return e;
}

template <int ND, int CAP>
cudaError_t go_small(const SmallLaunch& p, cudaStream_t s, int sms) {
  cudaError_t e = prepare_small<ND, CAP>();
  if (e != cudaSuccess) return e;
  SmallArgs<CAP> a;
  for (int r = 0; r < CAP; ++r) a.r.g[r] = r < p.r.nd ? p.r.grads[r] : nullptr;
  a.r.gsum = nullptr;  // the sums stay in shared memory
  a.r.n_vec = p.r.n_span / 8;
  a.r.n_valid = p.r.n_valid;
  a.r.st = p.r.scratch;
  a.r.loss_scale = p.r.loss_scale;
  a.r.clip = p.r.clip;
  a.r.hp = p.r.hp;
  a.r.nd = p.r.nd;
  a.r.finalize = 1;
  a.master = p.master;
  a.m = p.exp_avg;
  a.v = p.exp_avg_sq;
  a.p16 = static_cast<uint16_t*>(p.param16);
  a.vecs_per_cta = (a.r.n_vec + sms - 1) / sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)sms);  // one CTA per SM, all resident (cooperative)
  cfg.blockDim = dim3(kSmallThreads + 32);
  cfg.dynamicSmemBytes = kSmallSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_step_small<ND, CAP>, a);
}

}  // namespace

long long small_step_max_vecs() {
  static std::atomic<long long> cache[kMaxDevices];
  int dev = 0;
  const int sms = sm_count(&dev);
  if (dev >= 0 && dev < kMaxDevices) {
    const long long c = cache[dev].load(std::memory_order_relaxed);
    if (c != 0) return c > 0 ? c : 0;
  }
  // every instantiation must fit one CTA per SM; the generic one holds the most registers
  int occ = 0, occ8 = 0;
  cudaError_t e = prepare_small<0, 64>();
  if (e == cudaSuccess) e = prepare_small<8, 16>();
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_step_small<0, 64>,
                                                      kSmallThreads + 32, kSmallSmem);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ8, k_step_small<8, 16>,
                                                      kSmallThreads + 32, kSmallSmem);
  const long long v = (e == cudaSuccess && occ >= 1 && occ8 >= 1) ? (long long)sms * kWideVecs : -1;
  if (dev >= 0 && dev < kMaxDevices) cache[dev].store(v, std::memory_order_relaxed);
  return v > 0 ? v : 0;
}

cudaError_t launch_small_step(const SmallLaunch& p, cudaStream_t s) {
  const int sms = sm_count(nullptr);
  switch (p.r.nd) {
    case 1: return go_small<1, 16>(p, s, sms);
    case 2: return go_small<2, 16>(p, s, sms);
    case 4: return go_small<4, 16>(p, s, sms);
    case 8: return go_small<8, 16>(p, s, sms);
    case 16: return go_small<16, 16>(p, s, sms);
    case 32: return go_small<32, 64>(p, s, sms);
    case 64: return go_small<64, 64>(p, s, sms);
    default:
      if (p.r.nd <= 64) return go_small<0, 64>(p, s, sms);
      return cudaErrorInvalidValue;
  }
}

cudaError_t launch_next_scalars(DevScratch* scratch, const HostHParams& hp, cudaStream_t s) {
  k_next_scalars<<<1, 32, 0, s>>>(scratch, hp);
  return cudaGetLastError();
}

cudaError_t launch_finalize(DevScratch* scratch, float loss_scale, float clip,
                            const HostHParams& hp, cudaStream_t s) {
  k_finalize<<<1, 32, 0, s>>>(scratch, loss_scale, clip, hp);
  return cudaGetLastError();
}

cudaError_t launch_update(const UpdateLaunch& p, cudaStream_t s) {
  UpdateArgs a;
  a.gsum = p.gsum;
  a.master = p.master;
  a.m = p.exp_avg;
  a.v = p.exp_avg_sq;
  a.p16 = static_cast<uint16_t*>(p.param16);
  a.n_valid = p.n_valid;
  a.st = p.scratch;
  int dev = 0;
  const int sms = sm_count(&dev);
  static std::atomic<bool> attr_set[kMaxDevices];
  if (dev < 0 || dev >= kMaxDevices || !attr_set[dev].load(std::memory_order_relaxed)) {
    cudaError_t e = cudaFuncSetAttribute(k_update, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kUpdSmem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices) attr_set[dev].store(true, std::memory_order_relaxed);
  }
  const long long tiles = ((p.n_valid & ~7ll) + kUpdTile - 1) / kUpdTile;
  long long grid = tiles < sms ? tiles : sms;  // one CTA per SM, persistent
  if (grid < 1) grid = 1;
  if (p.grid > 0 && p.grid < grid) grid = p.grid;
  k_update<<<(int)grid, kUpdThreads, kUpdSmem, s>>>(a);
  return cudaGetLastError();
}

// This translation unit's bounds-fault words (see bounds.h): 0 and the words in a checked
// build, 1 (and zeros) in the normal one, -1 on a CUDA error.
int bounds_words_step(unsigned long long* out, bool reset) {
#ifdef ZERO_BOUNDS_CHECK
  return bounds_fault_words(out, reset);
#else
  (void)reset;
  out[0] = out[1] = 0;
  return 1;
#endif
}

}  // namespace zero
