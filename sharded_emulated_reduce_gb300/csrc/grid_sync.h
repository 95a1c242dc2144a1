// Grid-wide barrier with sums, for cooperative launches of the libzero kernels on sm_103a.
//
// Only for launches whose CTAs are all resident at once (cudaLaunchAttributeCooperative).
// W 64-bit "counting" words, zero before the launch, are both the barrier and the
// exchange of the CTAs' statistics: one thread of each CTA adds to word j, with one
// atomic add, its own value v_j (< 2^32) plus 2^48. Bits 48..63 of a word then count the
// CTAs that have added to it and bits 0..47 hold the sum of their values (no carry into
// the count for up to 65535 CTAs). Each word is exact on its own: a read that finds its
// count complete holds every CTA's value, whatever the order of the adds, and no order
// between the words is needed. A waiting warp reads the W words, one lane each, until
// every count is complete: one round trip to L2 after the last CTA's adds, which also
// brings the sums (an arrival counter followed by reads of per-CTA partials takes two).
// Every wait is bounded: it gives up after `polls` polls or about kWaitNs and returns
// false, so that the caller records a status and returns instead of spinning on.
#pragma once
#include <stdint.h>

#include "bulk_async.h"

namespace zero {

constexpr int kCountShift = 48;
constexpr unsigned long long kCountOne = 1ull << kCountShift;

__device__ __forceinline__ void red_add_u64(unsigned long long* p, unsigned long long x) {
  asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(x) : "memory");
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long x;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(x) : "l"(p) : "memory");
  return x;
}

// One thread of each CTA: adds v[j] (< 2^32) to word j (at words + j * stride), counted.
template <int W>
__device__ __forceinline__ void sum_arrive(unsigned long long* words, int stride,
                                           const unsigned long long (&v)[W]) {
#pragma unroll
  for (int j = 0; j < W; ++j) red_add_u64(words + j * stride, kCountOne | v[j]);
}

// One whole warp: waits until each of the W words (W <= 32) counts nblocks CTAs; lane
// j < W then gets word j's sum in *sum. Returns the same in every lane: false if the
// wait gave up.
template <int W>
__device__ __forceinline__ bool sum_wait(const unsigned long long* words, int stride,
                                         unsigned nblocks, unsigned polls,
                                         unsigned long long* sum) {
  static_assert(W >= 1 && W <= 32, "one word per lane");
  const int lane = threadIdx.x & 31;
  const unsigned long long t0 = global_ns();
  for (unsigned i = 0; i < polls; ++i) {
    const unsigned long long w =
        lane < W ? ld_relaxed_u64(words + lane * stride) : (unsigned long long)nblocks << kCountShift;
    if (__all_sync(0xffffffffu, (w >> kCountShift) == nblocks)) {
      *sum = w & (kCountOne - 1);
      return true;
    }
    __nanosleep(64);
    if ((i & 63u) == 63u && __any_sync(0xffffffffu, global_ns() - t0 > kWaitNs)) return false;
  }
  return false;
}

}  // namespace zero
