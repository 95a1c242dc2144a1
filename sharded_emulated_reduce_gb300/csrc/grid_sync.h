// Grid-wide barrier for cooperative launches of the libzero kernels on sm_103a.
//
// Only for launches whose CTAs are all resident at once (cudaLaunchAttributeCooperative).
// One thread per CTA arrives on a counter; the last to arrive resets it and advances a
// generation word that the others poll. Every poll is bounded: the barrier gives up after
// `polls` polls or about kWaitNs and returns false, so that the caller records a status
// and returns instead of spinning on.
#pragma once
#include <stdint.h>

#include "bulk_async.h"

namespace zero {

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned x;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(x) : "l"(p) : "memory");
  return x;
}

// One thread of each CTA. The CTA's earlier global writes are visible to every CTA once
// this returns true.
__device__ __forceinline__ bool grid_barrier(unsigned* count, unsigned* gen_word,
                                             unsigned nblocks, unsigned polls) {
  const unsigned gen = ld_acquire_u32(gen_word);
  __threadfence();
  if (atomicAdd(count, 1u) == nblocks - 1) {
    *count = 0;  // nobody touches the count again in this launch
    __threadfence();
    atomicAdd(gen_word, 1u);
    return true;
  }
  const unsigned long long t0 = global_ns();
  for (unsigned i = 0; i < polls; ++i) {
    if (ld_acquire_u32(gen_word) != gen) {
      __threadfence();
      return true;
    }
    __nanosleep(64);
    if ((i & 63u) == 63u && global_ns() - t0 > kWaitNs) return false;
  }
  return false;
}

}  // namespace zero
