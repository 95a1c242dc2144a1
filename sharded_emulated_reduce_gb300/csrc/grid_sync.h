// Grid-wide barrier for cooperative launches of the libzero kernels on sm_103a.
//
// Only for launches whose CTAs are all resident at once (cudaLaunchAttributeCooperative).
// One thread per CTA adds 1 to a 64-bit arrival counter that only ever grows: the k-th
// launch of an nblocks-CTA grid that uses the counter (since it was last zeroed) takes it
// from k*nblocks to (k+1)*nblocks. A CTA's own arrival returns the count before it, so
// the CTA knows the value that completes its launch's barrier (the next multiple of
// nblocks) and polls the counter until it gets there. Nothing is reset and no second
// word is released, which keeps the last arrival one atomic away from the others'
// departure. Every launch on a counter must use the same grid size, and a launch in which
// a CTA never arrives leaves the counter off that rhythm: the host zeroes it after a
// barrier reported an expiry. Every poll is bounded: the barrier gives up after `polls`
// polls or about kWaitNs and returns false, so that the caller records a status and
// returns instead of spinning on.
#pragma once
#include <stdint.h>

#include "bulk_async.h"

namespace zero {

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long x;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(x) : "l"(p) : "memory");
  return x;
}

struct NoAction {
  __device__ void operator()() const {}
};

// One thread of each CTA. The CTA's earlier global writes are visible to every CTA once
// this returns true. `after_arrive` runs once this CTA has arrived, before it waits.
template <typename F = NoAction>
__device__ __forceinline__ bool grid_barrier(unsigned long long* arrivals, unsigned nblocks,
                                             unsigned polls, F after_arrive = F()) {
  __threadfence();  // this CTA's writes before its arrival
  const unsigned long long old = atomicAdd(arrivals, 1ull);
  const unsigned long long target = old - old % nblocks + nblocks;
  after_arrive();
  if (old + 1 == target) {  // the last to arrive
    __threadfence();
    return true;
  }
  const unsigned long long t0 = global_ns();
  for (unsigned i = 0; i < polls; ++i) {
    if (ld_acquire_u64(arrivals) >= target) {
      __threadfence();
      return true;
    }
    __nanosleep(64);
    if ((i & 63u) == 63u && global_ns() - t0 > kWaitNs) return false;
  }
  return false;
}

}  // namespace zero
