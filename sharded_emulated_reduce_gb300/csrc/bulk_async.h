// Bulk-async (TMA 1-D) copies and mbarrier waits for the libzero kernels on sm_103a.
//
// cp.async.bulk moves a contiguous byte range between global and shared memory on the
// TMA engine: a load signals an mbarrier with its byte count (complete_tx), a store is
// tracked as a bulk group. Addresses must be 16-byte aligned and sizes multiples of 16.
// Every wait on an mbarrier is bounded in polls and in time: the caller gets false and
// must record a status and stop instead of spinning on.
#pragma once
#include <stdint.h>

namespace zero {

constexpr unsigned kWaitLimit = 1u << 22;             // try_wait polls before giving up
constexpr uint32_t kPollSuspendNs = 1000;             // longest suspension of one poll
constexpr unsigned long long kWaitNs = 2000000000ull;  // and at most ~2 s in all

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(b)),
               "r"(bytes) : "memory");
}
// Wait for the phase with the given parity to complete. Each poll suspends the thread for
// at most kPollSuspendNs; the wait gives up after `limit` polls or about kWaitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity,
                                          unsigned limit = kWaitLimit) {
  const uint32_t a = smem_addr(b);
  const unsigned long long t0 = global_ns();
  for (unsigned i = 0; i < limit; ++i) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done) : "r"(a), "r"(parity), "r"(kPollSuspendNs) : "memory");
    if (done) return true;
    if ((i & 63u) == 63u && global_ns() - t0 > kWaitNs) return false;
  }
  return false;
}
__device__ __forceinline__ void bulk_load(void* dst_smem, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_addr(dst_smem)), "l"(src), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void bulk_store(void* dst, const void* src_smem, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
               "r"(smem_addr(src_smem)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// all but the most recent bulk group have finished reading their shared memory
__device__ __forceinline__ void bulk_wait_read_all_but_one() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// every bulk group has finished reading its shared memory
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// every bulk group is complete (its global writes done)
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// order this thread's shared-memory accesses before later bulk (async-proxy) accesses
__device__ __forceinline__ void fence_to_async_proxy() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace zero
