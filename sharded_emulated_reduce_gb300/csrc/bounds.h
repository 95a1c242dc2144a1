// Bounds-checked builds of the libzero kernels (ZERO_BOUNDS_CHECK defined).
//
// No memory checker runs this project's GPU tests, so a checked build stands in for one
// on the kernels' own index arithmetic: before each global access of a kernel's main
// paths, the byte range it touches is tested against the extent of the buffer it belongs
// to, as the launch describes that buffer. A range outside it records the first fault
// (the access site and the offending offset from the buffer's start) in a device word of
// the translation unit and is skipped. A skipped bulk load leaves its stage incomplete,
// so the kernel's bounded wait then expires and reports a status; nothing faults. The host
// reads the words with zero_bounds_check. In the normal build every check is the
// constant true and compiles away.
#pragma once
#include <stddef.h>
#include <stdint.h>

namespace zero {

// Access sites, as recorded in a fault.
enum BoundsSite : unsigned {
  kSiteNone = 0,
  kSiteReduceLoad = 1,     // contributions, register loads (reduce, one-launch step)
  kSiteReduceStore = 2,    // fp32 sums (reduce kernels)
  kSiteBulkReduceLoad = 3, // contributions, bulk loads (bulk-load reduce)
  kSiteUpdateLoad = 4,     // sums and state, bulk loads (update)
  kSiteUpdateStore = 5,    // state and fp16 parameters, bulk stores (update)
  kSiteUpdateTail = 6,     // the last parameters, one by one (update, one-launch step)
  kSiteSmallState = 7,     // state, bulk loads (one-launch step)
  kSiteSmallStore = 8,     // state and fp16 parameters (one-launch step)
  kSiteGatherTile = 9,     // a tile of a copy segment, source and destination (gather)
  kSiteRealignLoad = 10,   // source blocks of a stretch, bulk loads (realigning gather)
  kSiteRealignStore = 11,  // destination vectors (realigning gather)
};

#ifdef ZERO_BOUNDS_CHECK
// {site, offset} of this translation unit's first fault; site 0: none
static __device__ unsigned long long g_bounds_fault[2];

__device__ __forceinline__ bool in_bounds(unsigned site, const void* p, size_t nbytes,
                                          const void* base, size_t extent) {
  const char* a = static_cast<const char*>(p);
  const char* b = static_cast<const char*>(base);
  if (a >= b && nbytes <= extent && static_cast<size_t>(a - b) <= extent - nbytes) return true;
  if (atomicCAS(&g_bounds_fault[0], 0ull, static_cast<unsigned long long>(site)) == 0ull)
    g_bounds_fault[1] = static_cast<unsigned long long>(a - b);
  return false;
}
#define ZERO_IN_BOUNDS(site, p, nbytes, base, extent) \
  ::zero::in_bounds((site), (p), (nbytes), (base), (extent))

// Host side: this translation unit's fault words into out[2] and, with reset, zero them.
static inline int bounds_fault_words(unsigned long long* out, bool reset) {
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_bounds_fault) != cudaSuccess) return -1;
  if (cudaMemcpy(out, addr, 2 * sizeof(unsigned long long), cudaMemcpyDeviceToHost) !=
      cudaSuccess)
    return -1;
  if (reset && cudaMemset(addr, 0, 2 * sizeof(unsigned long long)) != cudaSuccess) return -1;
  return 0;
}
#else
#define ZERO_IN_BOUNDS(site, p, nbytes, base, extent) true
#endif

}  // namespace zero
