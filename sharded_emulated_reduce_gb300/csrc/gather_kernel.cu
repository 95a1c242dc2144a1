// The ZeRO-3 parameter gather on sm_103a: fp16 shards copied into contiguous per-layer
// buffers (the arithmetic of the all-gather before forward).
//
// The host cuts every layer at shard boundaries into copy segments (at most
// n_layers + nd of them) and numbers fixed-size tiles across all segments. A
// persistent grid walks the tiles; each CTA finds its segment by binary search over
// the segment table, which sits in the kernel's parameter space, and copies the tile
// with 16-byte vectors when source and destination share their alignment modulo 16
// bytes. The few elements before the first aligned destination vector and after the
// last are copied one by one, and so is a tile whose source and destination are
// misaligned relative to each other.
#include "internal.h"

namespace zero {
namespace {

__device__ __forceinline__ int find_segment(const GatherLaunch& a, long long tile) {
  int lo = 0, hi = a.nseg - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a.seg[mid].tile_begin <= tile) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ void copy_tile(const uint16_t* __restrict__ src,
                                          uint16_t* __restrict__ dst, long long n) {
  const uintptr_t sa = reinterpret_cast<uintptr_t>(src);
  const uintptr_t da = reinterpret_cast<uintptr_t>(dst);
  long long head = (long long)(((16u - (unsigned)(da & 15u)) & 15u) >> 1);
  if (head > n) head = n;
  const bool vec = ((sa + 2 * head) & 15u) == 0;
  if (!vec) {
    for (long long j = threadIdx.x; j < n; j += kThreads) dst[j] = src[j];
    return;
  }
  const long long nvec = (n - head) >> 3;
  const uint4* s4 = reinterpret_cast<const uint4*>(src + head);
  uint4* d4 = reinterpret_cast<uint4*>(dst + head);
  // 4 vectors in flight per thread per round
  long long j = threadIdx.x;
  for (; j + 3 * kThreads < nvec; j += 4 * kThreads) {
    const uint4 w0 = __ldcs(s4 + j);
    const uint4 w1 = __ldcs(s4 + j + kThreads);
    const uint4 w2 = __ldcs(s4 + j + 2 * kThreads);
    const uint4 w3 = __ldcs(s4 + j + 3 * kThreads);
    __stcs(d4 + j, w0);
    __stcs(d4 + j + kThreads, w1);
    __stcs(d4 + j + 2 * kThreads, w2);
    __stcs(d4 + j + 3 * kThreads, w3);
  }
  for (; j < nvec; j += kThreads) __stcs(d4 + j, __ldcs(s4 + j));
  if (threadIdx.x < head) dst[threadIdx.x] = src[threadIdx.x];
  const long long tail0 = head + nvec * 8;
  if (tail0 + threadIdx.x < n) dst[tail0 + threadIdx.x] = src[tail0 + threadIdx.x];
}

__global__ void __launch_bounds__(kThreads) k_gather(const __grid_constant__ GatherLaunch a) {
  for (long long t = blockIdx.x; t < a.tiles; t += gridDim.x) {
    const GatherSeg& sg = a.seg[find_segment(a, t)];
    const long long e0 = (t - sg.tile_begin) * kGatherTile;
    long long n = sg.len - e0;
    if (n > kGatherTile) n = kGatherTile;
    copy_tile(sg.src + e0, sg.dst + e0, n);
  }
}

}  // namespace

int gather_grid(int64_t tiles) {
  int dev = 0, sms = 0, per_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_gather, kThreads, 0);
  if (per_sm < 1) per_sm = 1;
  long long g = (long long)sms * per_sm;
  if (g > tiles) g = tiles;
  return g < 1 ? 1 : (int)g;
}

cudaError_t launch_gather(const GatherLaunch& p, cudaStream_t s) {
  if (p.nseg == 0 || p.tiles == 0) return cudaSuccess;
  const int grid = p.grid > 0 ? p.grid : gather_grid(p.tiles);
  k_gather<<<grid, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace zero
