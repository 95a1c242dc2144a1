// The ZeRO-3 parameter gather on sm_103a: fp16 shards copied into contiguous per-layer
// buffers (the arithmetic of the all-gather before forward).
//
// The host cuts every layer at shard boundaries into copy segments (at most
// n_layers + nd of them) and numbers fixed-size tiles (64 KiB) across all segments. A
// persistent grid walks the tiles; the segment table sits in the kernel's parameter
// space, and a tile is copied with 16-byte vectors, 8 in flight per thread, when source
// and destination share their alignment modulo 16 bytes. The few elements before the first aligned destination vector and after the
// last are copied one by one, and so is a tile whose source and destination are
// misaligned relative to each other.
#include "internal.h"

namespace zero {
namespace {

__device__ __forceinline__ void copy_tile(const uint16_t* __restrict__ src,
                                          uint16_t* __restrict__ dst, long long n) {
  const uintptr_t sa = reinterpret_cast<uintptr_t>(src);
  const uintptr_t da = reinterpret_cast<uintptr_t>(dst);
  long long head = (long long)(((16u - (unsigned)(da & 15u)) & 15u) >> 1);
  if (head > n) head = n;
  const bool vec = ((sa + 2 * head) & 15u) == 0;
  if (!vec) {  // source and destination misaligned relative to each other
    for (long long j = threadIdx.x; j < n; j += kThreads) dst[j] = src[j];
    return;
  }
  const long long nvec = (n - head) >> 3;
  const uint4* s4 = reinterpret_cast<const uint4*>(src + head);
  uint4* d4 = reinterpret_cast<uint4*>(dst + head);
  // 8 vectors (128 bytes) in flight per thread per round
  long long j = threadIdx.x;
  for (; j + 7 * kThreads < nvec; j += 8 * kThreads) {
    uint4 w[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) w[u] = s4[j + u * kThreads];
#pragma unroll
    for (int u = 0; u < 8; ++u) d4[j + u * kThreads] = w[u];
  }
  for (; j < nvec; j += kThreads) d4[j] = s4[j];
  if (threadIdx.x < head) dst[threadIdx.x] = src[threadIdx.x];
  const long long tail0 = head + nvec * 8;
  if (tail0 + threadIdx.x < n) dst[tail0 + threadIdx.x] = src[tail0 + threadIdx.x];
}

// A CTA visits its tiles in increasing order, so the segment that holds a tile is found
// by advancing a running index through the table instead of searching it per tile.
__global__ void __launch_bounds__(kThreads) k_gather(const __grid_constant__ GatherLaunch a) {
  int seg = 0;
  for (long long t = blockIdx.x; t < a.tiles; t += gridDim.x) {
    while (seg + 1 < a.nseg && a.seg[seg + 1].tile_begin <= t) ++seg;
    const GatherSeg& sg = a.seg[seg];
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
