// The ZeRO-3 parameter gather on sm_103a: fp16 shards copied into contiguous per-layer
// buffers (the arithmetic of the all-gather before forward).
//
// The host cuts every layer at shard boundaries into copy segments (at most
// n_layers + nd of them) and numbers fixed-size tiles (64 KiB) across all segments; the
// segment table sits in the kernel's parameter space. One persistent CTA per SM walks
// its tiles. Where source and destination share their alignment modulo 16 bytes (every
// layout with layer offsets that are multiples of 8 elements), one thread moves the tile
// through a 4-stage ring of 32 KiB shared-memory buffers with TMA bulk copies: a bulk load
// into a free buffer, then a bulk store out of it once the load has landed, several in
// flight at once. The few elements before the first 16-byte-aligned destination address
// and after the last are copied by the other threads, and a tile whose source and
// destination are misaligned relative to each other is copied element by element.
#include "bulk_async.h"
#include "internal.h"

namespace zero {
namespace {

constexpr int kGatStages = 4;
constexpr uint32_t kGatChunk = 32768;  // bytes per ring buffer
constexpr int kGatThreads = 256;
constexpr size_t kGatSmem = (size_t)kGatStages * kGatChunk + kGatStages * sizeof(uint64_t);
constexpr int kMaxDevices = 64;

struct Ring {
  unsigned char* buf;
  uint64_t* full;
  long long q;  // chunks this CTA has moved through the ring so far
};

// One thread: copy `bytes` (a multiple of 16; both addresses 16-byte aligned) through the
// ring, keeping up to kGatStages bulk loads in flight. False if a load did not arrive.
__device__ bool ring_copy(Ring& r, const unsigned char* src, unsigned char* dst, long long bytes) {
  const long long nch = (bytes + kGatChunk - 1) / kGatChunk;
  const long long q0 = r.q;
  auto len = [&](long long i) {
    const long long left = bytes - i * (long long)kGatChunk;
    return (uint32_t)(left < (long long)kGatChunk ? left : (long long)kGatChunk);
  };
  auto issue = [&](long long i) {
    const int s = (int)((q0 + i) % kGatStages);
    bulk_wait_read_all();  // no bulk store is still reading buffer s
    mbar_expect_tx(&r.full[s], len(i));
    bulk_load(r.buf + (size_t)s * kGatChunk, src + i * (long long)kGatChunk, len(i), &r.full[s]);
  };
  long long issued = 0;
  while (issued < nch && issued < kGatStages) issue(issued++);
  for (long long i = 0; i < nch; ++i) {
    const long long q = q0 + i;
    const int s = (int)(q % kGatStages);
    if (!mbar_wait(&r.full[s], (uint32_t)((q / kGatStages) & 1))) {
      for (long long k = i + 1; k < issued; ++k) {  // let the other issued loads land
        const long long qq = q0 + k;
        mbar_wait(&r.full[(int)(qq % kGatStages)], (uint32_t)((qq / kGatStages) & 1));
      }
      return false;
    }
    bulk_store(dst + i * (long long)kGatChunk, r.buf + (size_t)s * kGatChunk, len(i));
    bulk_commit();
    if (issued < nch) issue(issued++);
  }
  r.q = q0 + nch;
  return true;
}

// A CTA visits its tiles in increasing order, so the segment that holds a tile is found
// by advancing a running index through the table.
__global__ void __launch_bounds__(kGatThreads, 1) k_gather(const __grid_constant__ GatherLaunch a) {
  extern __shared__ __align__(128) unsigned char smem[];
  Ring r{smem, reinterpret_cast<uint64_t*>(smem + (size_t)kGatStages * kGatChunk), 0};
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int s = 0; s < kGatStages; ++s) mbar_init(&r.full[s], 1);
    mbar_fence_init();
  }
  __syncthreads();
  int seg = 0;
  bool ok = true;
  for (long long t = blockIdx.x; t < a.tiles && ok; t += gridDim.x) {
    while (seg + 1 < a.nseg && a.seg[seg + 1].tile_begin <= t) ++seg;
    const GatherSeg& sg = a.seg[seg];
    const long long e0 = (t - sg.tile_begin) * kGatherTile;
    long long n = sg.len - e0;
    if (n > kGatherTile) n = kGatherTile;
    const uint16_t* src = sg.src + e0;
    uint16_t* dst = sg.dst + e0;
    const uintptr_t sa = reinterpret_cast<uintptr_t>(src);
    const uintptr_t da = reinterpret_cast<uintptr_t>(dst);
    long long head = (long long)(((16u - (unsigned)(da & 15u)) & 15u) >> 1);
    if (head > n) head = n;
    if (((sa + 2 * head) & 15u) != 0) {  // misaligned relative to each other
      for (long long j = tid; j < n; j += kGatThreads) dst[j] = src[j];
      continue;
    }
    const long long body = ((n - head) >> 3) << 3;  // elements moved by bulk copies
    if (tid < head) dst[tid] = src[tid];
    const long long tail0 = head + body;
    if (tail0 + tid < n) dst[tail0 + tid] = src[tail0 + tid];
    if (tid == 0 && body > 0)
      ok = ring_copy(r, reinterpret_cast<const unsigned char*>(src + head),
                     reinterpret_cast<unsigned char*>(dst + head), body * 2);
    ok = __syncthreads_and(ok);
  }
  if (tid == 0) {
    bulk_wait_all();
    if (!ok && a.status) atomicExch(a.status, kStatusGatherWait);
  }
}

int sm_count() {
  static int sms[kMaxDevices] = {};
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < kMaxDevices && sms[dev] > 0) return sms[dev];
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (dev >= 0 && dev < kMaxDevices) sms[dev] = n;
  return n;
}

}  // namespace

int gather_grid(int64_t tiles) {
  long long g = sm_count();  // one CTA per SM (the ring takes 128 KiB of shared memory)
  if (g > tiles) g = tiles;
  return g < 1 ? 1 : (int)g;
}

cudaError_t launch_gather(const GatherLaunch& p, cudaStream_t s) {
  if (p.nseg == 0 || p.tiles == 0) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool attr_set[kMaxDevices] = {};
  if (dev < 0 || dev >= kMaxDevices || !attr_set[dev]) {
    e = cudaFuncSetAttribute(k_gather, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGatSmem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices) attr_set[dev] = true;
  }
  const int grid = p.grid > 0 ? p.grid : gather_grid(p.tiles);
  k_gather<<<grid, kGatThreads, kGatSmem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace zero
