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
// and after the last are copied by the other threads. A tile whose source and destination
// are misaligned relative to each other is copied by all threads with 16-byte loads that
// are recombined in registers (funnel shifts) into aligned 16-byte stores.
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

// Bytes [d, d+16) of the 32-byte concatenation lo|hi, for an even d in 2..14 (little
// endian: lo.x holds bytes 0..3).
__device__ __forceinline__ uint4 realign(const uint4& lo, const uint4& hi, int d) {
  switch (d) {
    case 2: return make_uint4(__funnelshift_r(lo.x, lo.y, 16), __funnelshift_r(lo.y, lo.z, 16),
                              __funnelshift_r(lo.z, lo.w, 16), __funnelshift_r(lo.w, hi.x, 16));
    case 4: return make_uint4(lo.y, lo.z, lo.w, hi.x);
    case 6: return make_uint4(__funnelshift_r(lo.y, lo.z, 16), __funnelshift_r(lo.z, lo.w, 16),
                              __funnelshift_r(lo.w, hi.x, 16), __funnelshift_r(hi.x, hi.y, 16));
    case 8: return make_uint4(lo.z, lo.w, hi.x, hi.y);
    case 10: return make_uint4(__funnelshift_r(lo.z, lo.w, 16), __funnelshift_r(lo.w, hi.x, 16),
                               __funnelshift_r(hi.x, hi.y, 16), __funnelshift_r(hi.y, hi.z, 16));
    case 12: return make_uint4(lo.w, hi.x, hi.y, hi.z);
    default: return make_uint4(__funnelshift_r(lo.w, hi.x, 16), __funnelshift_r(hi.x, hi.y, 16),
                               __funnelshift_r(hi.y, hi.z, 16), __funnelshift_r(hi.z, hi.w, 16));
  }
}

// A tile whose source and destination differ in alignment modulo 16 bytes (all threads).
// Destination vector j (16-byte aligned) is bytes [d, d+16) of the two aligned source
// vectors W_j, W_{j+1} around it; a vector is used only when both lie inside the tile's
// source range, and the remaining edge elements are copied one by one.
__device__ void copy_realigned(const uint16_t* src, uint16_t* dst, long long n, long long head) {
  const uintptr_t s0 = reinterpret_cast<uintptr_t>(src);
  const uintptr_t s_body = s0 + 2 * head;              // source of the first aligned dst vector
  const int d = (int)(s_body & 15u);                   // 2..14
  const uintptr_t a = s_body - d;                      // aligned source base
  const uintptr_t s_end = s0 + 2 * n;
  const long long nvec = (n - head) >> 3;              // dst vectors in the tile
  const long long j_lo = a >= s0 ? 0 : 1;
  long long j_hi = s_end >= a + 16 ? (long long)((s_end - a - 16) >> 4) : 0;
  if (j_hi > nvec) j_hi = nvec;
  if (j_hi < j_lo) j_hi = j_lo;                        // no vector fits
  const uint4* w = reinterpret_cast<const uint4*>(a);
  uint4* out = reinterpret_cast<uint4*>(dst + head);
  // 8 destination vectors per thread per round: 16 loads in flight (W_{j+1} of one thread
  // is W_j of the next, so half of them are served by L1), then 8 aligned stores
  long long j = j_lo + threadIdx.x;
  for (; j + 7 * kGatThreads < j_hi; j += 8 * kGatThreads) {
    uint4 lo[8], hi[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      lo[u] = w[j + u * kGatThreads];
      hi[u] = w[j + u * kGatThreads + 1];
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) out[j + u * kGatThreads] = realign(lo[u], hi[u], d);
  }
  for (; j < j_hi; j += kGatThreads) out[j] = realign(w[j], w[j + 1], d);
  long long v0 = head + 8 * j_lo, v1 = head + 8 * j_hi;  // vectors cover [v0, v1)
  if (v0 > n) v0 = n;
  if (v1 > n) v1 = n;
  for (long long i = threadIdx.x; i < v0; i += kGatThreads) dst[i] = src[i];
  for (long long i = v1 + threadIdx.x; i < n; i += kGatThreads) dst[i] = src[i];
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
      copy_realigned(src, dst, n, head);
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
