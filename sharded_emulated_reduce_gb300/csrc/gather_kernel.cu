// The ZeRO-3 parameter gather on sm_103a: fp16 shards copied into contiguous per-layer
// buffers (the arithmetic of the all-gather before forward).
//
// The host cuts every layer at shard boundaries into copy segments (at most
// n_layers + nd of them) and numbers fixed-size tiles (64 KiB) across all segments; the
// segment table sits in the kernel's parameter space. One persistent CTA per SM walks
// its tiles. Where source and destination share their alignment modulo 16 bytes (every
// layout with layer offsets that are multiples of 8 elements), one thread streams the
// 16-byte-aligned bodies of all of its tiles through a ring of 32 KiB shared-memory
// buffers with TMA bulk copies: a bulk load into a free buffer, then a bulk store out of
// it once the load has landed, with all but one buffer's loads in flight and no drain
// between tiles. The few elements before the first 16-byte-aligned destination address
// and after the last are copied by the other warps. Segments whose source and
// destination are misaligned relative to each other go to a second kernel (the host sorts
// them into their own table): bulk loads bring the aligned 16-byte source blocks around
// each stretch of the tile into a shared-memory ring, and all threads recombine pairs of
// blocks (funnel shifts) into aligned 16-byte stores to global memory.
#include <atomic>

#include "bounds.h"
#include "bulk_async.h"
#include "internal.h"

namespace zero {
namespace {

#ifndef ZERO_GATHER_STAGES
#define ZERO_GATHER_STAGES 6
#endif
constexpr int kGatStages = ZERO_GATHER_STAGES;  // ring buffers of the aligned-copy kernel
constexpr uint32_t kGatChunk = 32768;            // bytes per ring buffer
constexpr int kGatThreads = 128;
constexpr size_t kGatSmem = (size_t)kGatStages * kGatChunk + kGatStages * sizeof(uint64_t);
static_assert(kGatStages >= 3 && kGatSmem <= 232448, "ring must fit one CTA's shared memory");
constexpr int kMaxDevices = 64;

// Geometry of one tile of the aligned-copy kernel: n elements from src to dst, the first
// `head` elements (up to the first 16-byte-aligned destination address) and the last
// n - head - body ones copied element by element, the `body` in between by bulk copies.
// body = 0 when source and destination differ in alignment modulo 16 bytes (the host
// sends such segments to the realigning kernel, so this does not occur in practice).
struct AlTile {
  const uint16_t* src;
  uint16_t* dst;
  long long n, head, body;
};

__device__ __forceinline__ AlTile al_tile(const GatherLaunch& a, int& seg, long long t) {
  while (seg + 1 < a.nseg && a.seg[seg + 1].tile_begin <= t) ++seg;
  const GatherSeg& sg = a.seg[seg];
  const long long e0 = (t - sg.tile_begin) * kGatherTileAl;
  AlTile m;
  m.n = sg.len - e0;
  if (m.n > kGatherTileAl) m.n = kGatherTileAl;
  m.src = sg.src + e0;
  m.dst = sg.dst + e0;
  const uintptr_t sa = reinterpret_cast<uintptr_t>(m.src);
  const uintptr_t da = reinterpret_cast<uintptr_t>(m.dst);
  m.head = (long long)(((16u - (unsigned)(da & 15u)) & 15u) >> 1);
  if (m.head > m.n) m.head = m.n;
  m.body = ((sa + 2 * m.head) & 15u) ? 0 : ((m.n - m.head) >> 3) << 3;
  // the tile's source and destination lie inside its segment (every copy of the tile,
  // bulk or element by element, is inside the tile)
  if (!ZERO_IN_BOUNDS(kSiteGatherTile, m.src, 2 * (size_t)m.n, sg.src, 2 * (size_t)sg.len) ||
      !ZERO_IN_BOUNDS(kSiteGatherTile, m.dst, 2 * (size_t)m.n, sg.dst, 2 * (size_t)sg.len))
    m.n = m.head = m.body = 0;
  return m;
}

// A tile body in thread 0's queue of claimed tiles.
struct Body {
  const unsigned char* src;
  unsigned char* dst;
  long long bytes;  // a positive multiple of 16; both addresses 16-byte aligned
};
constexpr int kGatQueue = kGatStages + 2;  // claimed tiles held at once (see k_gather)

// Bytes [D, D+16) of the 32-byte concatenation lo|hi, for an even D in 0..14 (little
// endian: lo.x holds bytes 0..3).
template <int D>
__device__ __forceinline__ uint4 realign(const uint4& lo, const uint4& hi) {
  const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  constexpr int q = D / 4;  // first word
  if constexpr (D % 4 == 0) {
    return make_uint4(w[q], w[q + 1], w[q + 2], w[q + 3]);
  } else {
    return make_uint4(__funnelshift_r(w[q], w[q + 1], 16), __funnelshift_r(w[q + 1], w[q + 2], 16),
                      __funnelshift_r(w[q + 2], w[q + 3], 16), __funnelshift_r(w[q + 3], w[q + 4], 16));
  }
}

// One stretch of nv destination vectors from the nv + 1 source blocks in shared memory
// (all threads; D fixed per tile, so the loop has no branch on it).
template <int D, int NT>
__device__ __forceinline__ void realign_stretch(const uint4* w, uint4* out, long long nv) {
  long long i = threadIdx.x;
  for (; i + 7 * NT < nv; i += 8 * NT) {
    uint4 r[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) r[u] = realign<D>(w[i + u * NT], w[i + u * NT + 1]);
#pragma unroll
    for (int u = 0; u < 8; ++u) out[i + u * NT] = r[u];
  }
  for (; i < nv; i += NT) out[i] = realign<D>(w[i], w[i + 1]);
}

// Geometry of a tile whose source and destination differ in alignment modulo 16 bytes.
// Destination vector j (16-byte aligned, at dst + head + 8j) is bytes [d, d+16) of the two
// aligned source blocks W_j, W_{j+1} (16 bytes each, from a); vector j is used only for
// j_lo <= j < j_hi, where both blocks lie inside the tile's source range, and the elements
// outside [v0, v1) are copied one by one.
struct MisTile {
  const uint16_t* src;
  uint16_t* dst;
  long long n, head, j_lo, j_hi, v0, v1;
  uintptr_t a;
  int d;  // 2..14
};

__device__ __forceinline__ MisTile mis_tile(const GatherLaunch& L, int& seg, long long t) {
  while (seg + 1 < L.nseg && L.seg[seg + 1].tile_begin <= t) ++seg;
  const GatherSeg& sg = L.seg[seg];
  const long long e0 = (t - sg.tile_begin) * kGatherTile;
  MisTile m;
  m.n = sg.len - e0;
  if (m.n > kGatherTile) m.n = kGatherTile;
  m.src = sg.src + e0;
  m.dst = sg.dst + e0;
  const uintptr_t s0 = reinterpret_cast<uintptr_t>(m.src);
  m.head = (long long)(((16u - (unsigned)(reinterpret_cast<uintptr_t>(m.dst) & 15u)) & 15u) >> 1);
  if (m.head > m.n) m.head = m.n;
  const uintptr_t s_body = s0 + 2 * m.head;  // source of the first aligned dst vector
  m.d = (int)(s_body & 15u);
  m.a = s_body - m.d;
  const uintptr_t s_end = s0 + 2 * m.n;
  const long long nvec = (m.n - m.head) >> 3;
  m.j_lo = m.a >= s0 ? 0 : 1;
  m.j_hi = s_end >= m.a + 16 ? (long long)((s_end - m.a - 16) >> 4) : 0;
  if (m.j_hi > nvec) m.j_hi = nvec;
  if (m.j_hi < m.j_lo) m.j_hi = m.j_lo;  // no vector fits
  m.v0 = m.head + 8 * m.j_lo;
  m.v1 = m.head + 8 * m.j_hi;
  if (m.v0 > m.n) m.v0 = m.n;
  if (m.v1 > m.n) m.v1 = m.n;
  // the tile's source and destination lie inside its segment
  if (!ZERO_IN_BOUNDS(kSiteGatherTile, m.src, 2 * (size_t)m.n, sg.src, 2 * (size_t)sg.len) ||
      !ZERO_IN_BOUNDS(kSiteGatherTile, m.dst, 2 * (size_t)m.n, sg.dst, 2 * (size_t)sg.len)) {
    m.n = m.head = m.j_lo = m.j_hi = m.v0 = m.v1 = 0;
  }
  return m;
}

// Thread 0 claims tiles one at a time from the launch's counter (an atomic add, so a CTA
// on a slower SM simply claims fewer and every CTA finishes at about the same time) and
// streams their 16-byte-aligned bodies, cut into chunks of at most kGatChunk bytes,
// through one ring of kGatStages buffers: kGatStages - 1 bulk loads stay in flight, each
// landed chunk leaves by a bulk store, and a buffer is refilled once the store before the
// newest one has finished reading it. The ring does not drain between tiles. Tiles
// without a body are not queued, so the queue never holds more than kGatStages tiles
// (the consumer's and one per chunk in flight). The other warps copy the unaligned edge
// elements of every tile of the launch, split statically over the CTAs (disjoint bytes
// from the bulk stores). The last CTA to finish resets the counter for the next launch.
__global__ void __launch_bounds__(kGatThreads, 1) k_gather(const __grid_constant__ GatherLaunch a) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)kGatStages * kGatChunk);
  const int tid = threadIdx.x;
  if (tid == 0) {
    bool ok = true;
    for (int s = 0; s < kGatStages; ++s) mbar_init(&full[s], 1);
    mbar_fence_init();
    Body q[kGatQueue];
    long long q_head = 0, q_tail = 0;  // the consumer's tile is q[q_head], the next free q[q_tail]
    long long p_idx = 0, p_off = 0;    // the producer's tile and byte offset in its body
    long long c_off = 0;               // the consumer's byte offset in q[q_head]
    int claim_seg = 0;
    bool claims_done = false;
    // one more tile with a body into the queue; false when none is left (or no room)
    auto claim = [&]() -> bool {
      while (!claims_done && q_tail - q_head < kGatQueue) {
        const long long t = (long long)atomicAdd(a.sched, 1ull);
        if (t >= a.tiles) {
          claims_done = true;
          break;
        }
        const AlTile m = al_tile(a, claim_seg, t);
        if (m.body == 0) continue;  // edges only: the other warps copy it
        Body& b = q[q_tail % kGatQueue];
        b.src = reinterpret_cast<const unsigned char*>(m.src + m.head);
        b.dst = reinterpret_cast<unsigned char*>(m.dst + m.head);
        b.bytes = 2 * m.body;
        ++q_tail;
        return true;
      }
      return false;
    };
    long long issued = 0, done = 0;
    // issue loads until kGatStages - 1 are in flight: load `issued` goes to buffer
    // issued % kGatStages, last read by the store of chunk issued - kGatStages <= done - 2
    auto fill = [&]() {
      while (issued - done < kGatStages - 1) {
        if (p_idx == q_tail && !claim()) return;
        const Body& b = q[p_idx % kGatQueue];
        const long long left = b.bytes - p_off;
        const uint32_t len = (uint32_t)(left < (long long)kGatChunk ? left : (long long)kGatChunk);
        const int s = (int)(issued % kGatStages);
        bulk_wait_read_all_but_one();
        mbar_expect_tx(&full[s], len);
        bulk_load(smem + (size_t)s * kGatChunk, b.src + p_off, len, &full[s]);
        ++issued;
        p_off += len;
        if (p_off == b.bytes) {
          ++p_idx;
          p_off = 0;
        }
      }
    };
    fill();
    while (done < issued) {
      const Body& b = q[q_head % kGatQueue];
      const long long left = b.bytes - c_off;
      const uint32_t len = (uint32_t)(left < (long long)kGatChunk ? left : (long long)kGatChunk);
      const int s = (int)(done % kGatStages);
      if (!mbar_wait(&full[s], (uint32_t)((done / kGatStages) & 1))) {
        ok = false;
        break;
      }
      bulk_store(b.dst + c_off, smem + (size_t)s * kGatChunk, len);
      bulk_commit();
      ++done;
      c_off += len;
      if (c_off == b.bytes) {
        ++q_head;
        c_off = 0;
      }
      fill();
    }
    // a wait that gave up: let every load still in flight land before the CTA exits
    for (long long k = done; k < issued; ++k)
      mbar_wait(&full[(int)(k % kGatStages)], (uint32_t)((k / kGatStages) & 1));
    bulk_wait_all();
    if (!ok && a.status) atomicExch(a.status, kStatusGatherWait);
    // this CTA claims nothing more; the last one to get here resets the counter
    __threadfence();
    if (atomicAdd(&a.sched[1], 1ull) == (unsigned long long)gridDim.x - 1) {
      a.sched[0] = 0;
      a.sched[1] = 0;
    }
  } else if (tid >= 32) {
    const int warp = tid / 32 - 1, lane = tid % 32, warps = kGatThreads / 32 - 1;
    int seg = 0;
    long long k = 0;
    for (long long t = blockIdx.x; t < a.tiles; t += gridDim.x, ++k) {
      const AlTile m = al_tile(a, seg, t);
      if (k % warps != warp) continue;
      if (m.body == 0) {  // no bulk part: the whole tile element by element
        for (long long i = lane; i < m.n; i += 32) m.dst[i] = m.src[i];
        continue;
      }
      if (lane < m.head) m.dst[lane] = m.src[lane];
      const long long t0 = m.head + m.body;
      if (t0 + lane < m.n) m.dst[t0 + lane] = m.src[t0 + lane];
    }
  }
}

// Segments whose source and destination differ in alignment modulo 16 bytes. A tile's
// vectors are cut into stretches of up to kMisVecs; thread 0 bulk-loads the kMisVecs + 1
// source blocks of a stretch into a ring stage (kMisStages stages, up to two tiles ahead),
// and after the stage has landed every thread builds its destination vectors from pairs of
// adjacent blocks and stores them. The stage is refilled once all threads are past it.
constexpr int kMisThreads = 256;
constexpr int kMisStages = 4;
constexpr long long kMisVecs = 2048;              // destination vectors per stretch
constexpr uint32_t kMisStageBytes = 32768 + 128;  // (kMisVecs + 1) blocks, rounded to 128 B
constexpr size_t kMisSmem = (size_t)kMisStages * kMisStageBytes + kMisStages * sizeof(uint64_t);

// Walks this CTA's tiles and their non-empty stretches in the order they are consumed.
struct StretchIt {
  long long t;
  long long h;  // next stretch of tile t
  int seg;
};

// Next stretch: source blocks [a + 16 jb, + bytes) for destination vectors jb.. of its tile.
__device__ __forceinline__ bool next_stretch(const GatherLaunch& L, StretchIt& it,
                                             const unsigned char** src, uint32_t* bytes) {
  while (it.t < L.tiles) {
    const MisTile m = mis_tile(L, it.seg, it.t);
    const long long jb = m.j_lo + it.h * kMisVecs;
    if (jb < m.j_hi) {
      long long nv = m.j_hi - jb;
      if (nv > kMisVecs) nv = kMisVecs;
      *src = reinterpret_cast<const unsigned char*>(m.a) + 16 * jb;
      *bytes = (uint32_t)(16 * (nv + 1));
      ++it.h;
      return true;
    }
    it.t += gridDim.x;
    it.h = 0;
  }
  return false;
}

__global__ void __launch_bounds__(kMisThreads, 1)
    k_gather_realign(const __grid_constant__ GatherLaunch L) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)kMisStages * kMisStageBytes);
  const int tid = threadIdx.x;
  StretchIt prod{(long long)blockIdx.x, 0, 0};  // thread 0's issue position
  long long issued = 0;                         // stretches issued (thread 0)
  auto issue = [&]() {
    const unsigned char* src;
    uint32_t bytes;
    if (!next_stretch(L, prod, &src, &bytes)) return;
    const GatherSeg& sg = L.seg[prod.seg];
    if (!ZERO_IN_BOUNDS(kSiteRealignLoad, src, bytes, sg.src, 2 * (size_t)sg.len)) return;
    const int s = (int)(issued % kMisStages);
    mbar_expect_tx(&full[s], bytes);
    bulk_load(smem + (size_t)s * kMisStageBytes, src, bytes, &full[s]);
    ++issued;
  };
  if (tid == 0) {
    for (int s = 0; s < kMisStages; ++s) mbar_init(&full[s], 1);
    mbar_fence_init();
    for (int s = 0; s < kMisStages; ++s) issue();
  }
  __syncthreads();
  long long q = 0;  // stretches consumed
  int seg = 0;
  bool ok = true;
  for (long long t = blockIdx.x; t < L.tiles && ok; t += gridDim.x) {
    const MisTile m = mis_tile(L, seg, t);
    for (long long i = tid; i < m.v0; i += kMisThreads) m.dst[i] = m.src[i];
    for (long long i = m.v1 + tid; i < m.n; i += kMisThreads) m.dst[i] = m.src[i];
    uint4* out = reinterpret_cast<uint4*>(m.dst + m.head);
    for (long long jb = m.j_lo; jb < m.j_hi && ok; jb += kMisVecs) {
      long long nv = m.j_hi - jb;
      if (nv > kMisVecs) nv = kMisVecs;
      const int s = (int)(q % kMisStages);
      bool landed = mbar_wait(&full[s], (uint32_t)((q / kMisStages) & 1));
      if (landed && ZERO_IN_BOUNDS(kSiteRealignStore, out + jb, 16 * (size_t)nv, L.seg[seg].dst,
                                   2 * (size_t)L.seg[seg].len)) {
        const uint4* w = reinterpret_cast<const uint4*>(smem + (size_t)s * kMisStageBytes);
        switch (m.d) {  // even byte offsets 2..14 (0 only in tiles without vectors)
          case 0: realign_stretch<0, kMisThreads>(w, out + jb, nv); break;
          case 2: realign_stretch<2, kMisThreads>(w, out + jb, nv); break;
          case 4: realign_stretch<4, kMisThreads>(w, out + jb, nv); break;
          case 6: realign_stretch<6, kMisThreads>(w, out + jb, nv); break;
          case 8: realign_stretch<8, kMisThreads>(w, out + jb, nv); break;
          case 10: realign_stretch<10, kMisThreads>(w, out + jb, nv); break;
          case 12: realign_stretch<12, kMisThreads>(w, out + jb, nv); break;
          default: realign_stretch<14, kMisThreads>(w, out + jb, nv); break;
        }
      }
      ok = __syncthreads_and(landed);  // every thread is done with stage s
      if (ok) {
        ++q;
        if (tid == 0) issue();  // into stage s, the one just freed
      }
    }
  }
  if (tid == 0) {
    // a wait that gave up: let every load still in flight land before the CTA exits
    for (long long k = q; k < issued; ++k)
      mbar_wait(&full[(int)(k % kMisStages)], (uint32_t)((k / kMisStages) & 1));
    if (!ok && L.status) atomicExch(L.status, kStatusGatherWait);
  }
}

// Per-device values below are computed once; several host threads may race to compute
// the same value, so they are relaxed atomics.
int sm_count() {
  static std::atomic<int> sms[kMaxDevices];
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < kMaxDevices) {
    n = sms[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
  }
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (dev >= 0 && dev < kMaxDevices) sms[dev].store(n, std::memory_order_relaxed);
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
  static std::atomic<bool> attr_set[kMaxDevices];
  if (dev < 0 || dev >= kMaxDevices || !attr_set[dev].load(std::memory_order_relaxed)) {
    e = cudaFuncSetAttribute(k_gather, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGatSmem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices) attr_set[dev].store(true, std::memory_order_relaxed);
  }
  if (p.realign) {
    static std::atomic<bool> mis_attr_set[kMaxDevices];
    if (dev < 0 || dev >= kMaxDevices || !mis_attr_set[dev].load(std::memory_order_relaxed)) {
      e = cudaFuncSetAttribute(k_gather_realign, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kMisSmem);
      if (e != cudaSuccess) return e;
      if (dev >= 0 && dev < kMaxDevices) mis_attr_set[dev].store(true, std::memory_order_relaxed);
    }
    const int grid = p.grid > 0 ? p.grid : gather_grid(p.tiles);
    k_gather_realign<<<grid, kMisThreads, kMisSmem, s>>>(p);
    return cudaGetLastError();
  }
  const int grid = p.grid > 0 ? p.grid : gather_grid(p.tiles);
  k_gather<<<grid, kGatThreads, kGatSmem, s>>>(p);
  return cudaGetLastError();
}

namespace {
// 64 bytes that the bounds self-test measures ranges against (never read or written)
__device__ uint16_t g_bounds_probe_buf[32];

// The bounds self-test: one range inside g_bounds_probe_buf and one reaching past its end
// (bytes 80..95 of a 64-byte buffer) are tested; neither is accessed.
__global__ void k_bounds_probe() {
  if (threadIdx.x != 0) return;
  const uint16_t* b = g_bounds_probe_buf;
  bool inside = ZERO_IN_BOUNDS(kSiteGatherTile, b + 8, 16, b, 64);
  bool outside = ZERO_IN_BOUNDS(kSiteRealignStore, b + 40, 16, b, 64);
  (void)inside;
  (void)outside;
}
}  // namespace

cudaError_t bounds_probe() {
  k_bounds_probe<<<1, 32>>>();
  const cudaError_t e = cudaGetLastError();
  return e != cudaSuccess ? e : cudaDeviceSynchronize();
}

// This translation unit's bounds-fault words (see bounds.h): 0 and the words in a checked
// build, 1 (and zeros) in the normal one, -1 on a CUDA error.
int bounds_words_gather(unsigned long long* out, bool reset) {
#ifdef ZERO_BOUNDS_CHECK
  return bounds_fault_words(out, reset);
#else
  (void)reset;
  out[0] = out[1] = 0;
  return 1;
#endif
}

}  // namespace zero
