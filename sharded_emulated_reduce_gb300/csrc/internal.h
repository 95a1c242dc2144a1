// Internal interface between the host side of libzero (plan.cpp) and its kernels
// (step_kernels.cu, gather_kernel.cu). Not part of the public ABI.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "zero.h"

namespace zero {

constexpr int kThreads = 256;        // threads per CTA for every kernel
constexpr int kMaxPartialBlocks = 1024;  // CTAs of the reduce kernel (one partial each)
constexpr int kGatherSegs = 128;     // copy segments per gather launch
constexpr int kGatherSlots = 64;     // tile-counter slots of the gather (a ring)
constexpr int kSmallWords = 5;       // counting sums of the one-launch step (4 limbs, count)
constexpr int kSumStride = 16;       // words from one counting sum to the next (128 bytes)

// Scalars of one step, written by the finalize stage and read by the update kernel.
struct DevScalars {
  int32_t overflow, skipped, status, pad;
  int64_t step;  // step counter after this step
  double ss, norm, clip_coef;
  float s, omb1, omb2, bc1, bc2, decay, lr, beta1, beta2, eps;
  float loss_scale;  // the scale this step's gradients carried
  float pad2;
};

// Dynamic loss scale kept on the device; growth_interval <= 0 means disabled.
struct DevScaler {
  float scale;
  int32_t good_steps;
  float growth, backoff;
  int32_t interval;
  int32_t pad;
};

// One reduce CTA's statistics: the 128-bit sum of squares and the non-finite count, which
// the last CTA of the reduce kernels combines.
struct alignas(16) DevPartial {
  unsigned long long lo, hi;
  long long bad;
  long long pad;
};

// The step's scalars that depend only on the step counter t and the hyperparameters.
// A CTA of the reduce kernel with no reduce work computes them for the next step (t + 1)
// while the others reduce, so that the serial combine at the end of the next step's
// reduce finds them ready; slot t & 1 holds those for t. The tag (t and the
// hyperparameters) decides whether a slot may be used.
struct DevPre {
  float omb1, omb2, bc1, bc2, decay;
  float lr, beta1, beta2, weight_decay;  // tag: the hyperparameters
  int32_t valid;                         // kPreValid once written (zeroed scratch: not)
  long long t;                           // tag: the step counter
};
constexpr int32_t kPreValid = 0x50524531;

// The plan's device scratch (one allocation, < 64 KiB).
struct DevScratch {
  long long stats[ZERO_STATS_WORDS];  // exchange buffer (see zero_shard_stats)
  DevScalars sc;
  DevPre pre[2];
  DevScaler scaler;
  long long step;       // optimizer step counter t
  unsigned int ticket;    // arrival counter of the reduce CTAs
  int32_t gather_status;  // 0, or kStatusGatherWait after a gather wait expired
  unsigned long long small_launch;  // launches of the one-launch step since the last reset
  unsigned long long reduce_next;   // next tile the bulk-load reduce claims (0 between launches)
  // the one-launch step's counting sums (grid_sync.h), one set per launch parity: the
  // four 32-bit limbs of the 128-bit sum of squares and the non-finite count, each word
  // in its own 128-byte line; launch k uses set k & 1 and clears set (k + 1) & 1
  alignas(128) unsigned long long small_sums[2][kSmallWords * kSumStride];
  // tile counters of the bulk-copy gather: {next tile to claim, CTAs finished} per slot;
  // each launch takes the next slot of the ring, and its last CTA resets the slot to 0
  unsigned long long gather_sched[kGatherSlots][2];
  DevPartial partials[kMaxPartialBlocks];
};

struct HostHParams {
  float lr, beta1, beta2, eps, weight_decay;
};

struct ReduceLaunch {
  const void* const* grads;  // host array of nd device pointers (span-relative)
  int nd;
  float* gsum;               // workspace, n_span floats
  int64_t n_span;            // elements in the span (multiple of 8)
  int64_t n_valid;           // real parameters at the start of the span
  DevScratch* scratch;
  bool finalize;             // compute the step scalars in the last CTA
  float loss_scale, clip;
  HostHParams hp;
  int grid;                  // CTAs (<= kMaxPartialBlocks)
};

struct UpdateLaunch {
  const float* gsum;
  float *master, *exp_avg, *exp_avg_sq;
  void* param16;
  int64_t n_span, n_valid;
  DevScratch* scratch;
  int grid;
};

struct GatherSeg {
  const uint16_t* src;
  uint16_t* dst;
  int64_t len;         // elements
  int64_t tile_begin;  // first global tile index of this segment
};

struct GatherLaunch {
  GatherSeg seg[kGatherSegs];
  int nseg;
  int64_t tiles;       // total tiles over all segments
  int grid;
  int32_t* status;     // set to kStatusGatherWait if a bounded wait expires
  unsigned long long* sched;  // this launch's {next tile, CTAs done} slot, zero at launch
  int realign;         // 1: every segment's source and destination differ in alignment
                       // modulo 16 bytes (k_gather_realign); 0: they agree (k_gather)
};

constexpr int64_t kGatherTile = 32768;    // elements per tile of the realigning gather (64 KiB)
constexpr int64_t kGatherTileAl = 16384;  // elements per tile of the bulk-copy gather (32 KiB)
constexpr int32_t kStatusGatherWait = 4;

// *spare_cta (if given) is set to 1 when the launch carried the spare CTA that computes
// the next step's t-only scalars (spans below one wave), else 0.
cudaError_t launch_reduce(const ReduceLaunch& p, cudaStream_t s, int* spare_cta = nullptr);
// One thread: the t-only scalars for the step counter now in the scratch, into their slot
// (a no-op when the slot holds them already).
cudaError_t launch_next_scalars(DevScratch* scratch, const HostHParams& hp, cudaStream_t s);
cudaError_t launch_finalize(DevScratch* scratch, float loss_scale, float clip,
                            const HostHParams& hp, cudaStream_t s);
cudaError_t launch_update(const UpdateLaunch& p, cudaStream_t s);

// The whole step as one cooperative launch, for spans of at most small_step_max_vecs()
// groups of 8 (see k_step_small). Same arguments as the reduce plus the bound state.
struct SmallLaunch {
  ReduceLaunch r;  // grads, nd, n_span, n_valid, scratch, loss_scale, clip, hp (gsum unused)
  float *master, *exp_avg, *exp_avg_sq;
  void* param16;
};
long long small_step_max_vecs();  // 0 when the device cannot run it
cudaError_t launch_small_step(const SmallLaunch& p, cudaStream_t s);
constexpr int32_t kStatusStepWait = 5;  // the fused step's grid barrier expired
cudaError_t launch_gather(const GatherLaunch& p, cudaStream_t s);

// The bounds-fault words {site, offset} of the step and gather kernels' translation units
// (bounds.h): return 0 in a bounds-checked build, 1 (zeros written) in the normal build,
// -1 on a CUDA error; `reset` zeroes them after the read.
int bounds_words_step(unsigned long long* out, bool reset);
int bounds_words_gather(unsigned long long* out, bool reset);
// Runs the bounds self-test kernel (gather_kernel.cu) and waits for it.
cudaError_t bounds_probe();

// Set the calling thread's zero_last_error() message; returns code.
int set_error(int code, const char* msg);

// Occupancy-derived persistent grid size of the gather for the current device.
int gather_grid(int64_t tiles);

}  // namespace zero
