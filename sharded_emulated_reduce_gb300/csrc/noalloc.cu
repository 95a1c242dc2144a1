// A shard step that allocates no memory: zero_shard_step_noalloc.
//
// Some callers cannot allocate device memory at the point where they run the optimizer
// step: a framework that reserved all of HBM for its own pool at start-up and forbids
// later cudaMalloc calls, an allocator hook that would re-enter its allocator, or a
// latency-bound loop in which cudaMalloc/cudaFree may synchronise the whole device.
// For them this entry point runs the same reduce and update kernels as zero_shard_step,
// but takes all of its scratch (the fp32 rank sums, the per-CTA partials, the step's
// scalars) from one file-scope device array instead of from a plan.
//
// The array is kNoallocSpanMax fp32 values plus the small control block: 16 MiB +
// ~35 KiB. Every GPU that loads this library holds it until the process exits. All calls
// share it, and it keeps the last call's contents, so two calls whose work overlaps on
// the GPU (different streams, or different host threads, without ordering between them)
// race on it and produce wrong results.
#include <mutex>

#include <cstddef>
#include <cstring>

#include "internal.h"

namespace zero {
namespace {

constexpr int64_t kNoallocSpanMax = int64_t(1) << 22;  // 4,194,304 parameters
constexpr size_t kCtrlBytes = (sizeof(DevScratch) + 255) / 256 * 256;
constexpr size_t kNoallocBytes = kCtrlBytes + sizeof(float) * kNoallocSpanMax;

// Device-resident scratch. In host code this name is only a stand-in for the symbol; the
// device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once per device
// (or, with lookup == false, only if it was looked up before; else *out = nullptr).
cudaError_t scratch_address(void** out, bool lookup = true) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_addr[dev] && lookup) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

}  // namespace

}  // namespace zero

extern "C" int zero_shard_step_noalloc(int32_t nd, int64_t n, int64_t n_valid,
                                       const void* const* grad_ptrs, float* master,
                                       float* exp_avg, float* exp_avg_sq, void* param16,
                                       int64_t* step_counter, const zero_adam_hparams* hp,
                                       float loss_scale, float clip, void* stream) {
  using namespace zero;
  auto bad = [](int code, const char* msg) { return set_error(code, msg); };
  set_error(ZERO_OK, "");
  if (nd < 1 || nd > ZERO_MAX_ND) return bad(ZERO_EINVAL, "nd must be in [1, ZERO_MAX_ND]");
  if (n < 8 || n % 8 != 0) return bad(ZERO_EINVAL, "n must be a positive multiple of 8");
  if (n > kNoallocSpanMax)
    return bad(ZERO_EINVAL, "n exceeds ZERO_NOALLOC_MAX_SPAN (4194304) elements");
  if (n_valid < 0 || n_valid > n) return bad(ZERO_EINVAL, "n_valid must be in [0, n]");
  if ((long double)n * nd * nd >= 140737488355328.0L)
    return bad(ZERO_EINVAL, "n * nd^2 must be below 2^47");
  if (!grad_ptrs || !master || !exp_avg || !exp_avg_sq || !param16 || !step_counter || !hp)
    return bad(ZERO_EINVAL, "NULL pointer argument");
  for (int k = 0; k < nd; ++k) {
    if (!grad_ptrs[k]) return bad(ZERO_EINVAL, "grad_ptrs has a NULL entry");
    if (reinterpret_cast<uintptr_t>(grad_ptrs[k]) & 15u)
      return bad(ZERO_EALIGN, "grad_ptrs entries must be 16-byte aligned");
  }
  const void* st_ptrs[4] = {master, exp_avg, exp_avg_sq, param16};
  for (const void* p : st_ptrs)
    if (reinterpret_cast<uintptr_t>(p) & 15u)
      return bad(ZERO_EALIGN, "state pointers must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(step_counter) & 7u)
    return bad(ZERO_EALIGN, "step_counter must be 8-byte aligned");
  if (!(loss_scale > 0.0f) || loss_scale == __builtin_inff())
    return bad(ZERO_EINVAL, "loss_scale must be finite and > 0");
  if (clip != clip || clip == __builtin_inff() || clip == -__builtin_inff())
    return bad(ZERO_EINVAL, "clip must be finite");
  const float f[5] = {hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay};
  for (float x : f)
    if (x != x || x == __builtin_inff() || x == -__builtin_inff())
      return bad(ZERO_EINVAL, "hyperparameters must be finite");
  if (hp->lr < 0 || hp->beta1 < 0 || hp->beta1 >= 1 || hp->beta2 < 0 || hp->beta2 >= 1 ||
      hp->eps <= 0 || hp->weight_decay < 0)
    return bad(ZERO_EINVAL, "need lr >= 0, 0 <= beta1, beta2 < 1, eps > 0, weight_decay >= 0");

  void* base = nullptr;
  cudaError_t e = scratch_address(&base);
  if (e != cudaSuccess) return bad(ZERO_ECUDA, "cudaGetSymbolAddress of the scratch array failed");
  DevScratch* st = static_cast<DevScratch*>(base);
  float* gsum = reinterpret_cast<float*>(static_cast<unsigned char*>(base) + kCtrlBytes);
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // The ticket of the last-arriving CTA, the one-launch step's launch count, the
  // reduce's tile counter and the one-launch step's counting sums (which follow it in
  // this order) must start at zero; the step counter is the caller's and is copied in and
  // out around the kernels.
  constexpr size_t first = offsetof(DevScratch, ticket);
  constexpr size_t end = offsetof(DevScratch, small_sums) + sizeof(DevScratch::small_sums);
  static_assert(offsetof(DevScratch, small_launch) > first &&
                    offsetof(DevScratch, reduce_next) > first &&
                    offsetof(DevScratch, small_sums) > first,
                "the counters follow the ticket");
  e = cudaMemsetAsync(reinterpret_cast<unsigned char*>(st) + first, 0, end - first, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(&st->step, step_counter, sizeof(int64_t), cudaMemcpyDeviceToDevice, s);
  if (e != cudaSuccess) return bad(ZERO_ECUDA, "scratch set-up copy failed");

  const HostHParams hpp = {hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay};
  if (nd <= 64 && n / 8 <= small_step_max_vecs()) {  // the whole step in one launch
    SmallLaunch sl{};
    sl.r.grads = grad_ptrs;
    sl.r.nd = nd;
    sl.r.gsum = nullptr;
    sl.r.n_span = n;
    sl.r.n_valid = n_valid;
    sl.r.scratch = st;
    sl.r.finalize = true;
    sl.r.loss_scale = loss_scale;
    sl.r.clip = clip;
    sl.r.hp = hpp;
    sl.master = master;
    sl.exp_avg = exp_avg;
    sl.exp_avg_sq = exp_avg_sq;
    sl.param16 = param16;
    e = launch_small_step(sl, s);
    if (e != cudaSuccess) return bad(ZERO_ECUDA, "fused step launch failed");
    e = cudaMemcpyAsync(step_counter, &st->step, sizeof(int64_t), cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return bad(ZERO_ECUDA, "step counter copy failed");
    return ZERO_OK;
  }

  ReduceLaunch rl{};
  rl.grads = grad_ptrs;
  rl.nd = nd;
  rl.gsum = gsum;
  rl.n_span = n;
  rl.n_valid = n_valid;
  rl.scratch = st;
  rl.finalize = true;
  rl.loss_scale = loss_scale;
  rl.clip = clip;
  rl.hp = hpp;
  rl.grid = 0;
  e = launch_reduce(rl, s);
  if (e != cudaSuccess) return bad(ZERO_ECUDA, "reduce launch failed");

  UpdateLaunch ul{};
  ul.gsum = gsum;
  ul.master = master;
  ul.exp_avg = exp_avg;
  ul.exp_avg_sq = exp_avg_sq;
  ul.param16 = param16;
  ul.n_span = n;
  ul.n_valid = n_valid;
  ul.scratch = st;
  ul.grid = 0;
  e = launch_update(ul, s);
  if (e != cudaSuccess) return bad(ZERO_ECUDA, "update launch failed");

  e = cudaMemcpyAsync(step_counter, &st->step, sizeof(int64_t), cudaMemcpyDeviceToDevice, s);
  if (e != cudaSuccess) return bad(ZERO_ECUDA, "step counter copy failed");
  return ZERO_OK;
}

extern "C" int zero_noalloc_step_result(void* stream, zero_step_info* out) {
  using namespace zero;
  set_error(ZERO_OK, "");
  if (!out) return set_error(ZERO_EINVAL, "out is NULL");
  void* base = nullptr;
  cudaError_t e = scratch_address(&base, false);
  if (e != cudaSuccess) return set_error(ZERO_ECUDA, "cudaGetDevice failed");
  if (!base)
    return set_error(ZERO_EUNBOUND, "no allocation-free step has run on the current device");
  const DevScratch* st = static_cast<const DevScratch*>(base);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DevScalars sc;  // pageable: the copy completes before cudaMemcpyAsync returns
  e = cudaMemcpyAsync(&sc, &st->sc, sizeof sc, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return set_error(ZERO_ECUDA, "copy of the step result failed");
  memset(out, 0, sizeof *out);
  out->overflow = sc.overflow;
  out->skipped = sc.skipped;
  out->status = sc.status;
  out->step = sc.step;
  out->global_norm = sc.norm;
  out->sum_sq = sc.ss;
  out->clip_coef = sc.clip_coef;
  out->scale = sc.s;
  out->bc1 = sc.bc1;
  out->bc2 = sc.bc2;
  out->loss_scale = sc.loss_scale;
  if (sc.status != 0)
    return set_error(ZERO_EDEVICE, "the allocation-free step reported a device failure");
  return ZERO_OK;
}
