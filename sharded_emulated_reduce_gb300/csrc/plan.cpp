// Host side of libzero: plans, argument checks, the gather's segment planner, kernel
// timing and the C ABI declared in include/zero.h.
//
// Every entry point checks all of its arguments before it makes any CUDA call, so an
// invalid call launches nothing and changes nothing.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstddef>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "internal.h"

using zero::DevScratch;

namespace {

thread_local std::string g_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_error = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(ZERO_ECUDA, "%s: %s (%d)", what, cudaGetErrorString(e), (int)e);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct EventPair {
  cudaEvent_t start = nullptr, stop = nullptr;
  int kind = 0;
};

constexpr size_t kMaxPendingEvents = 1 << 16;

}  // namespace

int zero::set_error(int code, const char* msg) {
  g_error = msg;
  return code;
}

struct zero_plan {
  int64_t n = 0, np = 0, s = 0;
  int32_t nd = 0, stage = 0, align = 0;
  zero::HostHParams hp{};

  bool bound = false;
  int32_t r0 = 0, r1 = 0;
  float *master = nullptr, *exp_avg = nullptr, *exp_avg_sq = nullptr;
  void* param16 = nullptr;
  float* workspace = nullptr;

  int device = -1;
  DevScratch* scratch = nullptr;
  zero::DevScalars* host_sc = nullptr;  // pinned
  cudaStream_t last_stream = nullptr;    // stream of the last step (zero_step_result)
  cudaStream_t gather_stream = nullptr;  // stream of the last gather (zero_gather_status)
  // second stream for the next step's t-only scalars, forked after a full-wave reduce
  // and joined before the caller's stream goes on
  cudaStream_t side = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  // second stream of the layer-by-layer gather (zero_gather_layers_events): every other
  // layer's copy runs there, so that it starts on the SMs the previous layer leaves
  cudaStream_t gside = nullptr;
  cudaEvent_t gev_fork = nullptr, gev_join = nullptr;
  unsigned gather_launches = 0;  // picks each bulk-copy gather launch's tile-counter slot
  bool stepped = false;

  bool scaler_on = false;  // host mirror of the device scaler's on/off switch

  bool prof = false;
  std::vector<EventPair> free_events, pending;
  double prof_ms[ZERO_PROF_KINDS] = {};
  int64_t prof_launches[ZERO_PROF_KINDS] = {};
};

namespace {

// Padded length and shard length; written independently of any other module from the
// definition: pad to a multiple of nd * align, split into nd equal shards.
void partition(int64_t n, int32_t nd, int32_t align, int64_t* np, int64_t* s) {
  const int64_t unit = (int64_t)nd * align;
  *np = (n + unit - 1) / unit * unit;
  *s = *np / nd;
}

int check_span(const zero_plan* p, int32_t r0, int32_t r1) {
  if (!p) return fail(ZERO_EINVAL, "plan is NULL");
  if (r0 < 0 || r1 > p->nd || r0 >= r1)
    return fail(ZERO_EINVAL, "rank range [%d, %d) is not a non-empty subrange of [0, %d)", r0,
                r1, p->nd);
  return ZERO_OK;
}

int check_bound(const zero_plan* p, int32_t r0, int32_t r1) {
  int rc = check_span(p, r0, r1);
  if (rc) return rc;
  if (!p->bound) return fail(ZERO_EUNBOUND, "no state is bound to the plan");
  if (r0 != p->r0 || r1 != p->r1)
    return fail(ZERO_EUNBOUND, "rank range [%d, %d) differs from the bound range [%d, %d)", r0,
                r1, p->r0, p->r1);
  return ZERO_OK;
}

int check_device(const zero_plan* p) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev != p->device)
    return fail(ZERO_EINVAL, "current device %d differs from the plan's device %d", dev,
                p->device);
  return ZERO_OK;
}

int check_grads(const zero_plan* p, const void* const* grads) {
  if (!grads) return fail(ZERO_EINVAL, "grad_ptrs is NULL");
  for (int k = 0; k < p->nd; ++k) {
    if (!grads[k]) return fail(ZERO_EINVAL, "grad_ptrs[%d] is NULL", k);
    if (!aligned16(grads[k])) return fail(ZERO_EALIGN, "grad_ptrs[%d] is not 16-byte aligned", k);
  }
  return ZERO_OK;
}

int check_scalars(const zero_plan* p, float loss_scale, float clip) {
  if (p->scaler_on) {
    if (loss_scale != 0.0f)
      return fail(ZERO_EINVAL, "the plan's dynamic loss scaler is on: pass loss_scale = 0");
  } else if (!std::isfinite(loss_scale) || loss_scale <= 0.0f) {
    return fail(ZERO_EINVAL, "loss_scale must be finite and > 0 (got %g)", (double)loss_scale);
  }
  if (!std::isfinite(clip)) return fail(ZERO_EINVAL, "clip must be finite (got %g)", (double)clip);
  return ZERO_OK;
}

void prof_begin(zero_plan* p, cudaStream_t s, EventPair* ev) {
  ev->start = nullptr;
  if (!p->prof || p->pending.size() >= kMaxPendingEvents) return;
  if (p->free_events.empty()) {
    EventPair e;
    if (cudaEventCreate(&e.start) != cudaSuccess) return;
    if (cudaEventCreate(&e.stop) != cudaSuccess) {
      cudaEventDestroy(e.start);
      return;
    }
    p->free_events.push_back(e);
  }
  *ev = p->free_events.back();
  p->free_events.pop_back();
  cudaEventRecord(ev->start, s);
}

void prof_end(zero_plan* p, cudaStream_t s, EventPair* ev, int kind) {
  if (!ev->start) return;
  cudaEventRecord(ev->stop, s);
  ev->kind = kind;
  p->pending.push_back(*ev);
}

// The plan's device scratch and pinned result buffer, allocated once on `dev`.
int ensure_scratch(zero_plan* p, int dev) {
  if (p->scratch) return ZERO_OK;
  DevScratch* sc = nullptr;
  cudaError_t e = cudaMalloc(&sc, sizeof(DevScratch));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(scratch)");
  e = cudaMemset(sc, 0, sizeof(DevScratch));
  if (e != cudaSuccess) {
    cudaFree(sc);
    return cuda_fail(e, "cudaMemset(scratch)");
  }
  zero::DevScalars* hs = nullptr;
  e = cudaMallocHost(&hs, sizeof(zero::DevScalars));
  if (e != cudaSuccess) {
    cudaFree(sc);
    return cuda_fail(e, "cudaMallocHost");
  }
  // the second stream for the next step's t-only scalars, made here (outside any graph
  // capture the caller may start later)
  cudaStream_t side = nullptr, gside = nullptr;
  cudaEvent_t ev[4] = {};
  e = cudaStreamCreateWithFlags(&side, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&gside, cudaStreamNonBlocking);
  for (int i = 0; i < 4 && e == cudaSuccess; ++i)
    e = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming);
  if (e != cudaSuccess) {
    for (cudaEvent_t x : ev)
      if (x) cudaEventDestroy(x);
    if (gside) cudaStreamDestroy(gside);
    if (side) cudaStreamDestroy(side);
    cudaFreeHost(hs);
    cudaFree(sc);
    return cuda_fail(e, "second streams");
  }
  p->scratch = sc;
  p->host_sc = hs;
  p->device = dev;
  p->side = side;
  p->ev_fork = ev[0];
  p->ev_join = ev[1];
  p->gside = gside;
  p->gev_fork = ev[2];
  p->gev_join = ev[3];
  return ZERO_OK;
}

int64_t n_valid_of_span(const zero_plan* p) {
  const int64_t first = (int64_t)p->r0 * p->s;
  const int64_t n_span = (int64_t)(p->r1 - p->r0) * p->s;
  return std::max<int64_t>(0, std::min<int64_t>(n_span, p->n - first));
}

int do_reduce(zero_plan* p, const void* const* grads, bool finalize, float loss_scale,
              float clip, cudaStream_t s, int* spare_cta = nullptr) {
  // contributions are span-relative: element i of rank k is flat index r0*S + i
  zero::ReduceLaunch rl{};
  rl.grads = grads;
  rl.nd = p->nd;
  rl.gsum = p->workspace;
  rl.n_span = (int64_t)(p->r1 - p->r0) * p->s;
  rl.n_valid = n_valid_of_span(p);
  rl.scratch = p->scratch;
  rl.finalize = finalize;
  rl.loss_scale = loss_scale;
  rl.clip = clip;
  rl.hp = p->hp;
  rl.grid = 0;
  EventPair ev;
  prof_begin(p, s, &ev);
  cudaError_t e = zero::launch_reduce(rl, s, spare_cta);
  prof_end(p, s, &ev, 0);
  if (e != cudaSuccess) return cuda_fail(e, "reduce launch");
  return ZERO_OK;
}

// The next step's t-only scalars on the plan's second stream: forked from s after the
// reduce (whose combine has advanced the step counter), joined back into s after the
// update, so the next operation on s finds them done. They run while the update runs.
int fork_next_scalars(zero_plan* p, cudaStream_t s) {
  cudaError_t e = cudaEventRecord(p->ev_fork, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(p->side, p->ev_fork, 0);
  if (e != cudaSuccess) return cuda_fail(e, "fork");
  EventPair ev;
  prof_begin(p, p->side, &ev);
  e = zero::launch_next_scalars(p->scratch, p->hp, p->side);
  prof_end(p, p->side, &ev, 2);
  if (e == cudaSuccess) e = cudaEventRecord(p->ev_join, p->side);
  if (e != cudaSuccess) return cuda_fail(e, "next-step scalars");
  return ZERO_OK;
}

// The whole step as one cooperative launch, when the span is small enough for the fused
// kernel (a graph capture records it as a cooperative kernel node).
bool small_step_fits(const zero_plan* p) {
  const int64_t n_vec = (int64_t)(p->r1 - p->r0) * p->s / 8;
  return p->nd <= 64 && n_vec <= zero::small_step_max_vecs();
}

int do_small_step(zero_plan* p, const void* const* grads, float loss_scale, float clip,
                  cudaStream_t s) {
  zero::SmallLaunch sl{};
  sl.r.grads = grads;
  sl.r.nd = p->nd;
  sl.r.gsum = nullptr;
  sl.r.n_span = (int64_t)(p->r1 - p->r0) * p->s;
  sl.r.n_valid = n_valid_of_span(p);
  sl.r.scratch = p->scratch;
  sl.r.finalize = true;
  sl.r.loss_scale = loss_scale;
  sl.r.clip = clip;
  sl.r.hp = p->hp;
  sl.master = p->master;
  sl.exp_avg = p->exp_avg;
  sl.exp_avg_sq = p->exp_avg_sq;
  sl.param16 = p->param16;
  EventPair ev;
  prof_begin(p, s, &ev);
  cudaError_t e = zero::launch_small_step(sl, s);
  prof_end(p, s, &ev, 4);
  if (e != cudaSuccess) return cuda_fail(e, "fused step launch");
  return ZERO_OK;
}

int join_next_scalars(zero_plan* p, cudaStream_t s) {
  cudaError_t e = cudaStreamWaitEvent(s, p->ev_join, 0);
  if (e != cudaSuccess) return cuda_fail(e, "join");
  return ZERO_OK;
}

int do_update(zero_plan* p, cudaStream_t s) {
  zero::UpdateLaunch ul{};
  ul.gsum = p->workspace;
  ul.master = p->master;
  ul.exp_avg = p->exp_avg;
  ul.exp_avg_sq = p->exp_avg_sq;
  ul.param16 = p->param16;
  ul.n_span = (int64_t)(p->r1 - p->r0) * p->s;
  ul.n_valid = n_valid_of_span(p);
  ul.scratch = p->scratch;
  ul.grid = 0;
  EventPair ev;
  prof_begin(p, s, &ev);
  cudaError_t e = zero::launch_update(ul, s);
  prof_end(p, s, &ev, 1);
  if (e != cudaSuccess) return cuda_fail(e, "update launch");
  return ZERO_OK;
}

// Arguments of a gather: checked in full before anything is enqueued. Allocates the
// plan's device scratch (which holds the gather's status word) on first use.
int check_gather(zero_plan* p, const int64_t* offs, int32_t n_layers, const void* const* shards,
                 void* const* dst) {
  if (!p) return fail(ZERO_EINVAL, "plan is NULL");
  if (!offs || !shards || !dst) return fail(ZERO_EINVAL, "NULL array argument");
  if (n_layers < 1) return fail(ZERO_EINVAL, "n_layers must be >= 1");
  if (offs[0] < 0) return fail(ZERO_EINVAL, "layer_offsets[0] must be >= 0");
  for (int l = 0; l < n_layers; ++l) {
    if (offs[l + 1] < offs[l]) return fail(ZERO_EINVAL, "layer_offsets must be non-decreasing");
    if (offs[l + 1] > offs[l]) {
      if (!dst[l]) return fail(ZERO_EINVAL, "layer_dst[%d] is NULL", l);
      if (reinterpret_cast<uintptr_t>(dst[l]) & 1u)
        return fail(ZERO_EALIGN, "layer_dst[%d] is not 2-byte aligned", l);
    }
  }
  if (offs[n_layers] > p->n)
    return fail(ZERO_EINVAL, "layer_offsets[%d] = %lld exceeds n_params = %lld", n_layers,
                (long long)offs[n_layers], (long long)p->n);
  for (int r = 0; r < p->nd; ++r) {
    if (!shards[r]) return fail(ZERO_EINVAL, "shard_ptrs[%d] is NULL", r);
    if (reinterpret_cast<uintptr_t>(shards[r]) & 1u)
      return fail(ZERO_EALIGN, "shard_ptrs[%d] is not 2-byte aligned", r);
  }
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (p->device >= 0 && dev != p->device)
    return fail(ZERO_EINVAL, "current device %d differs from the plan's device %d", dev, p->device);
  return ensure_scratch(p, dev);
}

// The two segment tables of a gather launch: source and destination equal modulo 16 bytes
// (t[0], k_gather), or not (t[1], k_gather_realign); tiles are numbered per table.
struct GatherTables {
  zero::GatherLaunch t[2];
  explicit GatherTables(zero_plan* p) {
    for (int k = 0; k < 2; ++k) {
      t[k].nseg = 0;
      t[k].tiles = 0;
      t[k].grid = 0;
      t[k].status = &p->scratch->gather_status;
      t[k].sched = nullptr;
      t[k].realign = k;
    }
  }
};

int flush_gather(zero_plan* p, zero::GatherLaunch& gl, cudaStream_t s) {
  if (gl.nseg == 0) return ZERO_OK;
  // the next slot of the ring of tile counters (each is zero again once its launch ends)
  gl.sched = p->scratch->gather_sched[p->gather_launches++ % zero::kGatherSlots];
  EventPair ev;
  prof_begin(p, s, &ev);
  cudaError_t e = zero::launch_gather(gl, s);
  prof_end(p, s, &ev, 3);
  gl.nseg = 0;
  gl.tiles = 0;
  if (e != cudaSuccess) return cuda_fail(e, "gather launch");
  return ZERO_OK;
}

// Cut layer l at shard boundaries into copy segments, each into the table of its alignment
// class; a full table is launched on s first.
int plan_layer(zero_plan* p, const int64_t* offs, int l, const void* const* shards,
               void* const* dst, GatherTables& gt, cudaStream_t s) {
  const int64_t a = offs[l], b = offs[l + 1];
  for (int64_t r = a / p->s; a < b && r * p->s < b; ++r) {
    const int64_t lo = std::max(a, r * p->s), hi = std::min(b, (r + 1) * p->s);
    if (hi <= lo) continue;
    const uint16_t* src = static_cast<const uint16_t*>(shards[r]) + (lo - r * p->s);
    uint16_t* dptr = static_cast<uint16_t*>(dst[l]) + (lo - a);
    const int k =
        ((reinterpret_cast<uintptr_t>(src) - reinterpret_cast<uintptr_t>(dptr)) & 15u) ? 1 : 0;
    zero::GatherLaunch& gl = gt.t[k];
    if (gl.nseg == zero::kGatherSegs) {
      int rc = flush_gather(p, gl, s);
      if (rc) return rc;
    }
    zero::GatherSeg& sg = gl.seg[gl.nseg++];
    sg.src = src;
    sg.dst = dptr;
    sg.len = hi - lo;
    sg.tile_begin = gl.tiles;
    const int64_t tile = k ? zero::kGatherTile : zero::kGatherTileAl;
    gl.tiles += (sg.len + tile - 1) / tile;
  }
  return ZERO_OK;
}

}  // namespace

extern "C" {

int zero_plan_create(int64_t n_params, int32_t nd, int32_t stage, int32_t align,
                     const zero_adam_hparams* hp, zero_plan** out) {
  g_error.clear();
  if (!out) return fail(ZERO_EINVAL, "out is NULL");
  *out = nullptr;
  if (n_params < 1) return fail(ZERO_EINVAL, "n_params must be >= 1");
  if (nd < 1 || nd > ZERO_MAX_ND) return fail(ZERO_EINVAL, "nd must be in [1, %d]", ZERO_MAX_ND);
  if (stage < 1 || stage > 3) return fail(ZERO_EINVAL, "stage must be 1, 2 or 3");
  if (align < 8 || align % 8 != 0) return fail(ZERO_EINVAL, "align must be a positive multiple of 8");
  if (!hp) return fail(ZERO_EINVAL, "hp is NULL");
  const float f[5] = {hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay};
  for (float x : f)
    if (!std::isfinite(x)) return fail(ZERO_EINVAL, "hyperparameters must be finite");
  if (hp->lr < 0 || hp->beta1 < 0 || hp->beta1 >= 1 || hp->beta2 < 0 || hp->beta2 >= 1 ||
      hp->eps <= 0 || hp->weight_decay < 0)
    return fail(ZERO_EINVAL, "need lr >= 0, 0 <= beta1, beta2 < 1, eps > 0, weight_decay >= 0");
  const int64_t unit = (int64_t)nd * align;
  if (n_params > INT64_MAX - unit) return fail(ZERO_EINVAL, "n_params too large");
  int64_t np, s;
  partition(n_params, nd, align, &np, &s);
  // exact sum of squares: Np * nd^2 * (65504 * 2^24 * (1 + 2^-20))^2 must stay below 2^128
  const long double bound = (long double)np * nd * nd;
  if (bound >= 140737488355328.0L)  // 2^47
    return fail(ZERO_EINVAL, "Np * nd^2 must be below 2^47 (Np = %lld, nd = %d)", (long long)np, nd);
  zero_plan* p = new (std::nothrow) zero_plan();
  if (!p) return fail(ZERO_EINVAL, "out of host memory");
  p->n = n_params;
  p->np = np;
  p->s = s;
  p->nd = nd;
  p->stage = stage;
  p->align = align;
  p->hp = {hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay};
  *out = p;
  return ZERO_OK;
}

void zero_plan_destroy(zero_plan* p) {
  if (!p) return;
  int prev = -1;
  const bool has_dev = p->device >= 0 && cudaGetDevice(&prev) == cudaSuccess;
  if (has_dev && prev != p->device) cudaSetDevice(p->device);
  for (auto& e : p->pending) p->free_events.push_back(e);
  for (auto& e : p->free_events) {
    cudaEventDestroy(e.start);
    cudaEventDestroy(e.stop);
  }
  if (p->side) cudaStreamDestroy(p->side);
  if (p->ev_fork) cudaEventDestroy(p->ev_fork);
  if (p->ev_join) cudaEventDestroy(p->ev_join);
  if (p->gside) cudaStreamDestroy(p->gside);
  if (p->gev_fork) cudaEventDestroy(p->gev_fork);
  if (p->gev_join) cudaEventDestroy(p->gev_join);
  if (p->scratch) cudaFree(p->scratch);
  if (p->host_sc) cudaFreeHost(p->host_sc);
  if (has_dev && prev != p->device) cudaSetDevice(prev);
  delete p;
}

int zero_plan_layout(const zero_plan* p, int64_t* padded_len, int64_t* shard_len) {
  g_error.clear();
  if (!p || !padded_len || !shard_len) return fail(ZERO_EINVAL, "NULL argument");
  *padded_len = p->np;
  *shard_len = p->s;
  return ZERO_OK;
}

int64_t zero_workspace_bytes(const zero_plan* p, int32_t r0, int32_t r1) {
  g_error.clear();
  int rc = check_span(p, r0, r1);
  if (rc) return rc;
  return 4 * (int64_t)(r1 - r0) * p->s;
}

int zero_plan_bind(zero_plan* p, int32_t r0, int32_t r1, float* master, float* exp_avg,
                   float* exp_avg_sq, void* param16, void* workspace, int64_t initial_step) {
  g_error.clear();
  int rc = check_span(p, r0, r1);
  if (rc) return rc;
  void* ptrs[5] = {master, exp_avg, exp_avg_sq, param16, workspace};
  const char* names[5] = {"master", "exp_avg", "exp_avg_sq", "param16", "workspace"};
  for (int i = 0; i < 5; ++i) {
    if (!ptrs[i]) return fail(ZERO_EINVAL, "%s is NULL", names[i]);
    if (!aligned16(ptrs[i])) return fail(ZERO_EALIGN, "%s is not 16-byte aligned", names[i]);
  }
  if (initial_step < 0) return fail(ZERO_EINVAL, "initial_step must be >= 0");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (p->scratch && dev != p->device)
    return fail(ZERO_EINVAL, "plan was bound on device %d; current device is %d", p->device, dev);
  rc = ensure_scratch(p, dev);
  if (rc) return rc;
  long long t = initial_step;
  e = cudaMemcpy(&p->scratch->step, &t, sizeof t, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(step)");
  p->bound = true;
  p->r0 = r0;
  p->r1 = r1;
  p->master = master;
  p->exp_avg = exp_avg;
  p->exp_avg_sq = exp_avg_sq;
  p->param16 = param16;
  p->workspace = static_cast<float*>(workspace);
  p->stepped = false;
  return ZERO_OK;
}

int zero_shard_step(zero_plan* p, int32_t r0, int32_t r1, const void* const* grads,
                    float loss_scale, float clip, void* stream) {
  g_error.clear();
  int rc = check_span(p, r0, r1);
  if (!rc) rc = check_grads(p, grads);
  if (!rc) rc = check_scalars(p, loss_scale, clip);
  if (!rc) rc = check_bound(p, r0, r1);
  if (!rc) rc = check_device(p);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (small_step_fits(p)) {
    rc = do_small_step(p, grads, loss_scale, clip, s);
    if (rc) return rc;
    p->last_stream = s;
    p->stepped = true;
    return ZERO_OK;
  }
  int spare = 0;
  rc = do_reduce(p, grads, true, loss_scale, clip, s, &spare);
  if (rc) return rc;
  // a full-wave reduce has no spare CTA for the next step's t-only scalars
  const bool side = !spare;
  if (side) rc = fork_next_scalars(p, s);
  if (rc) return rc;
  rc = do_update(p, s);
  if (!rc && side) rc = join_next_scalars(p, s);
  if (rc) return rc;
  p->last_stream = s;
  p->stepped = true;
  return ZERO_OK;
}

int zero_shard_reduce(zero_plan* p, int32_t r0, int32_t r1, const void* const* grads,
                      void* stream) {
  g_error.clear();
  int rc = check_span(p, r0, r1);
  if (!rc) rc = check_grads(p, grads);
  if (!rc) rc = check_bound(p, r0, r1);
  if (!rc) rc = check_device(p);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  rc = do_reduce(p, grads, false, 1.0f, 0.0f, s);
  if (rc) return rc;
  p->last_stream = s;
  return ZERO_OK;
}

int zero_shard_stats(zero_plan* p, void** dev_words) {
  g_error.clear();
  if (!p || !dev_words) return fail(ZERO_EINVAL, "NULL argument");
  if (!p->scratch) return fail(ZERO_EUNBOUND, "no state is bound to the plan");
  *dev_words = p->scratch->stats;
  return ZERO_OK;
}

int zero_shard_update(zero_plan* p, int32_t r0, int32_t r1, float loss_scale, float clip,
                      void* stream) {
  g_error.clear();
  int rc = check_span(p, r0, r1);
  if (!rc) rc = check_scalars(p, loss_scale, clip);
  if (!rc) rc = check_bound(p, r0, r1);
  if (!rc) rc = check_device(p);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  EventPair ev;
  prof_begin(p, s, &ev);
  cudaError_t e = zero::launch_finalize(p->scratch, loss_scale, clip, p->hp, s);
  prof_end(p, s, &ev, 2);
  if (e != cudaSuccess) return cuda_fail(e, "finalize launch");
  rc = do_update(p, s);
  if (rc) return rc;
  p->last_stream = s;
  p->stepped = true;
  return ZERO_OK;
}

int zero_step_result(zero_plan* p, zero_step_info* out) {
  g_error.clear();
  if (!p || !out) return fail(ZERO_EINVAL, "NULL argument");
  if (!p->bound || !p->stepped) return fail(ZERO_EUNBOUND, "the plan has not stepped yet");
  int rc = check_device(p);
  if (rc) return rc;
  cudaError_t e = cudaMemcpyAsync(p->host_sc, &p->scratch->sc, sizeof(zero::DevScalars),
                                  cudaMemcpyDeviceToHost, p->last_stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(p->last_stream);
  if (e != cudaSuccess) return cuda_fail(e, "step result");
  const zero::DevScalars& sc = *p->host_sc;
  std::memset(out, 0, sizeof *out);
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
  if (sc.status == zero::kStatusStepWait) {
    // the one-launch step's wait gave up: start its launch count and counting sums (and
    // the reduce's tile counter between them, zero between launches) from zero
    constexpr size_t first = offsetof(zero::DevScratch, small_launch);
    constexpr size_t end = offsetof(zero::DevScratch, small_sums) + sizeof(zero::DevScratch::small_sums);
    cudaMemsetAsync(reinterpret_cast<unsigned char*>(p->scratch) + first, 0, end - first,
                    p->last_stream);
    cudaStreamSynchronize(p->last_stream);
  }
  if (sc.status != 0) return fail(ZERO_EDEVICE, "device status %d", sc.status);
  return ZERO_OK;
}

int zero_gather_layers(zero_plan* p, const int64_t* offs, int32_t n_layers,
                       const void* const* shards, void* const* dst, void* stream) {
  g_error.clear();
  int rc = check_gather(p, offs, n_layers, shards, dst);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  GatherTables gt(p);
  for (int l = 0; l < n_layers && !rc; ++l) rc = plan_layer(p, offs, l, shards, dst, gt, s);
  if (!rc) rc = flush_gather(p, gt.t[0], s);
  if (!rc) rc = flush_gather(p, gt.t[1], s);
  if (!rc) p->gather_stream = s;
  return rc;
}

int zero_gather_layers_events(zero_plan* p, const int64_t* offs, int32_t n_layers,
                              const void* const* shards, void* const* dst,
                              void* const* layer_done, void* stream) {
  g_error.clear();
  if (!layer_done) return fail(ZERO_EINVAL, "layer_done is NULL");
  int rc = check_gather(p, offs, n_layers, shards, dst);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // layers 0, 2, 4, ... on the caller's stream, 1, 3, 5, ... on the plan's second gather
  // stream, which starts after the work already on `stream` and is joined back into it
  // at the end: consecutive layers overlap, so the next layer's CTAs take the SMs the
  // previous layer's last CTAs leave, and each layer's event marks that layer alone
  cudaError_t e = cudaEventRecord(p->gev_fork, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(p->gside, p->gev_fork, 0);
  if (e != cudaSuccess) return cuda_fail(e, "gather fork");
  GatherTables gt(p);
  for (int l = 0; l < n_layers && !rc; ++l) {
    cudaStream_t sl = (l & 1) ? p->gside : s;
    rc = plan_layer(p, offs, l, shards, dst, gt, sl);
    if (!rc) rc = flush_gather(p, gt.t[0], sl);
    if (!rc) rc = flush_gather(p, gt.t[1], sl);
    if (!rc && layer_done[l]) {
      e = cudaEventRecord(static_cast<cudaEvent_t>(layer_done[l]), sl);
      if (e != cudaSuccess)
        rc = fail(ZERO_ECUDA, "cudaEventRecord(layer_done[%d]): %s (%d)", l,
                  cudaGetErrorString(e), (int)e);
    }
  }
  // join even after an error, so that the caller's stream still orders after the work
  // already enqueued
  e = cudaEventRecord(p->gev_join, p->gside);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, p->gev_join, 0);
  if (!rc && e != cudaSuccess) rc = cuda_fail(e, "gather join");
  if (!rc) p->gather_stream = s;
  return rc;
}

int zero_gather_status(zero_plan* p, int32_t* status) {
  g_error.clear();
  if (!p || !status) return fail(ZERO_EINVAL, "NULL argument");
  if (!p->scratch) {
    *status = 0;  // no gather has run
    return ZERO_OK;
  }
  int rc = check_device(p);
  if (rc) return rc;
  cudaError_t e = cudaStreamSynchronize(p->gather_stream);
  int32_t st = 0;
  if (e == cudaSuccess)
    e = cudaMemcpy(&st, &p->scratch->gather_status, sizeof st, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && st != 0) e = cudaMemset(&p->scratch->gather_status, 0, sizeof st);
  if (e != cudaSuccess) return cuda_fail(e, "gather status");
  *status = st;
  if (st != 0) return fail(ZERO_EDEVICE, "a gather stopped early (status %d)", st);
  return ZERO_OK;
}

int zero_memory_bytes(int64_t n, int32_t nd, int32_t align, int32_t stage, int64_t* out) {
  g_error.clear();
  if (!out) return fail(ZERO_EINVAL, "out is NULL");
  if (n < 1 || nd < 1 || align < 1) return fail(ZERO_EINVAL, "need n >= 1, nd >= 1, align >= 1");
  int64_t np, s;
  partition(n, nd, align, &np, &s);
  switch (stage) {
    case 0: *out = 16 * n; break;          // replicated: 2 + 2 + 12 bytes per parameter
    case 1: *out = 4 * n + 12 * s; break;  // optimizer states partitioned
    case 2: *out = 2 * n + 14 * s; break;  // + gradients
    case 3: *out = 16 * s; break;          // + parameters
    default: return fail(ZERO_EINVAL, "stage must be 0, 1, 2 or 3");
  }
  return ZERO_OK;
}

int zero_bounds_check(int32_t reset, int32_t* enabled, int32_t* site, int64_t* offset) {
  g_error.clear();
  if (!enabled || !site || !offset) return fail(ZERO_EINVAL, "enabled, site and offset are required");
  unsigned long long a[2], b[2];
  const int ra = zero::bounds_words_step(a, reset != 0);
  const int rb = zero::bounds_words_gather(b, reset != 0);
  if (ra < 0 || rb < 0) return fail(ZERO_ECUDA, "reading the bounds-fault words failed");
  const unsigned long long* f = a[0] != 0 ? a : b;
  *enabled = ra == 0 ? 1 : 0;
  *site = static_cast<int32_t>(f[0]);
  *offset = static_cast<int64_t>(f[1]);
  return ZERO_OK;
}

int zero_selftest_bounds(void) {
  g_error.clear();
  const cudaError_t e = zero::bounds_probe();
  if (e != cudaSuccess) return cuda_fail(e, "bounds self-test");
  return ZERO_OK;
}

int zero_profile_enable(zero_plan* p, int32_t on) {
  g_error.clear();
  if (!p) return fail(ZERO_EINVAL, "plan is NULL");
  p->prof = on != 0;
  return ZERO_OK;
}

int zero_profile_read(zero_plan* p, double* ms, int64_t* launches, int32_t reset) {
  g_error.clear();
  if (!p) return fail(ZERO_EINVAL, "plan is NULL");
  for (auto& ev : p->pending) {
    cudaError_t e = cudaEventSynchronize(ev.stop);
    float t = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&t, ev.start, ev.stop);
    if (e != cudaSuccess) return cuda_fail(e, "profile events");
    p->prof_ms[ev.kind] += t;
    p->prof_launches[ev.kind] += 1;
    p->free_events.push_back(ev);
  }
  p->pending.clear();
  for (int k = 0; k < ZERO_PROF_KINDS; ++k) {
    if (ms) ms[k] = p->prof_ms[k];
    if (launches) launches[k] = p->prof_launches[k];
    if (reset) {
      p->prof_ms[k] = 0;
      p->prof_launches[k] = 0;
    }
  }
  return ZERO_OK;
}

namespace {

int check_scaler(const zero_loss_scaler* c) {
  if (!c) return fail(ZERO_EINVAL, "scaler is NULL");
  if (c->growth_interval < 0) return fail(ZERO_EINVAL, "growth_interval must be >= 0");
  if (c->growth_interval == 0) return ZERO_OK;  // off: the other fields are not used
  if (!std::isfinite(c->scale) || c->scale <= 0.0f)
    return fail(ZERO_EINVAL, "scale must be finite and > 0");
  if (c->good_steps < 0) return fail(ZERO_EINVAL, "good_steps must be >= 0");
  if (!std::isfinite(c->growth_factor) || c->growth_factor < 1.0f)
    return fail(ZERO_EINVAL, "growth_factor must be finite and >= 1");
  if (!(c->backoff_factor > 0.0f) || c->backoff_factor > 1.0f)
    return fail(ZERO_EINVAL, "backoff_factor must be in (0, 1]");
  return ZERO_OK;
}

int sync_last(zero_plan* p) {
  cudaError_t e = cudaStreamSynchronize(p->last_stream);
  return e == cudaSuccess ? ZERO_OK : cuda_fail(e, "cudaStreamSynchronize");
}

int write_scaler(zero_plan* p, const zero_loss_scaler* c) {
  zero::DevScaler d{};
  if (c->growth_interval > 0) {
    d.scale = c->scale;
    d.good_steps = c->good_steps;
    d.growth = c->growth_factor;
    d.backoff = c->backoff_factor;
    d.interval = c->growth_interval;
  }
  cudaError_t e = cudaMemcpy(&p->scratch->scaler, &d, sizeof d, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(scaler)");
  p->scaler_on = c->growth_interval > 0;
  return ZERO_OK;
}

}  // namespace

int zero_plan_set_scaler(zero_plan* p, const zero_loss_scaler* c) {
  g_error.clear();
  if (!p) return fail(ZERO_EINVAL, "plan is NULL");
  int rc = check_scaler(c);
  if (rc) return rc;
  if (!p->bound) return fail(ZERO_EUNBOUND, "no state is bound to the plan");
  rc = check_device(p);
  if (!rc) rc = sync_last(p);
  if (rc) return rc;
  return write_scaler(p, c);
}

int zero_loss_scale_ptr(zero_plan* p, float** dev_scale) {
  g_error.clear();
  if (!p || !dev_scale) return fail(ZERO_EINVAL, "NULL argument");
  if (!p->scratch) return fail(ZERO_EUNBOUND, "no state is bound to the plan");
  *dev_scale = &p->scratch->scaler.scale;
  return ZERO_OK;
}

int zero_plan_get_state(zero_plan* p, zero_plan_state* out) {
  g_error.clear();
  if (!p || !out) return fail(ZERO_EINVAL, "NULL argument");
  if (!p->bound) return fail(ZERO_EUNBOUND, "no state is bound to the plan");
  int rc = check_device(p);
  if (!rc) rc = sync_last(p);
  if (rc) return rc;
  long long t = 0;
  zero::DevScaler d{};
  cudaError_t e = cudaMemcpy(&t, &p->scratch->step, sizeof t, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(&d, &p->scratch->scaler, sizeof d, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(state)");
  std::memset(out, 0, sizeof *out);
  out->step = t;
  out->scaler.scale = d.scale;
  out->scaler.good_steps = d.good_steps;
  out->scaler.growth_factor = d.growth;
  out->scaler.backoff_factor = d.backoff;
  out->scaler.growth_interval = d.interval > 0 ? d.interval : 0;
  return ZERO_OK;
}

int zero_plan_set_state(zero_plan* p, const zero_plan_state* in) {
  g_error.clear();
  if (!p || !in) return fail(ZERO_EINVAL, "NULL argument");
  if (in->step < 0) return fail(ZERO_EINVAL, "step must be >= 0");
  int rc = check_scaler(&in->scaler);
  if (rc) return rc;
  if (!p->bound) return fail(ZERO_EUNBOUND, "no state is bound to the plan");
  rc = check_device(p);
  if (!rc) rc = sync_last(p);
  if (rc) return rc;
  long long t = in->step;
  cudaError_t e = cudaMemcpy(&p->scratch->step, &t, sizeof t, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(step)");
  return write_scaler(p, &in->scaler);
}

const char* zero_last_error(void) { return g_error.c_str(); }

}  // extern "C"
