/* libzero: the data-parallel hot path of ZeRO (Zero Redundancy Optimizer) on one GB300.
 *
 * ZeRO keeps data-parallel training but partitions the model states (optimizer states,
 * gradients, parameters) across the Nd data-parallel ranks instead of replicating them
 * ("ZeRO" method entry, codewithpapers.app/method/zero, description; ZeRO explainer,
 * papermap.vercel.app, "The 16 Bytes per Parameter Audit" and Chapter 02 "The Three
 * Stages"). This library computes what one device does in that scheme:
 *
 *   - the partition of a flat parameter buffer into Nd aligned shards;
 *   - the shard step: the sum of the Nd ranks' fp16 gradient contributions over the
 *     owned span (the arithmetic of the reduce-scatter after backward, Chapter 02,
 *     ZeRO-3 item), the inf/nan overflow check, unscaling by the loss scale, optional
 *     global-norm clipping, the mixed-precision AdamW update of the fp32 master weights
 *     and moments, and the fp16 cast (Chapter 02 "Memory per parameter");
 *   - the ZeRO-3 gather of fp16 shards into contiguous per-layer buffers (the
 *     arithmetic of the all-gather before forward, Chapter 02, ZeRO-3 item);
 *   - the per-rank memory accounting of the stage ladder (Chapter 02 "What each stage
 *     shards" and the stage table after Chapter 05).
 *
 * The Nd logical ranks are emulated on one device: their contributions are Nd device
 * buffers, and no inter-GPU collective is issued. A span of logical ranks [r0, r1) can
 * be split across processes; zero_shard_reduce / zero_shard_stats / zero_shard_update
 * expose the single exchange step (a sum of a few integers) for that case.
 *
 * Conventions for every call:
 *   - Device memory (gradients, state, workspace, shards, layer buffers) is allocated
 *     and owned by the caller; the library never frees it. "Device pointer" means an
 *     address the GPU can dereference: HBM, or pinned or registered host memory (on a
 *     GB300 the kernels then read and write it over NVLink-C2C, which is how optimizer
 *     state or fp16 shards can live in Grace memory — the offload variant of ZeRO). A
 *     plan owns only its host metadata, a small device scratch area (< 64 KiB, allocated
 *     by zero_plan_bind on the device current at that time, freed by zero_plan_destroy),
 *     two CUDA streams with their events, and a few pinned host bytes.
 *   - Element types: fp16 buffers are IEEE binary16 (as torch.float16), fp32 buffers
 *     are IEEE binary32. All buffers are contiguous 1-D.
 *   - Streams are cudaStream_t passed as void*; NULL is the legacy default stream.
 *     Launching calls are asynchronous and return once the work is enqueued.
 *   - Return codes: ZERO_OK (0) or a negative ZERO_E* code. On any error nothing is
 *     launched and no state changes; zero_last_error() then gives a message.
 *   - An overflow (inf/nan among the summed gradients) is not an error: the step is
 *     skipped on the device and zero_step_result reports it.
 *   - A plan is not thread-safe; use one plan per host thread.
 */
#ifndef ZERO_H
#define ZERO_H
#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ZERO_OK 0
#define ZERO_EINVAL (-1)   /* an argument is out of range or inconsistent            */
#define ZERO_EALIGN (-2)   /* a device pointer is not 16-byte aligned                */
#define ZERO_EUNBOUND (-3) /* the plan has no state bound for the requested span     */
#define ZERO_ECUDA (-4)    /* a CUDA runtime call failed                             */
#define ZERO_EDEVICE (-5)  /* a kernel reported a failure status (see step info)     */

#define ZERO_MAX_ND 256        /* largest supported number of logical ranks Nd         */
#define ZERO_STATS_WORDS 8     /* int64 words in the exchange buffer of zero_shard_stats */

/* AdamW hyperparameters (fp32). */
typedef struct {
  float lr, beta1, beta2, eps, weight_decay;
} zero_adam_hparams;

/* Result of the last step of a plan. */
typedef struct {
  int32_t overflow;   /* 1 if any summed gradient in the span was inf or nan          */
  int32_t skipped;    /* 1 if the update was not applied (overflow or status != 0)    */
  int32_t status;     /* 0, or a device-side failure code: 2 = a bulk load of the
                       * update did not arrive within its bounded wait; 3 = a bulk load
                       * or stage wait of the reduce (8 ranks or more) did not complete
                       * in time (the step is then skipped, the state untouched); 5 = the
                       * grid barrier of the one-launch small-span step gave up (the
                       * update may be partly applied). None is expected on a healthy GPU. */
  int32_t reserved;
  int64_t step;       /* optimizer step counter after the step                        */
  double global_norm; /* L2 norm of the unscaled summed gradient (+inf on overflow)   */
  double sum_sq;      /* exact sum of squares of the scaled summed gradient, rounded   */
  double clip_coef;   /* min(1, clip / (global_norm + 1e-6)), or 1 without clipping    */
  float scale;        /* fp32 factor applied to the summed gradient: clip_coef / loss_scale */
  float bc1, bc2;     /* fp32 bias corrections 1 - beta^step used by the update       */
  float loss_scale;   /* the loss scale the step's gradients carried                 */
} zero_step_info;

/* Dynamic loss scaling kept on the device (mixed-precision practice; the pages name
 * mixed precision but give no scaling policy). After each step: on an overflow the
 * scale is multiplied by backoff_factor and good_steps restarts at 0; otherwise
 * good_steps grows by one, and when it reaches growth_interval the scale is multiplied
 * by growth_factor (unless that product is not finite) and good_steps restarts. fp32
 * multiplies. */
typedef struct {
  float scale;             /* current loss scale: finite, > 0                          */
  int32_t good_steps;      /* applied steps since the scale last changed, >= 0         */
  float growth_factor;     /* >= 1                                                     */
  float backoff_factor;    /* in (0, 1]                                                */
  int32_t growth_interval; /* >= 1 turns the scaler on; 0 turns it off                 */
  int32_t reserved;
} zero_loss_scaler;

/* Everything a plan holds besides the caller's buffers: with the bound master, exp_avg,
 * exp_avg_sq and param16 it is a complete checkpoint of a span (ZeRO explainer, Legacy:
 * sharding multiplies failure domains, so each rank checkpoints its own partition). */
typedef struct {
  int64_t step;            /* optimizer step counter t                                 */
  zero_loss_scaler scaler;
} zero_plan_state;

typedef struct zero_plan zero_plan; /* opaque */

/* Create a plan for a flat buffer of n_params parameters partitioned over nd ranks.
 * Partition ("ZeRO" method entry, description: partition the model states): the buffer
 * is padded to Np = ceil(n_params / (nd * align)) * nd * align elements and shard r is
 * [r*S, (r+1)*S) with S = Np / nd; the shards concatenate exactly to the padded buffer,
 * and the padding [n_params, Np) holds no parameter.
 *   n_params >= 1; 1 <= nd <= ZERO_MAX_ND; stage in {1, 2, 3} (ZeRO-1/2/3: which state
 *   classes are partitioned; the step's arithmetic is the same for all three);
 *   align >= 8 and a multiple of 8 (elements); Np * nd^2 < 2^47 (keeps the exact sum of
 *   squares within 128 bits); hp non-NULL with 0 <= beta1, beta2 < 1, lr >= 0, eps > 0,
 *   weight_decay >= 0, all finite.
 * On success *out receives a new plan (free it with zero_plan_destroy). Host only: no
 * CUDA call is made. Errors: ZERO_EINVAL. */
int zero_plan_create(int64_t n_params, int32_t nd, int32_t stage, int32_t align,
                     const zero_adam_hparams* hp, zero_plan** out);

/* Free a plan and its device scratch. NULL is ignored. The caller's buffers are not
 * touched. Any work enqueued with the plan must have completed. */
void zero_plan_destroy(zero_plan* plan);

/* The plan's padded length Np and shard length S (shard r starts at r * S): the partition
 * of the flat buffer into Nd equal shards ("ZeRO" method entry, description; ZeRO
 * explainer, Chapter 02 "What each stage shards"), as zero_plan_create defines it. Host
 * only. Errors: ZERO_EINVAL (a NULL argument). */
int zero_plan_layout(const zero_plan* plan, int64_t* padded_len, int64_t* shard_len);

/* Bytes of fp32 workspace the step needs for the span of logical ranks [r0, r1):
 * 4 * (r1 - r0) * S, the span's summed gradients. The pages count the fp32 gradient copy
 * as transient, not as model state (ZeRO explainer, "The 16 Bytes per Parameter Audit":
 * 2 + 2 + 12 bytes per parameter); this is where it lives between the sum and the
 * update. Host only. Returns the byte count, or ZERO_EINVAL. */
int64_t zero_workspace_bytes(const zero_plan* plan, int32_t r0, int32_t r1);

/* Bind the optimizer state of the span [r0, r1) (0 <= r0 < r1 <= nd; n = (r1-r0)*S
 * elements, element i is flat index r0*S + i). These are the partitioned model states a
 * ZeRO rank keeps for its own partition only: the fp32 master weights, momentum and
 * variance (12 bytes per parameter) and the fp16 parameter copy (ZeRO explainer, "The 16
 * Bytes per Parameter Audit" and Chapter 02 "What each stage shards"):
 *   master, exp_avg, exp_avg_sq: fp32[n], device, read and written by the step;
 *   param16: fp16[n], device, written by the step (the fp16 parameter copy);
 *   workspace: zero_workspace_bytes(plan, r0, r1) bytes of device memory, scratch;
 *   initial_step: the optimizer step counter t before the first step (>= 0).
 * Every pointer must be non-NULL and 16-byte aligned (ZERO_EALIGN otherwise). The
 * padding elements of master, exp_avg, exp_avg_sq and param16 are never read or written
 * (gradient contributions there are read and ignored). The first bind allocates the plan's device
 * scratch on the current device; rebinding replaces the state pointers and resets the
 * step counter. Synchronous. Errors: ZERO_EINVAL, ZERO_EALIGN, ZERO_ECUDA. */
int zero_plan_bind(zero_plan* plan, int32_t r0, int32_t r1, float* master, float* exp_avg,
                   float* exp_avg_sq, void* param16, void* workspace, int64_t initial_step);

/* One shard step over the bound span [r0, r1) (must equal the bound span):
 *   grad_ptrs: host array of nd device pointers; grad_ptrs[k] is rank k's fp16
 *     gradient for the span, n elements, 16-byte aligned. Element i of every rank
 *     belongs to flat index r0*S + i.
 *   loss_scale: finite and > 0; the summed gradient is divided by it. With the plan's
 *     dynamic loss scaler on (zero_plan_set_scaler) it must be 0: the device scale is
 *     used and then updated.
 *   clip: global-norm threshold; <= 0 disables clipping. Must be finite.
 * Computes, on the device, gsum = the fp32 sum of the nd contributions in rank order
 * 0..nd-1 (the reduce-scatter's arithmetic), the overflow flag and the norm over the
 * span's real parameters, and, unless the flag is set, the AdamW update of master,
 * exp_avg and exp_avg_sq with the fp16 cast into param16; the step counter advances
 * only on an applied step. Enqueued on stream; no host synchronisation. A span of at
 * most 3072 groups of 8 parameters per SM (and nd <= 64) runs as one cooperative launch
 * that keeps the fp32 sums in shared memory; other spans run a reduce and an update
 * kernel. When the span
 * fills at least one wave of the reduce, a one-warp kernel computing the next step's
 * step-counter-only scalars runs on a second stream that the plan owns, forked from
 * `stream` after the reduce and joined back into it after the update (stream order for
 * the caller is unchanged). The launches contain no host-side decision, so the call can
 * be captured in a CUDA graph and replayed (the graph keeps the pointers it was captured
 * with); make one ordinary call on the device first, so that the kernels' one-time
 * per-device set-up happens outside the capture (the plan's second stream is made when
 * state is bound).
 * Errors: ZERO_EINVAL, ZERO_EALIGN, ZERO_EUNBOUND, ZERO_ECUDA. */
int zero_shard_step(zero_plan* plan, int32_t r0, int32_t r1, const void* const* grad_ptrs,
                    float loss_scale, float clip, void* stream);

/* First half of zero_shard_step for a span split across processes: the rank-order sum
 * into the workspace and the span's statistics into the plan's exchange buffer
 * (zero_shard_stats). Same arguments and errors as zero_shard_step. */
int zero_shard_reduce(zero_plan* plan, int32_t r0, int32_t r1, const void* const* grad_ptrs,
                      void* stream);

/* The plan's exchange buffer: ZERO_STATS_WORDS int64 on the device, written by
 * zero_shard_reduce: word 0 counts non-finite summed gradients, words 1..4 hold the
 * exact sum of squares of (gsum * 2^24) as four 32-bit limbs (least significant first),
 * word 5 counts reduce CTAs whose bounded wait expired (0 on a healthy GPU; such a CTA also
 * adds a large count to word 0, so the step is skipped), words 6..7 are zero. Summing the
 * buffers of all processes word by word (an integer all-reduce) gives the statistics of the
 * whole buffer. Valid after zero_plan_bind. */
int zero_shard_stats(zero_plan* plan, void** dev_words);

/* Second half of zero_shard_step: reads the (possibly all-reduced) exchange buffer,
 * decides skip, norm and clip coefficient, and applies the update to the bound span.
 * Errors as zero_shard_step. */
int zero_shard_update(zero_plan* plan, int32_t r0, int32_t r1, float loss_scale, float clip,
                      void* stream);

/* Wait for the plan's last step to finish and copy its result to *out: the overflow
 * flag and skip decision of the mixed-precision step (ZeRO explainer, "The
 * mixed-precision era" and Chapter 02 "Memory per parameter": fp16 gradients with fp32
 * master state; an inf/nan gradient skips the update), the global norm and clip
 * coefficient, the step counter and the device-side failure status. This is the only
 * step call that synchronises with the device. Errors: ZERO_EINVAL, ZERO_EUNBOUND (no
 * step yet), ZERO_ECUDA, ZERO_EDEVICE (out is still filled). */
int zero_step_result(zero_plan* plan, zero_step_info* out);

/* ZeRO-3 gather ("all-gather before forward", ZeRO explainer, Chapter 02): with flat =
 * the concatenation of the nd fp16 shards of S elements each, copies
 * layer_dst[l][j] = flat[layer_offsets[l] + j] for 0 <= j < layer_offsets[l+1] -
 * layer_offsets[l].
 *   layer_offsets: host int64[n_layers + 1], non-decreasing, 0 <= offsets <= n_params
 *     (offsets index the unpadded flat buffer);
 *   shard_ptrs: host array of nd device pointers, fp16[S] each (2-byte aligned);
 *   layer_dst: host array of n_layers device pointers (2-byte aligned; may be NULL for
 *     an empty layer). Destinations must not overlap the shards or each other.
 * For ZeRO-1/2 the parameter all-gather is this call with one layer [0, n_params).
 * Each layer is cut at shard boundaries into copy segments; segments whose source and
 * destination addresses agree modulo 16 bytes are copied by TMA bulk copies, the others
 * by a kernel that realigns 16-byte blocks in registers (same result, same traffic).
 * Enqueued on stream. The first call on a plan that was never bound allocates the
 * plan's small device scratch (which holds the gather's status word) on the current
 * device. The plan is not const: the call may allocate that scratch, and it records the
 * stream it used so that zero_gather_status can wait for it.
 * Errors: ZERO_EINVAL, ZERO_EALIGN, ZERO_ECUDA. */
int zero_gather_layers(zero_plan* plan, const int64_t* layer_offsets, int32_t n_layers,
                       const void* const* shard_ptrs, void* const* layer_dst, void* stream);

/* The ZeRO-3 gather layer by layer, with a completion event per layer: the "dynamic
 * communication schedule" of the ZeRO method entry (codewithpapers.app/method/zero,
 * description), in which the all-gather of later layers runs ahead while the work on an
 * earlier layer starts. Copies exactly what zero_gather_layers copies, with the same
 * arguments and checks, plus:
 *   layer_done: host array of n_layers cudaEvent_t handles passed as void* (the caller
 *     creates them on the plan's device and owns them; an entry may be NULL for "no
 *     event"). layer_done[l] is recorded once layer l's copy has been enqueued, so
 *     cudaStreamWaitEvent(other_stream, layer_done[l]) lets other work start on layer l
 *     while later layers are still being copied.
 * Layers are enqueued in order, each by its own launch(es): layers 0, 2, 4, ... on
 * `stream`, layers 1, 3, 5, ... on a second stream that the plan owns, which first waits
 * for the work already on `stream` and is joined back into `stream` at the end. So two
 * consecutive layers may run at the same time (the next one takes the SMs the previous
 * one leaves, which hides each launch's start and end), and layer_done[l] marks layer l
 * alone: it may complete before layer_done[l-1]. Work enqueued on `stream` after this call
 * starts after every layer; zero_gather_status covers the call. An event handle that is
 * not valid on the plan's device makes the call fail with ZERO_ECUDA after the earlier
 * layers have been enqueued (their copies still complete, and `stream` is still joined).
 * Errors: ZERO_EINVAL (also for layer_done == NULL), ZERO_EALIGN, ZERO_ECUDA. */
int zero_gather_layers_events(zero_plan* plan, const int64_t* layer_offsets, int32_t n_layers,
                              const void* const* shard_ptrs, void* const* layer_dst,
                              void* const* layer_done, void* stream);

/* Wait for the plan's last gather and report whether it finished (the library's own
 * failure reporting; the pages have no counterpart): *status is 0, or 4 if a
 * bulk copy did not arrive within its bounded wait and the gather stopped early (never
 * expected on a healthy GPU; the status is then cleared and ZERO_EDEVICE returned).
 * Errors: ZERO_EINVAL, ZERO_ECUDA, ZERO_EDEVICE. */
int zero_gather_status(zero_plan* plan, int32_t* status);

/* Per-rank model-state bytes (ZeRO explainer, "The 16 Bytes per Parameter Audit",
 * Chapter 02 and the stage table): 2 B fp16 parameter + 2 B fp16 gradient + 12 B of
 * optimizer state (fp32 master, momentum, variance) per parameter, with S the padded
 * shard length of create's partition:
 *   stage 0 (plain data parallel) 16 N; stage 1 4 N + 12 S; stage 2 2 N + 14 S;
 *   stage 3 16 S.
 * align (elements, >= 1) is an argument because a rank holds its whole padded shard:
 * S = Np / nd with Np = ceil(n_params / (nd * align)) * nd * align, as zero_plan_create
 * partitions, so the same n_params and nd give different per-rank bytes for different
 * alignments (for align = 1 and nd dividing n_params, S = n_params / nd exactly, the
 * pages' Psi / Nd). Host only. Errors: ZERO_EINVAL. */
int zero_memory_bytes(int64_t n_params, int32_t nd, int32_t align, int32_t stage,
                      int64_t* per_rank_bytes);

/* Kernel timing with CUDA events on the launching stream, for profiling (a measurement
 * facility; the pages have no counterpart). When enabled,
 * every kernel the plan launches is bracketed by two events; zero_profile_read
 * synchronises and returns, per kernel kind (0 reduce, 1 update, 2 scalars: the
 * finalize of a split step and the next step's step-counter-only scalars, 3 gather,
 * 4 step: a whole small-span step in one launch), the summed milliseconds and the
 * launch count, then clears them if reset != 0. Off by default. Errors: ZERO_EINVAL,
 * ZERO_ECUDA. */
#define ZERO_PROF_KINDS 5
int zero_profile_enable(zero_plan* plan, int32_t on);
int zero_profile_read(zero_plan* plan, double* ms, int64_t* launches, int32_t reset);

/* A shard step that allocates nothing. The pages have no counterpart: this is an interface
 * variant of zero_shard_step for callers that cannot allocate device memory when they step
 * (a framework that reserved all of HBM for its own pool at start-up and forbids later
 * cudaMalloc calls, an allocator hook that must not re-enter its allocator, or a loop in
 * which the device-wide synchronisation that cudaMalloc/cudaFree may cause is not
 * acceptable). It needs no plan and runs the same kernels as zero_shard_step (one
 * cooperative launch for a small span, else the reduce and update kernels).
 *   nd: ranks, 1..ZERO_MAX_ND; n: span length, a multiple of 8, 8 <= n <=
 *     ZERO_NOALLOC_MAX_SPAN; n_valid: real parameters at the start of the span (0..n);
 *     n * nd^2 < 2^47;
 *   grad_ptrs: host array of nd device pointers, fp16[n] each, 16-byte aligned;
 *   master, exp_avg, exp_avg_sq: fp32[n]; param16: fp16[n]; device, 16-byte aligned;
 *   step_counter: one int64 in device memory, the optimizer step counter t, read before
 *     and written after the step (it stays unchanged when the step is skipped);
 *   hp, loss_scale, clip: as for zero_plan_create and zero_shard_step.
 * The caller passes every input and output. Scratch comes from one device array inside
 * this library: ZERO_NOALLOC_MAX_SPAN fp32 values plus a control block of about 35 KiB
 * (16.03 MiB), which every GPU that loads the library holds until the process exits. The
 * first call on a device looks up that array's device address (cudaGetSymbolAddress) and
 * caches it; make that first call before any stream capture. Every call shares the array
 * and it keeps the last call's contents (the control words that must start at zero are
 * cleared by each call), so calls whose work overlaps on the GPU race and give wrong
 * results: order them on one stream or with events. Enqueued on stream; asynchronous: a
 * device-side failure is reported only through zero_noalloc_step_result.
 * Errors: ZERO_EINVAL (including n > ZERO_NOALLOC_MAX_SPAN), ZERO_EALIGN, ZERO_ECUDA;
 * nothing is launched on an error. */
#define ZERO_NOALLOC_MAX_SPAN 4194304
int zero_shard_step_noalloc(int32_t nd, int64_t n, int64_t n_valid, const void* const* grad_ptrs,
                            float* master, float* exp_avg, float* exp_avg_sq, void* param16,
                            int64_t* step_counter, const zero_adam_hparams* hp,
                            float loss_scale, float clip, void* stream);

/* Result of the last allocation-free step on the current device (a companion of
 * zero_shard_step_noalloc; the pages have no counterpart). Waits for `stream` (the stream
 * that step was enqueued on), then copies the step's overflow flag, skip decision, norm,
 * clip coefficient, scalars and step counter, and its device-side failure status, from the
 * library's scratch array into *out. This is the only way to see a failure inside that
 * step: status 2 (a bulk load of the update did not arrive within its bounded wait) or 5
 * (the grid barrier of the one-launch step gave up, so parts of the span may be updated and
 * others not); the step call itself returns ZERO_OK once its work is enqueued. Allocates
 * nothing. The array holds the result of whichever allocation-free step ran last on the
 * device. Errors: ZERO_EINVAL, ZERO_EUNBOUND (no allocation-free step has run on the
 * current device), ZERO_ECUDA, ZERO_EDEVICE (status != 0; *out is still filled). */
int zero_noalloc_step_result(void* stream, zero_step_info* out);

/* Configure the plan's device-resident loss scaler (see zero_loss_scaler) after
 * zero_plan_bind. While it is on, zero_shard_step and zero_shard_update must be given
 * loss_scale = 0 and use the device scale instead; zero_loss_scale_ptr gives its address
 * so that the caller can scale its loss on the device without a host round trip.
 * Waits for the plan's last stream, then writes the state (synchronous). Errors:
 * ZERO_EINVAL, ZERO_EUNBOUND, ZERO_ECUDA. */
int zero_plan_set_scaler(zero_plan* plan, const zero_loss_scaler* scaler);

/* Device address of the current loss scale (one fp32 value in the plan's scratch; part of
 * the dynamic scaler above, which the pages do not describe). Valid
 * after zero_plan_bind and until zero_plan_destroy. Errors: ZERO_EINVAL, ZERO_EUNBOUND. */
int zero_loss_scale_ptr(zero_plan* plan, float** dev_scale);

/* Read (get) or restore (set) the plan's step counter and scaler, for checkpoints: saving
 * the bound buffers and this state, then binding fresh buffers holding the saved bytes and
 * restoring the state, continues the run bit for bit. Both wait for the plan's last
 * stream (synchronous). Errors: ZERO_EINVAL, ZERO_EUNBOUND, ZERO_ECUDA. */
int zero_plan_get_state(zero_plan* plan, zero_plan_state* out);
int zero_plan_set_state(zero_plan* plan, const zero_plan_state* in);

/* Self-test of the bounded waits the bulk-copy kernels use (the pages have no
 * counterpart; this checks the library's own failure path). A one-warp kernel waits on a
 * shared-memory barrier that nothing completes, polling at most `polls` times (1..2^24,
 * each poll suspended at most 1 us, the whole wait at most about 2 s), and records that it
 * gave up; *expired receives 1 when the wait expired as it must, 0 if it (wrongly)
 * completed. Synchronises the device; the context stays usable. Errors: ZERO_EINVAL,
 * ZERO_ECUDA. */
int zero_selftest_wait(uint32_t polls, int32_t* expired);

/* Self-test of the grid barrier of the one-launch small-span step (a facility for failure
 * reporting; the pages have no counterpart): a cooperative launch of two CTAs meets at
 * the barrier, which also sums values over the CTAs, with the given poll limit
 * (1 .. 2^24 polls of about 64 ns). With skip_one != 0 the second CTA leaves without
 * arriving, so the first must give up; *expired is 1 if it gave up, 0 if the barrier was
 * met with the right sums and 2 if it was met with wrong ones. Synchronises the device.
 * Errors: ZERO_EINVAL, ZERO_ECUDA. */
int zero_selftest_grid_barrier(uint32_t polls, int32_t skip_one, int32_t* expired);

/* Bounds report of a bounds-checked build (a facility for testing; the pages have no
 * counterpart). A build compiled with ZERO_BOUNDS_CHECK tests the byte range of each
 * global access of the kernels' main paths against the extent of the buffer it belongs
 * to, skips an access outside it and records the first such fault on the current device.
 * *enabled: 1 in such a build, 0 in the normal one (where *site and *offset are always 0).
 * *site: 0, or the first faulting access site (1 contribution register loads, 2 fp32 sum
 * stores, 3 contribution bulk loads, 4 update loads, 5 update stores, 6 the last few
 * parameters, 7 one-launch state loads, 8 one-launch stores, 9 a gather tile, 10
 * realigning-gather loads, 11 realigning-gather stores); *offset: its byte offset from
 * the buffer's start. With reset != 0 the record is cleared after it is read. Synchronous
 * in a checked build. Errors: ZERO_EINVAL (a NULL output), ZERO_ECUDA. */
int zero_bounds_check(int32_t reset, int32_t* enabled, int32_t* site, int64_t* offset);

/* Self-test of those checks (the pages have no counterpart): one kernel tests a range
 * inside a 64-byte device buffer and one reaching past its end (bytes 80..95), accessing
 * neither. In a bounds-checked build zero_bounds_check then reports site 11 at offset 80
 * (unless an earlier fault is recorded); in the normal build it has no effect.
 * Synchronises the device. Errors: ZERO_ECUDA. */
int zero_selftest_bounds(void);

/* Message of the calling thread's last error ("" if none). Valid until the thread's
 * next libzero call. */
const char* zero_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* ZERO_H */
