/* The libzero C ABI driven from plain C11, as a C caller links it (no Python, no torch).
 *
 *   abi_demo cpu  -- host-only calls: partition layout, workspace and accounting sizes,
 *                    and the error codes of invalid arguments (no CUDA call is made);
 *   abi_demo gpu  -- on the current CUDA device: two shard steps of a 1M-parameter,
 *                    4-rank span (the second with an inf in one rank's contribution, so
 *                    it is skipped), then the ZeRO-3 gather of the step's fp16 output into
 *                    two layers, checked against the shards byte for byte.
 * Prints "ok" and exits 0 on success; prints the failing check and exits 1 otherwise. */
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "zero.h"

#define CHECK(cond)                                                           \
  do {                                                                        \
    if (!(cond)) {                                                            \
      fprintf(stderr, "check failed at line %d: %s (%s)\n", __LINE__, #cond,  \
              zero_last_error());                                             \
      return 1;                                                               \
    }                                                                         \
  } while (0)

static const zero_adam_hparams HP = {1e-3f, 0.9f, 0.999f, 1e-8f, 0.01f};

static int host_only(void) {
  zero_plan* p = NULL;
  CHECK(zero_plan_create(1000003, 4, 2, 8, &HP, &p) == ZERO_OK && p != NULL);
  int64_t np = 0, s = 0;
  CHECK(zero_plan_layout(p, &np, &s) == ZERO_OK);
  CHECK(np == 1000032 && s == 250008 && np == 4 * s);  /* ceil(N / 32) * 32 */
  CHECK(zero_workspace_bytes(p, 0, 4) >= (int64_t)(4 * s * 4));
  CHECK(zero_workspace_bytes(p, 2, 1) == ZERO_EINVAL);
  zero_plan_destroy(p);
  /* the pages' audit: 7B parameters at 16 bytes each, replicated (stage 0) */
  int64_t bytes = 0;
  CHECK(zero_memory_bytes(7000000000LL, 1, 1, 0, &bytes) == ZERO_OK);
  CHECK(bytes == 112000000000LL);
  /* invalid arguments return their code and create nothing */
  p = NULL;
  CHECK(zero_plan_create(100, 0, 2, 8, &HP, &p) == ZERO_EINVAL && p == NULL);
  CHECK(zero_plan_create(100, 4, 2, 12, &HP, &p) == ZERO_EINVAL && p == NULL);
  CHECK(zero_plan_create(100, 4, 4, 8, &HP, &p) == ZERO_EINVAL && p == NULL);
  CHECK(strlen(zero_last_error()) > 0);
  return 0;
}

/* fp16 bits of a small gradient value: +-(1 + k/1024) * 2^-12, k in 0..1023 */
static uint16_t grad_bits(int64_t i, int r) {
  const uint16_t k = (uint16_t)((i * 7 + r * 13) & 1023);
  const uint16_t sign = (uint16_t)(((i + r) & 1) << 15);
  return (uint16_t)(sign | (3u << 10) | k);  /* exponent field 3: 2^(3-15) */
}

static int device_steps(void) {
  const int64_t n = 1000000;
  const int nd = 4;
  zero_plan* p = NULL;
  CHECK(zero_plan_create(n, nd, 3, 8, &HP, &p) == ZERO_OK);
  int64_t np = 0, s = 0;
  CHECK(zero_plan_layout(p, &np, &s) == ZERO_OK);
  const int64_t span = nd * s;  /* this device owns all four logical ranks */
  uint16_t* host = (uint16_t*)malloc((size_t)span * 2);
  float* hm = (float*)malloc((size_t)span * 4);
  CHECK(host && hm);
  void* grads[4];
  for (int r = 0; r < nd; ++r) {
    for (int64_t i = 0; i < span; ++i) host[i] = i < n ? grad_bits(i, r) : 0;
    CHECK(cudaMalloc(&grads[r], (size_t)span * 2) == cudaSuccess);
    CHECK(cudaMemcpy(grads[r], host, (size_t)span * 2, cudaMemcpyHostToDevice) == cudaSuccess);
  }
  float *master, *m, *v;
  void *p16, *ws;
  const int64_t wsb = zero_workspace_bytes(p, 0, nd);
  CHECK(wsb > 0);
  CHECK(cudaMalloc((void**)&master, (size_t)span * 4) == cudaSuccess);
  CHECK(cudaMalloc((void**)&m, (size_t)span * 4) == cudaSuccess);
  CHECK(cudaMalloc((void**)&v, (size_t)span * 4) == cudaSuccess);
  CHECK(cudaMalloc(&p16, (size_t)span * 2) == cudaSuccess);
  CHECK(cudaMalloc(&ws, (size_t)wsb) == cudaSuccess);
  for (int64_t i = 0; i < span; ++i) hm[i] = i < n ? 0.02f * (float)((i % 201) - 100) / 100.0f : 0.0f;
  CHECK(cudaMemcpy(master, hm, (size_t)span * 4, cudaMemcpyHostToDevice) == cudaSuccess);
  CHECK(cudaMemset(m, 0, (size_t)span * 4) == cudaSuccess);
  CHECK(cudaMemset(v, 0, (size_t)span * 4) == cudaSuccess);
  CHECK(cudaMemset(p16, 0, (size_t)span * 2) == cudaSuccess);
  CHECK(zero_plan_bind(p, 0, nd, master, m, v, p16, ws, 0) == ZERO_OK);

  /* an applied step */
  zero_step_info info;
  CHECK(zero_shard_step(p, 0, nd, (const void* const*)grads, 1.0f, 1.0f, NULL) == ZERO_OK);
  CHECK(zero_step_result(p, &info) == ZERO_OK);
  CHECK(info.status == 0 && info.overflow == 0 && info.skipped == 0 && info.step == 1);
  CHECK(info.global_norm > 0.0 && isfinite(info.global_norm));
  CHECK(info.clip_coef > 0.0 && info.clip_coef <= 1.0);
  float* after = (float*)malloc((size_t)span * 4);
  CHECK(after);
  CHECK(cudaMemcpy(after, master, (size_t)span * 4, cudaMemcpyDeviceToHost) == cudaSuccess);
  int64_t changed = 0;
  for (int64_t i = 0; i < n; ++i) changed += after[i] != hm[i];
  CHECK(changed > n / 2);
  for (int64_t i = n; i < span; ++i) CHECK(after[i] == 0.0f);  /* padding untouched */

  /* an inf in rank 2's contribution: the step is skipped and the state keeps its bits */
  const uint16_t inf16 = 0x7C00;
  CHECK(cudaMemcpy((uint16_t*)grads[2] + 12345, &inf16, 2, cudaMemcpyHostToDevice) == cudaSuccess);
  CHECK(zero_shard_step(p, 0, nd, (const void* const*)grads, 1.0f, 1.0f, NULL) == ZERO_OK);
  CHECK(zero_step_result(p, &info) == ZERO_OK);
  CHECK(info.overflow == 1 && info.skipped == 1 && info.step == 1 && isinf(info.global_norm));
  float* again = (float*)malloc((size_t)span * 4);
  CHECK(again);
  CHECK(cudaMemcpy(again, master, (size_t)span * 4, cudaMemcpyDeviceToHost) == cudaSuccess);
  CHECK(memcmp(again, after, (size_t)span * 4) == 0);

  /* the ZeRO-3 gather of the fp16 parameters (the shards are consecutive in p16) into
   * two layers, the boundary inside shard 1 */
  const int64_t offs[3] = {0, 400001, n};
  const void* shards[4];
  for (int r = 0; r < nd; ++r) shards[r] = (const uint16_t*)p16 + r * s;
  void* dst[2];
  CHECK(cudaMalloc(&dst[0], (size_t)offs[1] * 2) == cudaSuccess);
  CHECK(cudaMalloc(&dst[1], (size_t)(offs[2] - offs[1]) * 2) == cudaSuccess);
  CHECK(zero_gather_layers(p, offs, 2, shards, dst, NULL) == ZERO_OK);
  CHECK(cudaDeviceSynchronize() == cudaSuccess);
  uint16_t* flat = (uint16_t*)malloc((size_t)n * 2);
  uint16_t* got = (uint16_t*)malloc((size_t)n * 2);
  CHECK(flat && got);
  CHECK(cudaMemcpy(flat, p16, (size_t)n * 2, cudaMemcpyDeviceToHost) == cudaSuccess);
  CHECK(cudaMemcpy(got, dst[0], (size_t)offs[1] * 2, cudaMemcpyDeviceToHost) == cudaSuccess);
  CHECK(cudaMemcpy(got + offs[1], dst[1], (size_t)(offs[2] - offs[1]) * 2,
                   cudaMemcpyDeviceToHost) == cudaSuccess);
  CHECK(memcmp(flat, got, (size_t)n * 2) == 0);

  zero_plan_destroy(p);
  for (int r = 0; r < nd; ++r) cudaFree(grads[r]);
  cudaFree(master);
  cudaFree(m);
  cudaFree(v);
  cudaFree(p16);
  cudaFree(ws);
  cudaFree(dst[0]);
  cudaFree(dst[1]);
  free(host);
  free(hm);
  free(after);
  free(again);
  free(flat);
  free(got);
  return 0;
}

int main(int argc, char** argv) {
  const int gpu = argc > 1 && strcmp(argv[1], "gpu") == 0;
  const int rc = gpu ? device_steps() : host_only();
  if (rc == 0) printf("ok\n");
  return rc;
}
