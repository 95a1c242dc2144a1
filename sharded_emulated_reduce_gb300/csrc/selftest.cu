// Self-tests of the bounded waits of the libzero kernels.
//
// zero_selftest_wait: a one-warp kernel initialises an mbarrier that nothing will ever
// complete and waits on it with a caller-given poll limit. The wait must give up, the
// kernel must record that and return, and the context must stay usable. This exercises
// the failure path of the bulk-copy kernels without faulting, trapping or hanging the GPU.
//
// zero_selftest_grid_barrier: a cooperative launch of two CTAs meets at the counting sums
// that are the one-launch step's grid barrier, each adding two values; CTA 0 checks the
// two sums. With skip_one set, CTA 1 leaves without adding, so CTA 0's wait must give up
// within its poll limit and record that.
#include "bulk_async.h"
#include "grid_sync.h"
#include "internal.h"

namespace zero {
namespace {

__global__ void k_wait_probe(unsigned polls, int32_t* out) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  __syncthreads();
  const bool arrived = mbar_wait(&bar, 0, polls);  // nothing arrives on `bar`
  if (threadIdx.x == 0) *out = arrived ? 0 : 1;
}

// One warp per CTA; *out = 0 if the sums were met and right, 1 if the wait gave up, 2 if
// they were met but wrong.
__global__ void k_barrier_probe(unsigned polls, int skip_one, unsigned long long* words,
                                int32_t* out) {
  if (skip_one && blockIdx.x == 1) return;  // never arrives
  if (threadIdx.x == 0) {
    const unsigned long long v[2] = {blockIdx.x + 1ull, 100ull + blockIdx.x};
    sum_arrive<2>(words, kSumStride, v);
  }
  unsigned long long sum = 0;
  const bool met = sum_wait<2>(words, kSumStride, gridDim.x, polls, &sum);
  const unsigned long long s0 = __shfl_sync(0xffffffffu, sum, 0);
  const unsigned long long s1 = __shfl_sync(0xffffffffu, sum, 1);
  if (blockIdx.x == 0 && threadIdx.x == 0) *out = !met ? 1 : (s0 == 3 && s1 == 201) ? 0 : 2;
}

// Result word of the probe; host code gets its device address from cudaGetSymbolAddress.
static __device__ int32_t g_probe_result;
static __device__ unsigned long long g_probe_words[2 * kSumStride];

}  // namespace
}  // namespace zero

extern "C" int zero_selftest_wait(uint32_t polls, int32_t* expired) {
  using namespace zero;
  if (!expired) return set_error(ZERO_EINVAL, "expired is NULL");
  if (polls < 1 || polls > (1u << 24)) return set_error(ZERO_EINVAL, "polls must be in [1, 2^24]");
  void* addr = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&addr, g_probe_result);
  if (e == cudaSuccess) e = cudaMemset(addr, 0xff, sizeof(int32_t));
  if (e != cudaSuccess) return set_error(ZERO_ECUDA, "self-test set-up failed");
  k_wait_probe<<<1, 32>>>(polls, static_cast<int32_t*>(addr));
  e = cudaGetLastError();
  int32_t r = -1;
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(&r, addr, sizeof r, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return set_error(ZERO_ECUDA, "self-test kernel failed");
  *expired = r;
  set_error(ZERO_OK, "");
  return ZERO_OK;
}

extern "C" int zero_selftest_grid_barrier(uint32_t polls, int32_t skip_one, int32_t* expired) {
  using namespace zero;
  if (!expired) return set_error(ZERO_EINVAL, "expired is NULL");
  if (polls < 1 || polls > (1u << 24)) return set_error(ZERO_EINVAL, "polls must be in [1, 2^24]");
  void* res = nullptr;
  void* words = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&res, g_probe_result);
  if (e == cudaSuccess) e = cudaGetSymbolAddress(&words, g_probe_words);
  if (e == cudaSuccess) e = cudaMemset(res, 0xff, sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMemset(words, 0, sizeof(unsigned long long) * 2 * kSumStride);
  if (e != cudaSuccess) return set_error(ZERO_ECUDA, "self-test set-up failed");
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(32);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, k_barrier_probe, (unsigned)polls, (int)(skip_one != 0),
                         static_cast<unsigned long long*>(words), static_cast<int32_t*>(res));
  int32_t r = -1;
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(&r, res, sizeof r, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return set_error(ZERO_ECUDA, "self-test kernel failed");
  *expired = r;
  set_error(ZERO_OK, "");
  return ZERO_OK;
}
