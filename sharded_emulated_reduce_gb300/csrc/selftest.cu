// Self-test of the bounded wait that every libzero kernel uses on its mbarriers.
//
// A one-warp kernel initialises an mbarrier that nothing will ever complete and waits on
// it with a caller-given poll limit. The wait must give up, the kernel must record that
// and return, and the context must stay usable. This exercises the failure path of the
// bulk-copy kernels without faulting, trapping or hanging the GPU.
#include "bulk_async.h"
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

// Result word of the probe; host code gets its device address from cudaGetSymbolAddress.
static __device__ int32_t g_probe_result;

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
