// Seeded synthetic inputs on the GPU: the device twin of the CPU generator in
// synth/__init__.py. It draws numbers only; none of the ZeRO step's arithmetic
// lives here.
//
// Element i of a stream with key k takes the SplitMix64 words for counters 2i and
// 2i+1 (word(c) = mix(k + G*(c+1)), mix = the SplitMix64 output function of Steele,
// Lea and Flood, OOPSLA 2014), sums their eight 16-bit lanes, centres the sum
// (Irwin-Hall(8)) and multiplies by an fp32 factor c in one IEEE multiply. fp16
// outputs round that product to nearest even. Indices at or past n_valid are 0.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr uint64_t kG = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ int lanes16(uint64_t w) {
  return (int)(w & 0xFFFF) + (int)((w >> 16) & 0xFFFF) + (int)((w >> 32) & 0xFFFF) +
         (int)(w >> 48);
}

__device__ __forceinline__ float draw(uint64_t key, int64_t idx, float c) {
  uint64_t base = key + kG * (2ull * (uint64_t)idx + 1ull);
  int z = lanes16(mix(base)) + lanes16(mix(base + kG)) - 4 * 65535;
  return __fmul_rn((float)z, c);
}

// mode 0: fp16, 1: fp32, 2: |fp32|
__global__ void fill_kernel(void* out, int mode, int64_t n, int64_t start, int64_t n_valid,
                            uint64_t key, float c) {
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += stride) {
    int64_t idx = start + j;
    float v = idx < n_valid ? draw(key, idx, c) : 0.0f;
    if (mode == 0) {
      reinterpret_cast<__half*>(out)[j] = __float2half_rn(v);
    } else {
      reinterpret_cast<float*>(out)[j] = mode == 2 ? fabsf(v) : v;
    }
  }
}

}  // namespace

extern "C" int synth_fill(void* out, int mode, int64_t n, int64_t start, int64_t n_valid,
                          uint64_t key, float c, int reserved, void* stream) {
  (void)reserved;
  if (n <= 0) return 0;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (n + 255) / 256;
  int64_t cap = (int64_t)sms * 16;
  if (blocks > cap) blocks = cap;
  fill_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(out, mode, n, start, n_valid,
                                                                   key, c);
  return (int)cudaGetLastError();
}
