/*
 * Device side of the seeded input generator: fills a device buffer with the
 * same values gen_host.c produces (built with --fmad=false; see gen_core.h).
 * Test and benchmark infrastructure only; no selective-scan arithmetic.
 */
#include <cstdint>
#include <cuda_runtime.h>
#include "gen_core.h"

template <bool BF16>
__global__ void gen_fill_normal_kernel(uint64_t key, double mean, double sd, int64_t start,
                                       int64_t count, void* out) {
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += stride) {
    float v = (float)(mean + sd * gen_normal(key, (uint64_t)(start + i)));
    if (BF16) ((uint16_t*)out)[i] = gen_f32_to_bf16(v);
    else ((float*)out)[i] = v;
  }
}

extern "C" int gen_dev_fill_normal(uint64_t seed, uint64_t tensor_id, double mean, double sd,
                                   int64_t start, int64_t count, int is_bf16, void* out,
                                   cudaStream_t stream) {
  if (count <= 0) return 0;
  if (out == nullptr) return 1;
  uint64_t key = gen_key(seed, tensor_id);
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (count + 255) / 256;
  int64_t cap = (int64_t)sms * 16;
  if (blocks > cap) blocks = cap;
  if (is_bf16)
    gen_fill_normal_kernel<true><<<(unsigned)blocks, 256, 0, stream>>>(key, mean, sd, start, count, out);
  else
    gen_fill_normal_kernel<false><<<(unsigned)blocks, 256, 0, stream>>>(key, mean, sd, start, count, out);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}
