// Internal launch interface between the C ABI layer (ssm_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace ssm {

struct ScanParams {
  const void* u;
  const void* delta;
  const float* A;
  const void* B;
  const void* C;
  const float* D;           // may be null
  const void* z;            // may be null
  const float* delta_bias;  // may be null
  int softplus;
  void* y;
  float* last_state;        // may be null
  const float* initial_state;  // may be null: the state before the first step is zero
  int64_t batch, L, d_inner;
  int d_state;
  // Time chunking: the sequence is cut into n_chunks chunks of chunk_len steps
  // (the last one may be shorter).  For n_chunks > 1 the workspace holds, per
  // (batch, chunk < n_chunks-1, channel), the chunk's delta sum and its end
  // state started from zero.
  int64_t chunk_len;
  int n_chunks;
  int lanes;  // 1 or 2 lanes per channel (which kernel runs)
  float* ws_S;  // [batch][n_chunks-1][d_inner]
  float* ws_h;  // [batch][n_chunks-1][d_inner][d_state]
};

struct DecodeParams {
  float* state;
  const void* u;
  const void* delta;
  const float* A;
  const void* B;
  const void* C;
  const float* D;
  const void* z;
  void* y;
  const float* delta_bias;
  int softplus;
  int64_t batch, d_inner;
  int d_state;
};

// Channels handled by one CTA of the scan kernels.
int scan_channels_per_cta();

// How a scan of these sizes runs on a device with `sms` SMs: the kernel (lanes per
// channel) and the time chunking.
struct ScanPlan {
  int lanes;
  int64_t chunk_len;
  int n_chunks;
};
void plan_scan(int64_t batch, int64_t L, int64_t d_inner, int sms, ScanPlan* plan);

cudaError_t launch_scan(const ScanParams& p, bool bf16, cudaStream_t stream);
cudaError_t launch_state_update(const DecodeParams& p, bool bf16, cudaStream_t stream);

}  // namespace ssm
