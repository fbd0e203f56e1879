// Single-token decode step (selective_state_update): one step of the selective
// recurrence on a carried fp32 state, updated in place, with the same step
// size, discretisation, readout and gate as the full scan.
// Source: ai-lab.club "机器学习基础算法", section "核心优势" (like an RNN, a
// new token costs constant work on a fixed-size state); the step itself is
// one iteration of the loop in youngju.dev "Mamba: Linear-Time Sequence
// Modeling with Selective State Spaces 论文分析", "解决方案：Kernel Fusion +
// Recomputation".
//
// The step is bound by HBM: per (batch, channel) it reads and writes d_state
// fp32 states and touches only a few bytes of activations.  One thread owns
// one channel's states; the state row is moved with 16-byte accesses when
// d_state is a multiple of 4.

#include "ssm_device.cuh"
#include "ssm_internal.h"

namespace ssm {

constexpr int kDecodeThreads = 256;

template <int N, typename T>
__global__ void __launch_bounds__(kDecodeThreads) state_update_kernel(const DecodeParams p) {
  const int64_t i = (int64_t)blockIdx.x * kDecodeThreads + threadIdx.x;  // b * d_inner + d
  if (i >= p.batch * p.d_inner) return;
  const int64_t b = i / p.d_inner, d = i % p.d_inner;
  const T* u = static_cast<const T*>(p.u);
  const T* dl = static_cast<const T*>(p.delta);
  const T* Bg = static_cast<const T*>(p.B) + b * N;
  const T* Cg = static_cast<const T*>(p.C) + b * N;
  const T* zg = static_cast<const T*>(p.z);

  const float x = to_f32(dl[i]) + (p.delta_bias ? p.delta_bias[d] : 0.f);
  const float dt = p.softplus ? softplus(x) : x;
  const float uu = to_f32(u[i]);
  const float w = dt * uu;

  float h[N];
  float* st = p.state + i * N;
  if constexpr (N % 4 == 0) {
#pragma unroll
    for (int q = 0; q < N / 4; q++) {
      const float4 v = reinterpret_cast<const float4*>(st)[q];
      h[4 * q] = v.x; h[4 * q + 1] = v.y; h[4 * q + 2] = v.z; h[4 * q + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int n = 0; n < N; n++) h[n] = st[n];
  }
  float acc = 0.f;
#pragma unroll
  for (int n = 0; n < N; n++) {
    const float dA = ex2(dt * (p.A[d * N + n] * kLog2e));
    h[n] = fmaf(dA, h[n], w * to_f32(Bg[n]));
    acc = fmaf(to_f32(Cg[n]), h[n], acc);
  }
  if constexpr (N % 4 == 0) {
#pragma unroll
    for (int q = 0; q < N / 4; q++)
      reinterpret_cast<float4*>(st)[q] = make_float4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
  } else {
#pragma unroll
    for (int n = 0; n < N; n++) st[n] = h[n];
  }
  if (p.D) acc = fmaf(p.D[d], uu, acc);
  if (zg) acc *= silu(to_f32(zg[i]));
  static_cast<T*>(p.y)[i] = from_f32<T>(acc);
}

template <int N, typename T>
static cudaError_t launch_t(const DecodeParams& p, cudaStream_t s) {
  const int64_t total = p.batch * p.d_inner;
  const int64_t blocks = (total + kDecodeThreads - 1) / kDecodeThreads;
  state_update_kernel<N, T><<<(unsigned)blocks, kDecodeThreads, 0, s>>>(p);
  return cudaGetLastError();
}

template <typename T>
static cudaError_t dispatch_n(const DecodeParams& p, cudaStream_t s) {
  switch (p.d_state) {
    case 1: return launch_t<1, T>(p, s);
    case 2: return launch_t<2, T>(p, s);
    case 3: return launch_t<3, T>(p, s);
    case 4: return launch_t<4, T>(p, s);
    case 5: return launch_t<5, T>(p, s);
    case 6: return launch_t<6, T>(p, s);
    case 7: return launch_t<7, T>(p, s);
    case 8: return launch_t<8, T>(p, s);
    case 9: return launch_t<9, T>(p, s);
    case 10: return launch_t<10, T>(p, s);
    case 11: return launch_t<11, T>(p, s);
    case 12: return launch_t<12, T>(p, s);
    case 13: return launch_t<13, T>(p, s);
    case 14: return launch_t<14, T>(p, s);
    case 15: return launch_t<15, T>(p, s);
    case 16: return launch_t<16, T>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_state_update(const DecodeParams& p, bool bf16, cudaStream_t stream) {
  return bf16 ? dispatch_n<__nv_bfloat16>(p, stream) : dispatch_n<float>(p, stream);
}

}  // namespace ssm
