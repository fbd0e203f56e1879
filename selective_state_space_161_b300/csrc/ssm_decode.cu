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
// fp32 states and touches only a few bytes of activations.

#include "ssm_device.cuh"
#include "ssm_internal.h"

#include <algorithm>
#include <cstdlib>

namespace ssm {

constexpr int kDecodeThreads = 64;  // swept 32-512 on the 256 x 5120 x 16 decode: 64 fastest

// SPL consecutive I/O elements -> fp32; multiples of 4 move as 16-byte (fp32) or 8-byte
// (bf16) pieces.
template <int SPL>
__device__ __forceinline__ void load_vals(const float* g, float* v) {
  if constexpr (SPL % 4 == 0) {
#pragma unroll
    for (int k = 0; k < SPL / 4; k++) {
      const float4 q = reinterpret_cast<const float4*>(g)[k];
      v[4 * k] = q.x; v[4 * k + 1] = q.y; v[4 * k + 2] = q.z; v[4 * k + 3] = q.w;
    }
  } else {
#pragma unroll
    for (int n = 0; n < SPL; n++) v[n] = g[n];
  }
}
template <int SPL>
__device__ __forceinline__ void load_vals(const __nv_bfloat16* g, float* v) {
  if constexpr (SPL % 4 == 0) {
#pragma unroll
    for (int k = 0; k < SPL / 4; k++) {
      const uint2 q = reinterpret_cast<const uint2*>(g)[k];
      v[4 * k] = __uint_as_float(q.x << 16); v[4 * k + 1] = __uint_as_float(q.x & 0xFFFF0000u);
      v[4 * k + 2] = __uint_as_float(q.y << 16); v[4 * k + 3] = __uint_as_float(q.y & 0xFFFF0000u);
    }
  } else {
#pragma unroll
    for (int n = 0; n < SPL; n++) v[n] = __bfloat162float(g[n]);
  }
}

// One batch row's operands of a thread's share of a step, loaded before any arithmetic.
template <int SPL>
struct RowOperands {
  float h[SPL], Bv[SPL], Cv[SPL];
  float xraw, uu, zraw;
};

// LPC lanes per (batch, channel), each owning SPL = N / LPC consecutive states, so that
// the state row, A row and B/C rows move as coalesced 16-byte (or 8-byte) pieces; the
// readout sum over states is finished with log2(LPC) shuffles.  The grid is 2-D (channels,
// batch rows), so no index needs an integer division.  A thread serves the same channel of
// two batch rows (b and b + gridDim.y): the A row is loaded once for both, and every load of
// both rows is issued before the first arithmetic that depends on one, so twice the state
// bytes are in flight per thread.  The state math runs on packed fp32 pairs.
template <int N, typename T, int LPC, bool kConv>
__global__ void __launch_bounds__(kDecodeThreads) state_update_kernel(const DecodeParams p) {
  constexpr int SPL = N / LPC;
  constexpr int kChPerCta = kDecodeThreads / LPC;
  // Launched as a programmatic dependent of the previous kernel in the stream: let the next
  // step's launch begin now (its CTAs take the SMs this grid's last CTAs leave), and wait until
  // the previous kernel has finished and its writes are visible before reading anything.
  // Without the launch attribute both are no-ops.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t d = (int64_t)blockIdx.x * kChPerCta + threadIdx.x / LPC;
  const int q = (int)(threadIdx.x % LPC);
  const bool valid = d < p.d_inner;
  const int64_t dc = valid ? d : 0;  // lanes past the end still join the shuffles
  const T* u = static_cast<const T*>(p.u);
  const T* dl = static_cast<const T*>(p.delta);
  const T* zg = static_cast<const T*>(p.z);
  float A[SPL];
  load_vals<SPL>(p.A + dc * N + q * SPL, A);
  const float bias = p.delta_bias ? p.delta_bias[dc] : 0.f;
  const float Dd = p.D ? p.D[dc] : 0.f;

  auto load_row = [&](int64_t b, RowOperands<SPL>& r) {
    const int64_t ic = b * p.d_inner + dc;
    load_vals<SPL>(p.state + ic * N + q * SPL, r.h);
    load_vals<SPL>(static_cast<const T*>(p.B) + b * N + q * SPL, r.Bv);
    load_vals<SPL>(static_cast<const T*>(p.C) + b * N + q * SPL, r.Cv);
    r.xraw = to_f32(dl[ic]);
    r.uu = to_f32(u[ic]);
    r.zraw = zg ? to_f32(zg[ic]) : 0.f;
  };
  auto step_row = [&](int64_t b, RowOperands<SPL>& r) {
    const int64_t ic = b * p.d_inner + dc;
    float uu = r.uu;
    float x_new = 0.f;
    if constexpr (kConv) {
      // u = silu(conv_b + sum_{j<K-1} w[j] * x_{t-(K-1)+j} + w[K-1] * x_t), the earlier inputs
      // coming from conv_state (every lane of the channel computes it; lane 0 shifts it below)
      const int K = p.d_conv;
      const float* cs = p.conv_state + ic * (K - 1);
      float c = p.conv_b ? p.conv_b[dc] : 0.f;
      for (int j = 0; j < K - 1; j++) c = fmaf(p.conv_w[dc * K + j], cs[j], c);
      x_new = uu;
      uu = silu(fmaf(p.conv_w[dc * K + K - 1], x_new, c));
    }
    const float x = r.xraw + bias;
    const float dt = p.softplus ? softplus(x) : x;
    const float w = dt * uu;
    float acc = 0.f;
    if constexpr (SPL % 2 == 0) {
      const float2 dt2 = make_float2(dt * kLog2e, dt * kLog2e), w2 = make_float2(w, w);
      float2 acc2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int n = 0; n < SPL; n += 2) {
        const float2 xa = __fmul2_rn(dt2, make_float2(A[n], A[n + 1]));
        const float2 dA = make_float2(ex2(xa.x), ex2(xa.y));
        const float2 hn = __ffma2_rn(dA, make_float2(r.h[n], r.h[n + 1]),
                                     __fmul2_rn(w2, make_float2(r.Bv[n], r.Bv[n + 1])));
        r.h[n] = hn.x;
        r.h[n + 1] = hn.y;
        acc2 = __ffma2_rn(make_float2(r.Cv[n], r.Cv[n + 1]), hn, acc2);
      }
      acc = acc2.x + acc2.y;
    } else {
#pragma unroll
      for (int n = 0; n < SPL; n++) {
        const float dA = ex2(dt * (A[n] * kLog2e));
        r.h[n] = fmaf(dA, r.h[n], w * r.Bv[n]);
        acc = fmaf(r.Cv[n], r.h[n], acc);
      }
    }
#pragma unroll
    for (int o = 1; o < LPC; o <<= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
    if (!valid) return;
    float* st = p.state + ic * N + q * SPL;
    if constexpr (SPL % 4 == 0) {
#pragma unroll
      for (int k = 0; k < SPL / 4; k++)
        reinterpret_cast<float4*>(st)[k] = make_float4(r.h[4 * k], r.h[4 * k + 1], r.h[4 * k + 2], r.h[4 * k + 3]);
    } else {
#pragma unroll
      for (int n = 0; n < SPL; n++) st[n] = r.h[n];
    }
    if constexpr (kConv) {
      if (q == 0 && p.d_conv > 1) {  // after the shuffle: every lane has read conv_state
        float* cs = p.conv_state + ic * (p.d_conv - 1);
        for (int j = 0; j < p.d_conv - 2; j++) cs[j] = cs[j + 1];
        cs[p.d_conv - 2] = x_new;
      }
    }
    if (q == 0) {
      acc = fmaf(Dd, uu, acc);
      if (zg) acc *= silu(r.zraw);
      static_cast<T*>(p.y)[ic] = from_f32<T>(acc);
    }
  };

  // rows b0 and b0 + gridDim.y together (one pass unless batch > 2 * 65535)
  for (int64_t b0 = blockIdx.y; b0 < p.batch; b0 += 2 * (int64_t)gridDim.y) {
    const int64_t b1 = b0 + gridDim.y;
    const bool two = b1 < p.batch;  // CTA-uniform
    RowOperands<SPL> r0, r1;
    load_row(b0, r0);
    if (two) load_row(b1, r1);
    step_row(b0, r0);
    if (two) step_row(b1, r1);
  }
}

// Programmatic dependent launch of the decode steps (SSM_DECODE_PDL=0 turns it off).
static bool decode_pdl() {
  const char* v = std::getenv("SSM_DECODE_PDL");
  return v == nullptr || std::atoi(v) != 0;
}

template <int N, typename T>
static cudaError_t launch_t(const DecodeParams& p, cudaStream_t s) {
  // Lanes per channel: a power of two (the shuffles pair lanes by xor) with 8 states
  // each where d_state allows (measured fastest at d_state 16: enough bytes in flight per
  // thread, 16-byte pieces, and twice the threads of one lane per channel).
  constexpr int LPC = (N % 8 == 0) ? N / 8 : 1;
  constexpr int kChPerCta = kDecodeThreads / LPC;
  const dim3 grid((unsigned)((p.d_inner + kChPerCta - 1) / kChPerCta),
                  (unsigned)std::min<int64_t>((p.batch + 1) / 2, 65535));
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kDecodeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = decode_pdl() ? 1 : 0;
  return p.conv_w != nullptr ? cudaLaunchKernelEx(&cfg, state_update_kernel<N, T, LPC, true>, p)
                             : cudaLaunchKernelEx(&cfg, state_update_kernel<N, T, LPC, false>, p);
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
