// Device-side helpers shared by the scan and decode kernels: the fast
// transcendental steps of the selective scan and I/O dtype conversion.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssm {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// 2^x on the SFU (MUFU.EX2); subnormal results flush to zero.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// softplus(x) = log(1 + e^x) = max(x, 0) + log1p(e^-|x|).
// With e = e^-|x| in (0, 1]: for e < 1/16 the Taylor series of log1p,
// e - e^2/2 + ... - e^6/6 (truncation below 1e-8 relative), keeps full
// relative accuracy where 1 + e would round away the small term; otherwise
// log2(1 + e) on the SFU, scaled by ln 2.
__device__ __forceinline__ float softplus(float x) {
  float e = ex2(-fabsf(x) * kLog2e);
  float series = e * (1.f - e * (0.5f - e * (1.f / 3.f - e * (0.25f - e * (0.2f - e * (1.f / 6.f))))));
  float viaLog = lg2(1.f + e) * kLn2;
  return fmaxf(x, 0.f) + (e < 0.0625f ? series : viaLog);
}

// softplus on two values at once (packed fp32x2 arithmetic; same steps as above,
// with the log1p series as Horner in e: e * (1 + e(-1/2 + e(1/3 + e(-1/4 + e/5))))).
__device__ __forceinline__ float2 softplus2(float2 x) {
  const float2 e = make_float2(ex2(-fabsf(x.x) * kLog2e), ex2(-fabsf(x.y) * kLog2e));
  float2 q = __ffma2_rn(e, make_float2(0.2f, 0.2f), make_float2(-0.25f, -0.25f));
  q = __ffma2_rn(e, q, make_float2(1.f / 3.f, 1.f / 3.f));
  q = __ffma2_rn(e, q, make_float2(-0.5f, -0.5f));
  q = __ffma2_rn(e, q, make_float2(1.f, 1.f));
  const float2 series = __fmul2_rn(e, q);
  const float2 ope = __fadd2_rn(e, make_float2(1.f, 1.f));
  const float2 viaLog = __fmul2_rn(make_float2(lg2(ope.x), lg2(ope.y)), make_float2(kLn2, kLn2));
  const float2 l = make_float2(e.x < 0.0625f ? series.x : viaLog.x, e.y < 0.0625f ? series.y : viaLog.y);
  return __fadd2_rn(make_float2(fmaxf(x.x, 0.f), fmaxf(x.y, 0.f)), l);
}

// silu on two values at once.
__device__ __forceinline__ float2 silu2(float2 z) {
  const float2 e = make_float2(ex2(-z.x * kLog2e), ex2(-z.y * kLog2e));
  const float2 d = __fadd2_rn(e, make_float2(1.f, 1.f));
  return __fmul2_rn(z, make_float2(rcp(d.x), rcp(d.y)));
}

// silu(z) = z * sigmoid(z) = z / (1 + e^-z).
__device__ __forceinline__ float silu(float z) { return z * rcp(1.f + ex2(-z * kLog2e)); }

// I/O element conversion.
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

}  // namespace ssm
