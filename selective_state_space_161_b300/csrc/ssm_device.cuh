// Device-side helpers shared by the scan and decode kernels: the fast
// transcendental steps of the selective scan and I/O dtype conversion.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssm {

constexpr float kLog2e = 1.4426950408889634f;

// 2^x on the SFU (MUFU.EX2); subnormal results flush to zero.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// log1p(e) for e in [0, 1], as e * q(e): q is a degree-9 polynomial from Chebyshev
// interpolation of log1p(e)/e on [0, 1] (nodes cos((2k+1)pi/20), k = 0..9, mapped to [0, 1];
// the power-basis coefficients rounded to float).  Evaluated by Horner's rule with fused
// multiply-adds in float it is within 1.4e-7 relative error of log1p on the whole interval,
// small e included (e * q(e) keeps full relative precision where 1 + e would lose it), and
// it needs no MUFU operation.
__device__ __forceinline__ float log1p_unit(float e) {
  float q = -0.0031760570127516985f;
  q = fmaf(q, e, 0.019542526453733444f);
  q = fmaf(q, e, -0.056373611092567444f);
  q = fmaf(q, e, 0.10543623566627502f);
  q = fmaf(q, e, -0.1526966691017151f);
  q = fmaf(q, e, 0.1966327428817749f);
  q = fmaf(q, e, -0.24951615929603577f);
  q = fmaf(q, e, 0.33329710364341736f);
  q = fmaf(q, e, -0.49999892711639404f);
  q = fmaf(q, e, 1.0f);
  return e * q;
}
__device__ __forceinline__ float2 log1p_unit2(float2 e) {
  float2 q = make_float2(-0.0031760570127516985f, -0.0031760570127516985f);
  q = __ffma2_rn(q, e, make_float2(0.019542526453733444f, 0.019542526453733444f));
  q = __ffma2_rn(q, e, make_float2(-0.056373611092567444f, -0.056373611092567444f));
  q = __ffma2_rn(q, e, make_float2(0.10543623566627502f, 0.10543623566627502f));
  q = __ffma2_rn(q, e, make_float2(-0.1526966691017151f, -0.1526966691017151f));
  q = __ffma2_rn(q, e, make_float2(0.1966327428817749f, 0.1966327428817749f));
  q = __ffma2_rn(q, e, make_float2(-0.24951615929603577f, -0.24951615929603577f));
  q = __ffma2_rn(q, e, make_float2(0.33329710364341736f, 0.33329710364341736f));
  q = __ffma2_rn(q, e, make_float2(-0.49999892711639404f, -0.49999892711639404f));
  q = __ffma2_rn(q, e, make_float2(1.f, 1.f));
  return __fmul2_rn(e, q);
}

// softplus(x) = log(1 + e^x) = max(x, 0) + log1p(e^-|x|), e^-|x| in (0, 1] on the SFU.
__device__ __forceinline__ float softplus(float x) {
  return fmaxf(x, 0.f) + log1p_unit(ex2(-fabsf(x) * kLog2e));
}

// softplus on two values at once (packed fp32x2 arithmetic).
__device__ __forceinline__ float2 softplus2(float2 x) {
  const float2 e = make_float2(ex2(-fabsf(x.x) * kLog2e), ex2(-fabsf(x.y) * kLog2e));
  return __fadd2_rn(make_float2(fmaxf(x.x, 0.f), fmaxf(x.y, 0.f)), log1p_unit2(e));
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
