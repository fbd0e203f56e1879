/*
 * Seeded synthetic-input generator shared by the test oracle and the CUDA
 * benchmarks.  It holds none of the selective-scan arithmetic: it only turns
 * (seed, tensor id, flat index) into a number.
 *
 * Bit-reproducibility contract: the same source compiles for the host (gcc,
 * -ffp-contract=off) and for the device (nvcc, --fmad=false), and every step
 * below is a correctly rounded IEEE double operation (+, -, *, /, sqrt) or
 * integer arithmetic, so a value drawn on the GPU equals the value drawn on
 * the CPU bit for bit.  No libm call is used for that reason; the natural
 * logarithm is evaluated from its atanh series.
 *
 * Counter-based stream: SplitMix64's output function (Steele, Lea & Flood,
 * "Fast splittable pseudorandom number generators", OOPSLA 2014) applied to a
 * Weyl sequence keyed by (seed, tensor id, counter).
 * Normal deviates: Marsaglia's polar method, with the k-th rejection attempt
 * for element i drawing counters 2*(64*i + k) and 2*(64*i + k) + 1.
 */
#ifndef SSM_INPUTGEN_CORE_H
#define SSM_INPUTGEN_CORE_H
#include <stdint.h>

#if defined(__CUDACC__)
#define GEN_HD __host__ __device__ __forceinline__
#else
#define GEN_HD static inline
#endif

#define GEN_GOLDEN 0x9E3779B97F4A7C15ULL

/* SplitMix64 output mix (the published constants and shifts). */
GEN_HD uint64_t gen_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* Stream key for one tensor of one workload. */
GEN_HD uint64_t gen_key(uint64_t seed, uint64_t tensor_id) {
  return gen_mix64(seed * GEN_GOLDEN + gen_mix64(tensor_id + 0x632BE59BD9B4E019ULL));
}

/* 64 random bits for counter c of the stream `key`. */
GEN_HD uint64_t gen_bits(uint64_t key, uint64_t c) {
  return gen_mix64(key + (c + 1ULL) * GEN_GOLDEN);
}

/* Uniform double in the open interval (0, 1): 53 random bits plus one half. */
GEN_HD double gen_uniform(uint64_t key, uint64_t c) {
  return ((double)(gen_bits(key, c) >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

/* Natural log of s in (0, 1] by s = m * 2^e, m in [sqrt(1/2), sqrt(2)),
 * log m = 2 atanh(f), f = (m - 1)/(m + 1), |f| < 0.1716; 12 odd terms of the
 * atanh series leave a truncation error below 1e-19. */
GEN_HD double gen_log(double s) {
  union { double d; uint64_t u; } v;
  v.d = s;
  int e = (int)((v.u >> 52) & 0x7FF) - 1023;
  v.u = (v.u & 0x000FFFFFFFFFFFFFULL) | 0x3FF0000000000000ULL; /* m in [1, 2) */
  double m = v.d;
  if (m > 1.4142135623730951) { m = m * 0.5; e += 1; }
  double f = (m - 1.0) / (m + 1.0);
  double f2 = f * f;
  double term = f, sum = 0.0;
  for (int k = 0; k < 12; k++) {
    sum = sum + term / (double)(2 * k + 1);
    term = term * f2;
  }
  return (double)e * 0.6931471805599453 + 2.0 * sum;
}

/* Standard normal deviate for element index i (polar method, <= 32 tries;
 * the chance that all 32 are rejected is below 1e-21 and then 0 is returned). */
GEN_HD double gen_normal(uint64_t key, uint64_t i) {
  for (uint64_t k = 0; k < 32; k++) {
    uint64_t c = 2ULL * (64ULL * i + k);
    double a = 2.0 * gen_uniform(key, c) - 1.0;
    double b = 2.0 * gen_uniform(key, c + 1ULL) - 1.0;
    double s = a * a + b * b;
    if (s < 1.0 && s > 0.0) {
      double r = -2.0 * gen_log(s) / s;
#if defined(__CUDA_ARCH__)
      return a * __dsqrt_rn(r);
#else
      return a * __builtin_sqrt(r);
#endif
    }
  }
  return 0.0;
}

/* float -> bfloat16 bits, round to nearest even (inputs are finite). */
GEN_HD uint16_t gen_f32_to_bf16(float x) {
  union { float f; uint32_t u; } v;
  v.f = x;
  uint32_t lsb = (v.u >> 16) & 1u;
  return (uint16_t)((v.u + 0x7FFFu + lsb) >> 16);
}

#endif
