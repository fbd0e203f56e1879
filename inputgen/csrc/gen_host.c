/*
 * Host side of the seeded input generator (plain C, OpenMP over elements).
 * Built with -ffp-contract=off so that every value matches the device fill
 * bit for bit (see gen_core.h).  Test and benchmark infrastructure only.
 */
#include <math.h>
#include <stdint.h>
#include "gen_core.h"

/* out[i] = fp32(mean + sd * N(0,1)) for flat indices start .. start+count-1. */
void gen_normal_f32(uint64_t seed, uint64_t tensor_id, double mean, double sd,
                    int64_t start, int64_t count, float* out) {
  uint64_t key = gen_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < count; i++)
    out[i] = (float)(mean + sd * gen_normal(key, (uint64_t)(start + i)));
}

/* Same values rounded once more to bfloat16 (round to nearest even). */
void gen_normal_bf16(uint64_t seed, uint64_t tensor_id, double mean, double sd,
                     int64_t start, int64_t count, uint16_t* out) {
  uint64_t key = gen_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < count; i++)
    out[i] = gen_f32_to_bf16((float)(mean + sd * gen_normal(key, (uint64_t)(start + i))));
}

/* Gather variants: element k is the value at flat index idx[k]. */
void gen_normal_f32_at(uint64_t seed, uint64_t tensor_id, double mean, double sd,
                       const int64_t* idx, int64_t count, float* out) {
  uint64_t key = gen_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < count; i++)
    out[i] = (float)(mean + sd * gen_normal(key, (uint64_t)idx[i]));
}

void gen_normal_bf16_at(uint64_t seed, uint64_t tensor_id, double mean, double sd,
                        const int64_t* idx, int64_t count, uint16_t* out) {
  uint64_t key = gen_key(seed, tensor_id);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < count; i++)
    out[i] = gen_f32_to_bf16((float)(mean + sd * gen_normal(key, (uint64_t)idx[i])));
}

/* Uniform draws in (0,1), as doubles, for host-only recipes. */
void gen_uniform_f64(uint64_t seed, uint64_t tensor_id, int64_t start, int64_t count,
                     double* out) {
  uint64_t key = gen_key(seed, tensor_id);
  for (int64_t i = 0; i < count; i++) out[i] = gen_uniform(key, (uint64_t)(start + i));
}

/* Step-size bias recipe: dt log-uniform on [dt_min, dt_max], bias = the
 * inverse of softplus at dt, i.e. dt + log(-expm1(-dt)), rounded to fp32.
 * Host only (uses libm); the device never draws this tensor. */
void gen_delta_bias_f32(uint64_t seed, uint64_t tensor_id, double dt_min, double dt_max,
                        int64_t count, float* out) {
  uint64_t key = gen_key(seed, tensor_id);
  double lo = log(dt_min), hi = log(dt_max);
  for (int64_t i = 0; i < count; i++) {
    double dt = exp(lo + (hi - lo) * gen_uniform(key, (uint64_t)i));
    out[i] = (float)(dt + log(-expm1(-dt)));
  }
}

/* bfloat16 bits -> fp32 (exact). */
void gen_bf16_to_f32(const uint16_t* in, int64_t count, float* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < count; i++) {
    union { uint32_t u; float f; } v;
    v.u = (uint32_t)in[i] << 16;
    out[i] = v.f;
  }
}
