// Forward states for the training backward pass (ssm_scan_bwd.cu): per-chunk summaries of
// the recurrence and the state before every 8 steps (kCkptSteps).  These are the forward
// recurrence of the selective scan (dA = exp(delta*A), dBu = delta*B*u,
// h_t = dA_t h_{t-1} + dBu_t; youngju.dev "Mamba: Linear-Time Sequence Modeling with
// Selective State Spaces 论文分析", "解决方案：Kernel Fusion + Recomputation", whose backward
// recomputes the intermediate states instead of storing them) without the readout.
//
// A CTA covers 32 consecutive channels of one batch row over one time chunk, one lane per
// channel with all of its states as fp32 pairs in registers.  Per tile of 16 steps, delta and
// u arrive in shared memory by cp.async (16-byte pieces) one tile ahead, and the B_t rows
// are fetched a tile ahead and read as shared-memory broadcasts.
//  - summary mode (every chunk but the last): the chunk from a zero state; writes
//    (sum of delta over the chunk, end state);
//  - checkpoint mode (every chunk): the chunk from its true start state (the initial state
//    folded with the summaries of the chunks before it, using the associativity of
//    (a, b) o (a', b') = (a a', a b' + b) and prod_t exp(delta_t A) = exp(A sum_t delta_t)),
//    storing the state before every 8 steps (two per tile).

#include "ssm_device.cuh"
#include "ssm_internal.h"

#include <algorithm>
#include <cstdlib>
#include <type_traits>

namespace ssm {

constexpr int kScanCh = 32;                          // channels per CTA
constexpr int kScanTile = 16;                        // time steps per pipelined tile
constexpr int kChunkAlign = 32;
static_assert(kScanTile == 2 * kCkptSteps, "two checkpoints per tile");

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  const int n = valid ? 16 : 0;  // n == 0: no global read, 16 zero bytes written
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
__device__ __forceinline__ void cp_async_wait_prev() { asm volatile("cp.async.wait_group 1;\n" ::); }

// 16 raw bytes of B/C -> fp32 values in shared memory.
__device__ __forceinline__ void store_bc_chunk(float* dst, uint4 v, float) {
  *reinterpret_cast<float4*>(dst) = make_float4(__uint_as_float(v.x), __uint_as_float(v.y),
                                                __uint_as_float(v.z), __uint_as_float(v.w));
}
__device__ __forceinline__ void store_bc_chunk(float* dst, uint4 v, __nv_bfloat16) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 2; q++)
    *reinterpret_cast<float4*>(dst + 4 * q) = make_float4(
        __uint_as_float(w[2 * q] << 16), __uint_as_float(w[2 * q] & 0xFFFF0000u),
        __uint_as_float(w[2 * q + 1] << 16), __uint_as_float(w[2 * q + 1] & 0xFFFF0000u));
}

// kCkpt == false: summary mode; kCkpt == true: checkpoint mode (see the file comment).
template <int N, typename T, bool kCkpt>
__global__ void __launch_bounds__(kScanCh)
scan_state_kernel(const ScanParams p) {
  constexpr bool kSummary = !kCkpt;
  constexpr int kS = sizeof(T);
  constexpr int kVec = 16 / kS;
  constexpr int kCPR = kScanCh / kVec;
  constexpr int kRowsPerPass = kScanCh / kCPR;
  constexpr int kPasses = kScanTile / kRowsPerPass;
  constexpr int NP = (N + 1) / 2;
  constexpr int NPAD = 2 * NP;
  constexpr bool kVecBC = (N * kS) % 16 == 0;
  constexpr int kBCChunks = kScanTile * N / kVec;
  constexpr int kBCChunksPerThread = kVecBC ? (kBCChunks + kScanCh - 1) / kScanCh : 1;
  constexpr int kBCVals = kScanTile * N;
  constexpr int kBCValsPerThread = kVecBC ? 1 : (kBCVals + kScanCh - 1) / kScanCh;
  __shared__ __align__(16) T sX[2][2][kScanTile][kScanCh];
  __shared__ __align__(16) float sB[2][kScanTile][NPAD];
  const int64_t n_dtiles = (p.d_inner + kScanCh - 1) / kScanCh;
  const int chunks = kSummary ? p.n_chunks - 1 : p.n_chunks;
  int64_t blk = blockIdx.x;
  const int64_t dtile = blk % n_dtiles;
  blk /= n_dtiles;
  const int c = (int)(blk % chunks);
  const int64_t b = blk / chunks;
  const int tid = threadIdx.x;
  const int64_t Dn = p.d_inner, L = p.L;
  const int64_t d0 = dtile * kScanCh;
  const int64_t d = d0 + tid;
  const bool active = d < Dn;
  const int64_t t0 = (int64_t)c * p.chunk_len;
  const int64_t t1 = min(t0 + p.chunk_len, L);
  const int ntiles = (int)((t1 - t0 + kScanTile - 1) / kScanTile);
  const T* __restrict__ Bg = static_cast<const T*>(p.B);
  const int ci = tid % kCPR, rb = tid / kCPR;
  const bool dvalid = d0 + (int64_t)ci * kVec < Dn;
  const int64_t row_bytes = Dn * kS;
  const char* xsrc[2] = {static_cast<const char*>(p.delta), static_cast<const char*>(p.u)};
  const int64_t x_off0 = ((b * L + t0 + rb) * Dn + d0 + (int64_t)ci * kVec) * kS;
  auto issue_x = [&](int tile, int stage) {
    const int64_t rows0 = (int64_t)tile * kScanTile + rb;
    const int64_t off = x_off0 + (int64_t)tile * kScanTile * row_bytes;
#pragma unroll
    for (int x = 0; x < 2; x++) {
#pragma unroll
      for (int m = 0; m < kPasses; m++) {
        const bool valid = dvalid && t0 + rows0 + m * kRowsPerPass < t1;
        const char* g = xsrc[x] + off + (int64_t)m * kRowsPerPass * row_bytes;
        cp_async16(&sX[stage][x][rb + m * kRowsPerPass][ci * kVec], valid ? g : xsrc[x], valid);
      }
    }
  };
  uint4 bcv[kBCChunksPerThread];
  float bcs[kBCValsPerThread];
  const int64_t bc_elems = p.batch * L * N;
  auto load_b = [&](int tile) {
    const int64_t e_row0 = (b * L + t0 + (int64_t)tile * kScanTile) * N;
    const int64_t rows_left = t1 - (t0 + (int64_t)tile * kScanTile);
    if constexpr (kVecBC) {
#pragma unroll
      for (int j = 0; j < kBCChunksPerThread; j++) {
        const int q = tid + j * kScanCh;
        const int e = q * kVec;
        bcv[j] = make_uint4(0, 0, 0, 0);
        if (q < kBCChunks && e / N < rows_left && e_row0 + e + kVec <= bc_elems)
          bcv[j] = *reinterpret_cast<const uint4*>(Bg + e_row0 + e);
      }
    } else {
#pragma unroll
      for (int j = 0; j < kBCValsPerThread; j++) {
        const int e = tid + j * kScanCh;
        bcs[j] = 0.f;
        if (e < kBCVals && e / N < rows_left) bcs[j] = to_f32(Bg[e_row0 + e]);
      }
    }
  };
  auto store_b = [&](int stage) {
    if constexpr (kVecBC) {
#pragma unroll
      for (int j = 0; j < kBCChunksPerThread; j++) {
        const int q = tid + j * kScanCh;
        if (q < kBCChunks) store_bc_chunk(&sB[stage][0][0] + q * kVec, bcv[j], T());
      }
    } else {
#pragma unroll
      for (int j = 0; j < kBCValsPerThread; j++) {
        const int e = tid + j * kScanCh;
        if (e < kBCVals) sB[stage][e / N][e % N] = bcs[j];
      }
    }
  };
  if constexpr (NPAD != N) {
    for (int i = tid; i < 2 * kScanTile; i += kScanCh) (&sB[0][0][0])[i * NPAD + N] = 0.f;
  }
  float2 A2[NP], h[NP];
#pragma unroll
  for (int j = 0; j < NP; j++) {
    const float a0 = active ? p.A[d * N + 2 * j] * kLog2e : 0.f;
    const float a1 = (active && 2 * j + 1 < N) ? p.A[d * N + 2 * j + 1] * kLog2e : 0.f;
    A2[j] = make_float2(a0, a1);
    h[j] = make_float2(0.f, 0.f);
    if (kCkpt && active && p.initial_state) {
      const float* h0 = p.initial_state + (b * Dn + d) * N;
      h[j] = make_float2(h0[2 * j], 2 * j + 1 < N ? h0[2 * j + 1] : 0.f);
    }
  }
  const float bias = (active && p.delta_bias) ? p.delta_bias[d] : 0.f;
  const bool sp = p.softplus != 0;
  if (ntiles > 0) { issue_x(0, 0); cp_async_commit(); load_b(0); store_b(0); }
  if (kCkpt && c > 0 && active) {  // fold the summaries of the chunks before this one
    const int64_t base = b * (p.n_chunks - 1);
    for (int j = 0; j < c; j++) {
      const float S = p.ws_S[(base + j) * Dn + d];
      const float* hj = p.ws_h + ((base + j) * Dn + d) * N;
#pragma unroll
      for (int q = 0; q < NP; q++) {
        const float e0 = hj[2 * q];
        const float e1 = (2 * q + 1 < N) ? hj[2 * q + 1] : 0.f;
        h[q].x = fmaf(ex2(A2[q].x * S), h[q].x, e0);
        h[q].y = fmaf(ex2(A2[q].y * S), h[q].y, e1);
      }
    }
  }
  float S = 0.f, S_comp = 0.f;  // compensated (Kahan) sum of delta (summary mode)
  // One recurrence step on all states (packed pairs), given the step size and delta*u.
  auto advance = [&](int stage, int k, float dt, float w) {
    if (kSummary) { const float yk = dt - S_comp; const float tk = S + yk; S_comp = (tk - S) - yk; S = tk; }
    const float2 dt2 = make_float2(dt, dt), w2 = make_float2(w, w);
    const float* Bk = sB[stage][k];
#pragma unroll
    for (int j = 0; j < NP; j++) {
      float2 Bv;
      if constexpr (NPAD % 4 == 0) {
        const float4 b4 = *reinterpret_cast<const float4*>(Bk + 4 * (j / 2));
        Bv = (j & 1) ? make_float2(b4.z, b4.w) : make_float2(b4.x, b4.y);
      } else {
        Bv = *reinterpret_cast<const float2*>(Bk + 2 * j);
      }
      const float2 xa = __fmul2_rn(dt2, A2[j]);
      const float2 dA = make_float2(ex2(xa.x), ex2(xa.y));
      h[j] = __ffma2_rn(dA, h[j], __fmul2_rn(w2, Bv));
    }
  };
  for (int tile = 0; tile < ntiles; tile++) {
    const int stage = tile & 1;
    if (tile + 1 < ntiles) { issue_x(tile + 1, stage ^ 1); load_b(tile + 1); }
    cp_async_commit();
    cp_async_wait_prev();
    __syncthreads();
    const int64_t ts = t0 + (int64_t)tile * kScanTile;
    // checkpoint mode: the state before step ts + q (q = 0 or kCkptSteps; chunks start on
    // tile boundaries)
    auto store_ckpt = [&](int q) {
      float* ck = p.ckpt_h + ((b * ((L + kCkptSteps - 1) / kCkptSteps) + (ts + q) / kCkptSteps) * Dn + d) * N;
      if constexpr (N % 4 == 0) {  // whole 16-byte pieces (a channel's row is 16-byte aligned)
#pragma unroll
        for (int j = 0; j < NP; j += 2)
          *reinterpret_cast<float4*>(ck + 2 * j) = make_float4(h[j].x, h[j].y, h[j + 1].x, h[j + 1].y);
      } else {
#pragma unroll
        for (int j = 0; j < NP; j++) { ck[2 * j] = h[j].x; if (2 * j + 1 < N) ck[2 * j + 1] = h[j].y; }
      }
    };
    if (kCkpt && active) store_ckpt(0);
    if (active) {
      if (ts + kScanTile <= t1) {
        // two steps' step sizes at once in packed fp32x2, then the two recurrence steps
#pragma unroll
        for (int k = 0; k < kScanTile; k += 2) {
          const float2 x = __fadd2_rn(make_float2(to_f32(sX[stage][0][k][tid]), to_f32(sX[stage][0][k + 1][tid])),
                                      make_float2(bias, bias));
          const float2 dt = sp ? softplus2(x) : x;
          const float2 w = __fmul2_rn(dt, make_float2(to_f32(sX[stage][1][k][tid]), to_f32(sX[stage][1][k + 1][tid])));
          advance(stage, k, dt.x, w.x);
          advance(stage, k + 1, dt.y, w.y);
          if (kCkpt && k + 2 == kCkptSteps) store_ckpt(kCkptSteps);
        }
      } else {
        const int steps = (int)(t1 - ts);
        for (int k = 0; k < steps; k++) {
          const float x = to_f32(sX[stage][0][k][tid]) + bias;
          const float dt = sp ? softplus(x) : x;
          advance(stage, k, dt, dt * to_f32(sX[stage][1][k][tid]));
          if (kCkpt && k + 1 == kCkptSteps && steps > kCkptSteps) store_ckpt(kCkptSteps);
        }
      }
    }
    __syncthreads();
    if (tile + 1 < ntiles) store_b(stage ^ 1);
  }
  if (kSummary && active) {
    const int64_t slot = (b * (p.n_chunks - 1) + c) * Dn + d;
    p.ws_S[slot] = S;
#pragma unroll
    for (int j = 0; j < NP; j++) { p.ws_h[slot * N + 2 * j] = h[j].x; if (2 * j + 1 < N) p.ws_h[slot * N + 2 * j + 1] = h[j].y; }
  }
}


int scan_channels_per_cta() { return kScanCh; }

static int64_t env_int(const char* name, int64_t fallback) {
  if (const char* v = std::getenv(name)) {
    const long long x = std::atoll(v);
    if (x > 0) return x;
  }
  return fallback;
}

void plan_scan(int64_t batch, int64_t L, int64_t d_inner, int sms, ScanPlan* plan) {
  // Time chunks of the backward pass: none when its gradient CTAs (64 channels each, about
  // three resident per SM) fill the GPU; otherwise about two waves of them, at least 64 steps
  // per chunk (measured on B300: the 2 x 2048 x 1536 shape at 0.30 ms with 16 chunks against
  // 0.35 with 8 or 32; the 8 x 2048 x 5120 shape fastest unchunked).
  const int64_t per_chunk = batch * ((d_inner + 63) / 64);
  const int64_t slots = (int64_t)sms * 3;
  int64_t G = 1;
  if (per_chunk > 0 && per_chunk < slots) G = (2 * slots + per_chunk - 1) / per_chunk;
  G = env_int("SSM_BWD_CHUNKS", G);  // tuning override
  G = std::min<int64_t>(G, std::max<int64_t>(1, L / 64));
  G = std::min<int64_t>(G, 4096);
  int64_t len = L > 0 ? (L + G - 1) / G : 1;
  len = (len + kChunkAlign - 1) / kChunkAlign * kChunkAlign;
  plan->lanes = 1;
  plan->chunk_len = len;
  plan->n_chunks = L > 0 ? (int)((L + len - 1) / len) : 1;
}

template <typename T>
static cudaError_t summary_only(const ScanParams& p, cudaStream_t s) {
  const int64_t blocks = (p.d_inner + kScanCh - 1) / kScanCh * (p.n_chunks - 1) * p.batch;
  switch (p.d_state) {
#define SSM_SUMMARY_CASE(NN) \
    case NN: scan_state_kernel<NN, T, false><<<(unsigned)blocks, kScanCh, 0, s>>>(p); break;
    SSM_SUMMARY_CASE(1) SSM_SUMMARY_CASE(2) SSM_SUMMARY_CASE(3) SSM_SUMMARY_CASE(4)
    SSM_SUMMARY_CASE(5) SSM_SUMMARY_CASE(6) SSM_SUMMARY_CASE(7) SSM_SUMMARY_CASE(8)
    SSM_SUMMARY_CASE(9) SSM_SUMMARY_CASE(10) SSM_SUMMARY_CASE(11) SSM_SUMMARY_CASE(12)
    SSM_SUMMARY_CASE(13) SSM_SUMMARY_CASE(14) SSM_SUMMARY_CASE(15) SSM_SUMMARY_CASE(16)
#undef SSM_SUMMARY_CASE
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

template <typename T>
static cudaError_t ckpt_only(const ScanParams& p, cudaStream_t s) {
  const int64_t blocks = (p.d_inner + kScanCh - 1) / kScanCh * p.n_chunks * p.batch;
  switch (p.d_state) {
#define SSM_CKPT_CASE(NN) \
    case NN: scan_state_kernel<NN, T, true><<<(unsigned)blocks, kScanCh, 0, s>>>(p); break;
    SSM_CKPT_CASE(1) SSM_CKPT_CASE(2) SSM_CKPT_CASE(3) SSM_CKPT_CASE(4)
    SSM_CKPT_CASE(5) SSM_CKPT_CASE(6) SSM_CKPT_CASE(7) SSM_CKPT_CASE(8)
    SSM_CKPT_CASE(9) SSM_CKPT_CASE(10) SSM_CKPT_CASE(11) SSM_CKPT_CASE(12)
    SSM_CKPT_CASE(13) SSM_CKPT_CASE(14) SSM_CKPT_CASE(15) SSM_CKPT_CASE(16)
#undef SSM_CKPT_CASE
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_scan_ckpt(const ScanParams& p, bool bf16, cudaStream_t stream) {
  return bf16 ? ckpt_only<__nv_bfloat16>(p, stream) : ckpt_only<float>(p, stream);
}

cudaError_t launch_scan_summary(const ScanParams& p, bool bf16, cudaStream_t stream) {
  if (p.n_chunks <= 1) return cudaSuccess;
  return bf16 ? summary_only<__nv_bfloat16>(p, stream) : summary_only<float>(p, stream);
}

}  // namespace ssm
