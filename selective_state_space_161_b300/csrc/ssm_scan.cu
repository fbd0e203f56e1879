// Selective-scan forward: fused softplus step size, zero-order-hold style
// discretisation (dA = exp(delta*A), dBu = delta*B*u), the linear recurrence
// over (batch, d_inner, d_state), the C.h + D.u readout and the SiLU(z) gate.
//
// Sources (page title, section): youngju.dev "Mamba: Linear-Time Sequence
// Modeling with Selective State Spaces 论文分析", "解决方案：Kernel Fusion +
// Recomputation" (the concept selective_scan: discretise, recur, read out with
// the updated state) and "Mamba 模块架构" (D, the SiLU gate, the biased delta
// projection); ai-lab.club "机器学习基础算法", discrete state equations.
// The pages' kernel keeps every intermediate (dA, dBu, h) out of HBM; here
// they live in registers and only u, delta, z, B, C in and y out touch HBM.
//
// Parallel structure.  A CTA covers 32 consecutive channels (d_inner) of one batch row
// over one time chunk and walks the chunk sequentially; the recurrence state never
// leaves registers.  Two kernels:
//  - one lane per channel (32-thread CTAs): a thread keeps all d_state states of its
//    channel as fp32 pairs and updates them with packed fp32x2 instructions;
//  - two lanes per channel (64-thread CTAs): each lane keeps half of the states, and the
//    per-step work that does not touch the state (step size, input, skip term, gate,
//    output) is split between the two lanes by step parity and exchanged by shuffles.
//    It doubles the warps for problems with few channels and short sequences.
// Per tile of 16 steps, delta, u (and z) are staged in shared memory by cp.async
// (16-byte pieces, coalesced along d_inner) one tile ahead, and the B_t/C_t rows (shared
// by every channel) are fetched a tile ahead and read as shared-memory broadcasts.
//
// Time chunks.  When batch * d_inner cannot fill the GPU, time is cut into chunks.  The
// recurrence is associative in the pairs (a, b) with (a2, b2) o (a1, b1) =
// (a2 a1, a2 b1 + b2), so a chunk is summarised by its decay prod_t dA_t =
// exp(A * sum_t delta_t) and its end state from zero.  Pass 1 writes those summaries
// for every chunk but the last; pass 2 folds the summaries of the chunks before its own
// into its start state (the given initial state, or zero, folded with every summary before
// it), then runs the exact recurrence and writes y.  No block waits on another block.

#include "ssm_device.cuh"
#include "ssm_internal.h"

#include <algorithm>
#include <cstdlib>
#include <type_traits>

namespace ssm {

constexpr int kScanCh = 32;                          // channels per CTA
constexpr int kScanThreads = 2 * kScanCh;            // two lanes per channel
constexpr int kScanTile = 16;                        // time steps per pipelined tile
constexpr int kChunkAlign = 32;

// How a channel's d_state states are split over its two lanes: each lane owns an
// even number kHalf of them (padding states, if any, have A = B = C = 0 and stay 0).
template <int N>
struct StateSplit {
  static constexpr int kHalf = ((N + 1) / 2 + 1) / 2 * 2;
  static constexpr int kPad = 2 * kHalf;
  static constexpr int kPairs = kHalf / 2;
};

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

__device__ __forceinline__ float shfl_pair(float v) { return __shfl_xor_sync(0xFFFFFFFFu, v, 1); }

// Programmatic dependent launch: the main pass is launched while the summary pass is still
// running; a main-pass CTA that needs summaries waits here until the summary grid has
// completed and its writes are visible (a hardware wait; returns at once without a
// prerequisite grid).  The summary pass lets the main grid launch once each of its CTAs
// has stored its summary.
__device__ __forceinline__ void wait_for_summaries() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_main_pass() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// One lane per channel: a 32-thread CTA covers kScanCh channels of one batch row over one
// time chunk; each thread keeps all of its channel's states (as fp32 pairs) in registers.
template <int N, typename T, bool kSummary, bool kConv, bool kCkpt>
__global__ void __launch_bounds__(kScanCh)
scan_chunk_kernel_1lane(const ScanParams p) {
  // kCkpt: the main pass's true states without any output, storing the state before every
  // tile of kScanTile steps into p.ckpt_h (the checkpoints of the training backward).
  constexpr bool kOut = !kSummary && !kCkpt;
  constexpr int kS = sizeof(T);
  constexpr int kVec = 16 / kS;
  constexpr int kCPR = kScanCh / kVec;
  constexpr int kRowsPerPass = kScanCh / kCPR;
  constexpr int kPasses = kScanTile / kRowsPerPass;
  constexpr int kNX = kOut ? 3 : 2;
  constexpr int kNBC = kOut ? 2 : 1;
  constexpr int NP = (N + 1) / 2;
  constexpr int NPAD = 2 * NP;
  constexpr bool kVecBC = (N * kS) % 16 == 0;
  constexpr int kBCChunks = kNBC * kScanTile * N / kVec;
  constexpr int kBCChunksPerThread = kVecBC ? (kBCChunks + kScanCh - 1) / kScanCh : 1;
  constexpr int kBCVals = kNBC * kScanTile * N;
  constexpr int kBCValsPerThread = kVecBC ? 1 : (kBCVals + kScanCh - 1) / kScanCh;
  __shared__ __align__(16) T sX[2][kNX][kScanTile][kScanCh];
  __shared__ __align__(16) float sBC[2][kNBC][kScanTile][NPAD];
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
  const T* __restrict__ Cg = static_cast<const T*>(p.C);
  const bool has_z = kOut && p.z != nullptr;
  const int nx = kOut ? (has_z ? 3 : 2) : 2;
  const int ci = tid % kCPR, rb = tid / kCPR;
  const bool dvalid = d0 + (int64_t)ci * kVec < Dn;
  const int64_t row_bytes = Dn * kS;
  const char* xsrc[3] = {static_cast<const char*>(p.delta), static_cast<const char*>(p.u), static_cast<const char*>(p.z)};
  const int64_t x_off0 = ((b * L + t0 + rb) * Dn + d0 + (int64_t)ci * kVec) * kS;
  auto issue_x = [&](int tile, int stage) {
    const int64_t rows0 = (int64_t)tile * kScanTile + rb;
    const int64_t off = x_off0 + (int64_t)tile * kScanTile * row_bytes;
#pragma unroll
    for (int x = 0; x < kNX; x++) {
      if (x >= nx) break;
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
  auto load_bc = [&](int tile) {
    const int64_t e_row0 = (b * L + t0 + (int64_t)tile * kScanTile) * N;
    const int64_t rows_left = t1 - (t0 + (int64_t)tile * kScanTile);
    if constexpr (kVecBC) {
#pragma unroll
      for (int j = 0; j < kBCChunksPerThread; j++) {
        const int q = tid + j * kScanCh;
        const int which = q / (kScanTile * N / kVec);
        const int e = (q % (kScanTile * N / kVec)) * kVec;
        bcv[j] = make_uint4(0, 0, 0, 0);
        if (q < kBCChunks && e / N < rows_left && e_row0 + e + kVec <= bc_elems)
          bcv[j] = *reinterpret_cast<const uint4*>((which ? Cg : Bg) + e_row0 + e);
      }
    } else {
#pragma unroll
      for (int j = 0; j < kBCValsPerThread; j++) {
        const int i = tid + j * kScanCh;
        const int which = i / (kScanTile * N), e = i % (kScanTile * N);
        bcs[j] = 0.f;
        if (i < kBCVals && e / N < rows_left) bcs[j] = to_f32((which ? Cg : Bg)[e_row0 + e]);
      }
    }
  };
  auto store_bc = [&](int stage) {
    if constexpr (kVecBC) {
#pragma unroll
      for (int j = 0; j < kBCChunksPerThread; j++) {
        const int q = tid + j * kScanCh;
        if (q < kBCChunks) {
          const int which = q / (kScanTile * N / kVec);
          const int e = (q % (kScanTile * N / kVec)) * kVec;
          store_bc_chunk(&sBC[stage][which][0][0] + e, bcv[j], T());
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < kBCValsPerThread; j++) {
        const int i = tid + j * kScanCh;
        if (i < kBCVals) {
          const int which = i / (kScanTile * N), e = i % (kScanTile * N);
          sBC[stage][which][e / N][e % N] = bcs[j];
        }
      }
    }
  };
  if constexpr (NPAD != N) {
    for (int i = tid; i < 2 * kNBC * kScanTile; i += kScanCh) (&sBC[0][0][0][0])[i * NPAD + N] = 0.f;
  }
  float2 A2[NP], h[NP];
#pragma unroll
  for (int j = 0; j < NP; j++) {
    const float a0 = active ? p.A[d * N + 2 * j] * kLog2e : 0.f;
    const float a1 = (active && 2 * j + 1 < N) ? p.A[d * N + 2 * j + 1] * kLog2e : 0.f;
    A2[j] = make_float2(a0, a1);
    h[j] = make_float2(0.f, 0.f);
    if (!kSummary && active && p.initial_state) {  // the main pass starts from the given state
      const float* h0 = p.initial_state + (b * Dn + d) * N;
      h[j] = make_float2(h0[2 * j], 2 * j + 1 < N ? h0[2 * j + 1] : 0.f);
    }
  }
  const float Dd = (active && p.D) ? p.D[d] : 0.f;
  const float bias = (active && p.delta_bias) ? p.delta_bias[d] : 0.f;
  const bool sp = p.softplus != 0;
  if (ntiles > 0) { issue_x(0, 0); cp_async_commit(); load_bc(0); store_bc(0); }
  if (!kSummary && c > 0) wait_for_summaries();
  if (!kSummary && c > 0 && active) {
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
  float S = 0.f, S_comp = 0.f;
  T* __restrict__ yg = static_cast<T*>(p.y);
  // Causal conv1d window (kConv): x at t-1, t-2, t-3 and the 4-tap weights, tap j
  // multiplying x[t-3+j] (kernels shorter than 4 get leading zero taps).
  float cw[4] = {0.f, 0.f, 0.f, 0.f}, cb = 0.f, xw1 = 0.f, xw2 = 0.f, xw3 = 0.f;
  if constexpr (kConv) {
    if (active) {
      const int K = p.d_conv;
#pragma unroll
      for (int j = 0; j < 4; j++)
        if (j >= 4 - K) cw[j] = p.conv_w[d * K + j - (4 - K)];
      cb = p.conv_b ? p.conv_b[d] : 0.f;
      const T* xg = static_cast<const T*>(p.u);
      if (t0 >= 1) xw1 = to_f32(xg[(b * L + t0 - 1) * Dn + d]);
      if (t0 >= 2) xw2 = to_f32(xg[(b * L + t0 - 2) * Dn + d]);
      if (t0 >= 3) xw3 = to_f32(xg[(b * L + t0 - 3) * Dn + d]);
    }
  }
  auto step = [&](int stage, int k, T* yrow) {
    const float x = to_f32(sX[stage][0][k][tid]) + bias;
    const float dt = sp ? softplus(x) : x;
    float uu = to_f32(sX[stage][1][k][tid]);
    if constexpr (kConv) {
      const float xt = uu;
      uu = silu(fmaf(cw[3], xt, fmaf(cw[2], xw1, fmaf(cw[1], xw2, fmaf(cw[0], xw3, cb)))));
      xw3 = xw2; xw2 = xw1; xw1 = xt;
      // u_out has y's layout: the same flat element index as this step's y
      if (kOut && p.u_out) static_cast<T*>(p.u_out)[yrow - static_cast<T*>(p.y)] = from_f32<T>(uu);
    }
    const float w = dt * uu;
    if (kSummary) { const float yk = dt - S_comp; const float tk = S + yk; S_comp = (tk - S) - yk; S = tk; }
    const float2 dt2 = make_float2(dt, dt), w2 = make_float2(w, w);
    const float* Bk = sBC[stage][0][k];
    const float* Ck = sBC[stage][kNBC - 1][k];
    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < NP; j++) {
      float2 Bv, Cv;
      if constexpr (NPAD % 4 == 0) {
        const float4 b4 = *reinterpret_cast<const float4*>(Bk + 4 * (j / 2));
        Bv = (j & 1) ? make_float2(b4.z, b4.w) : make_float2(b4.x, b4.y);
        if (kOut) { const float4 c4 = *reinterpret_cast<const float4*>(Ck + 4 * (j / 2)); Cv = (j & 1) ? make_float2(c4.z, c4.w) : make_float2(c4.x, c4.y); }
      } else {
        Bv = *reinterpret_cast<const float2*>(Bk + 2 * j);
        if (kOut) Cv = *reinterpret_cast<const float2*>(Ck + 2 * j);
      }
      const float2 xa = __fmul2_rn(dt2, A2[j]);
      const float2 dA = make_float2(ex2(xa.x), ex2(xa.y));
      h[j] = __ffma2_rn(dA, h[j], __fmul2_rn(w2, Bv));
      if (kOut) { if (j & 1) acc1 = __ffma2_rn(Cv, h[j], acc1); else acc0 = __ffma2_rn(Cv, h[j], acc0); }
    }
    if (kOut) {
      const float2 a = __fadd2_rn(acc0, acc1);
      float yv = fmaf(Dd, uu, a.x + a.y);
      if (has_z) yv *= silu(to_f32(sX[stage][kNX - 1][k][tid]));
      *yrow = from_f32<T>(yv);
    }
  };
  // Two steps at once for full tiles: the per-step work that does not touch the state
  // (step size, input, skip term, gate) in packed fp32x2 arithmetic, then the recurrence for
  // step k and step k + 1 in order.
  auto step_pair = [&](int stage, int k, T* yrow) {
    const float2 x = __fadd2_rn(make_float2(to_f32(sX[stage][0][k][tid]), to_f32(sX[stage][0][k + 1][tid])),
                                make_float2(bias, bias));
    const float2 dt = sp ? softplus2(x) : x;
    float2 uu = make_float2(to_f32(sX[stage][1][k][tid]), to_f32(sX[stage][1][k + 1][tid]));
    if constexpr (kConv) {
      const float x0 = uu.x, x1 = uu.y;
      const float2 pre = make_float2(fmaf(cw[3], x0, fmaf(cw[2], xw1, fmaf(cw[1], xw2, fmaf(cw[0], xw3, cb)))),
                                     fmaf(cw[3], x1, fmaf(cw[2], x0, fmaf(cw[1], xw1, fmaf(cw[0], xw2, cb)))));
      uu = silu2(pre);
      xw3 = xw1; xw2 = x0; xw1 = x1;
      if (kOut && p.u_out) {
        T* uo = static_cast<T*>(p.u_out) + (yrow - static_cast<T*>(p.y));
        uo[0] = from_f32<T>(uu.x);
        uo[Dn] = from_f32<T>(uu.y);
      }
    }
    const float2 w = __fmul2_rn(dt, uu);
    float2 g = make_float2(1.f, 1.f), du = make_float2(0.f, 0.f);
    if (kOut) {
      du = __fmul2_rn(make_float2(Dd, Dd), uu);
      if (has_z) g = silu2(make_float2(to_f32(sX[stage][kNX - 1][k][tid]), to_f32(sX[stage][kNX - 1][k + 1][tid])));
    }
#pragma unroll
    for (int e = 0; e < 2; e++) {
      const float dte = e ? dt.y : dt.x, we = e ? w.y : w.x;
      if (kSummary) { const float yk = dte - S_comp; const float tk = S + yk; S_comp = (tk - S) - yk; S = tk; }
      const float2 dt2 = make_float2(dte, dte), w2 = make_float2(we, we);
      const float* Bk = sBC[stage][0][k + e];
      const float* Ck = sBC[stage][kNBC - 1][k + e];
      float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
      for (int j = 0; j < NP; j++) {
        float2 Bv, Cv;
        if constexpr (NPAD % 4 == 0) {
          const float4 b4 = *reinterpret_cast<const float4*>(Bk + 4 * (j / 2));
          Bv = (j & 1) ? make_float2(b4.z, b4.w) : make_float2(b4.x, b4.y);
          if (kOut) { const float4 c4 = *reinterpret_cast<const float4*>(Ck + 4 * (j / 2)); Cv = (j & 1) ? make_float2(c4.z, c4.w) : make_float2(c4.x, c4.y); }
        } else {
          Bv = *reinterpret_cast<const float2*>(Bk + 2 * j);
          if (kOut) Cv = *reinterpret_cast<const float2*>(Ck + 2 * j);
        }
        const float2 xa = __fmul2_rn(dt2, A2[j]);
        const float2 dA = make_float2(ex2(xa.x), ex2(xa.y));
        h[j] = __ffma2_rn(dA, h[j], __fmul2_rn(w2, Bv));
        if (kOut) { if (j & 1) acc1 = __ffma2_rn(Cv, h[j], acc1); else acc0 = __ffma2_rn(Cv, h[j], acc0); }
      }
      if (kOut) {
        const float2 a = __fadd2_rn(acc0, acc1);
        const float yv = ((e ? du.y : du.x) + (a.x + a.y)) * (e ? g.y : g.x);
        yrow[e * Dn] = from_f32<T>(yv);
      }
    }
  };
  for (int tile = 0; tile < ntiles; tile++) {
    const int stage = tile & 1;
    if (tile + 1 < ntiles) { issue_x(tile + 1, stage ^ 1); load_bc(tile + 1); }
    cp_async_commit();
    cp_async_wait_prev();
    __syncthreads();
    const int64_t ts = t0 + (int64_t)tile * kScanTile;
    T* yrow = kOut ? yg + (b * L + ts) * Dn + d : nullptr;
    if constexpr (kCkpt) {  // the state before this tile (chunks start on tile boundaries)
      if (active) {
        float* ck = p.ckpt_h + ((b * ((L + kScanTile - 1) / kScanTile) + ts / kScanTile) * Dn + d) * N;
        if constexpr (N % 4 == 0) {  // whole 16-byte pieces (a channel's row is 16-byte aligned)
#pragma unroll
          for (int j = 0; j < NP; j += 2)
            *reinterpret_cast<float4*>(ck + 2 * j) = make_float4(h[j].x, h[j].y, h[j + 1].x, h[j + 1].y);
        } else {
#pragma unroll
          for (int j = 0; j < NP; j++) { ck[2 * j] = h[j].x; if (2 * j + 1 < N) ck[2 * j + 1] = h[j].y; }
        }
      }
    }
    if (active) {
      if (ts + kScanTile <= t1) {
#pragma unroll
        for (int k = 0; k < kScanTile; k += 2) step_pair(stage, k, yrow + k * Dn);
      } else {
        const int steps = (int)(t1 - ts);
        for (int k = 0; k < steps; k++) step(stage, k, yrow + k * Dn);
      }
    }
    __syncthreads();
    if (tile + 1 < ntiles) store_bc(stage ^ 1);
  }
  if (!active) return;
  if (kSummary) {
    const int64_t slot = (b * (p.n_chunks - 1) + c) * Dn + d;
    p.ws_S[slot] = S;
#pragma unroll
    for (int j = 0; j < NP; j++) { p.ws_h[slot * N + 2 * j] = h[j].x; if (2 * j + 1 < N) p.ws_h[slot * N + 2 * j + 1] = h[j].y; }
    allow_main_pass();
  } else if (kOut && c == p.n_chunks - 1 && p.last_state) {
    float* ls = p.last_state + (b * Dn + d) * N;
#pragma unroll
    for (int j = 0; j < NP; j++) { ls[2 * j] = h[j].x; if (2 * j + 1 < N) ls[2 * j + 1] = h[j].y; }
  }
}


// One CTA: kScanCh consecutive channels of one batch row over one time chunk.
// Lanes 2c and 2c+1 of a warp share channel c: each owns half of its states,
// and the per-step work that does not involve the state (step size, input,
// skip term, gate, output) is split between them by step parity and exchanged
// with one shuffle per value.  kSummary: the CTA writes the chunk's (sum of
// delta, end state from zero) instead of y.
//
// Data movement per tile of kScanTile steps: delta, u (and z) arrive in shared
// memory by cp.async (16-byte pieces, coalesced along d_inner) one tile ahead
// of use; the next tile's B/C rows are fetched into registers while the current
// tile is computed and converted to fp32 in shared memory.  So no step waits on
// HBM latency.  State pairs are updated with packed fp32x2 instructions.
template <int N, typename T, bool kSummary, bool kConv>
__global__ void __launch_bounds__(kScanThreads)
scan_chunk_kernel_2lane(const ScanParams p) {
  using SS = StateSplit<N>;
  constexpr int kHalf = SS::kHalf, NPAD = SS::kPad, kPairs = SS::kPairs;
  constexpr int kS = sizeof(T);
  constexpr int kVec = 16 / kS;                       // elements per 16-byte copy
  constexpr int kRow = kScanCh + (kS == 4 ? 16 : 0);  // fp32 rows padded: no bank conflict
  constexpr int kCPR = kScanCh / kVec;                // copies per activation row
  constexpr int kRowsPerPass = kScanThreads / kCPR;
  constexpr int kPasses = kScanTile / kRowsPerPass;
  constexpr int kNX = kSummary ? 2 : 3;               // delta, u (, z)
  constexpr int kNBC = kSummary ? 1 : 2;              // B (, C)
  constexpr int kHalfSteps = kScanTile / 2;
  // B/C rows move as 16-byte vectors when a row is a whole number of them and unpadded.
  constexpr bool kVecBC = (N * kS) % 16 == 0 && NPAD == N;
  constexpr int kBCChunks = kNBC * kScanTile * N / kVec;
  constexpr int kBCChunksPerThread = kVecBC ? (kBCChunks + kScanThreads - 1) / kScanThreads : 1;
  constexpr int kBCVals = kNBC * kScanTile * N;
  constexpr int kBCValsPerThread = kVecBC ? 1 : (kBCVals + kScanThreads - 1) / kScanThreads;
  static_assert(kScanTile % kRowsPerPass == 0 && kPasses >= 1, "tile rows must split evenly");
  __shared__ __align__(16) T sX[2][kNX][kScanTile][kRow];
  __shared__ __align__(16) float sBC[2][kNBC][kScanTile][NPAD];

  const int64_t n_dtiles = (p.d_inner + kScanCh - 1) / kScanCh;
  const int chunks = kSummary ? p.n_chunks - 1 : p.n_chunks;
  int64_t blk = blockIdx.x;
  const int64_t dtile = blk % n_dtiles;
  blk /= n_dtiles;
  const int c = (int)(blk % chunks);
  const int64_t b = blk / chunks;
  const int tid = threadIdx.x;
  const int cl = ((tid >> 5) << 4) | ((tid & 31) >> 1);  // channel within the CTA
  const int par = tid & 1;                                // this lane's half / step parity
  const int64_t Dn = p.d_inner, L = p.L;
  const int64_t d0 = dtile * kScanCh;
  const int64_t d = d0 + cl;
  const bool active = d < Dn;
  const int64_t t0 = (int64_t)c * p.chunk_len;
  const int64_t t1 = min(t0 + p.chunk_len, L);
  const int ntiles = (int)((t1 - t0 + kScanTile - 1) / kScanTile);

  const T* __restrict__ Bg = static_cast<const T*>(p.B);
  const T* __restrict__ Cg = static_cast<const T*>(p.C);
  const bool has_z = !kSummary && p.z != nullptr;
  const int nx = kSummary ? 2 : (has_z ? 3 : 2);

  // Activation copies: thread moves 16-byte piece ci of rows rb, rb + kRowsPerPass, ...
  const int ci = tid % kCPR, rb = tid / kCPR;
  const bool dvalid = d0 + (int64_t)ci * kVec < Dn;
  const int64_t row_bytes = Dn * kS;
  const char* xsrc[3] = {static_cast<const char*>(p.delta), static_cast<const char*>(p.u),
                         static_cast<const char*>(p.z)};
  const int64_t x_off0 = ((b * L + t0 + rb) * Dn + d0 + (int64_t)ci * kVec) * kS;
  auto issue_x = [&](int tile, int stage) {
    const int64_t rows0 = (int64_t)tile * kScanTile + rb;
    const int64_t off = x_off0 + (int64_t)tile * kScanTile * row_bytes;
#pragma unroll
    for (int x = 0; x < kNX; x++) {
      if (x >= nx) break;
#pragma unroll
      for (int m = 0; m < kPasses; m++) {
        const bool valid = dvalid && t0 + rows0 + m * kRowsPerPass < t1;
        const char* g = xsrc[x] + off + (int64_t)m * kRowsPerPass * row_bytes;
        cp_async16(&sX[stage][x][rb + m * kRowsPerPass][ci * kVec], valid ? g : xsrc[x], valid);
      }
    }
  };

  // B/C rows of a tile: global -> registers (a tile ahead) -> fp32 shared memory.
  uint4 bcv[kBCChunksPerThread];
  float bcs[kBCValsPerThread];
  const int64_t bc_elems = p.batch * L * N;
  auto load_bc = [&](int tile) {
    const int64_t e_row0 = (b * L + t0 + (int64_t)tile * kScanTile) * N;
    const int64_t rows_left = t1 - (t0 + (int64_t)tile * kScanTile);
    if constexpr (kVecBC) {
#pragma unroll
      for (int j = 0; j < kBCChunksPerThread; j++) {
        const int q = tid + j * kScanThreads;
        const int which = q / (kScanTile * N / kVec);
        const int e = (q % (kScanTile * N / kVec)) * kVec;  // element within the tile
        bcv[j] = make_uint4(0, 0, 0, 0);
        if (q < kBCChunks && e / N < rows_left && e_row0 + e + kVec <= bc_elems)
          bcv[j] = *reinterpret_cast<const uint4*>((which ? Cg : Bg) + e_row0 + e);
      }
    } else {
#pragma unroll
      for (int j = 0; j < kBCValsPerThread; j++) {
        const int i = tid + j * kScanThreads;
        const int which = i / (kScanTile * N), e = i % (kScanTile * N);
        bcs[j] = 0.f;
        if (i < kBCVals && e / N < rows_left) bcs[j] = to_f32((which ? Cg : Bg)[e_row0 + e]);
      }
    }
  };
  auto store_bc = [&](int stage) {
    if constexpr (kVecBC) {
#pragma unroll
      for (int j = 0; j < kBCChunksPerThread; j++) {
        const int q = tid + j * kScanThreads;
        if (q < kBCChunks) {
          const int which = q / (kScanTile * N / kVec);
          const int e = (q % (kScanTile * N / kVec)) * kVec;
          store_bc_chunk(&sBC[stage][which][0][0] + e, bcv[j], T());
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < kBCValsPerThread; j++) {
        const int i = tid + j * kScanThreads;
        if (i < kBCVals) {
          const int which = i / (kScanTile * N), e = i % (kScanTile * N);
          sBC[stage][which][e / N][e % N] = bcs[j];
        }
      }
    }
  };

  if constexpr (NPAD != N) {
    // padding states read B = C = 0 from columns that are never overwritten
    for (int i = tid; i < 2 * kNBC * kScanTile * (NPAD - N); i += kScanThreads)
      (&sBC[0][0][0][0])[(i / (NPAD - N)) * NPAD + N + i % (NPAD - N)] = 0.f;
  }

  // This lane's states: par * kHalf + 2j, +1 (j < kPairs).
  const int n0 = par * kHalf;
  float2 A2[kPairs], h[kPairs];
#pragma unroll
  for (int j = 0; j < kPairs; j++) {
    const int na = n0 + 2 * j, nb = na + 1;
    const float a0 = (active && na < N) ? p.A[d * N + na] * kLog2e : 0.f;  // e^x = 2^(x log2 e)
    const float a1 = (active && nb < N) ? p.A[d * N + nb] * kLog2e : 0.f;
    A2[j] = make_float2(a0, a1);
    h[j] = make_float2(0.f, 0.f);
    if (!kSummary && active && p.initial_state) {  // the main pass starts from the given state
      const float* h0 = p.initial_state + (b * Dn + d) * N;
      h[j] = make_float2(na < N ? h0[na] : 0.f, nb < N ? h0[nb] : 0.f);
    }
  }
  const float Dd = (active && p.D) ? p.D[d] : 0.f;
  const float bias = (active && p.delta_bias) ? p.delta_bias[d] : 0.f;
  const bool sp = p.softplus != 0;
  // Causal conv1d window (kConv): the 4-tap weights (tap j multiplies x[t-3+j]; shorter
  // kernels get leading zero taps) and x at the three steps before the current tile.
  float cw[4] = {0.f, 0.f, 0.f, 0.f}, cb = 0.f, xh1 = 0.f, xh2 = 0.f, xh3 = 0.f;
  if constexpr (kConv) {
    if (active) {
      const int K = p.d_conv;
#pragma unroll
      for (int j = 0; j < 4; j++)
        if (j >= 4 - K) cw[j] = p.conv_w[d * K + j - (4 - K)];
      cb = p.conv_b ? p.conv_b[d] : 0.f;
      const T* xg = static_cast<const T*>(p.u);
      if (t0 >= 1) xh1 = to_f32(xg[(b * L + t0 - 1) * Dn + d]);
      if (t0 >= 2) xh2 = to_f32(xg[(b * L + t0 - 2) * Dn + d]);
      if (t0 >= 3) xh3 = to_f32(xg[(b * L + t0 - 3) * Dn + d]);
    }
  }

  if (ntiles > 0) {
    issue_x(0, 0);
    cp_async_commit();
    load_bc(0);
    store_bc(0);
  }

  if (!kSummary && c > 0) wait_for_summaries();
  if (!kSummary && c > 0 && active) {
    // Start state of chunk c: fold the summaries of chunks 0 .. c-1 in order.
    const int64_t base = b * (p.n_chunks - 1);
    for (int j = 0; j < c; j++) {
      const float S = p.ws_S[(base + j) * Dn + d];
      const float* hj = p.ws_h + ((base + j) * Dn + d) * N;
#pragma unroll
      for (int q = 0; q < kPairs; q++) {
        const int na = n0 + 2 * q, nb = na + 1;
        h[q].x = fmaf(ex2(A2[q].x * S), h[q].x, na < N ? hj[na] : 0.f);
        h[q].y = fmaf(ex2(A2[q].y * S), h[q].y, nb < N ? hj[nb] : 0.f);
      }
    }
  }

  float S = 0.f, S_comp = 0.f;  // compensated (Kahan) sum of delta over the chunk
  T* __restrict__ yg = static_cast<T*>(p.y);

  for (int tile = 0; tile < ntiles; tile++) {
    const int stage = tile & 1;
    if (tile + 1 < ntiles) {
      issue_x(tile + 1, stage ^ 1);
      load_bc(tile + 1);
    }
    cp_async_commit();
    cp_async_wait_prev();  // this tile's copies have landed (only the newest group may pend)
    __syncthreads();
    const int64_t ts = t0 + (int64_t)tile * kScanTile;
    const int steps = (int)min((int64_t)kScanTile, t1 - ts);

    // (1) Own steps k = 2i + par: step size, input, skip term, gate (packed over i, i+1).
    float odt[kHalfSteps], ow[kHalfSteps], odu[kHalfSteps], og[kHalfSteps];
#pragma unroll
    for (int i = 0; i < kHalfSteps; i += 2) {
      const int k0 = 2 * i + par, k1 = k0 + 2;
      const float2 x = __fadd2_rn(make_float2(to_f32(sX[stage][0][k0][cl]), to_f32(sX[stage][0][k1][cl])),
                                  make_float2(bias, bias));
      const float2 dt = sp ? softplus2(x) : x;
      float2 uu = make_float2(to_f32(sX[stage][1][k0][cl]), to_f32(sX[stage][1][k1][cl]));
      if constexpr (kConv) {
        // x before the tile comes from the window carried in registers
        auto xv = [&](int k) -> float {
          return k >= 0 ? to_f32(sX[stage][1][k][cl]) : (k == -1 ? xh1 : (k == -2 ? xh2 : xh3));
        };
        const float2 pre = make_float2(
            fmaf(cw[3], uu.x, fmaf(cw[2], xv(k0 - 1), fmaf(cw[1], xv(k0 - 2), fmaf(cw[0], xv(k0 - 3), cb)))),
            fmaf(cw[3], uu.y, fmaf(cw[2], xv(k1 - 1), fmaf(cw[1], xv(k1 - 2), fmaf(cw[0], xv(k1 - 3), cb)))));
        uu = silu2(pre);
        if (!kSummary && p.u_out && active) {
          T* uo = static_cast<T*>(p.u_out) + (b * L + ts) * Dn + d;
          if (k0 < steps) uo[(int64_t)k0 * Dn] = from_f32<T>(uu.x);
          if (k1 < steps) uo[(int64_t)k1 * Dn] = from_f32<T>(uu.y);
        }
      }
      const float2 w = __fmul2_rn(dt, uu);
      odt[i] = dt.x; odt[i + 1] = dt.y;
      ow[i] = w.x; ow[i + 1] = w.y;
      if (!kSummary) {
        const float2 du = __fmul2_rn(make_float2(Dd, Dd), uu);
        odu[i] = du.x; odu[i + 1] = du.y;
        if (has_z) {
          const float2 g = silu2(make_float2(to_f32(sX[stage][kNX - 1][k0][cl]),
                                             to_f32(sX[stage][kNX - 1][k1][cl])));
          og[i] = g.x; og[i + 1] = g.y;
        }
      }
    }

    // (2) The recurrence over every step of the tile on this lane's states.  Full tiles take
    // the unguarded copy (straight-line code the scheduler can overlap across steps).
    float part[kScanTile];
    auto recur_tile = [&](auto guarded) {
      constexpr bool kGuard = decltype(guarded)::value;
#pragma unroll
      for (int i = 0; i < kHalfSteps; i++) {
        const float rdt = shfl_pair(odt[i]), rw = shfl_pair(ow[i]);
#pragma unroll
        for (int e = 0; e < 2; e++) {
          const int k = 2 * i + e;
          const bool mine = (e == par);
          const float dt = mine ? odt[i] : rdt;
          const float w = mine ? ow[i] : rw;
          if (!kGuard || k < steps) {
            if (kSummary) {
              const float yk = dt - S_comp;
              const float tk = S + yk;
              S_comp = (tk - S) - yk;
              S = tk;
            }
            const float2 dt2 = make_float2(dt, dt), w2 = make_float2(w, w);
            const float* Bk = &sBC[stage][0][k][n0];
            const float* Ck = &sBC[stage][kNBC - 1][k][n0];
            float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < kPairs; j++) {
              float2 Bv, Cv;
              if constexpr (kHalf % 4 == 0) {
                const float4 b4 = *reinterpret_cast<const float4*>(Bk + 4 * (j / 2));
                Bv = (j & 1) ? make_float2(b4.z, b4.w) : make_float2(b4.x, b4.y);
                if (!kSummary) {
                  const float4 c4 = *reinterpret_cast<const float4*>(Ck + 4 * (j / 2));
                  Cv = (j & 1) ? make_float2(c4.z, c4.w) : make_float2(c4.x, c4.y);
                }
              } else {
                Bv = *reinterpret_cast<const float2*>(Bk + 2 * j);
                if (!kSummary) Cv = *reinterpret_cast<const float2*>(Ck + 2 * j);
              }
              const float2 xa = __fmul2_rn(dt2, A2[j]);
              const float2 dA = make_float2(ex2(xa.x), ex2(xa.y));
              h[j] = __ffma2_rn(dA, h[j], __fmul2_rn(w2, Bv));
              if (!kSummary) {
                if (j & 1) acc1 = __ffma2_rn(Cv, h[j], acc1);
                else acc0 = __ffma2_rn(Cv, h[j], acc0);
              }
            }
            if (!kSummary) {
              const float2 a = __fadd2_rn(acc0, acc1);
              part[k] = a.x + a.y;
            }
          } else if (!kSummary) {
            part[k] = 0.f;
          }
        }
      }
    };
    if (steps == kScanTile) recur_tile(std::false_type{});
    else recur_tile(std::true_type{});

    // (3) Own output steps: add the partner lane's half of C.h, skip term and gate.
    if (!kSummary) {
      T* yrow = yg + (b * L + ts + par) * Dn + d;
#pragma unroll
      for (int i = 0; i < kHalfSteps; i++) {
        const float give = par ? part[2 * i] : part[2 * i + 1];
        const float keep = par ? part[2 * i + 1] : part[2 * i];
        float v = keep + shfl_pair(give) + odu[i];
        if (has_z) v *= og[i];
        if (active && 2 * i + par < steps) yrow[(int64_t)2 * i * Dn] = from_f32<T>(v);
      }
    }
    if constexpr (kConv) {  // the window for the next tile: this tile's last three inputs
      xh1 = to_f32(sX[stage][1][kScanTile - 1][cl]);
      xh2 = to_f32(sX[stage][1][kScanTile - 2][cl]);
      xh3 = to_f32(sX[stage][1][kScanTile - 3][cl]);
    }
    __syncthreads();  // stage is free for the tile after next
    if (tile + 1 < ntiles) store_bc(stage ^ 1);
  }

  if (!active) return;
  if (kSummary) {
    const int64_t slot = (b * (p.n_chunks - 1) + c) * Dn + d;
    if (par == 0) p.ws_S[slot] = S;
#pragma unroll
    for (int j = 0; j < kPairs; j++) {
      const int na = n0 + 2 * j, nb = na + 1;
      if (na < N) p.ws_h[slot * N + na] = h[j].x;
      if (nb < N) p.ws_h[slot * N + nb] = h[j].y;
    }
    allow_main_pass();
  } else if (c == p.n_chunks - 1 && p.last_state) {
    float* ls = p.last_state + (b * Dn + d) * N;
#pragma unroll
    for (int j = 0; j < kPairs; j++) {
      const int na = n0 + 2 * j, nb = na + 1;
      if (na < N) ls[na] = h[j].x;
      if (nb < N) ls[nb] = h[j].y;
    }
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
  // Kernel choice: two lanes per channel doubles the warps for short sequences over few
  // channels; long sequences get their parallelism from time chunks instead.
  const int64_t channels = batch * d_inner;
  int lanes = (L <= 16384 && channels < (int64_t)sms * 128) ? 2 : 1;
  lanes = (int)env_int("SSM_SCAN_LANES", lanes) == 2 ? 2 : 1;
  // Time chunks: none when the channels alone give each SM >= 8 warps; otherwise, since
  // chunking costs a summary pass over all but the last chunk whatever their number,
  // cut enough chunks for ~32 warps per SM (at least 64 steps per chunk).
  const int64_t threads = channels * lanes;
  const int64_t full = (int64_t)sms * env_int("SSM_SCAN_THREADS_PER_SM", 1024);
  int64_t G = 1;
  if (threads > 0 && threads < (int64_t)sms * 256) G = (full + threads - 1) / threads;
  G = env_int("SSM_SCAN_CHUNKS", G);  // tuning override
  G = std::min<int64_t>(G, std::max<int64_t>(1, L / 64));
  G = std::min<int64_t>(G, 4096);
  int64_t len = L > 0 ? (L + G - 1) / G : 1;
  len = (len + kChunkAlign - 1) / kChunkAlign * kChunkAlign;
  plan->lanes = lanes;
  plan->chunk_len = len;
  plan->n_chunks = L > 0 ? (int)((L + len - 1) / len) : 1;
}

// Summary pass (if there are several chunks), then the main pass; the main pass is a
// programmatic dependent launch so that it can start while the summary pass drains.
static cudaError_t launch_passes(void (*summary)(const ScanParams), void (*main_pass)(const ScanParams),
                                 const ScanParams& p, int threads, int64_t sblocks, int64_t mblocks,
                                 cudaStream_t stream) {
  if (p.n_chunks <= 1) {
    main_pass<<<(unsigned)mblocks, threads, 0, stream>>>(p);
    return cudaGetLastError();
  }
  summary<<<(unsigned)sblocks, threads, 0, stream>>>(p);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)mblocks);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, main_pass, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int N, typename T>
static cudaError_t launch_scan_t(const ScanParams& p, cudaStream_t stream) {
  const int64_t n_dtiles = (p.d_inner + kScanCh - 1) / kScanCh;
  const int64_t sblocks = n_dtiles * (p.n_chunks - 1) * p.batch;
  const int64_t mblocks = n_dtiles * p.n_chunks * p.batch;
  if (p.conv_w != nullptr) {  // conv1d + SiLU in front
    if (p.lanes == 2)
      return launch_passes(scan_chunk_kernel_2lane<N, T, true, true>,
                           scan_chunk_kernel_2lane<N, T, false, true>, p, kScanThreads, sblocks,
                           mblocks, stream);
    return launch_passes(scan_chunk_kernel_1lane<N, T, true, true, false>,
                         scan_chunk_kernel_1lane<N, T, false, true, false>, p, kScanCh, sblocks, mblocks,
                         stream);
  } else if (p.lanes == 2) {
    return launch_passes(scan_chunk_kernel_2lane<N, T, true, false>,
                         scan_chunk_kernel_2lane<N, T, false, false>, p, kScanThreads, sblocks,
                         mblocks, stream);
  }
  return launch_passes(scan_chunk_kernel_1lane<N, T, true, false, false>,
                       scan_chunk_kernel_1lane<N, T, false, false, false>, p, kScanCh, sblocks, mblocks,
                       stream);
}

template <typename T>
static cudaError_t dispatch_n(const ScanParams& p, cudaStream_t s) {
  switch (p.d_state) {
    case 1: return launch_scan_t<1, T>(p, s);
    case 2: return launch_scan_t<2, T>(p, s);
    case 3: return launch_scan_t<3, T>(p, s);
    case 4: return launch_scan_t<4, T>(p, s);
    case 5: return launch_scan_t<5, T>(p, s);
    case 6: return launch_scan_t<6, T>(p, s);
    case 7: return launch_scan_t<7, T>(p, s);
    case 8: return launch_scan_t<8, T>(p, s);
    case 9: return launch_scan_t<9, T>(p, s);
    case 10: return launch_scan_t<10, T>(p, s);
    case 11: return launch_scan_t<11, T>(p, s);
    case 12: return launch_scan_t<12, T>(p, s);
    case 13: return launch_scan_t<13, T>(p, s);
    case 14: return launch_scan_t<14, T>(p, s);
    case 15: return launch_scan_t<15, T>(p, s);
    case 16: return launch_scan_t<16, T>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
static cudaError_t summary_only(const ScanParams& p, cudaStream_t s) {
  const int64_t blocks = (p.d_inner + kScanCh - 1) / kScanCh * (p.n_chunks - 1) * p.batch;
  switch (p.d_state) {
#define SSM_SUMMARY_CASE(NN) \
    case NN: scan_chunk_kernel_1lane<NN, T, true, false, false><<<(unsigned)blocks, kScanCh, 0, s>>>(p); break;
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
    case NN: scan_chunk_kernel_1lane<NN, T, false, false, true><<<(unsigned)blocks, kScanCh, 0, s>>>(p); break;
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

cudaError_t launch_scan(const ScanParams& p, bool bf16, cudaStream_t stream) {
  return bf16 ? dispatch_n<__nv_bfloat16>(p, stream) : dispatch_n<float>(p, stream);
}

}  // namespace ssm
