// Backward pass of the selective scan: gradients with respect to u, delta_raw, A, B, C, D, z,
// delta_bias and the initial state, given dL/dy and (optionally) dL/dlast_state.
//
// The pages describe the backward only as "recompute the intermediate states in the backward
// pass instead of storing them" (youngju.dev, "Mamba: Linear-Time Sequence Modeling with
// Selective State Spaces 论文分析", section "解决方案：Kernel Fusion + Recomputation").  Here:
//  1. forward checkpoints: the forward scan's own kernels (its summary pass, then its
//     one-lane kernel in checkpoint mode) store the state before every 16-step tile — one
//     state per 16 steps, never the per-step states;
//  2. reverse summaries: the adjoint lambda_t = ds_t C_t + dA_{t+1} lambda_{t+1} runs
//     backwards in time with the same chunk decomposition; per chunk, its carry-out from a
//     zero carry-in and its decay exp(A sum delta);
//  3. gradients: one CTA per (batch row, time chunk, 32 or 16 channels) starts from the
//     adjoint carry entering its chunk from the right (dL/dlast_state folded with the
//     summaries of the later chunks) and walks the chunk's tiles backwards: per tile it
//     recomputes the 16 states into shared memory from the tile's checkpoint, then carries
//     the adjoint through the tile while forming every gradient.  dB and dC sum over
//     channels (a warp reduction, then one atomic add per lane).
// All arithmetic is fp32; one thread per (batch, channel), all d_state states in registers.

#include "ssm_device.cuh"
#include "ssm_internal.h"

#include <algorithm>

namespace ssm {

constexpr int kBwdCh = 32;    // channels per CTA (one warp)
constexpr int kBwdTile = 16;  // time steps per tile

template <typename T>
__device__ __forceinline__ float ldf(const void* p, int64_t i) {
  return to_f32(static_cast<const T*>(p)[i]);
}

// Step sizes of a tile, two at a time in packed fp32x2: dt_k = softplus(x_k + bias) (or
// x_k + bias without softplus).
__device__ __forceinline__ void tile_step_sizes(const float (&x)[kBwdTile], float bias, bool sp,
                                                float (&dt)[kBwdTile]) {
#pragma unroll
  for (int k = 0; k < kBwdTile; k += 2) {
    const float2 v = __fadd2_rn(make_float2(x[k], x[k + 1]), make_float2(bias, bias));
    const float2 d = sp ? softplus2(v) : v;
    dt[k] = d.x;
    dt[k + 1] = d.y;
  }
}

// ---------------------------------------------------------------------------------------
// 2. Reverse summaries.  Walking a chunk backwards from carry m (entering its last step):
//      lambda_t = m + ds_t C_t,   m <- dA_t lambda_t   (carry to step t - 1),
//    with ds_t = dy_t silu(z_t): from m = 0, store (sum delta, m after the chunk's first
//    step) for chunks >= 1.
template <int N, typename T>
__global__ void __launch_bounds__(kBwdCh) bwd_reverse_summary_kernel(const BwdArgs p) {
  constexpr bool kSummary = true;
  constexpr int NP = (N + 1) / 2;
  const int64_t n_dtiles = (p.d_inner + kBwdCh - 1) / kBwdCh;
  const int chunks = kSummary ? p.n_chunks - 1 : p.n_chunks;
  int64_t blk = blockIdx.x;
  const int64_t dtile = blk % n_dtiles;
  blk /= n_dtiles;
  const int c = (int)(blk % chunks) + (kSummary ? 1 : 0);
  const int64_t b = blk / chunks;
  const int lane = threadIdx.x;
  const int64_t Dn = p.d_inner, L = p.L, d = dtile * kBwdCh + lane;
  const bool active = d < Dn;
  const int64_t dc = active ? d : 0;
  const int64_t t0 = (int64_t)c * p.chunk_len, t1 = min(t0 + p.chunk_len, L);
  __shared__ __align__(16) float sC[kBwdTile][2 * NP];

  float2 A2[NP], m[NP];
#pragma unroll
  for (int j = 0; j < NP; j++) {
    const int n0 = 2 * j, n1 = n0 + 1;
    A2[j] = make_float2(p.A[dc * N + n0] * kLog2e, n1 < N ? p.A[dc * N + n1] * kLog2e : 0.f);
    m[j] = make_float2(0.f, 0.f);
  }
  if (2 * NP != N)
    for (int i = lane; i < kBwdTile; i += kBwdCh) sC[i][N] = 0.f;
  const float bias = p.delta_bias ? p.delta_bias[dc] : 0.f;
  float S = 0.f, S_comp = 0.f;
  const int64_t first_tile = t0 / kBwdTile, last_tile = (t1 - 1) / kBwdTile;
  // per tile: delta_raw, dy, z in registers, loaded at once, next tile prefetched
  float xr[kBwdTile], dr[kBwdTile], zr[kBwdTile];
  auto load_tile = [&](int64_t tl, float* xa, float* da, float* za) {
    const int64_t ts = tl * kBwdTile;
    const int steps = (int)min((int64_t)kBwdTile, t1 - ts);
#pragma unroll
    for (int k = 0; k < kBwdTile; k++) {
      const int64_t e = (b * L + ts + min(k, steps - 1)) * Dn + dc;
      xa[k] = ldf<T>(p.delta, e);
      da[k] = ldf<T>(p.dy, e);
      za[k] = p.z ? ldf<T>(p.z, e) : 0.f;
    }
  };
  if (t0 < t1) load_tile(last_tile, xr, dr, zr);
  for (int64_t tl = last_tile; tl >= first_tile; tl--) {
    const int64_t ts = tl * kBwdTile;
    const int steps = (int)min((int64_t)kBwdTile, t1 - ts);
    float xn[kBwdTile], dn[kBwdTile], zn[kBwdTile];
    const bool more = tl > first_tile;
    if (more) load_tile(tl - 1, xn, dn, zn);
    __syncwarp();
    for (int i = lane; i < steps * N; i += kBwdCh) sC[i / N][i % N] = ldf<T>(p.C, (b * L + ts) * N + i);
    __syncwarp();
    float dts[kBwdTile];
    tile_step_sizes(xr, bias, p.softplus != 0, dts);
#pragma unroll
    for (int k = kBwdTile - 1; k >= 0; k--) {
      if (k < steps) {
        const float dt = dts[k];
        if (kSummary) {
          const float yk = dt - S_comp;
          const float tk = S + yk;
          S_comp = (tk - S) - yk;
          S = tk;
        }
        const float ds = p.z ? dr[k] * silu(zr[k]) : dr[k];
        const float2 dt2 = make_float2(dt, dt), ds2 = make_float2(ds, ds);
#pragma unroll
        for (int j = 0; j < NP; j++) {
          const float2 xa = __fmul2_rn(dt2, A2[j]);
          m[j] = __fmul2_rn(make_float2(ex2(xa.x), ex2(xa.y)),
                            __ffma2_rn(ds2, *reinterpret_cast<const float2*>(&sC[k][2 * j]), m[j]));
        }
      }
    }
    __syncwarp();
    if (more) {
#pragma unroll
      for (int k = 0; k < kBwdTile; k++) { xr[k] = xn[k]; dr[k] = dn[k]; zr[k] = zn[k]; }
    }
  }
  if (kSummary && active) {
    const int64_t slot = (b * p.n_chunks + c) * Dn + d;
    p.rws_S[slot] = S;
#pragma unroll
    for (int j = 0; j < NP; j++) {
      p.rws_m[slot * N + 2 * j] = m[j].x;
      if (2 * j + 1 < N) p.rws_m[slot * N + 2 * j + 1] = m[j].y;
    }
  }
}

// ---------------------------------------------------------------------------------------
// 3. Gradients for one tile.  Lane = channel; the 2N per-step partials of dB (lambda dt u) and
//    dC (ds h) are summed over the 32 channels by a reduce-scatter: after five halving
//    exchanges lane j holds the warp's total of value j, and adds it to global memory.
template <int N>
__device__ __forceinline__ void warp_reduce_scatter_add(float (&v)[32], int lane, float* dB_row,
                                                        float* dC_row) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int j = 0; j < o; j++) {
      const float send = upper ? v[j] : v[j + o];
      const float keep = upper ? v[j + o] : v[j];
      v[j] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, o);
    }
  }
  if (lane < N) atomicAdd(dB_row + lane, v[0]);
  else if (lane < 2 * N) atomicAdd(dC_row + lane - N, v[0]);
}

// The adjoint carry entering chunk c from the right for states nb + 2j, nb + 2j + 1 (j < NP):
// dL/dlast_state (or zero) folded with the reverse summaries of chunks n_chunks - 1 .. c + 1.
template <int N, int NP>
__device__ __forceinline__ void chunk_carry_in(const BwdArgs& p, int64_t b, int64_t dc, int c, int nb,
                                               const float2 (&A2)[NP], float2 (&m)[NP]) {
  const int64_t Dn = p.d_inner;
#pragma unroll
  for (int j = 0; j < NP; j++) m[j] = make_float2(0.f, 0.f);
  if (p.dlast) {
    const float* dl = p.dlast + (b * Dn + dc) * N + nb;
#pragma unroll
    for (int j = 0; j < NP; j++) m[j] = make_float2(dl[2 * j], nb + 2 * j + 1 < N ? dl[2 * j + 1] : 0.f);
  }
  for (int jc = p.n_chunks - 1; jc > c; jc--) {
    const int64_t slot = (b * p.n_chunks + jc) * Dn + dc;
    const float S = p.rws_S[slot];
    const float* ms = p.rws_m + slot * N + nb;
#pragma unroll
    for (int j = 0; j < NP; j++) {
      m[j].x = fmaf(ex2(A2[j].x * S), m[j].x, ms[2 * j]);
      m[j].y = fmaf(ex2(A2[j].y * S), m[j].y, nb + 2 * j + 1 < N ? ms[2 * j + 1] : 0.f);
    }
  }
}

template <int N, typename T>
__global__ void __launch_bounds__(kBwdCh) bwd_grad_kernel(const BwdArgs p) {
  static_assert(2 * N <= 32, "dB/dC partials must fit one value per lane");
  constexpr int NP = (N + 1) / 2;          // state pairs (packed fp32x2 arithmetic)
  constexpr int NQ = (2 * NP + 3) / 4;     // groups of 4 states in the shared state rows
  const int64_t n_dtiles = (p.d_inner + kBwdCh - 1) / kBwdCh;
  const int64_t tiles = (p.L + kBwdTile - 1) / kBwdTile;
  int64_t blk = blockIdx.x;
  const int64_t dtile = blk % n_dtiles;
  blk /= n_dtiles;
  const int c = (int)(blk % p.n_chunks);
  const int64_t b = blk / p.n_chunks;
  const int lane = threadIdx.x;
  const int64_t Dn = p.d_inner, L = p.L, d = dtile * kBwdCh + lane;
  const bool active = d < Dn;
  const int64_t dc = active ? d : 0;
  const int64_t t0 = (int64_t)c * p.chunk_len, t1 = min(t0 + p.chunk_len, L);
  const int64_t tl_lo = t0 / kBwdTile, tl_hi = (t1 - 1) / kBwdTile;  // chunks hold whole tiles
  __shared__ __align__(16) float sB[kBwdTile][4 * NQ], sC[kBwdTile][4 * NQ];
  // states after each step of the tile: [step][group of 4 states][lane][4] (16-byte rows)
  __shared__ __align__(16) float4 sH[kBwdTile][NQ][kBwdCh];

  float2 A2[NP], Af[NP], m[NP], dAacc[NP];
#pragma unroll
  for (int j = 0; j < NP; j++) {
    const int n0 = 2 * j, n1 = 2 * j + 1;
    const float a0 = p.A[dc * N + n0], a1 = n1 < N ? p.A[dc * N + n1] : 0.f;
    Af[j] = make_float2(a0, a1);
    A2[j] = make_float2(a0 * kLog2e, a1 * kLog2e);
    dAacc[j] = make_float2(0.f, 0.f);
  }
  chunk_carry_in<N, NP>(p, b, dc, c, 0, A2, m);
  if (2 * NP != 4 * NQ || 2 * NP != N) {  // zero the padding columns of the B/C rows
    for (int i = lane; i < kBwdTile * 4 * NQ; i += kBwdCh) { sB[i / (4 * NQ)][i % (4 * NQ)] = 0.f; sC[i / (4 * NQ)][i % (4 * NQ)] = 0.f; }
  }
  const float bias = p.delta_bias ? p.delta_bias[dc] : 0.f;
  const float Dd = p.D ? p.D[dc] : 0.f;
  float dDacc = 0.f, dbacc = 0.f;
  auto hrow = [&](int k, int j) -> float2 {
    const float4 q = sH[k][j / 2][lane];
    return (j & 1) ? make_float2(q.z, q.w) : make_float2(q.x, q.y);
  };
  auto pair_of = [&](const float* row, int j) -> float2 {
    return *reinterpret_cast<const float2*>(row + 2 * j);
  };

  for (int64_t tl = tl_hi; tl >= tl_lo; tl--) {
    const int64_t ts = tl * kBwdTile;
    const int steps = (int)min((int64_t)kBwdTile, L - ts);
    float xs[kBwdTile], us[kBwdTile], dys[kBwdTile], zs[kBwdTile];
#pragma unroll
    for (int k = 0; k < kBwdTile; k++) {
      const int64_t e = (b * L + ts + min(k, steps - 1)) * Dn + dc;
      xs[k] = ldf<T>(p.delta, e) + bias;
      us[k] = ldf<T>(p.u, e);
      dys[k] = ldf<T>(p.dy, e);
      zs[k] = p.z ? ldf<T>(p.z, e) : 0.f;
    }
    __syncwarp();
    for (int i = lane; i < steps * N; i += kBwdCh) {
      sB[i / N][i % N] = ldf<T>(p.B, (b * L + ts) * N + i);
      sC[i / N][i % N] = ldf<T>(p.C, (b * L + ts) * N + i);
    }
    float2 h0[NP];
    {
      const float* hk = p.ckpt_h + ((b * tiles + tl) * Dn + dc) * N;
#pragma unroll
      for (int j = 0; j < NP; j++)
        h0[j] = active ? make_float2(hk[2 * j], 2 * j + 1 < N ? hk[2 * j + 1] : 0.f) : make_float2(0.f, 0.f);
    }
    __syncwarp();
    float dts[kBwdTile];
    tile_step_sizes(xs, 0.f, p.softplus != 0, dts);  // xs hold delta_raw + bias

    // forward recompute of the tile's states into shared memory
    {
      float2 h[NP];
#pragma unroll
      for (int j = 0; j < NP; j++) h[j] = h0[j];
#pragma unroll
      for (int k = 0; k < kBwdTile; k++) {
        if (k < steps) {
          const float2 dt2 = make_float2(dts[k], dts[k]);
          const float w = dts[k] * us[k];
          const float2 w2 = make_float2(w, w);
#pragma unroll
          for (int j = 0; j < NP; j++) {
            const float2 xa = __fmul2_rn(dt2, A2[j]);
            h[j] = __ffma2_rn(make_float2(ex2(xa.x), ex2(xa.y)), h[j], __fmul2_rn(w2, pair_of(sB[k], j)));
          }
#pragma unroll
          for (int q = 0; q < NQ; q++)
            sH[k][q][lane] = make_float4(h[2 * q].x, h[2 * q].y, 2 * q + 1 < NP ? h[2 * q + 1].x : 0.f,
                                         2 * q + 1 < NP ? h[2 * q + 1].y : 0.f);
        }
      }
    }
    __syncwarp();

    // reverse over the tile; hk holds the state after step k, loaded one step ahead
    float2 hk[NP];
#pragma unroll
    for (int j = 0; j < NP; j++) hk[j] = hrow(kBwdTile - 1 < steps ? kBwdTile - 1 : 0, j);
#pragma unroll
    for (int k = kBwdTile - 1; k >= 0; k--) {
      if (k >= steps) {
        if (k - 1 >= 0 && k - 1 < steps) {
#pragma unroll
          for (int j = 0; j < NP; j++) hk[j] = hrow(k - 1, j);
        }
        continue;
      }
      const int64_t e = (b * L + ts + k) * Dn + dc;
      float2 hp[NP];
#pragma unroll
      for (int j = 0; j < NP; j++) hp[j] = k > 0 ? hrow(k - 1, j) : h0[j];
      float2 s2 = make_float2(Dd * us[k], 0.f);
#pragma unroll
      for (int j = 0; j < NP; j++) s2 = __ffma2_rn(pair_of(sC[k], j), hk[j], s2);
      const float s = s2.x + s2.y;
      float g = 1.f;
      if (p.z) {
        const float sg = rcp(1.f + ex2(-zs[k] * kLog2e));
        g = zs[k] * sg;
        if (active) static_cast<T*>(p.dz)[e] = from_f32<T>(dys[k] * s * sg * fmaf(zs[k], 1.f - sg, 1.f));
      }
      const float ds = dys[k] * g;
      dDacc = fmaf(ds, us[k], dDacc);
      const float dt = dts[k];
      const float2 dt2 = make_float2(dt, dt), ds2 = make_float2(ds, ds), u2 = make_float2(us[k], us[k]);
      const float dtu = dt * us[k];
      const float2 dtu2 = make_float2(active ? dtu : 0.f, active ? dtu : 0.f);
      const float2 dsa = make_float2(active ? ds : 0.f, active ? ds : 0.f);
      float2 ddt2 = make_float2(0.f, 0.f), slb2 = make_float2(0.f, 0.f);
      float v[32];
#pragma unroll
      for (int j = 0; j < NP; j++) {
        const float2 Bv = pair_of(sB[k], j);
        const float2 lam = __ffma2_rn(ds2, pair_of(sC[k], j), m[j]);
        const float2 xa = __fmul2_rn(dt2, A2[j]);
        const float2 dA = make_float2(ex2(xa.x), ex2(xa.y));
        const float2 t1 = __fmul2_rn(__fmul2_rn(lam, hp[j]), dA);
        ddt2 = __ffma2_rn(t1, Af[j], __ffma2_rn(lam, __fmul2_rn(Bv, u2), ddt2));
        dAacc[j] = __ffma2_rn(t1, dt2, dAacc[j]);
        slb2 = __ffma2_rn(lam, Bv, slb2);
        const float2 pb = __fmul2_rn(lam, dtu2), pc = __fmul2_rn(dsa, hk[j]);
        v[2 * j] = pb.x;
        if (2 * j + 1 < N) v[2 * j + 1] = pb.y;
        v[N + 2 * j] = pc.x;
        if (2 * j + 1 < N) v[N + 2 * j + 1] = pc.y;
        m[j] = __fmul2_rn(dA, lam);
        hk[j] = hp[j];
      }
#pragma unroll
      for (int j = 2 * N; j < 32; j++) v[j] = 0.f;
      const float ddt = ddt2.x + ddt2.y;
      const float dx = p.softplus ? ddt * rcp(1.f + ex2(-xs[k] * kLog2e)) : ddt;
      dbacc += dx;
      if (active) {
        static_cast<T*>(p.du)[e] = from_f32<T>(fmaf(ds, Dd, dt * (slb2.x + slb2.y)));
        static_cast<T*>(p.ddelta)[e] = from_f32<T>(dx);
      }
      warp_reduce_scatter_add<N>(v, lane, p.dB + (b * L + ts + k) * N, p.dC + (b * L + ts + k) * N);
    }
    __syncwarp();
  }
  if (!active) return;
#pragma unroll
  for (int j = 0; j < NP; j++) {
    atomicAdd(p.dA + d * N + 2 * j, dAacc[j].x);
    if (2 * j + 1 < N) atomicAdd(p.dA + d * N + 2 * j + 1, dAacc[j].y);
  }
  if (p.dD) atomicAdd(p.dD + d, dDacc);
  if (p.dbias) atomicAdd(p.dbias + d, dbacc);
  if (p.dinit && tl_lo == 0) {
#pragma unroll
    for (int j = 0; j < NP; j++) {
      p.dinit[(b * Dn + d) * N + 2 * j] = m[j].x;
      if (2 * j + 1 < N) p.dinit[(b * Dn + d) * N + 2 * j + 1] = m[j].y;
    }
  }
}

// ---------------------------------------------------------------------------------------
// 3b. Gradients with two lanes per channel (d_state a multiple of 8): lane 2c + q of the warp
//     holds states [q N/2, (q + 1) N/2) of channel c, so a CTA covers 16 channels with half
//     the per-lane registers and half the shared state tile of the one-lane kernel per warp
//     (about twice the warps per SM).  The per-step readout and the step-size and u gradients
//     add the two halves with one shfl.xor each; dB and dC are summed over the 16 channels
//     through a transpose in shared memory (each lane stores its N partials as one row, then
//     sums one column over the 16 lanes of its parity) and added atomically, one value per
//     lane.
constexpr int kBwdCh2 = 16;  // channels per CTA of the two-lane gradient kernel

template <int N, typename T>
__global__ void __launch_bounds__(32, 10) bwd_grad_kernel2(const BwdArgs p) {
  static_assert(N % 8 == 0 && N <= 16, "two lanes of whole float4 state groups");
  constexpr int NL = N / 2;        // states per lane
  constexpr int NP = NL / 2;       // state pairs per lane (packed fp32x2 arithmetic)
  constexpr int NQ = NL / 4;       // float4 groups per lane in the shared state rows
  constexpr int kPitch = N + 4;    // reduction rows: N partials + padding (16-byte aligned)
  const int64_t n_dtiles = (p.d_inner + kBwdCh2 - 1) / kBwdCh2;
  const int64_t tiles = (p.L + kBwdTile - 1) / kBwdTile;
  int64_t blk = blockIdx.x;
  const int64_t dtile = blk % n_dtiles;
  blk /= n_dtiles;
  const int c = (int)(blk % p.n_chunks);
  const int64_t b = blk / p.n_chunks;
  const int lane = threadIdx.x, q = lane & 1;
  const int64_t Dn = p.d_inner, L = p.L, d = dtile * kBwdCh2 + (lane >> 1);
  const bool active = d < Dn;
  const int64_t dc = active ? d : 0;
  const int nb = q * NL;  // first state of this lane
  const int64_t t0 = (int64_t)c * p.chunk_len, t1 = min(t0 + p.chunk_len, L);
  const int64_t tl_lo = t0 / kBwdTile, tl_hi = (t1 - 1) / kBwdTile;  // chunks hold whole tiles
  __shared__ __align__(16) float sB[kBwdTile][N], sC[kBwdTile][N];
  __shared__ __align__(16) float4 sH[kBwdTile][NQ][32];  // this lane's states after each step
  __shared__ __align__(16) float sR[32][kPitch];          // dB/dC partials, one row per lane
  // the reduced value this lane adds: output o = lane (o < N: dB[o], else dC[o - N]), the sum
  // over channels of column (o < N ? 0 : NL) + o mod NL of the rows of parity (o mod N) / NL
  const int o_col = (lane < N ? 0 : NL) + (lane % N) % NL, o_par = (lane % N) / NL;

  float2 A2[NP], Af[NP], m[NP], dAacc[NP];
#pragma unroll
  for (int j = 0; j < NP; j++) {
    const float a0 = p.A[dc * N + nb + 2 * j], a1 = p.A[dc * N + nb + 2 * j + 1];
    Af[j] = make_float2(a0, a1);
    A2[j] = make_float2(a0 * kLog2e, a1 * kLog2e);
    dAacc[j] = make_float2(0.f, 0.f);
  }
  chunk_carry_in<N, NP>(p, b, dc, c, nb, A2, m);
  const float bias = p.delta_bias ? p.delta_bias[dc] : 0.f;
  const float Dd = p.D ? p.D[dc] : 0.f;
  float dDacc = 0.f, dbacc = 0.f;
  auto hrow = [&](int k, int j) -> float2 {
    const float4 v = sH[k][j / 2][lane];
    return (j & 1) ? make_float2(v.z, v.w) : make_float2(v.x, v.y);
  };
  auto pair_of = [&](const float* row, int j) -> float2 {
    return *reinterpret_cast<const float2*>(row + nb + 2 * j);
  };

  for (int64_t tl = tl_hi; tl >= tl_lo; tl--) {
    const int64_t ts = tl * kBwdTile;
    const int steps = (int)min((int64_t)kBwdTile, L - ts);
    float xs[kBwdTile], us[kBwdTile], dys[kBwdTile], zs[kBwdTile];
#pragma unroll
    for (int k = 0; k < kBwdTile; k++) {
      const int64_t e = (b * L + ts + min(k, steps - 1)) * Dn + dc;
      xs[k] = ldf<T>(p.delta, e) + bias;
      us[k] = ldf<T>(p.u, e);
      dys[k] = ldf<T>(p.dy, e);
      zs[k] = p.z ? ldf<T>(p.z, e) : 0.f;
    }
    __syncwarp();
    for (int i = lane; i < steps * N; i += 32) {
      sB[i / N][i % N] = ldf<T>(p.B, (b * L + ts) * N + i);
      sC[i / N][i % N] = ldf<T>(p.C, (b * L + ts) * N + i);
    }
    float2 h0[NP];
    {
      const float* hk = p.ckpt_h + ((b * tiles + tl) * Dn + dc) * N + nb;
#pragma unroll
      for (int j = 0; j < NP; j++) h0[j] = active ? make_float2(hk[2 * j], hk[2 * j + 1]) : make_float2(0.f, 0.f);
    }
    __syncwarp();
    float dts[kBwdTile];
    tile_step_sizes(xs, 0.f, p.softplus != 0, dts);  // xs hold delta_raw + bias

    // forward recompute of this lane's states over the tile into shared memory
    {
      float2 h[NP];
#pragma unroll
      for (int j = 0; j < NP; j++) h[j] = h0[j];
#pragma unroll
      for (int k = 0; k < kBwdTile; k++) {
        if (k < steps) {
          const float2 dt2 = make_float2(dts[k], dts[k]);
          const float w = dts[k] * us[k];
          const float2 w2 = make_float2(w, w);
#pragma unroll
          for (int j = 0; j < NP; j++) {
            const float2 xa = __fmul2_rn(dt2, A2[j]);
            h[j] = __ffma2_rn(make_float2(ex2(xa.x), ex2(xa.y)), h[j], __fmul2_rn(w2, pair_of(sB[k], j)));
          }
#pragma unroll
          for (int g = 0; g < NQ; g++) sH[k][g][lane] = make_float4(h[2 * g].x, h[2 * g].y, h[2 * g + 1].x, h[2 * g + 1].y);
        }
      }
    }
    __syncwarp();

    // reverse over the tile; hk holds the state after step k
    float2 hk[NP];
#pragma unroll
    for (int j = 0; j < NP; j++) hk[j] = hrow(kBwdTile - 1 < steps ? kBwdTile - 1 : 0, j);
#pragma unroll
    for (int k = kBwdTile - 1; k >= 0; k--) {
      if (k >= steps) {
        if (k - 1 >= 0 && k - 1 < steps) {
#pragma unroll
          for (int j = 0; j < NP; j++) hk[j] = hrow(k - 1, j);
        }
        continue;
      }
      const int64_t e = (b * L + ts + k) * Dn + dc;
      float2 hp[NP];
#pragma unroll
      for (int j = 0; j < NP; j++) hp[j] = k > 0 ? hrow(k - 1, j) : h0[j];
      float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int j = 0; j < NP; j++) s2 = __ffma2_rn(pair_of(sC[k], j), hk[j], s2);
      const float s_half = s2.x + s2.y;
      const float s = s_half + __shfl_xor_sync(0xFFFFFFFFu, s_half, 1) + Dd * us[k];
      float g = 1.f;
      if (p.z) {
        const float sg = rcp(1.f + ex2(-zs[k] * kLog2e));
        g = zs[k] * sg;
        if (active && q == 0) static_cast<T*>(p.dz)[e] = from_f32<T>(dys[k] * s * sg * fmaf(zs[k], 1.f - sg, 1.f));
      }
      const float ds = dys[k] * g;
      dDacc = fmaf(ds, us[k], dDacc);
      const float dt = dts[k];
      const float2 dt2 = make_float2(dt, dt), ds2 = make_float2(ds, ds), u2 = make_float2(us[k], us[k]);
      const float dtu = dt * us[k];
      const float2 dtu2 = make_float2(active ? dtu : 0.f, active ? dtu : 0.f);
      const float2 dsa = make_float2(active ? ds : 0.f, active ? ds : 0.f);
      float2 ddt2 = make_float2(0.f, 0.f), slb2 = make_float2(0.f, 0.f);
      float v[N];  // dB partials of this lane's states, then dC partials
#pragma unroll
      for (int j = 0; j < NP; j++) {
        const float2 Bv = pair_of(sB[k], j);
        const float2 lam = __ffma2_rn(ds2, pair_of(sC[k], j), m[j]);
        const float2 xa = __fmul2_rn(dt2, A2[j]);
        const float2 dA = make_float2(ex2(xa.x), ex2(xa.y));
        const float2 t1 = __fmul2_rn(__fmul2_rn(lam, hp[j]), dA);
        ddt2 = __ffma2_rn(t1, Af[j], __ffma2_rn(lam, __fmul2_rn(Bv, u2), ddt2));
        dAacc[j] = __ffma2_rn(t1, dt2, dAacc[j]);
        slb2 = __ffma2_rn(lam, Bv, slb2);
        const float2 pb = __fmul2_rn(lam, dtu2), pc = __fmul2_rn(dsa, hk[j]);
        v[2 * j] = pb.x;
        v[2 * j + 1] = pb.y;
        v[NL + 2 * j] = pc.x;
        v[NL + 2 * j + 1] = pc.y;
        m[j] = __fmul2_rn(dA, lam);
        hk[j] = hp[j];
      }
      const float ddt_half = ddt2.x + ddt2.y, slb_half = slb2.x + slb2.y;
      const float ddt = ddt_half + __shfl_xor_sync(0xFFFFFFFFu, ddt_half, 1);
      const float slb = slb_half + __shfl_xor_sync(0xFFFFFFFFu, slb_half, 1);
      const float dx = p.softplus ? ddt * rcp(1.f + ex2(-xs[k] * kLog2e)) : ddt;
      dbacc += dx;
      if (active) {
        if (q == 0) static_cast<T*>(p.du)[e] = from_f32<T>(fmaf(ds, Dd, dt * slb));
        else static_cast<T*>(p.ddelta)[e] = from_f32<T>(dx);
      }
      // dB / dC: sum the partials over the 16 channels through shared memory
#pragma unroll
      for (int c4 = 0; c4 < N / 4; c4++)
        *reinterpret_cast<float4*>(&sR[lane][4 * c4]) = make_float4(v[4 * c4], v[4 * c4 + 1], v[4 * c4 + 2], v[4 * c4 + 3]);
      __syncwarp();
      if (lane < 2 * N) {
        float acc = 0.f;
#pragma unroll
        for (int c = 0; c < kBwdCh2; c++) acc += sR[2 * c + o_par][o_col];
        float* row = (lane < N ? p.dB : p.dC) + (b * L + ts + k) * N;
        atomicAdd(row + lane % N, acc);
      }
      __syncwarp();
    }
    __syncwarp();
  }
  if (!active) return;
#pragma unroll
  for (int j = 0; j < NP; j++) {
    atomicAdd(p.dA + d * N + nb + 2 * j, dAacc[j].x);
    atomicAdd(p.dA + d * N + nb + 2 * j + 1, dAacc[j].y);
  }
  if (q == 0) {  // per-channel sums: both lanes hold them
    if (p.dD) atomicAdd(p.dD + d, dDacc);
    if (p.dbias) atomicAdd(p.dbias + d, dbacc);
  }
  if (p.dinit && tl_lo == 0) {
#pragma unroll
    for (int j = 0; j < NP; j++) {
      p.dinit[(b * Dn + d) * N + nb + 2 * j] = m[j].x;
      p.dinit[(b * Dn + d) * N + nb + 2 * j + 1] = m[j].y;
    }
  }
}

// ---------------------------------------------------------------------------------------

size_t bwd_workspace_floats(int64_t batch, int64_t L, int64_t d_inner, int d_state, int n_chunks) {
  const int64_t tiles = (L + kBwdTile - 1) / kBwdTile;
  const int64_t ck = batch * tiles * d_inner * d_state;                 // forward checkpoints
  const int64_t fws = batch * (int64_t)std::max(n_chunks - 1, 0) * d_inner * (d_state + 1);
  const int64_t rws = batch * (int64_t)n_chunks * d_inner * (d_state + 1);
  return (size_t)(ck + fws + rws);
}

template <int N, typename T>
static cudaError_t launch_bwd_t(const BwdArgs& a, const ScanParams& fwd, cudaStream_t s) {
  const int64_t n_dtiles = (a.d_inner + kBwdCh - 1) / kBwdCh;
  if (a.n_chunks > 1) {
    // forward chunk summaries: the forward scan's own summary pass
    cudaError_t e = launch_scan_summary(fwd, sizeof(T) == 2, s);
    if (e != cudaSuccess) return e;
    bwd_reverse_summary_kernel<N, T><<<(unsigned)(n_dtiles * (a.n_chunks - 1) * a.batch), kBwdCh, 0, s>>>(a);
  }
  {  // forward checkpoints: the forward scan's own kernel in its checkpoint mode
    ScanParams f = fwd;
    f.ckpt_h = a.ckpt_h;
    const cudaError_t e = launch_scan_ckpt(f, sizeof(T) == 2, s);
    if (e != cudaSuccess) return e;
  }
  if constexpr (N % 8 == 0) {  // two lanes per channel
    const int64_t n_dtiles2 = (a.d_inner + kBwdCh2 - 1) / kBwdCh2;
    bwd_grad_kernel2<N, T><<<(unsigned)(n_dtiles2 * a.n_chunks * a.batch), 32, 0, s>>>(a);
  } else {
    bwd_grad_kernel<N, T><<<(unsigned)(n_dtiles * a.n_chunks * a.batch), kBwdCh, 0, s>>>(a);
  }
  return cudaGetLastError();
}

template <typename T>
static cudaError_t dispatch_bwd(const BwdArgs& a, const ScanParams& fwd, cudaStream_t s) {
  switch (a.d_state) {
    case 1: return launch_bwd_t<1, T>(a, fwd, s);
    case 2: return launch_bwd_t<2, T>(a, fwd, s);
    case 3: return launch_bwd_t<3, T>(a, fwd, s);
    case 4: return launch_bwd_t<4, T>(a, fwd, s);
    case 5: return launch_bwd_t<5, T>(a, fwd, s);
    case 6: return launch_bwd_t<6, T>(a, fwd, s);
    case 7: return launch_bwd_t<7, T>(a, fwd, s);
    case 8: return launch_bwd_t<8, T>(a, fwd, s);
    case 9: return launch_bwd_t<9, T>(a, fwd, s);
    case 10: return launch_bwd_t<10, T>(a, fwd, s);
    case 11: return launch_bwd_t<11, T>(a, fwd, s);
    case 12: return launch_bwd_t<12, T>(a, fwd, s);
    case 13: return launch_bwd_t<13, T>(a, fwd, s);
    case 14: return launch_bwd_t<14, T>(a, fwd, s);
    case 15: return launch_bwd_t<15, T>(a, fwd, s);
    case 16: return launch_bwd_t<16, T>(a, fwd, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_scan_bwd(const BwdArgs& a, const ScanParams& fwd, bool bf16, cudaStream_t s) {
  return bf16 ? dispatch_bwd<__nv_bfloat16>(a, fwd, s) : dispatch_bwd<float>(a, fwd, s);
}

}  // namespace ssm
