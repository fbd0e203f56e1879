// Backward pass of the selective scan: gradients with respect to u, delta_raw, A, B, C, D, z,
// delta_bias and the initial state, given dL/dy and (optionally) dL/dlast_state.
//
// The pages describe the backward only as "recompute the intermediate states in the backward
// pass instead of storing them" (youngju.dev, "Mamba: Linear-Time Sequence Modeling with
// Selective State Spaces 论文分析", section "解决方案：Kernel Fusion + Recomputation").  Here:
//  1. forward checkpoints: the forward scan's look-back kernel in its checkpoint form
//     (ssm_scan_fwd.cu) stores the state before every 8 steps — never the per-step states;
//  2. reverse summaries (time-chunked plans only): the adjoint
//     lambda_t = ds_t C_t + dA_{t+1} lambda_{t+1} runs backwards over each chunk from a zero
//     carry; per chunk, its carry-out and its decay exp(A sum delta);
//  3. gradients: one CTA per (batch row, time chunk, 64 channels) walks the chunk's 8-step
//     tiles backwards from the adjoint carry entering it from the right, recomputing each
//     tile's states from its checkpoint (section 3 below).
// All arithmetic is fp32.

#include "ssm_device.cuh"
#include "ssm_internal.h"

#include <algorithm>
#include <cstdlib>
#include <type_traits>

namespace ssm {

constexpr int kBwdCh = 32;    // channels per CTA of the reverse-summary kernel (one warp)
constexpr int kBwdTile = 16;  // its time steps per tile

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
// 3. Gradients.  A CTA covers 64 consecutive channels of one batch row over one time chunk
//    and walks the chunk's 8-step tiles backwards, starting from the adjoint carry that
//    enters the chunk from the right.  Each thread owns a channel pair (d, d+1) and 4 of the
//    pair's states; the L lanes of a pair (L = 1, 2 or 4) split its 4L >= d_state states, and
//    state arithmetic runs on packed fp32 pairs of adjacent states.  Per tile:
//     - delta, u, z and dy rows (64 channels, 8 steps) are in shared memory (cp.async, issued
//       while the previous tile ran), B/C rows as fp32 (prefetched into registers);
//     - pre-phase: lane l does the per-element work of the steps k = l (mod L) once: step
//       size, delta*u, the gated output gradient ds = dy silu(z), and keeps the factors of
//       dz and of the softplus derivative for its own steps;
//     - forward recompute from the tile's checkpoint; the states after the odd steps go to
//       shared memory.  The reverse walk rebuilds each even step's state from the odd one
//       before it with one recurrence step: it needs that step's exp(delta A) anyway;
//     - reverse walk: lambda_t = m + ds_t C_t, the gradients of every input, m <- dA_t lambda_t.
//       Sums over states (delta, u and z gradients) go through shared memory per 4-step group;
//       so do dB and dC (sums over channels): per 4-step group each warp sums its pairs' values
//       in its own block, the warps' sums are added at the end of the tile and the tile's rows
//       go to global memory as float4 atomics.
namespace bwd {

constexpr int kCh = 64;   // channels per CTA
constexpr int kCP = 32;   // channel pairs per CTA
constexpr int kT = kCkptSteps;  // steps per tile (one checkpoint per tile)
constexpr int kOG = 4;    // steps per output group
static_assert(kT == 8, "the reverse walk is written for 8-step tiles");

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  const int n = valid ? 16 : 0;  // n == 0: no global read, 16 zero bytes written
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* q) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(q) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u64(unsigned long long* q, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(q), "l"(v) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::); }

template <typename T> struct PairIO;
template <> struct PairIO<float> {
  static __device__ __forceinline__ float2 load(const unsigned char* p) {
    return *reinterpret_cast<const float2*>(p);
  }
  static __device__ __forceinline__ void store(void* p, float2 v) { *reinterpret_cast<float2*>(p) = v; }
};
template <> struct PairIO<__nv_bfloat16> {
  static __device__ __forceinline__ float2 load(const unsigned char* p) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  }
  static __device__ __forceinline__ void store(void* p, float2 v) {
    *reinterpret_cast<__nv_bfloat162*>(p) = __float22bfloat162_rn(v);
  }
};

// softplus(x) and its derivative sigmoid(x) from one exponential e = exp(-|x|):
// softplus = max(x, 0) + log1p(e), sigmoid = (x >= 0 ? 1 : e) / (1 + e).
__device__ __forceinline__ void softplus_sigmoid2(float2 x, float2& sp, float2& sg) {
  const float2 e = make_float2(ex2(-fabsf(x.x) * kLog2e), ex2(-fabsf(x.y) * kLog2e));
  sp = __fadd2_rn(make_float2(fmaxf(x.x, 0.f), fmaxf(x.y, 0.f)), log1p_unit2(e));
  const float2 r = make_float2(rcp(1.f + e.x), rcp(1.f + e.y));
  sg = make_float2(x.x >= 0.f ? r.x : e.x * r.x, x.y >= 0.f ? r.y : e.y * r.y);
}

template <int L, typename T>
struct Cfg {
  static constexpr int kThreads = 32 * L;
  static constexpr int kWarps = L;
  static constexpr int kNP = 4 * L;                 // states held per pair (>= d_state)
  static constexpr int kTS = (int)sizeof(T);
  static constexpr int kRowB = kCh * kTS;            // one activation row of the CTA's channels
  static constexpr int kChunks = kRowB / 16;         // 16-byte pieces per row
  static constexpr int kPairB = 2 * kTS;
  static constexpr int kSwz = 8 / L;                 // row swizzle step
  static constexpr int kXB = 4 * kT * kRowB;         // delta, u, z, dy rows of one tile
  static constexpr int kBCB = 2 * kT * kNP * 4;      // B, C rows (fp32)
  static constexpr int kQB = 2 * kT * kCP * 16;      // per step and pair: (dt, dt*u), (ds, u)
  static constexpr int kHB = (kT / 2) * 2 * kThreads * 16;  // states after the odd steps
  // per-lane partial sums, [step of the group][lane of the pair][pair ^ swizzle]
  static constexpr int kP4B = kOG * L * kCP * 16;    // (ddt, u-gradient) sums
  static constexpr int kP2B = kOG * L * kCP * 8;     // readouts
  static constexpr int kWB = kWarps * kOG * 2 * 32 * 16;  // per warp: dB/dC values of its lanes
  static constexpr int kRB = kT * kWarps * 2 * kNP * 4;   // dB/dC rows per warp
  static constexpr int kSmem = kXB + kBCB + kQB + kHB + kP4B + kP2B + kWB + kRB;
};

template <int L, typename T>
__global__ void __launch_bounds__(32 * L, L == 4 ? 3 : (L == 2 ? 6 : 12)) grad_kernel(const BwdArgs p) {
  using K = Cfg<L, T>;
  constexpr int kNP = K::kNP;
  extern __shared__ __align__(16) unsigned char smem[];
  unsigned char* sX = smem;                                                    // [4][kT][kRowB]
  float* sBC = reinterpret_cast<float*>(smem + K::kXB);                        // [2][kT][kNP]
  float4* sQ = reinterpret_cast<float4*>(smem + K::kXB + K::kBCB);              // [kT][2][kCP]
  float4* sH = reinterpret_cast<float4*>(smem + K::kXB + K::kBCB + K::kQB);     // [kT/2][2][kThreads]
  float4* sP4 = reinterpret_cast<float4*>(smem + K::kXB + K::kBCB + K::kQB + K::kHB);  // [kOG][L][kCP]
  float2* sP2 = reinterpret_cast<float2*>(smem + K::kXB + K::kBCB + K::kQB + K::kHB + K::kP4B);
  float4* sW = reinterpret_cast<float4*>(smem + K::kXB + K::kBCB + K::kQB + K::kHB + K::kP4B + K::kP2B);
  float* sR = reinterpret_cast<float*>(smem + K::kXB + K::kBCB + K::kQB + K::kHB + K::kP4B + K::kP2B + K::kWB);

  const int N = p.d_state;
  const int64_t Dn = p.d_inner, Ls = p.L;
  const int64_t n_dt = (Dn + kCh - 1) / kCh;
  int64_t blk = blockIdx.x;
  const int64_t dtile = blk % n_dt;
  blk /= n_dt;
  // hand-over plans number the CTAs from the last chunk back, so that the CTA a chunk waits
  // for (the chunk after it) was dispatched before it
  const int c = p.handover ? p.n_chunks - 1 - (int)(blk / p.batch) : (int)(blk % p.n_chunks);
  const int64_t b = p.handover ? blk % p.batch : blk / p.n_chunks;
  const bool wait_carry = p.handover && c + 1 < p.n_chunks;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int l = lane % L;
  const int P = warp * (32 / L) + lane / L;
  const int64_t d0 = dtile * kCh;
  const int64_t d = d0 + 2 * P;
  const bool active = d < Dn;
  const int n0 = 4 * l;
  // partial-sum slot of (step kg of the group, lane mm of the pair, pair P): the XOR keeps both
  // the writes (lanes of a pair at one step) and the reads (one lane per step) on distinct banks
  //   slot = (kg L + mm) kCP + (P ^ (((kg ^ mm) & (L - 1)) c)), c = 8/L (float4) or 16/L (float2);
  // the XOR separates, so this lane's part (l c) is folded in once.
  const int Pl4 = P ^ (l * (8 / L)), Pl2 = P ^ (l * (16 / L));
  // written by lane l at step kg (compile-time) of the group
  auto p4w = [&](int kg) { return (kg * L + l) * kCP + (Pl4 ^ ((kg & (L - 1)) * (8 / L))); };
  auto p2w = [&](int kg) { return (kg * L + l) * kCP + (Pl2 ^ ((kg & (L - 1)) * (16 / L))); };
  // read by lane l for its own step kg = i L + l of the group, lane mm's part
  auto p4r = [&](int i, int mm) { return ((i * L + l) * L + mm) * kCP + (Pl4 ^ (mm * (8 / L))); };
  auto p2r = [&](int i, int mm) { return ((i * L + l) * L + mm) * kCP + (Pl2 ^ (mm * (16 / L))); };
  const int64_t t0 = (int64_t)c * p.chunk_len, t1 = min(t0 + p.chunk_len, Ls);
  const int64_t tiles = (Ls + kT - 1) / kT;
  const int64_t tl_lo = t0 / kT, tl_hi = (t1 - 1) / kT;  // chunks hold whole tiles

  // Index s = 2c + j: channel d + c, states n0 + 2j, n0 + 2j + 1.
  float2 A2[4], Af[4], m[4], dAacc[4];
#pragma unroll
  for (int s = 0; s < 4; s++) {
    const int cc = s / 2, n = n0 + 2 * (s % 2);
    const float* Ar = p.A + (active ? (d + cc) * N : 0);
    const float a0 = (active && n < N) ? Ar[n] : 0.f, a1 = (active && n + 1 < N) ? Ar[n + 1] : 0.f;
    Af[s] = make_float2(a0, a1);
    A2[s] = make_float2(a0 * kLog2e, a1 * kLog2e);
    dAacc[s] = make_float2(0.f, 0.f);
    m[s] = make_float2(0.f, 0.f);
    if (!active) continue;
    // adjoint carry entering the chunk: dL/dlast_state folded with the reverse summaries of
    // the chunks after it
    if (p.dlast && !wait_carry) {
      const float* dl = p.dlast + (b * Dn + d + cc) * N;
      m[s] = make_float2(n < N ? dl[n] : 0.f, n + 1 < N ? dl[n + 1] : 0.f);
    }
    for (int jc = p.n_chunks - 1; jc > c && !p.handover; jc--) {
      const int64_t slot = (b * p.n_chunks + jc) * Dn + d + cc;
      const float S = p.rws_S[slot];
      const float* ms = p.rws_m + slot * N;
      m[s].x = fmaf(ex2(A2[s].x * S), m[s].x, n < N ? ms[n] : 0.f);
      m[s].y = fmaf(ex2(A2[s].y * S), m[s].y, n + 1 < N ? ms[n + 1] : 0.f);
    }
  }
  const float2 bias2 = (active && p.delta_bias) ? make_float2(p.delta_bias[d], p.delta_bias[d + 1])
                                                : make_float2(0.f, 0.f);
  const float2 D2 = (active && p.D) ? make_float2(p.D[d], p.D[d + 1]) : make_float2(0.f, 0.f);
  const bool sp = p.softplus != 0;
  const bool has_z = p.z != nullptr;
  float2 dDacc = make_float2(0.f, 0.f), dbacc = make_float2(0.f, 0.f);

  if (kNP > N) {  // padding state columns of the B/C rows read as zero
    for (int i = tid; i < 2 * kT * (kNP - N); i += K::kThreads)
      sBC[(i / (kNP - N)) * kNP + N + i % (kNP - N)] = 0.f;
  }

  const int pchunk = (P * K::kPairB) / 16, pwithin = (P * K::kPairB) % 16;
  const char* xsrc[4] = {static_cast<const char*>(p.delta), static_cast<const char*>(p.u),
                         static_cast<const char*>(p.z), static_cast<const char*>(p.dy)};
  // One tile's activation rows: 16-byte piece ch of row r of array x lands at piece
  // ch ^ ((r % L) * kSwz), so that the L rows the lanes of a pair read at once hit distinct banks.
  auto issue_tile = [&](int64_t tl) {
    const int64_t ts = tl * kT;
    constexpr int kPieces = kT * K::kChunks;
#pragma unroll
    for (int x = 0; x < 4; x++) {
      if (x == 2 && !has_z) continue;
      const char* g0 = xsrc[x] + ((b * Ls + ts) * Dn + d0) * K::kTS;
#pragma unroll
      for (int j = 0; j < (kPieces + K::kThreads - 1) / K::kThreads; j++) {
        const int q = tid + j * K::kThreads;
        if (kPieces % K::kThreads == 0 || q < kPieces) {
          const int r = q / K::kChunks, ch = q % K::kChunks;
          const bool valid = ts + r < t1 && d0 + ch * (16 / K::kTS) < Dn;
          cp_async16(sX + (x * kT + r) * K::kRowB + ((ch ^ ((r % L) * K::kSwz)) * 16),
                     valid ? g0 + (int64_t)r * Dn * K::kTS + ch * 16 : xsrc[x], valid);
        }
      }
    }
  };
  // this pair's bytes in row i L + l (the pre-phase's rows) of array x
  const int xl = l * K::kRowB + ((pchunk ^ (l * K::kSwz)) * 16) + pwithin;
  auto xrow = [&](int x, int i) { return sX + (x * kT + i * L) * K::kRowB + xl; };

  // B/C rows of a tile: global -> registers -> fp32 shared memory.  Whole 16-byte pieces when
  // the rows are exactly the padded width and 16-byte multiples, element by element otherwise.
  const T* __restrict__ Bg = static_cast<const T*>(p.B);
  const T* __restrict__ Cg = static_cast<const T*>(p.C);
  constexpr int kVec = 16 / K::kTS;
  constexpr int kBCVals = 2 * kT * kNP;
  constexpr int kVecPT = (kBCVals / kVec + K::kThreads - 1) / K::kThreads;
  constexpr int kScPT = (kBCVals + K::kThreads - 1) / K::kThreads;
  const bool vec_bc = N == kNP && (N * K::kTS) % 16 == 0;
  uint4 bcv[kVecPT];
  float bcs[kScPT];
  auto load_bc = [&](int64_t tl) {
    const int64_t ts = tl * kT;
    const int64_t e0 = (b * Ls + ts) * N;
    const int64_t rows = min((int64_t)kT, t1 - ts);
    if (vec_bc) {
#pragma unroll
      for (int j = 0; j < kVecPT; j++) {
        const int e = (tid + j * K::kThreads) * kVec;  // element of [which][k][n]
        const int which = e / (kT * N), ew = e % (kT * N);
        bcv[j] = make_uint4(0, 0, 0, 0);
        if (e < kBCVals && ew / N < rows) bcv[j] = __ldg(reinterpret_cast<const uint4*>((which ? Cg : Bg) + e0 + ew));
      }
    } else {
#pragma unroll
      for (int j = 0; j < kScPT; j++) {
        const int e = tid + j * K::kThreads;
        const int which = e / (kT * N), ew = e % (kT * N);
        bcs[j] = 0.f;
        if (e < 2 * kT * N && ew / N < rows) bcs[j] = to_f32((which ? Cg : Bg)[e0 + ew]);
      }
    }
  };
  auto store_bc = [&]() {
    if (vec_bc) {
#pragma unroll
      for (int j = 0; j < kVecPT; j++) {
        const int e = (tid + j * K::kThreads) * kVec;
        if (e < kBCVals) {
          float* dst = sBC + e;  // N == kNP: the layouts agree
          const uint4 v = bcv[j];
          if constexpr (K::kTS == 4) {
            *reinterpret_cast<float4*>(dst) = make_float4(__uint_as_float(v.x), __uint_as_float(v.y),
                                                          __uint_as_float(v.z), __uint_as_float(v.w));
          } else {
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 2; q++)
              *reinterpret_cast<float4*>(dst + 4 * q) = make_float4(
                  __uint_as_float(w4[2 * q] << 16), __uint_as_float(w4[2 * q] & 0xFFFF0000u),
                  __uint_as_float(w4[2 * q + 1] << 16), __uint_as_float(w4[2 * q + 1] & 0xFFFF0000u));
          }
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < kScPT; j++) {
        const int e = tid + j * K::kThreads;
        if (e < 2 * kT * N) {
          const int which = e / (kT * N), ew = e % (kT * N);
          sBC[(which * kT + ew / N) * kNP + ew % N] = bcs[j];
        }
      }
    }
  };

  // The state before a tile (its checkpoint) for this thread's 4 states of both channels.
  float2 h0[4], h0n[4];
  auto load_ckpt = [&](int64_t tl, float2 (&h)[4]) {
#pragma unroll
    for (int s = 0; s < 4; s++) h[s] = make_float2(0.f, 0.f);
    if (!active) return;
#pragma unroll
    for (int cc = 0; cc < 2; cc++) {
      const float* ck = p.ckpt_h + ((b * tiles + tl) * Dn + d + cc) * N;
      if (N % 4 == 0) {
        if (n0 < N) {
          const float4 v = __ldcg(reinterpret_cast<const float4*>(ck + n0));
          h[2 * cc] = make_float2(v.x, v.y);
          h[2 * cc + 1] = make_float2(v.z, v.w);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 2; j++) {
          const int n = n0 + 2 * j;
          h[2 * cc + j] = make_float2(n < N ? ck[n] : 0.f, n + 1 < N ? ck[n + 1] : 0.f);
        }
      }
    }
  };

  // pair-of-step quantities (both channels) of step k, from the pre-phase
  auto q_dt = [&](int k) { return sQ[(k * 2 + 0) * kCP + (P ^ ((k % L) * K::kSwz))]; };  // dt0 dt1 dtu0 dtu1
  auto q_ds = [&](int k) { return sQ[(k * 2 + 1) * kCP + (P ^ ((k % L) * K::kSwz))]; };  // ds0 ds1 u0 u1
  // the same for this lane's own step i L + l (rows written by this lane in the pre-phase)
  const int qwl = l * 2 * kCP + (P ^ (l * K::kSwz));
  auto q_own = [&](int i, int w) { return sQ + (i * L * 2 + w) * kCP + qwl; };
  auto brow = [&](int k) { return *reinterpret_cast<const float4*>(sBC + (0 * kT + k) * kNP + n0); };
  auto crow = [&](int k) { return *reinterpret_cast<const float4*>(sBC + (1 * kT + k) * kNP + n0); };

  // exp(dt A) for the 4 state pairs at step k
  auto decays = [&](const float4 q, float2 (&dA)[4]) {
#pragma unroll
    for (int s = 0; s < 4; s++) {
      const float dtc = s < 2 ? q.x : q.y;
      const float2 xa = __fmul2_rn(make_float2(dtc, dtc), A2[s]);
      dA[s] = make_float2(ex2(xa.x), ex2(xa.y));
    }
  };
  // one forward step: h <- dA h + dt u B
  auto fwd_step = [&](const float4 q, const float4 Bq, const float2 (&dA)[4], const float2 (&hin)[4], float2 (&hout)[4]) {
    const float2 Bp[2] = {make_float2(Bq.x, Bq.y), make_float2(Bq.z, Bq.w)};
#pragma unroll
    for (int s = 0; s < 4; s++) {
      const float w = s < 2 ? q.z : q.w;
      hout[s] = __ffma2_rn(dA[s], hin[s], __fmul2_rn(make_float2(w, w), Bp[s % 2]));
    }
  };

  float4 own[kT / L];  // per own step: (dz factor, softplus derivative) of both channels

  // one reverse step at step k: hk = state after step k, hp = before, dA = exp(dt_k A)
  auto rev_step = [&](int k, const float2 (&hk)[4], const float2 (&hp)[4], const float2 (&dA)[4]) {
    const float4 q0 = q_dt(k), q1 = q_ds(k);
    const float4 Bq = brow(k), Cq = crow(k);
    const float2 Bp[2] = {make_float2(Bq.x, Bq.y), make_float2(Bq.z, Bq.w)};
    const float2 Cp[2] = {make_float2(Cq.x, Cq.y), make_float2(Cq.z, Cq.w)};
    float2 ddt[2], slb[2], rd[2], pbs[2], pcs[2];
#pragma unroll
    for (int cc = 0; cc < 2; cc++) {
      const float dt = cc ? q0.y : q0.x, dtu = cc ? q0.w : q0.z;
      const float ds = cc ? q1.y : q1.x, uu = cc ? q1.w : q1.z;
      const float2 dt2 = make_float2(dt, dt), dtu2 = make_float2(dtu, dtu), ds2 = make_float2(ds, ds),
                   u2 = make_float2(uu, uu);
      ddt[cc] = slb[cc] = rd[cc] = make_float2(0.f, 0.f);
#pragma unroll
      for (int j = 0; j < 2; j++) {
        const int s = 2 * cc + j;
        const float2 lam = __ffma2_rn(ds2, Cp[j], m[s]);
        const float2 t1 = __fmul2_rn(__fmul2_rn(lam, hp[s]), dA[s]);
        ddt[cc] = __ffma2_rn(t1, Af[s], __ffma2_rn(lam, __fmul2_rn(Bp[j], u2), ddt[cc]));
        dAacc[s] = __ffma2_rn(t1, dt2, dAacc[s]);
        slb[cc] = __ffma2_rn(lam, Bp[j], slb[cc]);
        rd[cc] = __ffma2_rn(Cp[j], hk[s], rd[cc]);
        const float2 pb = __fmul2_rn(lam, dtu2), pc = __fmul2_rn(ds2, hk[s]);
        pbs[j] = cc ? __fadd2_rn(pbs[j], pb) : pb;
        pcs[j] = cc ? __fadd2_rn(pcs[j], pc) : pc;
        m[s] = __fmul2_rn(dA[s], lam);
      }
    }
    // this lane's share of the per-channel sums over states
    const int kg = k % kOG;
    sP4[p4w(kg)] = make_float4(ddt[0].x + ddt[0].y, ddt[1].x + ddt[1].y,
                                              slb[0].x + slb[0].y, slb[1].x + slb[1].y);
    sP2[p2w(kg)] = make_float2(rd[0].x + rd[0].y, rd[1].x + rd[1].y);
    // dB (states n0..n0+3) and dC (same) of the pair, to this warp's block; lane position
    // XOR-swizzled per (step, dB|dC) so that the group's column sums read distinct banks
#pragma unroll
    for (int h = 0; h < 2; h++)
      sW[((warp * kOG + kg) * 2 + h) * 32 + (lane ^ (((2 * kg + h) * L) % 8))] =
          h ? make_float4(pcs[0].x, pcs[0].y, pcs[1].x, pcs[1].y) : make_float4(pbs[0].x, pbs[0].y, pbs[1].x, pbs[1].y);
  };

  // dB/dC of the steps k0 .. k0+kOG-1 summed over the warp's pairs: lane o takes (step, dB|dC,
  // state slice) and adds the 32/L pairs' values; the warps' sums go to sR.
  auto warp_bc_sums = [&](int k0) {
    constexpr int kOut = kOG * 2 * L;  // float4 outputs per warp and group
    if (lane < kOut) {
      const int kg = lane / (2 * L), h = (lane / L) % 2, lq = lane % L;
      const float4* src = sW + ((warp * kOG + kg) * 2 + h) * 32;
      const int sw = ((2 * kg + h) * L) % 8;
      const float4 v0 = src[lq ^ sw];
      float2 a01 = make_float2(v0.x, v0.y), a23 = make_float2(v0.z, v0.w);
#pragma unroll
      for (int pp = 1; pp < 32 / L; pp++) {
        const float4 v = src[(pp * L + lq) ^ sw];
        a01 = __fadd2_rn(a01, make_float2(v.x, v.y));
        a23 = __fadd2_rn(a23, make_float2(v.z, v.w));
      }
      *reinterpret_cast<float4*>(sR + ((k0 + kg) * K::kWarps + warp) * 2 * kNP + h * kNP + 4 * lq) =
          make_float4(a01.x, a01.y, a23.x, a23.y);
    }
  };

  // Outputs of the steps k0 .. k0+kOG-1: lane l finishes its own steps from the L lanes'
  // partial sums.
  int64_t ebase = 0;
  auto output_group = [&](auto k0_tag, int steps) {
    constexpr int k0 = decltype(k0_tag)::value;
#pragma unroll
    for (int i = 0; i < kOG / L; i++) {
      const int k = k0 + i * L + l;
      if (k < steps && active) {
        float4 a = sP4[p4r(i, 0)];
        float2 r = sP2[p2r(i, 0)];
#pragma unroll
        for (int mm = 1; mm < L; mm++) {
          const float4 a2 = sP4[p4r(i, mm)];
          const float2 r2 = sP2[p2r(i, mm)];
          a = make_float4(a.x + a2.x, a.y + a2.y, a.z + a2.z, a.w + a2.w);
          r = make_float2(r.x + r2.x, r.y + r2.y);
        }
        const float4 q0 = *q_own(k0 / L + i, 0), q1 = *q_own(k0 / L + i, 1);
        const float4 f = own[k0 / L + i];
        const float2 ddt = make_float2(a.x, a.y), slb = make_float2(a.z, a.w);
        const float2 dx = sp ? __fmul2_rn(ddt, make_float2(f.z, f.w)) : ddt;
        const float2 ds = make_float2(q1.x, q1.y), uu = make_float2(q1.z, q1.w), dt = make_float2(q0.x, q0.y);
        const float2 du = __ffma2_rn(ds, D2, __fmul2_rn(dt, slb));
        const int64_t e = ebase + (int64_t)(k0 + i * L) * Dn * K::kTS;
        PairIO<T>::store(static_cast<char*>(p.du) + e, du);
        PairIO<T>::store(static_cast<char*>(p.ddelta) + e, dx);
        if (has_z) {
          const float2 s = __ffma2_rn(D2, uu, r);  // the output before the gate
          PairIO<T>::store(static_cast<char*>(p.dz) + e, __fmul2_rn(s, make_float2(f.x, f.y)));
        }
        dbacc = __fadd2_rn(dbacc, dx);
      }
    }
  };

  if (tl_hi >= tl_lo) {
    issue_tile(tl_hi);
    cp_async_commit();
    load_bc(tl_hi);
    store_bc();
    load_ckpt(tl_hi, h0);
  }
  if (wait_carry) {
    // hand-over plans: the carry entering this chunk from the right is the one the next chunk
    // left at its first step; wait for its tag (bounded: a wait that runs out records code 7
    // in the status word and the walk goes on from what is there), then read it
    if (tid == 0) {
      const unsigned long long* f = p.hflags + ((b * p.n_chunks + c + 1) * n_dt + dtile);
      bool ok = false;
      unsigned ns = 32;
      for (unsigned it = 0; it < p.max_polls; it++) {
        if (ld_acquire_u64(f) == p.wait_tag) {
          ok = true;
          break;
        }
        __nanosleep(ns);
        ns = ns < 1024 ? 2 * ns : 1024;
      }
      if (!ok && p.header != nullptr) atomicMax(p.header, (p.tag << 8) | 7ull);
    }
    __syncthreads();
    if (active) {
#pragma unroll
      for (int s = 0; s < 4; s++) {
        const int cc = s / 2, n = n0 + 2 * (s % 2);
        const float* hm = p.rws_m + ((b * p.n_chunks + c + 1) * Dn + d + cc) * N;
        m[s] = make_float2(n < N ? __ldcg(hm + n) : 0.f, n + 1 < N ? __ldcg(hm + n + 1) : 0.f);
      }
    }
  }
  for (int64_t tl = tl_hi; tl >= tl_lo; tl--) {
    const int64_t ts = tl * kT;
    const int steps = (int)min((int64_t)kT, t1 - ts);
    cp_async_wait_all();
    __syncthreads();  // this tile's rows and B/C are in shared memory

    // this lane's output row base: step ts + l, channel d
    ebase = ((b * Ls + ts + l) * Dn + d) * K::kTS;
    // pre-phase: the per-element work of steps k = l (mod L)
#pragma unroll
    for (int i = 0; i < kT / L; i++) {
      const int k = i * L + l;
      const float2 xr = __fadd2_rn(PairIO<T>::load(xrow(0, i)), bias2);
      float2 spx, sgx;
      softplus_sigmoid2(xr, spx, sgx);
      float2 dt = sp ? spx : xr;
      if (k >= steps) dt = make_float2(0.f, 0.f);  // steps past the end: identity steps
      const float2 uu = PairIO<T>::load(xrow(1, i));
      const float2 dy = PairIO<T>::load(xrow(3, i));
      float2 ds = dy, zf = make_float2(0.f, 0.f);
      if (has_z) {
        const float2 zz = PairIO<T>::load(xrow(2, i));
        const float2 sz = make_float2(rcp(1.f + ex2(-zz.x * kLog2e)), rcp(1.f + ex2(-zz.y * kLog2e)));
        ds = __fmul2_rn(dy, __fmul2_rn(zz, sz));  // dy * silu(z)
        // d silu / dz = sigmoid(z) (1 + z (1 - sigmoid(z)))
        const float2 one = make_float2(1.f, 1.f);
        zf = __fmul2_rn(__fmul2_rn(dy, sz), __ffma2_rn(zz, make_float2(1.f - sz.x, 1.f - sz.y), one));
      }
      const float2 dtu = __fmul2_rn(dt, uu);
      *q_own(i, 0) = make_float4(dt.x, dt.y, dtu.x, dtu.y);
      *q_own(i, 1) = make_float4(ds.x, ds.y, uu.x, uu.y);
      own[i] = make_float4(zf.x, zf.y, sgx.x, sgx.y);
      dDacc = __ffma2_rn(ds, uu, dDacc);
    }
    __syncthreads();  // sQ complete; the staged rows are free
    if (tl > tl_lo) {
      issue_tile(tl - 1);
      cp_async_commit();
      load_bc(tl - 1);
      load_ckpt(tl - 1, h0n);
    }

    // forward recompute: the states after the odd steps to shared memory
    {
      float2 h[4];
#pragma unroll
      for (int s = 0; s < 4; s++) h[s] = h0[s];
#pragma unroll 1
      for (int k = 0; k < kT; k += 2) {
#pragma unroll
        for (int e = 0; e < 2; e++) {
          const float4 q = q_dt(k + e);
          float2 dA[4];
          decays(q, dA);
          fwd_step(q, brow(k + e), dA, h, h);
        }
        sH[((k / 2) * 2 + 0) * K::kThreads + tid] = make_float4(h[0].x, h[0].y, h[1].x, h[1].y);
        sH[((k / 2) * 2 + 1) * K::kThreads + tid] = make_float4(h[2].x, h[2].y, h[3].x, h[3].y);
      }
    }

    // reverse walk, two steps at a time: (k, k-1) with k odd
#pragma unroll
    for (int k = kT - 1; k >= 1; k -= 2) {
      float2 hk[4], hpp[4], hm[4], dAk[4], dAm[4];
      {
        const float4 a0 = sH[((k / 2) * 2 + 0) * K::kThreads + tid], a1 = sH[((k / 2) * 2 + 1) * K::kThreads + tid];
        hk[0] = make_float2(a0.x, a0.y); hk[1] = make_float2(a0.z, a0.w);
        hk[2] = make_float2(a1.x, a1.y); hk[3] = make_float2(a1.z, a1.w);
      }
      if (k >= 3) {
        const float4 a0 = sH[((k / 2 - 1) * 2 + 0) * K::kThreads + tid], a1 = sH[((k / 2 - 1) * 2 + 1) * K::kThreads + tid];
        hpp[0] = make_float2(a0.x, a0.y); hpp[1] = make_float2(a0.z, a0.w);
        hpp[2] = make_float2(a1.x, a1.y); hpp[3] = make_float2(a1.z, a1.w);
      } else {
#pragma unroll
        for (int s = 0; s < 4; s++) hpp[s] = h0[s];
      }
      const float4 qm = q_dt(k - 1);
      decays(qm, dAm);
      fwd_step(qm, brow(k - 1), dAm, hpp, hm);  // the state after step k-1
      decays(q_dt(k), dAk);
      rev_step(k, hk, hm, dAk);
      rev_step(k - 1, hm, hpp, dAm);
      if ((k - 1) % kOG == 0) {
        __syncwarp();
        if (k - 1 == kOG) output_group(std::integral_constant<int, kOG>{}, steps);
        else output_group(std::integral_constant<int, 0>{}, steps);  // k - 1 == 0
        warp_bc_sums(k - 1);
        __syncwarp();
      }
    }
    __syncthreads();  // sR complete; sBC, sH, sQ free

    // dB, dC rows of this tile: the warps' sums, added to global memory
    {
      constexpr int kGroups = kT * 2 * kNP / 4;
      if (tid < kGroups) {
        const int k = tid / (2 * kNP / 4), og = tid % (2 * kNP / 4);
        float4 acc = *reinterpret_cast<const float4*>(sR + (k * K::kWarps + 0) * 2 * kNP + 4 * og);
#pragma unroll
        for (int w = 1; w < K::kWarps; w++) {
          const float4 a2 = *reinterpret_cast<const float4*>(sR + (k * K::kWarps + w) * 2 * kNP + 4 * og);
          acc = make_float4(acc.x + a2.x, acc.y + a2.y, acc.z + a2.z, acc.w + a2.w);
        }
        const bool isC = og >= kNP / 4;
        const int nb = 4 * (isC ? og - kNP / 4 : og);
        if (k < steps && nb < N) {
          float* row = (isC ? p.dC : p.dB) + (b * Ls + ts + k) * N + nb;
          if (N % 4 == 0) {
            atomicAdd(reinterpret_cast<float4*>(row), acc);
          } else {
            const float vals[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
            for (int q = 0; q < 4; q++)
              if (nb + q < N) atomicAdd(row + q, vals[q]);
          }
        }
      }
    }
    if (tl > tl_lo) {
      store_bc();
#pragma unroll
      for (int s = 0; s < 4; s++) h0[s] = h0n[s];
    }
  }

  // per-channel sums over the lanes of the pair, then one atomic per output
#pragma unroll
  for (int o = 1; o < L; o <<= 1) {
    dDacc.x += __shfl_xor_sync(0xFFFFFFFFu, dDacc.x, o);
    dDacc.y += __shfl_xor_sync(0xFFFFFFFFu, dDacc.y, o);
    dbacc.x += __shfl_xor_sync(0xFFFFFFFFu, dbacc.x, o);
    dbacc.y += __shfl_xor_sync(0xFFFFFFFFu, dbacc.y, o);
  }
  if (p.handover && c > 0) {
    // hand the carry before this chunk's first step to the chunk before it
    if (active) {
#pragma unroll
      for (int s = 0; s < 4; s++) {
        const int cc = s / 2, n = n0 + 2 * (s % 2);
        float* hm = p.rws_m + ((b * p.n_chunks + c) * Dn + d + cc) * N;
        if (n < N) __stcg(hm + n, m[s].x);
        if (n + 1 < N) __stcg(hm + n + 1, m[s].y);
      }
    }
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      st_release_u64(p.hflags + ((b * p.n_chunks + c) * n_dt + dtile), p.tag);
    }
  }
  if (!active) return;
  if (l == 0) {
    if (p.dD) { atomicAdd(p.dD + d, dDacc.x); atomicAdd(p.dD + d + 1, dDacc.y); }
    if (p.dbias) { atomicAdd(p.dbias + d, dbacc.x); atomicAdd(p.dbias + d + 1, dbacc.y); }
  }
#pragma unroll
  for (int cc = 0; cc < 2; cc++) {
    float* row = p.dA + (d + cc) * N;
    if (N % 4 == 0) {
      if (n0 < N)
        atomicAdd(reinterpret_cast<float4*>(row + n0),
                  make_float4(dAacc[2 * cc].x, dAacc[2 * cc].y, dAacc[2 * cc + 1].x, dAacc[2 * cc + 1].y));
    } else {
#pragma unroll
      for (int j = 0; j < 2; j++) {
        const int n = n0 + 2 * j;
        if (n < N) atomicAdd(row + n, dAacc[2 * cc + j].x);
        if (n + 1 < N) atomicAdd(row + n + 1, dAacc[2 * cc + j].y);
      }
    }
  }
  if (p.dinit && tl_lo == 0) {  // the adjoint carry before step 0
#pragma unroll
    for (int cc = 0; cc < 2; cc++) {
      float* row = p.dinit + (b * Dn + d + cc) * N;
#pragma unroll
      for (int j = 0; j < 2; j++) {
        const int n = n0 + 2 * j;
        if (n < N) row[n] = m[2 * cc + j].x;
        if (n + 1 < N) row[n + 1] = m[2 * cc + j].y;
      }
    }
  }
}

}  // namespace bwd

// ---------------------------------------------------------------------------------------

static int64_t env_int(const char* name, int64_t fallback) {
  if (const char* v = std::getenv(name)) {
    const long long x = std::atoll(v);
    if (x > 0) return x;
  }
  return fallback;
}

void plan_scan_bwd(int64_t batch, int64_t L, int64_t d_inner, int sms, BwdPlan* plan) {
  plan->handover = 0;
  // Time chunks of the gradient kernel: none when its CTAs (64 channels each, about three
  // resident per SM) fill the GPU; otherwise about two waves of them, at least 64 steps per
  // chunk (measured on B300: the 2 x 2048 x 1536 shape at 0.30 ms with 16 chunks against 0.35
  // with 8 or 32; the 8 x 2048 x 5120 shape fastest unchunked).
  constexpr int64_t kAlign = 32;
  const int64_t per_chunk = batch * ((d_inner + bwd::kCh - 1) / bwd::kCh);
  const int64_t slots = (int64_t)sms * 3;
  int64_t G = 1;
  if (per_chunk > 0 && per_chunk < slots) G = (2 * slots + per_chunk - 1) / per_chunk;
  // More CTAs than one wave, but not whole waves: three chunks run as a chain (the last
  // third of the sequence first, each handing its adjoint carry to the chunk before it), which
  // needs no reverse summaries and lets the pieces fill the SMs the partial wave would leave
  // idle (8 x 2048 x 5120 x 16: 2.09 ms against 2.14 with two chunks, 2.12 with four).
  if (G == 1 && per_chunk > slots && per_chunk % slots != 0 && L >= 192) {
    G = 3;
    plan->handover = 1;
  }
  G = env_int("SSM_BWD_CHUNKS", G);  // tuning override
  if (const char* v = std::getenv("SSM_BWD_HANDOVER")) plan->handover = std::atoi(v) == 1;
  G = std::min<int64_t>(G, std::max<int64_t>(1, L / 64));
  G = std::min<int64_t>(G, 4096);
  int64_t len = L > 0 ? (L + G - 1) / G : 1;
  len = (len + kAlign - 1) / kAlign * kAlign;
  plan->chunk_len = len;
  plan->n_chunks = L > 0 ? (int)((L + len - 1) / len) : 1;
}

size_t bwd_workspace_floats(int64_t batch, int64_t L, int64_t d_inner, int d_state, int n_chunks) {
  const int64_t tiles = (L + kCkptSteps - 1) / kCkptSteps;
  const int64_t ck = batch * tiles * d_inner * d_state;                 // forward checkpoints
  const int64_t rws = batch * (int64_t)n_chunks * d_inner * (d_state + 1);  // reverse summaries
  const int64_t flags = 2 * batch * (int64_t)n_chunks * ((d_inner + bwd::kCh - 1) / bwd::kCh);  // u64 tags
  return (size_t)(ck + rws + flags);
}

template <int L, typename T>
static cudaError_t launch_grad(const BwdArgs& a, cudaStream_t s) {
  using K = bwd::Cfg<L, T>;
  const cudaError_t e = cudaFuncSetAttribute(bwd::grad_kernel<L, T>, cudaFuncAttributeMaxDynamicSharedMemorySize, K::kSmem);
  if (e != cudaSuccess) return e;
  const int64_t n_dt = (a.d_inner + bwd::kCh - 1) / bwd::kCh;
  bwd::grad_kernel<L, T><<<(unsigned)(n_dt * a.n_chunks * a.batch), K::kThreads, K::kSmem, s>>>(a);
  return cudaGetLastError();
}

template <int N, typename T>
static cudaError_t launch_bwd_t(const BwdArgs& a, const FwdLaunch& ckpt, cudaStream_t s) {
  if (a.n_chunks > 1 && !a.handover) {  // reverse chunk summaries
    const int64_t n_dtiles = (a.d_inner + kBwdCh - 1) / kBwdCh;
    bwd_reverse_summary_kernel<N, T><<<(unsigned)(n_dtiles * (a.n_chunks - 1) * a.batch), kBwdCh, 0, s>>>(a);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  // forward checkpoints: the forward scan's look-back kernel in its checkpoint form
  const cudaError_t e = launch_scan_fwd(ckpt, sizeof(T) == 2, s);
  if (e != cudaSuccess) return e;
  // lanes per channel pair: 4 states each, 4L >= d_state
  return N <= 4 ? launch_grad<1, T>(a, s) : N <= 8 ? launch_grad<2, T>(a, s) : launch_grad<4, T>(a, s);
}

template <typename T>
static cudaError_t dispatch_bwd(const BwdArgs& a, const FwdLaunch& ckpt, cudaStream_t s) {
  switch (a.d_state) {
#define SSM_BWD_CASE(NN) \
    case NN: return launch_bwd_t<NN, T>(a, ckpt, s);
    SSM_BWD_CASE(1) SSM_BWD_CASE(2) SSM_BWD_CASE(3) SSM_BWD_CASE(4)
    SSM_BWD_CASE(5) SSM_BWD_CASE(6) SSM_BWD_CASE(7) SSM_BWD_CASE(8)
    SSM_BWD_CASE(9) SSM_BWD_CASE(10) SSM_BWD_CASE(11) SSM_BWD_CASE(12)
    SSM_BWD_CASE(13) SSM_BWD_CASE(14) SSM_BWD_CASE(15) SSM_BWD_CASE(16)
#undef SSM_BWD_CASE
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_scan_bwd(const BwdArgs& a, const FwdLaunch& ckpt, bool bf16, cudaStream_t s) {
  return bf16 ? dispatch_bwd<__nv_bfloat16>(a, ckpt, s) : dispatch_bwd<float>(a, ckpt, s);
}

}  // namespace ssm
