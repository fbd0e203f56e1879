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
// Parallel structure.  One thread owns one (batch, channel) and all d_state
// states of it in registers, and walks its time chunk sequentially; a warp
// covers 32 consecutive channels, so the per-step loads of u, delta, z and
// the store of y are coalesced along d_inner, and the per-step rows B_t, C_t
// (shared by every channel) are staged once per CTA in shared memory and read
// as broadcasts.  When batch * d_inner is too small to fill the GPU, time is
// cut into chunks.  The recurrence is associative in the pairs (a, b) with
// (a2, b2) o (a1, b1) = (a2 a1, a2 b1 + b2), so a chunk is summarised by its
// decay prod_t dA_t = exp(A * sum_t delta_t) and its end state from zero.
// Pass 1 writes those summaries; pass 2 composes the summaries of the chunks
// before its own to get its start state, then runs the exact recurrence and
// writes y.  No kernel waits on another block.

#include "ssm_device.cuh"
#include "ssm_internal.h"

#include <algorithm>
#include <cstdlib>

namespace ssm {

constexpr int kScanCh = 64;    // channels (threads) per CTA
constexpr int kScanTile = 16;  // time steps per pipelined tile
constexpr int kChunkAlign = 32;

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  const int n = valid ? 16 : 0;  // n == 0: no global read, 16 zero bytes written
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
__device__ __forceinline__ void cp_async_wait_prev() { asm volatile("cp.async.wait_group 1;\n" ::); }

// One CTA: kScanCh consecutive channels of one batch row, one time chunk.
// kSummary: write the chunk's (sum of delta, end state from zero) instead of y.
//
// Per tile of kScanTile steps, the activations delta, u (and z) arrive in
// shared memory by cp.async (16-byte, coalesced along d_inner) one tile
// ahead of use, and the B/C rows of the next tile are fetched into registers
// while the current tile is computed; so no step waits on HBM latency.
template <int N, typename T, bool kSummary>
__global__ void __launch_bounds__(kScanCh)
scan_chunk_kernel(const ScanParams p) {
  constexpr int kVec = 16 / sizeof(T);            // elements per 16-byte copy
  constexpr int kCopiesPerRow = kScanCh / kVec;
  constexpr int kNX = kSummary ? 2 : 3;           // delta, u (, z)
  constexpr int kNBC = kSummary ? 1 : 2;          // B (, C)
  constexpr int kBCVals = kScanTile * N * kNBC;
  constexpr int kBCPerThread = (kBCVals + kScanCh - 1) / kScanCh;
  __shared__ __align__(16) T sX[2][kNX][kScanTile][kScanCh];
  __shared__ __align__(16) float sBC[2][kNBC][kScanTile][N];

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

  const T* __restrict__ u = static_cast<const T*>(p.u);
  const T* __restrict__ dl = static_cast<const T*>(p.delta);
  const T* __restrict__ Bg = static_cast<const T*>(p.B);
  const T* __restrict__ Cg = static_cast<const T*>(p.C);
  const T* __restrict__ zg = static_cast<const T*>(p.z);
  T* __restrict__ yg = static_cast<T*>(p.y);
  const bool has_z = !kSummary && zg != nullptr;

  auto issue_x = [&](int tile, int stage) {
    const int64_t ts = t0 + (int64_t)tile * kScanTile;
    const int nx = kSummary ? 2 : (has_z ? 3 : 2);
    for (int i = tid; i < nx * kScanTile * kCopiesPerRow; i += kScanCh) {
      const int x = i / (kScanTile * kCopiesPerRow);
      const int r = (i / kCopiesPerRow) % kScanTile;
      const int ci = i % kCopiesPerRow;
      const int64_t t = ts + r;
      const int64_t dd = d0 + (int64_t)ci * kVec;
      const bool valid = t < t1 && dd < Dn;
      const T* src = x == 0 ? dl : (x == 1 ? u : zg);
      cp_async16(&sX[stage][x][r][ci * kVec], valid ? src + (b * L + t) * Dn + dd : src, valid);
    }
  };
  float bc[kBCPerThread];
  auto load_bc = [&](int tile) {
    const int64_t ts = t0 + (int64_t)tile * kScanTile;
#pragma unroll
    for (int j = 0; j < kBCPerThread; j++) {
      const int i = tid + j * kScanCh;
      float v = 0.f;
      if (i < kBCVals) {
        const int which = i / (kScanTile * N), r = (i / N) % kScanTile, n = i % N;
        const int64_t t = ts + r;
        if (t < t1) v = to_f32((which ? Cg : Bg)[(b * L + t) * N + n]);
      }
      bc[j] = v;
    }
  };
  auto store_bc = [&](int stage) {
#pragma unroll
    for (int j = 0; j < kBCPerThread; j++) {
      const int i = tid + j * kScanCh;
      if (i < kBCVals) sBC[stage][i / (kScanTile * N)][(i / N) % kScanTile][i % N] = bc[j];
    }
  };

  float A2[N], h[N];
#pragma unroll
  for (int n = 0; n < N; n++) {
    A2[n] = active ? p.A[d * N + n] * kLog2e : 0.f;  // exp(x) = 2^(x log2 e)
    h[n] = 0.f;
  }
  const float Dd = (active && p.D) ? p.D[d] : 0.f;
  const float bias = (active && p.delta_bias) ? p.delta_bias[d] : 0.f;
  const bool sp = p.softplus != 0;

  if (ntiles > 0) {
    issue_x(0, 0);
    cp_async_commit();
    load_bc(0);
    store_bc(0);
  }

  if (!kSummary && c > 0 && active) {
    // Start state of chunk c: fold the summaries of chunks 0 .. c-1 in order.
    const int64_t base = b * (p.n_chunks - 1);
    for (int j = 0; j < c; j++) {
      const float S = p.ws_S[(base + j) * Dn + d];
      const float* hj = p.ws_h + ((base + j) * Dn + d) * N;
#pragma unroll
      for (int n = 0; n < N; n++) h[n] = fmaf(ex2(A2[n] * S), h[n], hj[n]);
    }
  }

  float S = 0.f, S_comp = 0.f;  // compensated (Kahan) sum of delta over the chunk

  // One time step of the recurrence for this thread's channel.
  auto step = [&](int stage, int k, int64_t t) {
    const float x = to_f32(sX[stage][0][k][tid]) + bias;
    const float dt = sp ? softplus(x) : x;
    const float uu = to_f32(sX[stage][1][k][tid]);
    const float w = dt * uu;
    if (kSummary) {
      const float yk = dt - S_comp;
      const float tk = S + yk;
      S_comp = (tk - S) - yk;
      S = tk;
    }
    const float* Bk = sBC[stage][0][k];
    float acc = 0.f;
#pragma unroll
    for (int n = 0; n < N; n++) {
      const float dA = ex2(dt * A2[n]);
      h[n] = fmaf(dA, h[n], w * Bk[n]);
      if (!kSummary) acc = fmaf(sBC[stage][kNBC - 1][k][n], h[n], acc);
    }
    if (!kSummary) {
      acc = fmaf(Dd, uu, acc);
      if (has_z) acc *= silu(to_f32(sX[stage][kNX - 1][k][tid]));
      yg[(b * L + t) * Dn + d] = from_f32<T>(acc);
    }
  };

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
    if (active) {
      if (ts + kScanTile <= t1) {
#pragma unroll 4
        for (int k = 0; k < kScanTile; k++) step(stage, k, ts + k);
      } else {
        const int steps = (int)(t1 - ts);
        for (int k = 0; k < steps; k++) step(stage, k, ts + k);
      }
    }
    __syncthreads();  // stage is free for the tile after next
    if (tile + 1 < ntiles) store_bc(stage ^ 1);
  }

  if (!active) return;
  if (kSummary) {
    const int64_t slot = (b * (p.n_chunks - 1) + c) * Dn + d;
    p.ws_S[slot] = S;
#pragma unroll
    for (int n = 0; n < N; n++) p.ws_h[slot * N + n] = h[n];
  } else if (c == p.n_chunks - 1 && p.last_state) {
#pragma unroll
    for (int n = 0; n < N; n++) p.last_state[(b * Dn + d) * N + n] = h[n];
  }
}

int scan_channels_per_cta() { return kScanCh; }

void plan_scan_chunks(int64_t batch, int64_t L, int64_t d_inner, int sms, int64_t* chunk_len,
                      int* n_chunks) {
  // Aim for at least `target` resident threads (channels x chunks); chunking
  // costs a second pass over all but the last chunk, so split only when the
  // channels alone leave the GPU short of warps.
  int64_t target_threads_per_sm = 256;
  if (const char* env = std::getenv("SSM_SCAN_THREADS_PER_SM")) {
    const long v = std::atol(env);
    if (v > 0) target_threads_per_sm = v;
  }
  const int64_t channels = batch * d_inner;
  const int64_t target = (int64_t)sms * target_threads_per_sm;
  int64_t G = 1;
  if (channels > 0 && channels < target) G = (target + channels - 1) / channels;
  const int64_t min_chunk = 64;
  G = std::min<int64_t>(G, std::max<int64_t>(1, L / min_chunk));
  G = std::min<int64_t>(G, 4096);
  int64_t len = L > 0 ? (L + G - 1) / G : 1;
  len = (len + kChunkAlign - 1) / kChunkAlign * kChunkAlign;
  *chunk_len = len;
  *n_chunks = L > 0 ? (int)((L + len - 1) / len) : 1;
}

template <int N, typename T>
static cudaError_t launch_scan_t(const ScanParams& p, cudaStream_t stream) {
  const int64_t n_dtiles = (p.d_inner + kScanCh - 1) / kScanCh;
  if (p.n_chunks > 1) {
    const int64_t blocks = n_dtiles * (p.n_chunks - 1) * p.batch;
    scan_chunk_kernel<N, T, true><<<(unsigned)blocks, kScanCh, 0, stream>>>(p);
  }
  const int64_t blocks = n_dtiles * p.n_chunks * p.batch;
  scan_chunk_kernel<N, T, false><<<(unsigned)blocks, kScanCh, 0, stream>>>(p);
  return cudaGetLastError();
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

cudaError_t launch_scan(const ScanParams& p, bool bf16, cudaStream_t stream) {
  return bf16 ? dispatch_n<__nv_bfloat16>(p, stream) : dispatch_n<float>(p, stream);
}

}  // namespace ssm
