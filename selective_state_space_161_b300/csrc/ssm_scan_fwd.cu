// Selective-scan forward in one pass: the softplus step size, the discretisation
// dA = exp(delta*A), dBu = delta*B*u, the recurrence h_t = dA_t h_{t-1} + dBu_t over
// (batch, d_inner, d_state), the readout y_t = C_t.h_t + D u_t and the SiLU(z) gate,
// with time chunks joined by a decoupled look-back.
//
// Sources (page title, section): youngju.dev "Mamba: Linear-Time Sequence Modeling with
// Selective State Spaces 论文分析", "解决方案：Kernel Fusion + Recomputation" (discretise,
// recur, read out with the updated state; nothing intermediate goes to HBM) and
// "Mamba 模块架构" (D, the SiLU gate, the biased step-size projection); ai-lab.club
// "机器学习基础算法", discrete state equations; the chunk carry is the associative form of
// the recurrence that "Mamba一作最新大發長文！", "(3) 訓練效率", and "看懂Mamba…", "3. 状态空间",
// describe as a parallel scan.
//
// Work layout.  A CTA covers 64 consecutive channels of one batch row over one time chunk.
// Each thread owns two adjacent channels (d, d+1) and S of the states of both; the L lanes
// of a channel pair (L = 1, 2 or 4) split the pair's L*S states, so a state update is one
// packed fp32x2 operation on (channel d, channel d+1).  Per tile of 16 steps:
//  - delta, u, z rows (64 channels) arrive in shared memory by cp.async, one tile ahead,
//    in 16-byte pieces whose position is XOR-swizzled by the row so that the lanes of a
//    warp, which read L different rows at once, hit distinct banks;
//  - B_t, C_t rows (shared by every channel) are fetched a tile ahead into registers and
//    stored as fp32 in shared memory;
//  - pre-phase: lane l of a pair computes the per-element work of the steps k = l (mod L)
//    once (step size, delta*u, the gate, D*u*gate) and leaves it in shared memory;
//  - recurrence: every lane runs all steps on its S states; for L > 1 the partial readouts
//    go through shared memory and lane l sums them for its own steps and writes y.
//
// Time chunks.  When batch * d_inner cannot fill the GPU, the sequence is cut into G
// chunks, one CTA per (chunk, batch row, channel tile), all resident at once.  The
// recurrence is associative in (a, b) with (a2, b2) o (a1, b1) = (a2 a1, a2 b1 + b2), and a
// chunk's decay prod_t exp(delta_t A) equals exp(A sum_t delta_t).  A CTA of a middle chunk
// first runs its chunk from a zero state (no readout) and publishes the aggregate
// (sum of delta, end state); then it looks back over its predecessors' records, newest
// first, folding aggregates until it meets an inclusive prefix (the true state at the end of
// that chunk), publishes its own inclusive prefix and runs its chunk again from the true
// carry, now with the readout.  Chunk 0 starts from the initial state at once and publishes
// its inclusive prefix at its end (it is shorter than the others, so that it finishes about
// when they finish their aggregates); the last chunk skips the aggregate.  Records carry a
// per-call tag, so a workspace needs no clearing.  CTAs are numbered chunk-major, so every
// CTA a CTA waits for was dispatched before it.  Waits are bounded: a CTA that polls too
// long records SSM_ERR_LOOKBACK_TIMEOUT in the workspace header, carries on with what it
// has and never hangs.

#include "ssm_device.cuh"
#include "ssm_internal.h"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <type_traits>

#ifndef SSM_FWD_UNROLL
#define SSM_FWD_UNROLL 4
#endif

namespace ssm {
namespace fwd {

constexpr int kStepUnroll = SSM_FWD_UNROLL;  // steps per iteration of the one-lane step loop

constexpr int kCh = 64;   // channels per CTA
constexpr int kCP = 32;   // channel pairs per CTA
constexpr int kT = 16;    // steps per tile
static_assert(kT == 2 * kCkptSteps, "two checkpoints per tile");
constexpr int kModeAgg = 0, kModeMain = 1;

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  const int n = valid ? 16 : 0;  // n == 0: no global read, 16 zero bytes written
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
__device__ __forceinline__ void cp_async_wait_prev() { asm volatile("cp.async.wait_group 1;\n" ::); }

__device__ __forceinline__ unsigned long long ld_acquire(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ float2 sub2(float2 a, float2 b) { return make_float2(a.x - b.x, a.y - b.y); }

// A channel pair of the I/O dtype <-> two fp32 values.
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

template <int L, int S, typename T, bool kConv>
struct Cfg {
  static constexpr int kHalo = kConv ? 3 : 0;         // rows before the tile (conv window)
  static constexpr int kRows = kT + kHalo;
  static constexpr int kThreads = 32 * L;
  static constexpr int kNP = L * S;                  // states held per pair (>= d_state; padding is 0)
  static constexpr int kTS = (int)sizeof(T);
  static constexpr int kRowB = kCh * kTS;             // one activation row of the CTA's channels
  static constexpr int kChunks = kRowB / 16;          // 16-byte pieces per row
  static constexpr int kPairB = 2 * kTS;
  static constexpr int kSwz = 8 / L;                  // row swizzle step (pieces / float4 slots)
  static constexpr int kLS = L == 4 ? 72 : L == 2 ? 80 : 64;     // partial buffer: lane stride (floats)
  static constexpr int kRS = L == 4 ? 296 : L == 2 ? 176 : 64;   // partial buffer: row stride (floats)
  static constexpr int kAggF = (2 + 2 * S + 3) / 4 * 4;  // floats per thread of an aggregate record
  static constexpr int kInclF = 2 * S;                    // floats per thread of an inclusive record
  // One stage of activation rows: delta (kT rows), u or the conv input (kRows rows: the kHalo
  // rows before the tile first), z (kT rows).
  static constexpr int kOffU = kT * kRowB;
  static constexpr int kOffZ = (kT + kRows) * kRowB;
  static constexpr int kStageB = (2 * kT + kRows) * kRowB;
  static constexpr int kXB = 2 * kStageB;
  static constexpr int kBCB = 2 * 2 * kT * kNP * 4;
  static constexpr int kDWB = L > 1 ? kT * kCP * 16 : 0;  // (delta, delta*u) pairs per step (L > 1)
  // steps per output group (partial readouts reduced in shared memory): 8, or 4 for fp32 I/O
  // on four lanes, whose larger staging tiles would otherwise allow only 4 CTAs per SM, not 5
  static constexpr int kOG = (kTS == 4 && L == 4) ? 4 : 8;
  static constexpr int kPB = L > 1 ? kOG * kRS * 4 : 0;    // partial readouts per step group (L > 1)
  static constexpr int kSmem = kXB + kBCB + kDWB + kPB + 16;
  static_assert(S % 4 == 0 && kNP <= 16, "states per lane must be a multiple of 4, at most 16 per pair");
};

struct Args {
  const void* u;
  const void* delta;
  const float* A;
  const void* B;
  const void* C;
  const float* D;
  const void* z;
  const float* delta_bias;
  int softplus;
  void* y;
  float* last_state;
  const float* initial_state;
  const float* conv_w;          // [d_inner][d_conv] (conv kernels only)
  const float* conv_b;          // [d_inner], may be null
  int d_conv;
  void* u_out;                  // may be null: the conv output u, I/O dtype
  float* ckpt;                  // checkpoint kernels: [batch][ceil(L/kCkptSteps)][d_inner][d_state]
  int64_t batch, L, d_inner;
  int N;
  int G;                        // time chunks
  int chain;                    // 1: no aggregates; every chunk continues from its predecessor's end state
  int64_t len0, len;            // length of chunk 0, of the others (the last may be shorter)
  unsigned long long* header;   // status word: (tag << 8) | error code
  unsigned long long* flags;    // [G-1][batch][channel tiles]: (tag << 2) | 1 aggregate, 2 inclusive
  float* agg;                   // aggregate records (per thread: sum of delta pair, end states from zero)
  float* incl;                  // inclusive records (per thread: true end states)
  unsigned long long tag;       // this call's tag (54 bits)
  unsigned long long wait_tag;  // the tag look-back accepts (== tag except in the wait self-test)
  unsigned max_polls;           // look-back polls before giving up
};

// Register allocation: 12 resident warps per SM for one lane per pair (three per scheduler,
// up to 168 registers: its 16 state pairs, A and B/C live at once), 16 for two lanes, 20 for
// four.
// kCkpt: the backward pass's checkpoint kernel.  The same chunks and look-back, but its last
// pass stores the state before every kCkptSteps steps instead of reading out y (no C, no
// z, no outputs).
template <int L, int S, typename T, bool kConv, bool kCkpt = false>
__global__ void __launch_bounds__(32 * L, L == 1 ? 12 : (L == 2 ? 8 : 5)) scan_fwd_kernel(const Args a) {
  static_assert(!(kConv && kCkpt), "the checkpoint kernels take the scan input u directly");
  using K = Cfg<L, S, T, kConv>;
  extern __shared__ __align__(16) unsigned char smem[];
  unsigned char* sX = smem;                                                  // [2][kStageB]
  float* sBC = reinterpret_cast<float*>(smem + K::kXB);                      // [2][2][kT][kNP]
  float4* sDW = reinterpret_cast<float4*>(smem + K::kXB + K::kBCB);          // [kT][kCP]
  float* sP = reinterpret_cast<float*>(smem + K::kXB + K::kBCB + K::kDWB);    // [K::kOG][kRS]
  int* sInfo = reinterpret_cast<int*>(smem + K::kXB + K::kBCB + K::kDWB + K::kPB);

  const int64_t Dn = a.d_inner, Ls = a.L;
  const int N = a.N;
  const int64_t n_dt = (Dn + kCh - 1) / kCh;
  int64_t blk = blockIdx.x;
  const int64_t dtile = blk % n_dt;
  blk /= n_dt;
  const int64_t b = blk % a.batch;
  const int c = (int)(blk / a.batch);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int l = lane % L;                       // this lane's share of the pair's states
  const int P = warp * (32 / L) + lane / L;     // channel pair within the CTA
  const int64_t d0 = dtile * kCh;
  const int64_t d = d0 + 2 * P;                 // first channel of the pair (d_inner is even)
  const bool active = d < Dn;
  const int64_t t0 = c == 0 ? 0 : a.len0 + (int64_t)(c - 1) * a.len;
  const int64_t t1 = min(t0 + (c == 0 ? a.len0 : a.len), Ls);
  const int ntiles = (int)((t1 - t0 + kT - 1) / kT);
  const int64_t rec = ((int64_t)c * a.batch + b) * n_dt + dtile;  // record of this chunk (c < G-1)

  if (blockIdx.x == 0 && tid == 0 && a.header != nullptr) atomicExch(a.header, a.tag << 8);

  // Per-lane constants: A * log2(e) for the lane's states (0 for padding states and inactive
  // channels).  Index s = c * (S/2) + j holds channel d + c, states n0 + 2j and n0 + 2j + 1 as
  // one fp32 pair, so that a state pair meets a (B_n, B_n+1) or (C_n, C_n+1) pair read
  // straight from shared memory.
  constexpr int kHP = S / 2;  // state pairs per channel
  const int n0 = S * l;
  float2 A2[S], h[S];
#pragma unroll
  for (int s = 0; s < S; s++) {
    const int c = s / kHP, n = n0 + 2 * (s % kHP);
    const float* Ar = a.A + (d + c) * N;
    A2[s] = make_float2((active && n < N) ? Ar[n] * kLog2e : 0.f, (active && n + 1 < N) ? Ar[n + 1] * kLog2e : 0.f);
    h[s] = make_float2(0.f, 0.f);
  }
  const float2 bias2 = (active && a.delta_bias) ? make_float2(a.delta_bias[d], a.delta_bias[d + 1])
                                                : make_float2(0.f, 0.f);
  const float2 D2 = (active && a.D) ? make_float2(a.D[d], a.D[d + 1]) : make_float2(0.f, 0.f);
  const bool sp = a.softplus != 0;
  const bool has_z = a.z != nullptr;

  // Padding state columns of the B/C tiles read as zero (the tile stores never touch them).
  if (K::kNP > N) {
    for (int i = tid; i < 2 * 2 * kT * (K::kNP - N); i += K::kThreads)
      sBC[(i / (K::kNP - N)) * K::kNP + N + i % (K::kNP - N)] = 0.f;
  }

  // This pair's 16-byte piece of an activation row, and its byte offset within the piece.
  const int pchunk = (P * K::kPairB) / 16, pwithin = (P * K::kPairB) % 16;
  // Causal conv1d taps (kConv): cw[j] multiplies x[t - 3 + j]; shorter kernels get leading
  // zero taps.
  float2 cw[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  float2 cb2 = make_float2(0.f, 0.f);
  if constexpr (kConv) {
    if (active) {
      const int Kc = a.d_conv;
#pragma unroll
      for (int j = 0; j < 4; j++)
        if (j >= 4 - Kc) cw[j] = make_float2(a.conv_w[d * Kc + j - (4 - Kc)], a.conv_w[(d + 1) * Kc + j - (4 - Kc)]);
      if (a.conv_b) cb2 = make_float2(a.conv_b[d], a.conv_b[d + 1]);
    }
  }
  const char* xd = static_cast<const char*>(a.delta);
  const char* xu = static_cast<const char*>(a.u);
  const char* xz = static_cast<const char*>(a.z);
  const T* __restrict__ Bg = static_cast<const T*>(a.B);
  const T* __restrict__ Cg = static_cast<const T*>(a.C);

  // One pass over the chunk: kMode == kModeAgg runs from the current h without readout
  // and sums delta; kModeMain runs from the current h and writes y.
  float2 Ssum = make_float2(0.f, 0.f), Scomp = make_float2(0.f, 0.f);
  auto run = [&](auto mode_tag) {
    constexpr int kMode = decltype(mode_tag)::value;
    constexpr bool kMain = kMode == kModeMain && !kCkpt;  // the pass that reads out y
    constexpr bool kStore = kMode == kModeMain && kCkpt;  // the pass that stores checkpoints
    const int nbc = kMain ? 2 : 1;

    // Activation rows of a tile: delta and z (kT rows), u or the conv input x (kRows rows,
    // the kHalo rows before the tile first); 16-byte piece ch of row r of an array lands at
    // piece ch ^ ((r % L) * kSwz).
    auto issue_rows = [&](auto rows_tag, const char* base, int off, int64_t tfirst) {
      constexpr int kR = decltype(rows_tag)::value;
      constexpr int kPieces = kR * K::kChunks;
      const char* g0 = base + ((b * Ls + tfirst) * Dn + d0) * K::kTS;  // row tfirst, channel d0
      const int64_t row_bytes = Dn * K::kTS;
#pragma unroll
      for (int j = 0; j < (kPieces + K::kThreads - 1) / K::kThreads; j++) {
        const int q = tid + j * K::kThreads;
        if (kPieces % K::kThreads == 0 || q < kPieces) {
          const int r = q / K::kChunks, ch = q % K::kChunks;  // kChunks is a power of two
          const int64_t t = tfirst + r;
          const bool valid = t >= 0 && t < t1 && d0 + ch * (16 / K::kTS) < Dn;
          const char* g = g0 + r * row_bytes + ch * 16;
          cp_async16(sX + off + r * K::kRowB + ((ch ^ ((r % L) * K::kSwz)) * 16), valid ? g : base, valid);
        }
      }
    };
    auto issue_x = [&](int tile, int stage) {
      const int64_t ts = t0 + (int64_t)tile * kT;
      const int so = stage * K::kStageB;
      issue_rows(std::integral_constant<int, kT>{}, xd, so, ts);
      issue_rows(std::integral_constant<int, K::kRows>{}, xu, so + K::kOffU, ts - K::kHalo);
      if (kMain && has_z) issue_rows(std::integral_constant<int, kT>{}, xz, so + K::kOffZ, ts);
    };

    // B/C rows of a tile: global -> registers (a tile ahead) -> fp32 shared memory.  Which
    // elements a thread moves is the same for every tile; their offsets are worked out once.
    constexpr int kVec = 16 / K::kTS;
    constexpr int kMaxEl = 2 * kT * K::kNP;
    constexpr int kVecPT = (kMaxEl / kVec + K::kThreads - 1) / K::kThreads;
    constexpr int kScPT = (kMaxEl + K::kThreads - 1) / K::kThreads;
    const bool vec_bc = (N * K::kTS) % 16 == 0;
    const int bc_el = nbc * kT * N;
    // vector path (d_state a multiple of 16 bytes): per-thread offsets fixed for every tile
    int bc_src[kVecPT], bc_dst[kVecPT], bc_row[kVecPT];  // element in the B (or C) rows, smem slot, row
    bool bc_isC[kVecPT];
#pragma unroll
    for (int j = 0; j < kVecPT; j++) {
      const int e = (tid + j * K::kThreads) * kVec;
      const int which = e / (kT * N), ew = e % (kT * N);
      const bool ok = vec_bc && e < bc_el;
      bc_src[j] = ew;
      bc_row[j] = ok ? ew / N : kT;  // kT: never loaded
      bc_dst[j] = ok ? ((which * kT + ew / N) * K::kNP + ew % N) : -1;
      bc_isC[j] = which != 0;
    }
    uint4 bcv[kVecPT];
    float bcs[kScPT];
    auto load_bc = [&](int tile) {
      const int64_t ts = t0 + (int64_t)tile * kT;
      const int64_t e0 = (b * Ls + ts) * N;
      const int64_t rows_left = t1 - ts;
      if (vec_bc) {
#pragma unroll
        for (int j = 0; j < kVecPT; j++) {
          bcv[j] = make_uint4(0, 0, 0, 0);
          if (bc_row[j] < rows_left) bcv[j] = __ldg(reinterpret_cast<const uint4*>((bc_isC[j] ? Cg : Bg) + e0 + bc_src[j]));
        }
      } else {
#pragma unroll
        for (int j = 0; j < kScPT; j++) {  // any d_state: element by element
          const int e = tid + j * K::kThreads;
          const int which = e / (kT * N), ew = e % (kT * N);
          bcs[j] = 0.f;
          if (e < bc_el && ew / N < rows_left) bcs[j] = to_f32((which ? Cg : Bg)[e0 + ew]);
        }
      }
    };
    auto store_bc = [&](int stage) {
      float* base = sBC + stage * 2 * kT * K::kNP;
      if (vec_bc) {
#pragma unroll
        for (int j = 0; j < kVecPT; j++) {
          if (bc_dst[j] >= 0) {
            float* dst = base + bc_dst[j];
            const uint4 v = bcv[j];
            if constexpr (K::kTS == 4) {
              *reinterpret_cast<float4*>(dst) = make_float4(__uint_as_float(v.x), __uint_as_float(v.y),
                                                            __uint_as_float(v.z), __uint_as_float(v.w));
            } else {
              const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
              for (int m = 0; m < 2; m++)
                *reinterpret_cast<float4*>(dst + 4 * m) = make_float4(
                    __uint_as_float(w4[2 * m] << 16), __uint_as_float(w4[2 * m] & 0xFFFF0000u),
                    __uint_as_float(w4[2 * m + 1] << 16), __uint_as_float(w4[2 * m + 1] & 0xFFFF0000u));
            }
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < kScPT; j++) {
          const int e = tid + j * K::kThreads;
          if (e < bc_el) {
            const int which = e / (kT * N), ew = e % (kT * N);
            base[(which * kT + ew / N) * K::kNP + ew % N] = bcs[j];
          }
        }
      }
    };

    T* __restrict__ yg = static_cast<T*>(a.y);
    if (ntiles > 0) {
      issue_x(0, 0);
      cp_async_commit();
      load_bc(0);
      store_bc(0);
    }
    for (int tile = 0; tile < ntiles; tile++) {
      const int stage = tile & 1;
      if (tile + 1 < ntiles) {
        issue_x(tile + 1, stage ^ 1);
        load_bc(tile + 1);
      }
      cp_async_commit();
      cp_async_wait_prev();  // this tile's pieces have landed (only the newest group may pend)
      __syncthreads();
      const int64_t ts = t0 + (int64_t)tile * kT;
      const int steps = (int)min((int64_t)kT, t1 - ts);
      // checkpoint kernels: this lane's states of both channels, the state before step t
      auto store_ckpt = [&](int64_t t) {
        if (!active) return;
        const int64_t row0 = (b * ((Ls + kCkptSteps - 1) / kCkptSteps) + t / kCkptSteps) * Dn + d;
#pragma unroll
        for (int c = 0; c < 2; c++) {
          float* dst = a.ckpt + (row0 + c) * N + n0;
#pragma unroll
          for (int q = 0; q < S / 4; q++) {
            const float2 h0 = h[c * kHP + 2 * q], h1 = h[c * kHP + 2 * q + 1];
            const int n = n0 + 4 * q;
            if (N % 4 == 0) {
              if (n < N) *reinterpret_cast<float4*>(dst + 4 * q) = make_float4(h0.x, h0.y, h1.x, h1.y);
            } else {
              const float v[4] = {h0.x, h0.y, h1.x, h1.y};
#pragma unroll
              for (int e = 0; e < 4; e++)
                if (n + e < N) dst[4 * q + e] = v[e];
            }
          }
        }
      };
      if constexpr (kStore) store_ckpt(ts);

      // The per-element work of step k for this lane's channel pair (step size, delta*u, and
      // for the main pass the gate and D*u*gate), from the staged rows of stage `stage`.
      auto element = [&](int k, float2& dlt, float2& w, float2& g, float2& dug) {
        auto xrow = [&](int off, int r) {  // this pair's bytes in row r of the array at off
          return sX + stage * K::kStageB + off + r * K::kRowB + (((pchunk ^ ((r % L) * K::kSwz)) * 16) + pwithin);
        };
        const int ku = k + K::kHalo;  // row of step k in the u (conv input) array
        const float2 xr = __fadd2_rn(PairIO<T>::load(xrow(0, k)), bias2);
        const float2 spx = softplus2(xr);  // computed either way, selected without a branch
        dlt = make_float2(sp ? spx.x : xr.x, sp ? spx.y : xr.y);
        float2 uu = PairIO<T>::load(xrow(K::kOffU, ku));
        if constexpr (kConv) {  // u = silu(conv_b + sum_j cw[j] x[t - 3 + j])
          float2 pre = __ffma2_rn(cw[3], uu, cb2);
          pre = __ffma2_rn(cw[2], PairIO<T>::load(xrow(K::kOffU, ku - 1)), pre);
          pre = __ffma2_rn(cw[1], PairIO<T>::load(xrow(K::kOffU, ku - 2)), pre);
          pre = __ffma2_rn(cw[0], PairIO<T>::load(xrow(K::kOffU, ku - 3)), pre);
          uu = silu2(pre);
          if (kMain && a.u_out != nullptr && active && k < steps)
            PairIO<T>::store(static_cast<T*>(a.u_out) + (b * Ls + ts + k) * Dn + d, uu);
        }
        w = __fmul2_rn(dlt, uu);
        if constexpr (kMain) {
          // without z the row was never staged; silu of whatever it holds is computed and
          // discarded by the select
          const float2 sz = silu2(PairIO<T>::load(xrow(K::kOffZ, k)));
          g = make_float2(has_z ? sz.x : 1.f, has_z ? sz.y : 1.f);
          dug = __fmul2_rn(__fmul2_rn(D2, uu), g);
        } else if (kMode == kModeAgg && k < steps) {  // compensated (Kahan) sum of delta over the chunk
          const float2 yk = sub2(dlt, Scomp);
          const float2 tk = make_float2(Ssum.x + yk.x, Ssum.y + yk.y);
          Scomp = sub2(sub2(tk, Ssum), yk);
          Ssum = tk;
        }
      };

      // One recurrence step on this lane's S states of the pair; returns the partial readout
      // (main pass), summed over independent accumulators to keep the chains short.
      auto advance = [&](int k, float2 dt2, float2 w2) {
        constexpr int kAcc = S >= 8 ? 2 : 1;  // accumulators per channel
        const float* Bk = sBC + ((stage * 2 + 0) * kT + k) * K::kNP + n0;
        const float* Ck = sBC + ((stage * 2 + 1) * kT + k) * K::kNP + n0;
        float2 acc[2][kAcc];
#pragma unroll
        for (int c = 0; c < 2; c++)
#pragma unroll
          for (int m = 0; m < kAcc; m++) acc[c][m] = make_float2(0.f, 0.f);
#pragma unroll
        for (int q = 0; q < S / 4; q++) {
          const float4 b4 = *reinterpret_cast<const float4*>(Bk + 4 * q);
          const float2 bp[2] = {make_float2(b4.x, b4.y), make_float2(b4.z, b4.w)};
          float2 cp[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
          if constexpr (kMain) {
            const float4 c4 = *reinterpret_cast<const float4*>(Ck + 4 * q);
            cp[0] = make_float2(c4.x, c4.y);
            cp[1] = make_float2(c4.z, c4.w);
          }
#pragma unroll
          for (int c = 0; c < 2; c++) {
            const float2 dtc = c ? make_float2(dt2.y, dt2.y) : make_float2(dt2.x, dt2.x);
            const float2 wc = c ? make_float2(w2.y, w2.y) : make_float2(w2.x, w2.x);
#pragma unroll
            for (int e = 0; e < 2; e++) {
              const int j = 2 * q + e, s = c * kHP + j;
              const float2 xa = __fmul2_rn(dtc, A2[s]);
              const float2 dA = make_float2(ex2(xa.x), ex2(xa.y));
              h[s] = __ffma2_rn(dA, h[s], __fmul2_rn(wc, bp[e]));
              if constexpr (kMain) acc[c][j % kAcc] = __ffma2_rn(cp[e], h[s], acc[c][j % kAcc]);
            }
          }
        }
        float2 r[2];
#pragma unroll
        for (int c = 0; c < 2; c++) {
#pragma unroll
          for (int m = 1; m < kAcc; m++) acc[c][0] = __fadd2_rn(acc[c][0], acc[c][m]);
          r[c] = acc[c][0];
        }
        return make_float2(r[0].x + r[0].y, r[1].x + r[1].y);
      };

      if constexpr (L == 1) {
        // One lane owns the pair and all of its states: the per-element work inline, step by step.
        T* yk = yg + (b * Ls + ts) * Dn + d;  // y of step k, advanced by one row per step
        auto step1 = [&](int k) {
          float2 dlt, w, g, dug;
          element(k, dlt, w, g, dug);
          const float2 part = advance(k, dlt, w);
          if constexpr (kMain) {
            if (active) PairIO<T>::store(yk, __ffma2_rn(part, g, dug));
            yk += Dn;
          }
          if constexpr (kStore) {
            if (k == kCkptSteps - 1 && steps > kCkptSteps) store_ckpt(ts + kCkptSteps);
          }
        };
        // Four steps per loop iteration: enough independent work for the scheduler, and code
        // small enough to stay in the instruction cache (a fully unrolled tile does not).
        if (steps == kT) {
#pragma unroll kStepUnroll
          for (int k = 0; k < kT; k++) step1(k);
        } else {
          for (int k = 0; k < steps; k++) step1(k);
        }
      } else {
        // Pre-phase: lane l does the per-element work of the steps k = l (mod L) once and leaves
        // (delta, delta*u) in shared memory for the pair's L lanes; it keeps (gate, D*u*gate) of
        // its own steps in registers for their outputs.
        float4 gd[kT / L];
#pragma unroll
        for (int i = 0; i < kT / L; i++) {
          const int k = i * L + l;
          float2 dlt, w, g, dug;
          element(k, dlt, w, g, dug);
          sDW[k * kCP + (P ^ (l * K::kSwz))] = make_float4(dlt.x, dlt.y, w.x, w.y);
          gd[i] = make_float4(g.x, g.y, dug.x, dug.y);
        }
        __syncwarp();

        // Output of the steps k0 .. k0+K::kOG-1: lane l sums the partial readouts of its own steps
        // over the pair's L lanes and applies the skip term and the gate.
        auto output_group = [&](int k0) {
#pragma unroll
          for (int i = 0; i < K::kOG / L; i++) {
            const int k = k0 + i * L + l;
            if (k < steps && active) {
              const float* pr = sP + (k - k0) * K::kRS + 2 * P;
              float2 sum = *reinterpret_cast<const float2*>(pr);
#pragma unroll
              for (int m = 1; m < L; m++) sum = __fadd2_rn(sum, *reinterpret_cast<const float2*>(pr + m * K::kLS));
              const float4 q = gd[k0 / L + i];
              PairIO<T>::store(yg + (b * Ls + ts + k) * Dn + d,
                               __ffma2_rn(sum, make_float2(q.x, q.y), make_float2(q.z, q.w)));
            }
          }
        };

        // Recurrence over the tile's steps on this lane's states.
        auto recur = [&](auto guarded) {
          constexpr bool kGuard = decltype(guarded)::value;
#pragma unroll
          for (int k = 0; k < kT; k++) {
            if (kGuard && k >= steps) break;
            const float4 dw = sDW[k * kCP + (P ^ ((k % L) * K::kSwz))];
            const float2 part = advance(k, make_float2(dw.x, dw.y), make_float2(dw.z, dw.w));
            if constexpr (kStore) {
              if (k == kCkptSteps - 1 && steps > kCkptSteps) store_ckpt(ts + kCkptSteps);
            }
            if constexpr (kMain) {
              *reinterpret_cast<float2*>(sP + (k % K::kOG) * K::kRS + l * K::kLS + 2 * P) = part;
              if (k % K::kOG == K::kOG - 1 || (kGuard && k == steps - 1)) {
                __syncwarp();
                output_group(k - k % K::kOG);
                __syncwarp();
              }
            }
          }
        };
        if (steps == kT) recur(std::false_type{});
        else recur(std::true_type{});
      }
      __syncthreads();  // this stage and the per-tile buffers are free again
      if (tile + 1 < ntiles) store_bc(stage ^ 1);
    }
  };

  const bool chunked = a.G > 1;
  const bool last_chunk = c == a.G - 1;
  // a chain of chunks (the four-lane plain and checkpoint kernels only): no aggregate pass;
  // every chunk waits for its predecessor's end state, published when its main pass ends
  const bool chain = !kConv && L == 4 && a.chain != 0;
  float2 S2 = make_float2(0.f, 0.f);  // sum of delta over this chunk (aggregate pass)
  float2 hagg[S];
#pragma unroll
  for (int s = 0; s < S; s++) hagg[s] = make_float2(0.f, 0.f);

  if (c > 0 && !last_chunk && !chain) {
    // Aggregate: the chunk from a zero state, published for the chunks after it.
    run(std::integral_constant<int, kModeAgg>{});
    S2 = sub2(Ssum, Scomp);
#pragma unroll
    for (int m = 1; m < L; m <<= 1)
      S2 = make_float2(S2.x + __shfl_xor_sync(0xFFFFFFFFu, S2.x, m), S2.y + __shfl_xor_sync(0xFFFFFFFFu, S2.y, m));
    float* dst = a.agg + (rec * K::kThreads + tid) * K::kAggF;
    float v[K::kAggF];
    v[0] = S2.x;
    v[1] = S2.y;
#pragma unroll
    for (int s = 0; s < S; s++) { v[2 + 2 * s] = h[s].x; v[3 + 2 * s] = h[s].y; hagg[s] = h[s]; }
#pragma unroll
    for (int m = 2 + 2 * S; m < K::kAggF; m++) v[m] = 0.f;
#pragma unroll
    for (int m = 0; m < K::kAggF; m += 4) *reinterpret_cast<float4*>(dst + m) = make_float4(v[m], v[m + 1], v[m + 2], v[m + 3]);
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      st_release(a.flags + rec, (a.tag << 2) | 1ull);
    }
  }

  if (c > 0) {
    // Look-back: find the newest predecessor j0 whose inclusive prefix is published, every
    // chunk after it (up to c-1) having published at least its aggregate; then fold forward
    // from it, h = exp(A S_j) h + h0_j for j = j0+1 .. c-1.  That is the arithmetic, in the
    // order, by which those chunks form their own inclusive prefixes, so the carry is the
    // same to the last bit whichever prefix the look-back happens to meet first.
    if (warp == 0) {
      int64_t jtop = c - 1;  // newest predecessor not yet examined
      int j0 = -1;
      bool gave_up = false;
      unsigned polls = 0, ns = 32;
      while (jtop >= 0) {
        const int64_t j = jtop - lane;
        int st = 0;
        if (j >= 0) {
          const unsigned long long f = ld_acquire(a.flags + ((j * a.batch + b) * n_dt + dtile));
          st = (f >> 2) == a.wait_tag ? (int)(f & 3ull) : 0;
        }
        const unsigned incl = __ballot_sync(0xFFFFFFFFu, st == 2);
        const unsigned ready = __ballot_sync(0xFFFFFFFFu, st >= 1);
        const int avail = (int)min((int64_t)32, jtop + 1);
        const int first_incl = incl ? __ffs(incl) - 1 : -1;
        const int n_need = first_incl >= 0 ? first_incl + 1 : avail;
        const unsigned mask = n_need >= 32 ? 0xFFFFFFFFu : ((1u << n_need) - 1u);
        if ((ready & mask) == mask) {
          if (first_incl >= 0) {
            j0 = (int)(jtop - first_incl);
            break;
          }
          jtop -= avail;  // a window of aggregates: look further back
          continue;
        }
        if (++polls > a.max_polls) {  // give up: this call's results are invalid
          gave_up = true;
          break;
        }
        __nanosleep(ns);
        ns = ns < 1024 ? 2 * ns : 1024;
      }
      if (lane == 0) {
        sInfo[0] = gave_up ? c : j0;  // giving up folds nothing
        if (gave_up && a.header != nullptr)
          atomicMax(a.header, (a.tag << 8) | (unsigned long long)kLookbackTimeoutCode);
      }
    }
    __syncthreads();
    const int j0 = sInfo[0];
    if (j0 >= 0 && j0 < c) {
      const float* src = a.incl + (((int64_t)j0 * a.batch + b) * n_dt * K::kThreads + dtile * K::kThreads + tid) * K::kInclF;
#pragma unroll
      for (int s = 0; s < S; s += 2) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(src + 2 * s));
        h[s] = make_float2(v.x, v.y);
        h[s + 1] = make_float2(v.z, v.w);
      }
    }
    constexpr int kAhead = S <= 4 ? 4 : S <= 8 ? 2 : 1;  // records loaded ahead of their fold
    for (int64_t j = (int64_t)j0 + 1; j < c; j += kAhead) {
      float v[kAhead][K::kAggF];
#pragma unroll
      for (int u = 0; u < kAhead; u++) {
        if (j + u < c) {
          const float* src = a.agg + (((j + u) * a.batch + b) * n_dt * K::kThreads + dtile * K::kThreads + tid) * K::kAggF;
#pragma unroll
          for (int m = 0; m < K::kAggF; m += 4) {
            const float4 q = __ldcg(reinterpret_cast<const float4*>(src + m));
            v[u][m] = q.x; v[u][m + 1] = q.y; v[u][m + 2] = q.z; v[u][m + 3] = q.w;
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kAhead; u++) {
        if (j + u < c) {
#pragma unroll
          for (int s = 0; s < S; s++) {
            const float Sc = v[u][s / kHP];  // the chunk's delta sum for this state's channel
            const float2 xa = __fmul2_rn(A2[s], make_float2(Sc, Sc));
            h[s] = __ffma2_rn(make_float2(ex2(xa.x), ex2(xa.y)), h[s], make_float2(v[u][2 + 2 * s], v[u][3 + 2 * s]));
          }
        }
      }
    }
    if (!last_chunk && !chain) {
      // Inclusive prefix of this chunk: its aggregate applied to the carry.
      float* dst = a.incl + (rec * K::kThreads + tid) * K::kInclF;
#pragma unroll
      for (int s = 0; s < S; s += 2) {
        const float S0 = s / kHP ? S2.y : S2.x, S1 = (s + 1) / kHP ? S2.y : S2.x;
        const float2 xa0 = __fmul2_rn(A2[s], make_float2(S0, S0)), xa1 = __fmul2_rn(A2[s + 1], make_float2(S1, S1));
        const float2 e0 = __ffma2_rn(make_float2(ex2(xa0.x), ex2(xa0.y)), h[s], hagg[s]);
        const float2 e1 = __ffma2_rn(make_float2(ex2(xa1.x), ex2(xa1.y)), h[s + 1], hagg[s + 1]);
        *reinterpret_cast<float4*>(dst + 2 * s) = make_float4(e0.x, e0.y, e1.x, e1.y);
      }
      __syncthreads();
      if (tid == 0) {
        __threadfence();
        st_release(a.flags + rec, (a.tag << 2) | 2ull);
      }
    }
  } else if (a.initial_state != nullptr && active) {
#pragma unroll
    for (int s = 0; s < S; s++) {
      const int c = s / kHP, n = n0 + 2 * (s % kHP);
      const float* hr = a.initial_state + (b * Dn + d + c) * N;
      h[s] = make_float2(n < N ? hr[n] : 0.f, n + 1 < N ? hr[n + 1] : 0.f);
    }
  }

  run(std::integral_constant<int, kModeMain>{});

  if (chain ? (chunked && !last_chunk) : (c == 0 && chunked)) {
    // Chunk 0's inclusive prefix is its true end state.
    float* dst = a.incl + (rec * K::kThreads + tid) * K::kInclF;
#pragma unroll
    for (int s = 0; s < S; s += 2)
      *reinterpret_cast<float4*>(dst + 2 * s) = make_float4(h[s].x, h[s].y, h[s + 1].x, h[s + 1].y);
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      st_release(a.flags + rec, (a.tag << 2) | 2ull);
    }
  }
  if (last_chunk && a.last_state != nullptr && active) {
#pragma unroll
    for (int s = 0; s < S; s++) {
      const int c = s / kHP, n = n0 + 2 * (s % kHP);
      float* lr = a.last_state + (b * Dn + d + c) * N;
      if (n < N) lr[n] = h[s].x;
      if (n + 1 < N) lr[n + 1] = h[s].y;
    }
  }
}

}  // namespace fwd

// ---------------------------------------------------------------------------------------
// Host side: the plan (lanes, states per lane, time chunks) and the launch.

namespace {

using KernelFn = void (*)(const fwd::Args);

struct Variant {
  KernelFn fn;
  int smem;
  int threads;
};

template <int L, int S, typename T, bool kConv, bool kCkpt>
Variant make_variant() {
  return Variant{fwd::scan_fwd_kernel<L, S, T, kConv, kCkpt>, fwd::Cfg<L, S, T, kConv>::kSmem, 32 * L};
}

// The kernel variants: (lanes, states per lane) in {(1,4), (1,8), (1,16), (2,4), (2,8), (4,4)}.
constexpr int kNumLS = 6;
int ls_index(int L, int S) {
  return L == 1 ? (S == 4 ? 0 : S == 8 ? 1 : S == 16 ? 2 : -1) : L == 2 ? (S == 4 ? 3 : S == 8 ? 4 : -1) : (L == 4 && S == 4) ? 5 : -1;
}

template <typename T, bool kConv, bool kCkpt>
Variant variant_t(int idx) {
  switch (idx) {
    case 0: return make_variant<1, 4, T, kConv, kCkpt>();
    case 1: return make_variant<1, 8, T, kConv, kCkpt>();
    case 2: return make_variant<1, 16, T, kConv, kCkpt>();
    case 3: return make_variant<2, 4, T, kConv, kCkpt>();
    case 4: return make_variant<2, 8, T, kConv, kCkpt>();
    case 5: return make_variant<4, 4, T, kConv, kCkpt>();
  }
  return Variant{nullptr, 0, 0};
}

template <typename T>
Variant variant_kind(int idx, int kind) {
  return kind == kFwdConv ? variant_t<T, true, false>(idx)
         : kind == kFwdCkpt ? variant_t<T, false, true>(idx)
                            : variant_t<T, false, false>(idx);
}

Variant variant(int L, int S, bool bf16, int kind) {
  const int idx = ls_index(L, S);
  return bf16 ? variant_kind<__nv_bfloat16>(idx, kind) : variant_kind<float>(idx, kind);
}

int64_t env_int(const char* name, int64_t fallback) {
  if (const char* v = std::getenv(name)) {
    const long long x = std::atoll(v);
    if (x > 0) return x;
  }
  return fallback;
}

double env_double(const char* name, double fallback) {
  if (const char* v = std::getenv(name)) {
    const double x = std::atof(v);
    if (x > 0) return x;
  }
  return fallback;
}

// Per device and variant: the dynamic shared-memory limit raised once, and the resident CTAs
// per SM (0: not prepared yet).
constexpr int kMaxDev = 64;
std::atomic<int> g_resident[kMaxDev][kNumLS * 2 * 3];

// Resident CTAs per SM of a kernel variant on the current device (0 on error); the first call
// per device raises the variant's dynamic shared-memory limit.
int prepare_variant(const Variant& v, int L, int S, bool bf16, int kind) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  const int slot = (ls_index(L, S) * 2 + (bf16 ? 1 : 0)) * 3 + kind;
  if (dev < kMaxDev) {
    const int r = g_resident[dev][slot].load(std::memory_order_relaxed);
    if (r > 0) return r;
  }
  if (cudaFuncSetAttribute(v.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, v.smem) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, v.fn, v.threads, v.smem) != cudaSuccess) return 0;
  if (dev < kMaxDev && n > 0) g_resident[dev][slot].store(n, std::memory_order_relaxed);
  return n;
}

}  // namespace

int fwd_channels_per_cta() { return fwd::kCh; }

bool plan_scan_fwd(int64_t batch, int64_t L, int64_t d_inner, int d_state, bool bf16, int kind,
                   int sms, FwdPlan* plan) {
  // Lanes per channel pair: the pair's states split over 1, 2 or 4 lanes.  Four lanes (4 states
  // each) give a GPU-filling batch of channels enough warps and keep time chunks long when
  // chunking is needed; one lane per pair (all states in one thread, no exchange between
  // lanes) issues the fewest instructions per element and wins when few channels run a long
  // sequence (measured on B300: 1 x 1,048,576 x 2048 x 16 at 15.2 ms with one lane against
  // 17.8 ms with four; 8 x 2048 x 5120 x 16 at 0.47 ms with four against 0.60-0.65 with one).
  int lanes = d_state <= 4 ? 1 : d_state <= 8 ? 2 : 4;
  if (d_state > 8 && L >= 16384 && batch * d_inner < (int64_t)sms * 12 * fwd::kCh / 2) lanes = 1;
  const int forced = (int)env_int("SSM_SCAN_LANES", 0);
  if (forced == 1 || forced == 2 || forced == 4) lanes = forced;
  int S = (d_state + lanes - 1) / lanes;
  S = S <= 4 ? 4 : S <= 8 ? 8 : 16;
  if (lanes * S > 16) { lanes = 4; S = 4; }
  const Variant v = variant(lanes, S, bf16, kind);
  if (v.fn == nullptr) return false;
  const int per_sm = prepare_variant(v, lanes, S, bf16, kind);
  if (per_sm <= 0) return false;
  const int64_t n_dt = (d_inner + fwd::kCh - 1) / fwd::kCh;
  const int64_t per_chunk = batch * n_dt;
  const int64_t slots = (int64_t)sms * per_sm;
  // Time chunks: none when the channels fill the GPU; otherwise as many as one full wave of
  // resident CTAs holds (every CTA resident at once), with chunks of at least 128 steps.
  int64_t G = 1;
  if (per_chunk > 0 && per_chunk < slots) G = slots / per_chunk;
  // One wave that does not spread evenly over the SMs (some hold one CTA more than others, and
  // those set the time): two chunks.  Two chunks need no aggregate pass (the second waits for
  // the first's end state), so the work is unchanged, and the pieces spread over the SMs as
  // the first ones finish (measured on B300 at 8 x 2048 x 5120 x 16, 640 CTAs in 740 slots:
  // 0.438 ms against 0.476 in one chunk).
  // The four-lane plain and checkpoint kernels go one step further there: three equal chunks
  // as a chain, each continuing from its predecessor's end state, with no aggregate pass at
  // all (0.428 ms against 0.438 for the two-chunk plan, same binary and box); the fused conv
  // variant keeps two chunks (the chain's branch would push it over its registers).
  bool chain = false;
  if (G == 1 && per_chunk > 0 && per_chunk <= slots && per_chunk % sms != 0) {
    G = 2;
    if (lanes == 4 && kind != kFwdConv && L >= 3 * 128) {
      G = 3;
      chain = true;
    }
  }
  G = std::min<int64_t>(G, std::max<int64_t>(1, L / 128));
  G = env_int("SSM_SCAN_CHUNKS", G);
  G = std::max<int64_t>(1, std::min<int64_t>(G, 4096));
  if (const char* v = std::getenv("SSM_SCAN_CHAIN")) chain = std::atoi(v) == 1;
  chain = chain && G > 1 && lanes == 4 && kind != kFwdConv;
  int64_t len0 = L, len = L;
  if (G > 1) {
    // Chunk 0 runs only its main pass.  With three or more chunks it is shorter than the
    // others, so that its inclusive prefix is out about when the others finish their
    // aggregates: the others start their main passes then, and the longer chunk 0 the shorter
    // all chunks.  The best fraction is about the cost of an aggregate step relative to a main
    // step, which is higher with several lanes per pair (their per-element pre-phase is paid in
    // both passes): measured on B300, 0.5 for one lane (1 x 1,048,576 x 2048 x 16: 15.25 ms
    // against 15.41 at 0.7) and 0.8 for four (2 x 2048 x 1536 x 16: 0.0704 ms against 0.0744 at
    // 0.5).  With two chunks nobody runs an aggregate and the second chunk waits for the
    // first's end state anyway; the first chunk's CTAs start at once and the second's fill in as
    // they finish, so a shorter second chunk shortens the tail: 1.5 (8 x 2048 x 5120 x 16:
    // 0.429 ms against 0.439 for equal halves and 0.446 at 3).
    const double alpha = env_double("SSM_SCAN_ALPHA", chain ? 1.0 : G == 2 ? 1.5 : (lanes == 1 ? 0.5 : 0.8));
    len = (int64_t)std::ceil((double)L / ((double)(G - 1) + alpha));
    len = (len + fwd::kT - 1) / fwd::kT * fwd::kT;
    len0 = std::max<int64_t>(fwd::kT, (int64_t)(alpha * (double)len) / fwd::kT * fwd::kT);
    if (len0 >= L) {
      G = 1;
      len0 = len = L;
    } else {
      G = 1 + (L - len0 + len - 1) / len;
    }
  }
  plan->lanes = lanes;
  plan->states_per_lane = S;
  plan->G = (int)G;
  plan->chain = chain && G > 1 ? 1 : 0;
  plan->len0 = len0;
  plan->len = len;
  plan->threads = v.threads;
  return true;
}

size_t fwd_workspace_bytes(int64_t batch, int64_t d_inner, const FwdPlan& plan) {
  const int64_t n_dt = (d_inner + fwd::kCh - 1) / fwd::kCh;
  const int64_t n_rec = (int64_t)(plan.G - 1) * batch * n_dt;
  const int64_t agg_f = (2 + 2 * plan.states_per_lane + 3) / 4 * 4;
  const int64_t incl_f = 2 * plan.states_per_lane;
  const size_t flags = ((size_t)n_rec * 8 + 255) / 256 * 256;
  return kFwdHeaderBytes + flags + (size_t)n_rec * plan.threads * (agg_f + incl_f) * sizeof(float);
}

cudaError_t launch_scan_fwd(const FwdLaunch& f, bool bf16, cudaStream_t stream) {
  const FwdPlan& plan = f.plan;
  const int kind = f.ckpt != nullptr ? kFwdCkpt : f.conv_w != nullptr ? kFwdConv : kFwdPlain;
  const Variant v = variant(plan.lanes, plan.states_per_lane, bf16, kind);
  if (v.fn == nullptr || prepare_variant(v, plan.lanes, plan.states_per_lane, bf16, kind) <= 0)
    return cudaErrorInvalidValue;
  const int64_t n_dt = (f.d_inner + fwd::kCh - 1) / fwd::kCh;
  const int64_t n_rec = (int64_t)(plan.G - 1) * f.batch * n_dt;
  const int64_t agg_f = (2 + 2 * plan.states_per_lane + 3) / 4 * 4;
  fwd::Args a{};
  a.u = f.u; a.delta = f.delta; a.A = f.A; a.B = f.B; a.C = f.C; a.D = f.D; a.z = f.z;
  a.delta_bias = f.delta_bias; a.softplus = f.softplus; a.y = f.y; a.last_state = f.last_state;
  a.initial_state = f.initial_state;
  a.conv_w = f.conv_w; a.conv_b = f.conv_b; a.d_conv = f.d_conv; a.u_out = f.u_out; a.ckpt = f.ckpt;
  a.batch = f.batch; a.L = f.L; a.d_inner = f.d_inner; a.N = f.d_state;
  a.G = plan.G; a.len0 = plan.len0; a.len = plan.len; a.chain = plan.chain;
  unsigned char* ws = static_cast<unsigned char*>(f.workspace);
  a.header = reinterpret_cast<unsigned long long*>(ws);
  a.flags = reinterpret_cast<unsigned long long*>(ws + kFwdHeaderBytes);
  float* recs = reinterpret_cast<float*>(ws + kFwdHeaderBytes + ((size_t)n_rec * 8 + 255) / 256 * 256);
  a.agg = recs;
  a.incl = recs + (size_t)n_rec * plan.threads * agg_f;
  a.tag = f.tag;
  a.wait_tag = f.wait_tag;
  a.max_polls = f.max_polls;
  const int64_t blocks = (int64_t)plan.G * f.batch * n_dt;
  v.fn<<<(unsigned)blocks, v.threads, v.smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace ssm
