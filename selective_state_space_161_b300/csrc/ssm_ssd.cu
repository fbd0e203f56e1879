// Chunked "state space duality" (SSD) form of the selective scan, on the tensor cores.
//
// youngju.dev, "Mamba: Linear-Time Sequence Modeling with Selective State Spaces 论文分析",
// section "后续研究：Mamba-2 与混合架构" names Mamba-2's State Space Duality — the same
// recurrence written as attention-like matrix products — without its equations.  The
// reading used here: when A is one scalar per head (A[d, n] = a_h for the head's P channels
// and every state) and the step size is one per head (delta[b, t, h]), the selective scan of
// the other kernels becomes, per chunk of Q steps with S_i = sum_{j <= i} delta_j a_h:
//   y_i  = sum_{j <= i} exp(S_i - S_j) delta_j (C_i . B_j) x_j      (intra-chunk, Q x Q)
//        + exp(S_i) C_i . H_in                                      (state entering the chunk)
//   H_out = exp(S_{Q-1}) H_in + sum_j exp(S_{Q-1} - S_j) delta_j x_j B_j^T   (P x N)
// followed by y = (y + D x) silu(z), exactly the recurrence h_t = exp(delta a) h + delta B x,
// y = C h + D x of the scan (the oracle checks it through that equivalence).
//
// One launch, one CTA of 4 warps per (batch, head), walking the head's chunks in order with
// the P x N state in registers: it never leaves the SM until the last state is written, so
// HBM sees only x, z, dt, B, C in and y out.  Per chunk:
//   G = C B^T (only the 16 x 8 tiles on or below the diagonal), masked and decayed into
//   M = G delta_j 2^(S_i - S_j), staged in shared memory;  Y = 2^(S_i) C H_in^T + M X;
//   y = (Y + D x) silu(z);  H = 2^(S_last) H + (w X)^T B, w_j = delta_j 2^(S_last - S_j).
// Warp w owns channels p in [16 w, 16 w + 16) of H, Y and y.  The accumulator layout of the
// mma.sync tile holding H (rows p, columns n) is exactly the B-operand layout that C H^T needs
// (k = n, column = p), so the state feeds the next chunk's readout straight from registers.
// Tensor-core tiles: mma.sync m16n8k16, bf16 operands, fp32 accumulation, fed from padded
// shared-memory tiles by ldmatrix.  The inputs x, B, C are bf16 already; the computed operands
// (M, w x, the carried state) go in as a bf16 hi part plus a bf16 lo part (the rounding
// remainder), two products each, so their rounding error is ~2^-16 rather than bf16's 2^-8.
//
// Time parts.  When the (batch, head) chains do not spread evenly over the SMs (a partial
// wave), each chain is cut into parts of whole chunks, one CTA each: part k walks its chunks
// from the state part k - 1 hands over through the workspace (a release store of a per-call,
// per-part tag), after starting its first copies and decays and waiting (acquire loads,
// bounded) for that tag; part 0 starts from zero.  The work is the same; the parts are finer
// pieces for the SMs to share.  CTAs are numbered part-major, so the CTA a part waits for was
// dispatched before it.

#include "ssm_device.cuh"
#include "ssm_internal.h"

#include <algorithm>
#include <cstdlib>
#include <cstring>

namespace ssm {

constexpr int kQ = 64;            // steps per chunk
constexpr int kP = 64;            // channels per head
constexpr int kSsdThreads = 128;  // 4 warps; warp w owns rows 16w .. 16w + 15 of each 64-row product
constexpr int kRowPad = 8;        // bf16 padding per shared-memory row (conflict-free ldmatrix)

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(smem_u32(p)));
}
// D += A (16x16, row) * B (16x8, col), bf16 in, fp32 accumulate.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  // not volatile: a pure function of its registers, so the compiler may interleave
  // independent products (back-to-back dependent ones would wait on the pipe's latency)
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Raw step sizes of steps t0 + 2 lane and t0 + 2 lane + 1 (warp 0 holds a whole chunk; steps
// at or past the sequence end read as 0 and are masked below).
__device__ __forceinline__ float2 load_dt_pair(const SsdParams& p, int64_t b, int h, int64_t t0, int lane) {
  float2 v = make_float2(0.f, 0.f);
  const int64_t t = t0 + 2 * lane;
  if (t < p.L) v.x = __bfloat162float(p.dt[(b * p.L + t) * p.heads + h]);
  if (t + 1 < p.L) v.y = __bfloat162float(p.dt[(b * p.L + t + 1) * p.heads + h]);
  return v;
}

// Warp 0: step sizes delta_t, the running decay S_i in log2 units (inclusive prefix sum of
// delta a log2 e) and the state-update weights w_j of one chunk, from the raw pair loaded
// above, into shared memory.
__device__ __forceinline__ void chunk_decays(const SsdParams& p, int h, int64_t t0, float2 raw, int lane,
                                             float* sDt, float* sS, float* sW) {
  const float bias = p.dt_bias ? p.dt_bias[h] : 0.f;
  const int64_t t = t0 + 2 * lane;
  float d0 = raw.x + bias, d1 = raw.y + bias;
  if (p.softplus) { d0 = softplus(d0); d1 = softplus(d1); }
  if (t >= p.L) d0 = 0.f;
  if (t + 1 >= p.L) d1 = 0.f;
  const float a = p.A[h] * kLog2e;
  const float e0 = d0 * a, e1 = d1 * a;
  float run = e0 + e1;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float v = __shfl_up_sync(0xFFFFFFFFu, run, o);
    if (lane >= o) run += v;
  }
  const float s_last = __shfl_sync(0xFFFFFFFFu, run, 31);
  sDt[2 * lane] = d0;
  sDt[2 * lane + 1] = d1;
  sS[2 * lane] = run - e1;
  sS[2 * lane + 1] = run;
  sW[2 * lane] = d0 * ex2(s_last - (run - e1));  // w_j = delta_j 2^(S_last - S_j)
  sW[2 * lane + 1] = d1 * ex2(s_last - run);
}

__device__ __forceinline__ void ldsm_x2(uint32_t (&r)[2], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n"
               : "=r"(r[0]), "=r"(r[1]) : "r"(smem_u32(p)));
}
// 16-byte global -> shared copy; src_bytes 0 fills the destination with zeros.
__device__ __forceinline__ void ssd_cp_async16(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n"
               :: "r"(smem_u32(dst)), "l"(src), "r"(src_bytes));
}
__device__ __forceinline__ void ssd_cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int kPending>
__device__ __forceinline__ void ssd_cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" :: "n"(kPending) : "memory");
}
// bf16 hi part of a pair, and the bf16 of what it leaves over.
__device__ __forceinline__ void split_pair(float v0, float v1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(v0, v1);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = pack_bf16(v0 - __bfloat162float(h.x), v1 - __bfloat162float(h.y));
}

// Rows [0, 64) x cols [0, W) of a bf16 matrix with row stride ld (elements) into shared memory
// (row stride W + kRowPad) by 16-byte asynchronous copies; rows at or past `rows` are zero.
template <int W>
__device__ __forceinline__ void load_tile_async(__nv_bfloat16* s, const __nv_bfloat16* g, int64_t ld,
                                                int rows) {
  constexpr int kPerRow = W / 8;  // 16-byte pieces per row
  static_assert((kQ * kPerRow) % kSsdThreads == 0, "whole pieces per thread");
  const int r0 = threadIdx.x / kPerRow, c = (threadIdx.x % kPerRow) * 8;
  constexpr int kRowStep = kSsdThreads / kPerRow;
#pragma unroll
  for (int k = 0; k < kQ * kPerRow / kSsdThreads; k++) {
    const int r = r0 + k * kRowStep;
    const bool in = r < rows;
    ssd_cp_async16(s + r * (W + kRowPad) + c, in ? g + r * ld + c : g, in ? 16 : 0);
  }
}

template <int N>
struct SsdSmem {
  float dt[2][kQ], S[2][kQ], W[2][kQ];          // per chunk parity: step sizes, running log2 decay, w_j
  float D[kP];                                  // D of the head's channels (0 if absent)
  __nv_bfloat16 X[kQ][kP + kRowPad];            // x tile [step][channel]
  __nv_bfloat16 Z[kQ][kP + kRowPad];            // z tile [step][channel]
  __nv_bfloat16 B[kQ][N + kRowPad];             // B tile [step][state]
  __nv_bfloat16 C[kQ][N + kRowPad];             // C tile [step][state]
  __nv_bfloat16 M[kQ][kQ + kRowPad], Mlo[kQ][kQ + kRowPad];  // masked decayed C B^T, hi / lo
};

// The lower-triangular 16 x 8 tiles (r, jt) of G (jt <= 2 r + 1: 20 tiles), five per warp,
// grouped so that a warp's tiles share as few row blocks r as possible:
//   warp 0: r3 j0-4 | warp 1: r3 j5-7, r0 j0-1 | warp 2: r2 j0-4 | warp 3: r2 j5, r1 j0-3
// Compile-time per warp, so that every shared-memory address and mask below folds.
__host__ __device__ constexpr int g_tile_r(int w, int s) {
  return w == 0 ? 3 : w == 1 ? (s < 3 ? 3 : 0) : w == 2 ? 2 : (s == 0 ? 2 : 1);
}
__host__ __device__ constexpr int g_tile_j(int w, int s) {
  return w == 0 ? s : w == 1 ? (s < 3 ? 5 + s : s - 3) : w == 2 ? s : (s == 0 ? 5 : s - 1);
}

// Warp WARP's five tiles of the chunk's Gram matrix G = C B^T (computed for all heads at once
// by the tensor-core kernel of ssm_ssd_gram.cu), in the m16n8 accumulator layout: G[s][0..1]
// at row 16 r + g, columns 8 jt + 2 tq (+1); G[s][2..3] eight rows below.  Loaded from L2 at
// the start of a chunk, so the latency hides behind the chunk's copies and barrier.
template <int WARP>
__device__ __forceinline__ void load_g(const float* Gc, int lane, float (&G)[5][4]) {
  const int g = lane / 4, tq = lane % 4;
#pragma unroll
  for (int s = 0; s < 5; s++) {
    const int r = g_tile_r(WARP, s), jt = g_tile_j(WARP, s);
    const float* row = Gc + (16 * r + g) * kQ + 8 * jt + 2 * tq;
    const float2 lo = __ldcg(reinterpret_cast<const float2*>(row));
    const float2 hi = __ldcg(reinterpret_cast<const float2*>(row + 8 * kQ));
    G[s][0] = lo.x; G[s][1] = lo.y; G[s][2] = hi.x; G[s][3] = hi.y;
  }
}

// Warp WARP's five tiles of G, masked (j <= i) and decayed into
// M[i][j] = G[i][j] delta_j 2^(S_i - S_j), stored as bf16 hi and lo.
template <int N, int WARP>
__device__ __forceinline__ void g_phase(SsdSmem<N>& sm, const float* sS, const float* sDt, int lane,
                                        const float (&G)[5][4]) {
  const int g = lane / 4, tq = lane % 4;
#pragma unroll
  for (int s = 0; s < 5; s++) {
    const int r = g_tile_r(WARP, s), jt = g_tile_j(WARP, s);
    const int j = 8 * jt + 2 * tq;
    const float2 sj = *reinterpret_cast<const float2*>(&sS[j]);
    const float2 dj = *reinterpret_cast<const float2*>(&sDt[j]);
#pragma unroll
    for (int half = 0; half < 2; half++) {
      const int i = 16 * r + g + 8 * half;
      const float si = sS[i];
      float m0 = G[s][2 * half] * dj.x * ex2(si - sj.x);
      float m1 = G[s][2 * half + 1] * dj.y * ex2(si - sj.y);
      if (jt >= 2 * r) {  // tiles on the diagonal: the causal mask
        if (j > i) m0 = 0.f;
        if (j + 1 > i) m1 = 0.f;
      }
      uint32_t hi, lo;
      split_pair(m0, m1, hi, lo);
      *reinterpret_cast<uint32_t*>(&sm.M[i][j]) = hi;
      *reinterpret_cast<uint32_t*>(&sm.Mlo[i][j]) = lo;
    }
  }
}

__device__ __forceinline__ unsigned long long ssd_ld_acquire(const unsigned long long* q) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(q) : "memory");
  return v;
}
__device__ __forceinline__ void ssd_st_release(unsigned long long* q, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(q), "l"(v) : "memory");
}

// part_len: steps per time part (a multiple of kQ; >= p.L for one part).
template <int N>
__global__ void __launch_bounds__(kSsdThreads, 3) ssd_fused_kernel(const SsdParams p, int64_t part_len) {
  extern __shared__ __align__(16) unsigned char ssd_smem[];
  SsdSmem<N>& sm = *reinterpret_cast<SsdSmem<N>*>(ssd_smem);
  const int64_t chains = p.batch * p.heads;
  const int64_t chain = blockIdx.x % chains;
  const int part = (int)(blockIdx.x / chains);
  const int64_t t_begin = (int64_t)part * part_len;
  const int64_t t_end = min(t_begin + part_len, p.L);
  const bool hands_over = t_end < p.L;  // a later part continues from this one's end state
  const int h = (int)(chain % p.heads);
  const int64_t b = chain / p.heads;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int g = lane / 4, tq = lane % 4;
  const int p0 = 16 * warp;  // this warp's channels within the head
  // (tile addresses are rebuilt from the kernel parameters where used: fewer live registers)

  if (threadIdx.x < kP) sm.D[threadIdx.x] = p.D ? p.D[h * kP + threadIdx.x] : 0.f;  // read after the first barrier

  float H[N / 8][4];  // state: rows p0 + g (+8), columns n = 8 nt + 2 tq (+1)
#pragma unroll
  for (int nt = 0; nt < N / 8; nt++) H[nt][0] = H[nt][1] = H[nt][2] = H[nt][3] = 0.f;

  // Pipeline: B, C of a chunk are requested while the previous chunk finishes (M X and the
  // outputs), x, z at the chunk's start; warp 0 computes the next chunk's step sizes and decays
  // (into the other parity's arrays) while the current chunk runs, from raw step sizes loaded
  // a chunk earlier still.
  load_tile_async<N>(&sm.B[0][0], p.B + (b * p.L + t_begin) * N, N, (int)min((int64_t)kQ, p.L - t_begin));
  load_tile_async<N>(&sm.C[0][0], p.C + (b * p.L + t_begin) * N, N, (int)min((int64_t)kQ, p.L - t_begin));
  ssd_cp_async_commit();
  float2 dt_raw = make_float2(0.f, 0.f);
  if (warp == 0) {
    chunk_decays(p, h, t_begin, load_dt_pair(p, b, h, t_begin, lane), lane, sm.dt[0], sm.S[0], sm.W[0]);
    if (t_begin + kQ < t_end) dt_raw = load_dt_pair(p, b, h, t_begin + kQ, lane);
  }

  if (part > 0) {
    // The state at t_begin, from the part before: wait for its tag (bounded: a wait that runs
    // out records code 7 in the status word, and the walk goes on from what is there).
    if (threadIdx.x == 0) {
      bool ok = false;
      unsigned ns = 32;
      const unsigned long long want = (p.wait_tag << 8) | (unsigned long long)part;
      for (unsigned it = 0; it < p.max_polls; it++) {
        if (ssd_ld_acquire(p.flags + chain) == want) {
          ok = true;
          break;
        }
        __nanosleep(ns);
        ns = ns < 1024 ? 2 * ns : 1024;
      }
      if (!ok) atomicMax(p.header, (p.tag << 8) | 7ull);
    }
    __syncthreads();
    const float* in = p.hand + (b * p.d_inner + (int64_t)h * kP + p0) * N;
#pragma unroll
    for (int nt = 0; nt < N / 8; nt++) {
      const int col = 8 * nt + 2 * tq;
      const float2 v0 = __ldcg(reinterpret_cast<const float2*>(in + g * N + col));
      const float2 v1 = __ldcg(reinterpret_cast<const float2*>(in + (g + 8) * N + col));
      H[nt][0] = v0.x; H[nt][1] = v0.y; H[nt][2] = v1.x; H[nt][3] = v1.y;
    }
  }

  int par = 0;  // parity of the current chunk's decay arrays
  for (int64_t t0 = t_begin; t0 < t_end; t0 += kQ, par ^= 1) {
    const int rows = (int)min((int64_t)kQ, p.L - t0);
    float G[5][4];  // this warp's tiles of the chunk's Gram matrix
    {
      const float* Gc = p.G + (b * ((p.L + kQ - 1) / kQ) + t0 / kQ) * kQ * kQ;
      switch (warp) {
        case 0: load_g<0>(Gc, lane, G); break;
        case 1: load_g<1>(Gc, lane, G); break;
        case 2: load_g<2>(Gc, lane, G); break;
        default: load_g<3>(Gc, lane, G); break;
      }
    }
    const float* sDt = sm.dt[par];
    const float* sS = sm.S[par];
    const float* sW = sm.W[par];
    const int64_t act0 = (b * p.L + t0) * p.d_inner + h * kP;  // this chunk's x / z / y tile
    load_tile_async<kP>(&sm.X[0][0], p.x + act0, p.d_inner, rows);
    if (p.z) load_tile_async<kP>(&sm.Z[0][0], p.z + act0, p.d_inner, rows);
    ssd_cp_async_commit();
    ssd_cp_async_wait<1>();  // this chunk's B, C have landed (x, z may still be in flight)
    __syncthreads();         // ... and this chunk's decays (written during the previous chunk)
    if (warp == 0 && t0 + kQ < t_end) {
      chunk_decays(p, h, t0 + kQ, dt_raw, lane, sm.dt[par ^ 1], sm.S[par ^ 1], sm.W[par ^ 1]);
      if (t0 + 2 * kQ < t_end) dt_raw = load_dt_pair(p, b, h, t0 + 2 * kQ, lane);
    }

    // ---- M (hi, lo) from this warp's tiles of G into shared memory
    switch (warp) {
      case 0: g_phase<N, 0>(sm, sS, sDt, lane, G); break;
      case 1: g_phase<N, 1>(sm, sS, sDt, lane, G); break;
      case 2: g_phase<N, 2>(sm, sS, sDt, lane, G); break;
      default: g_phase<N, 3>(sm, sS, sDt, lane, G); break;
    }

    // ---- Y = 2^(S_i) C H_in^T: rows i (four 16-row blocks) x this warp's 16 channels
    float Y[4][2][4];
#pragma unroll
    for (int r = 0; r < 4; r++)
#pragma unroll
      for (int pt = 0; pt < 2; pt++) Y[r][pt][0] = Y[r][pt][1] = Y[r][pt][2] = Y[r][pt][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < N / 16; kk++) {
      // B operand (k = n, column = p) straight from the state's accumulator tiles 2 kk, 2 kk + 1
      uint32_t bh[2][2], bl[2][2];
#pragma unroll
      for (int pt = 0; pt < 2; pt++) {
        split_pair(H[2 * kk][2 * pt], H[2 * kk][2 * pt + 1], bh[pt][0], bl[pt][0]);
        split_pair(H[2 * kk + 1][2 * pt], H[2 * kk + 1][2 * pt + 1], bh[pt][1], bl[pt][1]);
      }
#pragma unroll
      for (int r = 0; r < 4; r++) {
        uint32_t a[4];
        ldsm_x4(a, &sm.C[16 * r + (lane % 16)][kk * 16 + 8 * (lane / 16)]);
#pragma unroll
        for (int pt = 0; pt < 2; pt++) mma16816(Y[r][pt], a, bh[pt][0], bh[pt][1]);
#pragma unroll
        for (int pt = 0; pt < 2; pt++) mma16816(Y[r][pt], a, bl[pt][0], bl[pt][1]);
      }
    }
#pragma unroll
    for (int r = 0; r < 4; r++) {
      const float e0 = ex2(sS[16 * r + g]), e1 = ex2(sS[16 * r + g + 8]);
#pragma unroll
      for (int pt = 0; pt < 2; pt++) {
        Y[r][pt][0] *= e0; Y[r][pt][1] *= e0;
        Y[r][pt][2] *= e1; Y[r][pt][3] *= e1;
      }
    }
    ssd_cp_async_wait<0>();  // x, z have landed
    __syncthreads();         // M and x visible to every warp

    // ---- H = 2^(S_last) H + (w X)^T B: rows p (this warp's 16), columns n.  The weights w_j
    // scale the A fragments in registers (w X as bf16 hi + lo); B goes in as loaded.
    {
      const float decay = ex2(sS[kQ - 1]);
#pragma unroll
      for (int nt = 0; nt < N / 8; nt++) {
        H[nt][0] *= decay; H[nt][1] *= decay; H[nt][2] *= decay; H[nt][3] *= decay;
      }
#pragma unroll
      for (int kk = 0; kk < kQ / 16; kk++) {
        uint32_t a[4];  // A = X^T (rows p, k = j): transposed 8 x 8 blocks of X[j][p]
        ldsm_x4_t(a, &sm.X[kk * 16 + (lane % 8) + 8 * (lane / 16)][p0 + 8 * ((lane / 8) % 2)]);
        // a0, a1 hold k = j = 16 kk + 2 tq (+1); a2, a3 hold j + 8 (+1)
        const float2 w0 = *reinterpret_cast<const float2*>(&sW[kk * 16 + 2 * tq]);
        const float2 w1 = *reinterpret_cast<const float2*>(&sW[kk * 16 + 8 + 2 * tq]);
        uint32_t ah[4], al[4];
#pragma unroll
        for (int q = 0; q < 4; q++) {
          const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&a[q]);
          const float2 w = q < 2 ? w0 : w1;
          split_pair(__bfloat162float(v.x) * w.x, __bfloat162float(v.y) * w.y, ah[q], al[q]);
        }
#pragma unroll
        for (int nt = 0; nt < N / 8; nt += 2) {
          uint32_t bb[4];  // B operand (k = j, column = n) = B[j][n]
          ldsm_x4_t(bb, &sm.B[kk * 16 + (lane % 8) + 8 * ((lane / 8) % 2)][8 * nt + 8 * (lane / 16)]);
          mma16816(H[nt], ah, bb[0], bb[1]);
          mma16816(H[nt + 1], ah, bb[2], bb[3]);
          mma16816(H[nt], al, bb[0], bb[1]);
          mma16816(H[nt + 1], al, bb[2], bb[3]);
        }
      }
    }
    __syncthreads();  // every warp is done with the B and C tiles: request the next chunk's
    if (t0 + kQ < t_end) {
      const int next_rows = (int)min((int64_t)kQ, p.L - t0 - kQ);
      load_tile_async<N>(&sm.B[0][0], p.B + (b * p.L + t0 + kQ) * N, N, next_rows);
      load_tile_async<N>(&sm.C[0][0], p.C + (b * p.L + t0 + kQ) * N, N, next_rows);
    }
    ssd_cp_async_commit();

    // ---- Y += M X over the blocks on or below the diagonal
#pragma unroll
    for (int kk = 0; kk < kQ / 16; kk++) {
      uint32_t bx[4];  // B operand (k = j, column = p) = X[j][p], two 8-channel tiles
      ldsm_x4_t(bx, &sm.X[kk * 16 + (lane % 8) + 8 * ((lane / 8) % 2)][p0 + 8 * (lane / 16)]);
#pragma unroll
      for (int r = kk; r < 4; r++) {
        uint32_t a[4], al[4];
        ldsm_x4(a, &sm.M[16 * r + (lane % 16)][kk * 16 + 8 * (lane / 16)]);
        ldsm_x4(al, &sm.Mlo[16 * r + (lane % 16)][kk * 16 + 8 * (lane / 16)]);
#pragma unroll
        for (int pt = 0; pt < 2; pt++) mma16816(Y[r][pt], a, bx[2 * pt], bx[2 * pt + 1]);
#pragma unroll
        for (int pt = 0; pt < 2; pt++) mma16816(Y[r][pt], al, bx[2 * pt], bx[2 * pt + 1]);
      }
    }

    // ---- y = (Y + D x) silu(z), staged in this warp's own columns of the z tile (each value
    // over the z it was gated by), then written as 16-byte pieces: whole 32-byte sectors
#pragma unroll
    for (int r = 0; r < 4; r++) {
#pragma unroll
      for (int pt = 0; pt < 2; pt++) {
#pragma unroll
        for (int half = 0; half < 2; half++) {
          const int i = 16 * r + g + 8 * half;
          const int pp = p0 + 8 * pt + 2 * tq;
          const __nv_bfloat162 xx = *reinterpret_cast<const __nv_bfloat162*>(&sm.X[i][pp]);
          const float2 dd = *reinterpret_cast<const float2*>(&sm.D[pp]);
          float v0 = fmaf(dd.x, __bfloat162float(xx.x), Y[r][pt][2 * half]);
          float v1 = fmaf(dd.y, __bfloat162float(xx.y), Y[r][pt][2 * half + 1]);
          __nv_bfloat162* zy = reinterpret_cast<__nv_bfloat162*>(&sm.Z[i][pp]);
          if (p.z) {
            const __nv_bfloat162 zz = *zy;
            v0 *= silu(__bfloat162float(zz.x));
            v1 *= silu(__bfloat162float(zz.y));
          }
          *zy = __floats2bfloat162_rn(v0, v1);
        }
      }
    }
    __syncwarp();
    {
      __nv_bfloat16* yc = p.y + act0 + p0 + 8 * (lane % 2);
#pragma unroll
      for (int k = 0; k < 4; k++) {
        const int i = lane / 2 + 16 * k;
        if (i < rows)
          *reinterpret_cast<uint4*>(yc + (int64_t)i * p.d_inner) =
              *reinterpret_cast<const uint4*>(&sm.Z[i][p0 + 8 * (lane % 2)]);
      }
    }
    __syncthreads();  // x, z, M free for the next chunk
  }
  ssd_cp_async_wait<0>();  // nothing left in flight (the last commit is an empty group)

  if (hands_over) {
    float* out = p.hand + (b * p.d_inner + (int64_t)h * kP + p0) * N;
#pragma unroll
    for (int nt = 0; nt < N / 8; nt++) {
      const int col = 8 * nt + 2 * tq;
      __stcg(reinterpret_cast<float2*>(out + g * N + col), make_float2(H[nt][0], H[nt][1]));
      __stcg(reinterpret_cast<float2*>(out + (g + 8) * N + col), make_float2(H[nt][2], H[nt][3]));
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      ssd_st_release(p.flags + chain, (p.tag << 8) | (unsigned long long)(part + 1));
    }
    return;
  }
  if (p.last_state) {
    float* out = p.last_state + (b * p.d_inner + (int64_t)h * kP + p0) * N;
#pragma unroll
    for (int nt = 0; nt < N / 8; nt++) {
      const int col = 8 * nt + 2 * tq;
      *reinterpret_cast<float2*>(out + g * N + col) = make_float2(H[nt][0], H[nt][1]);
      *reinterpret_cast<float2*>(out + (g + 8) * N + col) = make_float2(H[nt][2], H[nt][3]);
    }
  }
}

template <int N>
static cudaError_t launch_ssd_n(const SsdParams& p, cudaStream_t s) {
  const int smem = (int)sizeof(SsdSmem<N>);
  cudaError_t e = cudaFuncSetAttribute(ssd_fused_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(ssd_fused_kernel<N>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ssd_fused_kernel<N>, kSsdThreads, smem);
  if (e != cudaSuccess) return e;
  // Two time parts unless the chains already spread evenly: whole waves of resident CTAs, or
  // one wave with the same number of CTAs on every SM (measured on B300 at 8 x 2048 x 5120 x
  // 128, 640 chains in 444 slots: see the design notes).
  const int64_t chains = p.batch * p.heads;
  const int64_t n_chunks = (p.L + kQ - 1) / kQ;
  const int64_t slots = (int64_t)std::max(1, p.sms) * std::max(1, per_sm);
  const bool even = chains % slots == 0 || (chains <= slots && chains % std::max(1, p.sms) == 0);
  int parts = even ? 1 : 2;
  if (const char* v = std::getenv("SSM_SSD_PARTS")) {
    const int f = std::atoi(v);
    if (f >= 1 && f <= 64) parts = f;
  }
  while (parts > 1 && (int64_t)parts * chains > 0x7FFFFFFF) parts--;  // grid size limit
  const int64_t chunks_per_part = (n_chunks + std::max(1, parts) - 1) / std::max(1, parts);
  const int64_t part_len = chunks_per_part * kQ;
  parts = (int)((n_chunks + chunks_per_part - 1) / chunks_per_part);  // none empty
  ssd_fused_kernel<N><<<(unsigned)(parts * chains), kSsdThreads, smem, s>>>(p, part_len);
  return cudaGetLastError();
}

int ssd_head_dim() { return kP; }

size_t ssd_flags_offset(int64_t batch, int64_t L) { return kFwdHeaderBytes + ssd_gram_bytes(batch, L); }

size_t ssd_hand_offset(int64_t batch, int64_t L, int64_t d_inner) {
  const int64_t chains = batch * (d_inner / kP);
  return ssd_flags_offset(batch, L) + ((size_t)chains * 8 + 255) / 256 * 256;
}

size_t ssd_workspace_bytes(int64_t batch, int64_t L, int64_t d_inner, int N) {
  return ssd_hand_offset(batch, L, d_inner) + (size_t)batch * d_inner * N * sizeof(float);
}

cudaError_t launch_ssd(const SsdParams& p, cudaStream_t s) {
  // SSM_SSD_KERNEL=tc: the per-head chain with every product on tcgen05 (ssm_ssd_tc.cu; measured
  // slower on B300, 0.57 ms against 0.44 ms at the 8 x 2048 x 5120 x 128 shape)
  const char* k = std::getenv("SSM_SSD_KERNEL");
  if (k != nullptr && std::strcmp(k, "tc") == 0) return launch_ssd_tc(p, s);
  // the chunk Gram matrices of every batch row first (tensor-core kernel), then the heads
  const cudaError_t e = launch_ssd_gram(p.C, p.B, p.G, p.batch, p.L, p.N, p.header, p.tag, s);
  if (e != cudaSuccess) return e;
  switch (p.N) {
    case 16: return launch_ssd_n<16>(p, s);
    case 32: return launch_ssd_n<32>(p, s);
    case 64: return launch_ssd_n<64>(p, s);
    case 128: return launch_ssd_n<128>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ssm
