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
// Three launches: (A) each chunk's local end state X^T (w * B) on the tensor cores;
// (B) the states entering every chunk, an elementwise scan over chunks; (C) the outputs:
// C B^T masked with the decays, times X, plus C H_in^T scaled by exp(S_i), on the tensor
// cores.  Tensor-core tiles: mma.sync m16n8k16, bf16 operands, fp32 accumulation, fed from
// padded shared-memory tiles by ldmatrix.  The inputs x, B, C are bf16 already; the computed
// operands (the masked decay matrix, w * B, the carried-in state) go in as a bf16 hi part
// plus a bf16 lo part (the rounding remainder), two products each, so their rounding error
// is ~2^-16 rather than bf16's 2^-8.

#include "ssm_device.cuh"
#include "ssm_internal.h"

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
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Per chunk: step sizes, and the running decay S_i in log2 units (sum of delta a log2 e),
// both into shared memory; steps past the sequence end get delta = 0.
__device__ __forceinline__ void chunk_decays(const SsdParams& p, int64_t b, int h, int64_t t0,
                                             float* sDt, float* sS) {
  const int tid = threadIdx.x;
  if (tid < kQ) {
    const int64_t t = t0 + tid;
    float dt = 0.f;
    if (t < p.L) {
      const float x = __bfloat162float(p.dt[(b * p.L + t) * p.heads + h]) + (p.dt_bias ? p.dt_bias[h] : 0.f);
      dt = p.softplus ? softplus(x) : x;
    }
    sDt[tid] = dt;
    sS[tid] = dt * p.A[h] * kLog2e;
  }
  __syncthreads();
  if (tid < 32) {  // inclusive prefix sum of 64 values: 2 per lane, then a warp scan
    const float a = sS[2 * tid], c = sS[2 * tid + 1];
    float run = a + c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float v = __shfl_up_sync(0xFFFFFFFFu, run, o);
      if (tid >= o) run += v;
    }
    const float before = run - (a + c);
    sS[2 * tid] = before + a;
    sS[2 * tid + 1] = run;
  }
  __syncthreads();
}

// Rows [0, 64) x cols [0, W) of a bf16 matrix with row stride ld (elements) into shared memory
// (row stride W + kRowPad); rows at or past `rows` are zero.
template <int W>
__device__ __forceinline__ void load_tile(__nv_bfloat16* s, const __nv_bfloat16* g, int64_t ld, int rows) {
  constexpr int kPerRow = W / 8;  // 16-byte pieces per row
  for (int i = threadIdx.x; i < kQ * kPerRow; i += kSsdThreads) {
    const int r = i / kPerRow, c = (i % kPerRow) * 8;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < rows) v = *reinterpret_cast<const uint4*>(g + r * ld + c);
    *reinterpret_cast<uint4*>(s + r * (W + kRowPad) + c) = v;
  }
}

// (A) local end state of a chunk: H_loc[p][n] = sum_j X[j][p] w_j B[j][n], w_j = delta_j 2^(S_last - S_j).
template <int N>
__global__ void __launch_bounds__(kSsdThreads) ssd_chunk_state_kernel(const SsdParams p) {
  const int c = blockIdx.x % p.nchunks;
  const int h = (blockIdx.x / p.nchunks) % p.heads;
  const int64_t b = blockIdx.x / ((int64_t)p.nchunks * p.heads);
  const int64_t t0 = (int64_t)c * kQ;
  const int rows = (int)min((int64_t)kQ, p.L - t0);
  __shared__ float sDt[kQ], sS[kQ];
  __shared__ __align__(16) __nv_bfloat16 sX[kQ][kP + kRowPad];
  __shared__ __align__(16) __nv_bfloat16 sB[kQ][N + kRowPad], sBlo[kQ][N + kRowPad];
  chunk_decays(p, b, h, t0, sDt, sS);
  load_tile<kP>(&sX[0][0], p.x + (b * p.L + t0) * p.d_inner + h * kP, p.d_inner, rows);
  const float s_last = sS[kQ - 1];
  for (int i = threadIdx.x; i < kQ * N; i += kSsdThreads) {  // B scaled by w_j, as bf16 hi + lo
    const int r = i / N, n = i % N;
    float v = 0.f;
    if (r < rows) v = __bfloat162float(p.B[(b * p.L + t0 + r) * N + n]) * sDt[r] * ex2(s_last - sS[r]);
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    sB[r][n] = hi;
    sBlo[r][n] = __float2bfloat16_rn(v - __bfloat162float(hi));
  }
  __syncthreads();

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int g = lane / 4, tq = lane % 4;
  float acc[N / 8][4];
#pragma unroll
  for (int nt = 0; nt < N / 8; nt++) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
  for (int kk = 0; kk < kQ / 16; kk++) {
    // A = X^T (rows p, cols j): transposed 8x8 blocks of sX[j][p]
    uint32_t a[4];
    ldsm_x4_t(a, &sX[kk * 16 + (lane % 8) + 8 * (lane / 16)][16 * warp + 8 * ((lane / 8) % 2)]);
#pragma unroll
    for (int nt = 0; nt < N / 8; nt += 2) {
      // B = sB[j][n] (j = k, n contiguous): transposed loads give the K-major fragments
      uint32_t bb[4], bl[4];
      ldsm_x4_t(bb, &sB[kk * 16 + (lane % 8) + 8 * ((lane / 8) % 2)][8 * nt + 8 * (lane / 16)]);
      ldsm_x4_t(bl, &sBlo[kk * 16 + (lane % 8) + 8 * ((lane / 8) % 2)][8 * nt + 8 * (lane / 16)]);
      mma16816(acc[nt], a, bb[0], bb[1]);
      mma16816(acc[nt + 1], a, bb[2], bb[3]);
      mma16816(acc[nt], a, bl[0], bl[1]);
      mma16816(acc[nt + 1], a, bl[2], bl[3]);
    }
  }
  float* Ho = p.Hs + (((b * p.heads + h) * p.nchunks + c) * kP) * N;
#pragma unroll
  for (int nt = 0; nt < N / 8; nt++) {
    const int row = 16 * warp + g, col = 8 * nt + 2 * tq;
    *reinterpret_cast<float2*>(Ho + row * N + col) = make_float2(acc[nt][0], acc[nt][1]);
    *reinterpret_cast<float2*>(Ho + (row + 8) * N + col) = make_float2(acc[nt][2], acc[nt][3]);
  }
  if (threadIdx.x == 0) p.Sc[(b * p.heads + h) * p.nchunks + c] = s_last;
}

// (B) states entering each chunk: H_in(0) = 0, H_in(c+1) = 2^(S_last(c)) H_in(c) + H_loc(c),
// written over H_loc; the state after the last chunk is last_state.
__global__ void __launch_bounds__(256) ssd_state_scan_kernel(const SsdParams p) {
  const int64_t per_head = (int64_t)kP * p.N;
  const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;  // over batch * heads * P * N
  if (i >= p.batch * p.heads * per_head) return;
  const int64_t bh = i / per_head, e = i % per_head;
  float H = 0.f;
  for (int c = 0; c < p.nchunks; c++) {
    float* slot = p.Hs + (bh * p.nchunks + c) * per_head + e;
    const float loc = *slot;
    *slot = H;
    H = fmaf(ex2(p.Sc[bh * p.nchunks + c]), H, loc);
  }
  if (p.last_state) {
    const int64_t b = bh / p.heads, h = bh % p.heads, pp = e / p.N, n = e % p.N;
    p.last_state[(b * p.d_inner + h * kP + pp) * p.N + n] = H;
  }
}

// (C) outputs of a chunk.
template <int N>
__global__ void __launch_bounds__(kSsdThreads) ssd_output_kernel(const SsdParams p) {
  const int c = blockIdx.x % p.nchunks;
  const int h = (blockIdx.x / p.nchunks) % p.heads;
  const int64_t b = blockIdx.x / ((int64_t)p.nchunks * p.heads);
  const int64_t t0 = (int64_t)c * kQ;
  const int rows = (int)min((int64_t)kQ, p.L - t0);
  // shared memory (dynamic: 61 KB at N = 128): step sizes, decays, X, B, C and H_in tiles
  extern __shared__ __align__(16) unsigned char ssd_smem[];
  float* sDt = reinterpret_cast<float*>(ssd_smem);
  float* sS = sDt + kQ;
  auto* sX = reinterpret_cast<__nv_bfloat16(*)[kP + kRowPad]>(sS + kQ);
  auto* sB = reinterpret_cast<__nv_bfloat16(*)[N + kRowPad]>(&sX[kQ][0]);
  auto* sC = reinterpret_cast<__nv_bfloat16(*)[N + kRowPad]>(&sB[kQ][0]);
  auto* sH = reinterpret_cast<__nv_bfloat16(*)[N + kRowPad]>(&sC[kQ][0]);
  auto* sHlo = reinterpret_cast<__nv_bfloat16(*)[N + kRowPad]>(&sH[kP][0]);
  chunk_decays(p, b, h, t0, sDt, sS);
  load_tile<kP>(&sX[0][0], p.x + (b * p.L + t0) * p.d_inner + h * kP, p.d_inner, rows);
  load_tile<N>(&sB[0][0], p.B + (b * p.L + t0) * N, N, rows);
  load_tile<N>(&sC[0][0], p.C + (b * p.L + t0) * N, N, rows);
  const float* Hin = p.Hs + (((b * p.heads + h) * p.nchunks + c) * kP) * N;
  for (int i = threadIdx.x; i < kP * N / 2; i += kSsdThreads) {
    const float2 v = reinterpret_cast<const float2*>(Hin)[i];
    const int r = (2 * i) / N, n = (2 * i) % N;
    const __nv_bfloat162 hi = __floats2bfloat162_rn(v.x, v.y);  // H_in as bf16 hi + lo
    *reinterpret_cast<__nv_bfloat162*>(&sH[r][n]) = hi;
    *reinterpret_cast<__nv_bfloat162*>(&sHlo[r][n]) =
        __floats2bfloat162_rn(v.x - __bfloat162float(hi.x), v.y - __bfloat162float(hi.y));
  }
  __syncthreads();

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int g = lane / 4, tq = lane % 4;
  const int i0 = 16 * warp + g, i1 = i0 + 8;  // this lane's two output rows (steps)

  // G = C B^T (rows i, cols j), K = N
  float G[kQ / 8][4];
#pragma unroll
  for (int jt = 0; jt < kQ / 8; jt++) G[jt][0] = G[jt][1] = G[jt][2] = G[jt][3] = 0.f;
  // Yi = C H_in^T (rows i, cols p), K = N
  float Yi[kP / 8][4];
#pragma unroll
  for (int pt = 0; pt < kP / 8; pt++) Yi[pt][0] = Yi[pt][1] = Yi[pt][2] = Yi[pt][3] = 0.f;
#pragma unroll
  for (int kk = 0; kk < N / 16; kk++) {
    uint32_t a[4];
    ldsm_x4(a, &sC[16 * warp + (lane % 16)][kk * 16 + 8 * (lane / 16)]);
#pragma unroll
    for (int jt = 0; jt < kQ / 8; jt += 2) {  // B operand (n, j) = sB[j][n]: n contiguous
      uint32_t bb[4];
      ldsm_x4(bb, &sB[8 * jt + (lane % 8) + 8 * (lane / 16)][kk * 16 + 8 * ((lane / 8) % 2)]);
      mma16816(G[jt], a, bb[0], bb[1]);
      mma16816(G[jt + 1], a, bb[2], bb[3]);
    }
#pragma unroll
    for (int pt = 0; pt < kP / 8; pt += 2) {  // B operand (n, p) = sH[p][n] (+ the lo part)
      uint32_t bb[4], bl[4];
      ldsm_x4(bb, &sH[8 * pt + (lane % 8) + 8 * (lane / 16)][kk * 16 + 8 * ((lane / 8) % 2)]);
      ldsm_x4(bl, &sHlo[8 * pt + (lane % 8) + 8 * (lane / 16)][kk * 16 + 8 * ((lane / 8) % 2)]);
      mma16816(Yi[pt], a, bb[0], bb[1]);
      mma16816(Yi[pt + 1], a, bb[2], bb[3]);
      mma16816(Yi[pt], a, bl[0], bl[1]);
      mma16816(Yi[pt + 1], a, bl[2], bl[3]);
    }
  }
  // causal mask and decays: M[i][j] = G[i][j] delta_j 2^(S_i - S_j) for j <= i
  const float s_i0 = sS[i0], s_i1 = sS[i1];
#pragma unroll
  for (int jt = 0; jt < kQ / 8; jt++) {
#pragma unroll
    for (int q = 0; q < 2; q++) {
      const int j = 8 * jt + 2 * tq + q;
      const float dj = sDt[j], sj = sS[j];
      G[jt][q] = j <= i0 ? G[jt][q] * dj * ex2(s_i0 - sj) : 0.f;
      G[jt][2 + q] = j <= i1 ? G[jt][2 + q] * dj * ex2(s_i1 - sj) : 0.f;
    }
  }
  // Y = M X (rows i, cols p), K = j; the M fragments come straight from G's accumulators
  float Y[kP / 8][4];
#pragma unroll
  for (int pt = 0; pt < kP / 8; pt++) {
    const float e0 = ex2(s_i0), e1 = ex2(s_i1);
    Y[pt][0] = Yi[pt][0] * e0; Y[pt][1] = Yi[pt][1] * e0;
    Y[pt][2] = Yi[pt][2] * e1; Y[pt][3] = Yi[pt][3] * e1;
  }
#pragma unroll
  for (int kk = 0; kk < kQ / 16; kk++) {
    // M as bf16 hi + lo fragments (the products are exact in fp32 accumulation)
    const float* g0 = G[2 * kk];
    const float* g1 = G[2 * kk + 1];
    uint32_t a[4], al[4];
    a[0] = pack_bf16(g0[0], g0[1]);
    a[1] = pack_bf16(g0[2], g0[3]);
    a[2] = pack_bf16(g1[0], g1[1]);
    a[3] = pack_bf16(g1[2], g1[3]);
    auto lo_of = [](float v0, float v1, uint32_t hi) {
      const __nv_bfloat162 h2 = *reinterpret_cast<const __nv_bfloat162*>(&hi);
      return pack_bf16(v0 - __bfloat162float(h2.x), v1 - __bfloat162float(h2.y));
    };
    al[0] = lo_of(g0[0], g0[1], a[0]);
    al[1] = lo_of(g0[2], g0[3], a[1]);
    al[2] = lo_of(g1[0], g1[1], a[2]);
    al[3] = lo_of(g1[2], g1[3], a[3]);
#pragma unroll
    for (int pt = 0; pt < kP / 8; pt += 2) {  // B operand (j, p) = sX[j][p]: p contiguous
      uint32_t bb[4];
      ldsm_x4_t(bb, &sX[kk * 16 + (lane % 8) + 8 * ((lane / 8) % 2)][8 * pt + 8 * (lane / 16)]);
      mma16816(Y[pt], a, bb[0], bb[1]);
      mma16816(Y[pt + 1], a, bb[2], bb[3]);
      mma16816(Y[pt], al, bb[0], bb[1]);
      mma16816(Y[pt + 1], al, bb[2], bb[3]);
    }
  }
  // y = (Y + D x) silu(z)
#pragma unroll
  for (int pt = 0; pt < kP / 8; pt++) {
#pragma unroll
    for (int half = 0; half < 2; half++) {
      const int i = half ? i1 : i0;
      if (i >= rows) continue;
      const int pp = 8 * pt + 2 * tq;
      const int64_t d0 = (int64_t)h * kP + pp;
      const int64_t e = (b * p.L + t0 + i) * p.d_inner + d0;
      float v0 = Y[pt][2 * half], v1 = Y[pt][2 * half + 1];
      if (p.D) {
        v0 = fmaf(p.D[d0], __bfloat162float(sX[i][pp]), v0);
        v1 = fmaf(p.D[d0 + 1], __bfloat162float(sX[i][pp + 1]), v1);
      }
      if (p.z) {
        const __nv_bfloat162 zz = *reinterpret_cast<const __nv_bfloat162*>(p.z + e);
        v0 *= silu(__bfloat162float(zz.x));
        v1 *= silu(__bfloat162float(zz.y));
      }
      *reinterpret_cast<__nv_bfloat162*>(p.y + e) = __floats2bfloat162_rn(v0, v1);
    }
  }
}

template <int N>
static size_t ssd_output_smem() {
  return 2 * kQ * sizeof(float) + (size_t)kQ * (kP + kRowPad) * 2 + 4 * (size_t)kQ * (N + kRowPad) * 2;
}

template <int N>
static cudaError_t launch_ssd_n(const SsdParams& p, cudaStream_t s) {
  static_assert(kP == kQ, "the H_in tile reuses the chunk-row layout");
  static bool attr_set = false;  // opt in to > 48 KB of dynamic shared memory once
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(ssd_output_kernel<N>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)ssd_output_smem<N>());
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int64_t blocks = p.batch * p.heads * p.nchunks;
  ssd_chunk_state_kernel<N><<<(unsigned)blocks, kSsdThreads, 0, s>>>(p);
  const int64_t elems = p.batch * p.heads * (int64_t)kP * N;
  ssd_state_scan_kernel<<<(unsigned)((elems + 255) / 256), 256, 0, s>>>(p);
  ssd_output_kernel<N><<<(unsigned)blocks, kSsdThreads, ssd_output_smem<N>(), s>>>(p);
  return cudaGetLastError();
}

size_t ssd_workspace_floats(int64_t batch, int64_t L, int heads, int N) {
  const int64_t chunks = (L + kQ - 1) / kQ;
  return (size_t)(batch * heads * chunks * ((int64_t)kP * N + 1));
}

int ssd_head_dim() { return kP; }

cudaError_t launch_ssd(const SsdParams& p, cudaStream_t s) {
  switch (p.N) {
    case 16: return launch_ssd_n<16>(p, s);
    case 32: return launch_ssd_n<32>(p, s);
    case 64: return launch_ssd_n<64>(p, s);
    case 128: return launch_ssd_n<128>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ssm
