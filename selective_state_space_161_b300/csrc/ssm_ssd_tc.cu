// Chunked SSD: the per-head chain on the 5th-generation tensor cores.
//
// The same chunked form as ssm_ssd.cu (youngju.dev, "Mamba: Linear-Time Sequence Modeling with
// Selective State Spaces 论文分析", section "后续研究：Mamba-2 与混合架构"; the reading and the
// equations are spelled out there): per chunk of 64 steps, with S_i the running log2 decay,
//   S  = (w X)^T B                          the chunk's own contribution to the state (P x N)
//   Yo = C H_in^T,   Yd = M X               the carried state's readout and the intra-chunk mix
//   y  = (2^{S_i} Yo + Yd + D x) silu(z),   H = 2^{S_last} H + S.
// One CTA of 8 warps per (batch row, head) walks the head's chunks in order.  All three products
// run on tcgen05.mma (M = 64, bf16 operands from shared memory, fp32 accumulators in tensor
// memory: S in columns [0, N), Yo in [128, 192), Yd in [192, 256)), issued by one thread and
// completed through an mbarrier.  The operands are laid out for the tensor core as they arrive:
// C (rows t, states contiguous) is K-major, B and x (rows t, states or channels contiguous) are
// MN-major, so cp.async puts them straight into the canonical no-swizzle core-matrix layout;
// the computed operands (w x, M, the carried state) go in as a bf16 hi part plus a bf16 lo part
// (two products each, rounding error ~2^-16).  The M = 64 accumulators are read back with
// tcgen05.ld.16x256b, which hands each thread the same elements as an m16n8 accumulator
// fragment: the state H stays in registers in that layout from chunk to chunk.  Warps w and
// w + 4 read the same lanes (rows 16 (w % 4) + g and + 8), each half of the columns.  Every wait on the
// mbarrier is bounded; a wait that runs out ends the walk (the outputs are then invalid) and
// never hangs.

#include "ssm_device.cuh"
#include "ssm_internal.h"

#include <algorithm>
#include <cstdlib>

namespace ssm {
namespace ssdtc {

constexpr int kQ = 64;          // steps per chunk
constexpr int kP = 64;          // channels per head
constexpr int kThreads = 256;  // 8 warps: warps w and w + 4 share a quadrant of TMEM lanes, each half the columns
constexpr int kColS = 0, kColYo = 128, kColYd = 192, kTmemCols = 256;
constexpr unsigned kMaxPolls = 1u << 24;
constexpr int kStageRow = kP + 8;  // bf16 per row of the output staging tile

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// Shared-memory matrix descriptor (no swizzle): start address, the byte distance between core
// matrices along K (leading) and along M/N (stride), descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46);
}
__device__ __forceinline__ void mma_f16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
               ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (unsigned it = 0; it < kMaxPolls; it++) {
    uint32_t done;
    asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
                 : "=r"(done) : "r"(bar), "r"(parity) : "memory");
    if (done) return true;
    if (it > 64) __nanosleep(64);
  }
  return false;
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)), "l"(src), "r"(valid ? 16 : 0));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld_16x256b_x1(uint32_t taddr, uint32_t (&r)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x1.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_16x256b_x2(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x2.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_16x256b_x4(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_16x256b_x8(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_16x256b_x16(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
               : "r"(taddr));
}

template <int R>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t (&r)[4 * R]) {
  if constexpr (R == 1) tmem_ld_16x256b_x1(taddr, r);
  else if constexpr (R == 2) tmem_ld_16x256b_x2(taddr, r);
  else if constexpr (R == 4) tmem_ld_16x256b_x4(taddr, r);
  else if constexpr (R == 8) tmem_ld_16x256b_x8(taddr, r);
  else tmem_ld_16x256b_x16(taddr, r);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
// bf16 hi part of a pair and the bf16 of what it leaves over
__device__ __forceinline__ void split_pair(float v0, float v1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 hv = __floats2bfloat162_rn(v0, v1);
  hi = *reinterpret_cast<const uint32_t*>(&hv);
  lo = pack_bf16(v0 - __bfloat162float(hv.x), v1 - __bfloat162float(hv.y));
}

// Byte offsets of the CTA's shared memory (every buffer 128-byte aligned).
template <int N>
struct Smem {
  static constexpr int kC = 0;                          // C: K-major [t][n]
  static constexpr int kB = kC + kQ * N * 2;            // B: MN-major [t][n]
  static constexpr int kX = kB + kQ * N * 2;            // x: MN-major [t][p]
  static constexpr int kWXh = kX + kQ * kP * 2;         // w x, hi / lo: MN-major [t][p]
  static constexpr int kWXl = kWXh + kQ * kP * 2;
  static constexpr int kMh = kWXl + kQ * kP * 2;        // M, hi / lo: K-major [t][s]
  static constexpr int kMl = kMh + kQ * kQ * 2;
  static constexpr int kHh = kMl + kQ * kQ * 2;         // carried state, hi / lo: K-major [p][n]
  static constexpr int kHl = kHh + kP * N * 2;
  static constexpr int kF = kHl + kP * N * 2;           // floats: dt, S, w [2][64] each, D [64]
  static constexpr int kBar = kF + (3 * 2 * kQ + kP) * 4;
  static constexpr int kBytes = kBar + 16;
  // at most two CTAs per SM (the tensor-memory columns of two), whatever the state size
  static constexpr int kAlloc = kBytes > 80 * 1024 ? kBytes : 80 * 1024;
  static_assert(kQ * kStageRow * 2 <= 2 * kQ * kQ * 2, "the output staging tile fits in the M buffers");
};

// Warp 0: step sizes, running log2 decay S_i (inclusive prefix sum of delta a log2 e) and the
// state-update weights w_j = delta_j 2^{S_last - S_j} of one chunk (steps past the end: delta 0).
__device__ __forceinline__ float2 load_dt_pair(const SsdParams& p, int64_t b, int h, int64_t t0, int lane) {
  float2 v = make_float2(0.f, 0.f);
  const int64_t t = t0 + 2 * lane;
  if (t < p.L) v.x = __bfloat162float(p.dt[(b * p.L + t) * p.heads + h]);
  if (t + 1 < p.L) v.y = __bfloat162float(p.dt[(b * p.L + t + 1) * p.heads + h]);
  return v;
}
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
  sW[2 * lane] = d0 * ex2(s_last - (run - e1));
  sW[2 * lane + 1] = d1 * ex2(s_last - run);
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* q) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(q) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u64(unsigned long long* q, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(q), "l"(v) : "memory");
}

constexpr int kIssuer = 128;  // thread that issues the MMAs: lane 0 of warp 4 (warp 0 computes decays)

// part_len: steps per time part of a chain (a multiple of kQ; >= p.L for one part).  Part k of a
// chain starts from the state part k - 1 hands over through the workspace, as in ssm_ssd.cu.
template <int N>
__global__ void __launch_bounds__(kThreads, 2) ssd_tc_kernel(const SsdParams p, int64_t part_len) {
  using SM = Smem<N>;
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* sC = smem + SM::kC;
  unsigned char* sB = smem + SM::kB;
  unsigned char* sX = smem + SM::kX;
  unsigned char* sWXh = smem + SM::kWXh;
  unsigned char* sWXl = smem + SM::kWXl;
  unsigned char* sMh = smem + SM::kMh;
  unsigned char* sMl = smem + SM::kMl;
  unsigned char* sHh = smem + SM::kHh;
  unsigned char* sHl = smem + SM::kHl;
  float* sF = reinterpret_cast<float*>(smem + SM::kF);
  float* sDt = sF;                 // [2][kQ]
  float* sS = sF + 2 * kQ;         // [2][kQ]
  float* sW = sF + 4 * kQ;         // [2][kQ]
  float* sD = sF + 6 * kQ;         // [kP]
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + SM::kBar);
  uint32_t* taddr = reinterpret_cast<uint32_t*>(smem + SM::kBar + 8);
  __nv_bfloat16* sY = reinterpret_cast<__nv_bfloat16*>(sMh);  // output staging [kQ][kStageRow]

  const int64_t chains = p.batch * p.heads;
  const int64_t chain = blockIdx.x % chains;
  const int part = (int)(blockIdx.x / chains);
  const int64_t t_begin = (int64_t)part * part_len;
  const int64_t t_end = min(t_begin + part_len, p.L);
  const int h = (int)(chain % p.heads);
  const int64_t b = chain / p.heads;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int g = lane / 4, tq = lane % 4;
  const int qd = warp % 4, ch = warp / 4;      // lane quadrant, column half
  const int rA = 16 * qd + g, rB = rA + 8;     // this thread's rows of every M = 64 product

  if (blockIdx.x == 0 && tid == 0) atomicExch(p.header, p.tag << 8);  // this call's status: ok
  if (tid < kP) sD[tid] = p.D ? p.D[h * kP + tid] : 0.f;
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(bar)));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(taddr)), "n"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }

  // This thread's half of the carried state (columns n0 + [0, N/2)), in the m16n8 fragment
  // layout: H[j] = (rA, n0 + 8j + 2tq), (rA, +1), (rB, n0 + 8j + 2tq), (rB, +1).
  constexpr int kHJ = N / 16;
  const int n0 = ch * (N / 2);
  float H[kHJ][4];
#pragma unroll
  for (int j = 0; j < kHJ; j++) H[j][0] = H[j][1] = H[j][2] = H[j][3] = 0.f;
  // H as the B operand of C H^T: K-major [p][n], core (p/8, n/8) at (p/8) 128 + (n/8) 1024
  auto store_state = [&]() {
#pragma unroll
    for (int j = 0; j < kHJ; j++) {
#pragma unroll
      for (int half = 0; half < 2; half++) {
        const int r = half ? rB : rA;
        uint32_t hi, lo;
        split_pair(H[j][2 * half], H[j][2 * half + 1], hi, lo);
        const int off = (r / 8) * 128 + (n0 / 8 + j) * 1024 + 16 * (r % 8) + 4 * tq;
        *reinterpret_cast<uint32_t*>(sHh + off) = hi;
        *reinterpret_cast<uint32_t*>(sHl + off) = lo;
      }
    }
  };
  store_state();

  // One chunk's B, C (rows t, N states) and x (rows t, 64 channels) into their tensor-core
  // layouts, as 16-byte pieces; rows past the end read as zero.  Pieces go 8 rows x 4 pieces per
  // warp instruction: whole 64-byte runs of each row from global memory, distinct banks in shared.
  auto load_bc = [&](int64_t t0) {
    const int rows = (int)min((int64_t)kQ, p.L - t0);
    constexpr int kPieces = kQ * N / 8;
#pragma unroll
    for (int i = 0; i < (kPieces + kThreads - 1) / kThreads; i++) {
      const int q = tid + i * kThreads;
      if (kPieces % kThreads != 0 && q >= kPieces) break;
      const int t = (q % 8) + 8 * (q / (8 * (N / 8))), j = (q / 8) % (N / 8);
      const bool in = t < rows;
      const int64_t src = (b * p.L + t0 + (in ? t : 0)) * N + 8 * j;
      cp_async16(sC + (t / 8) * 128 + j * 1024 + 16 * (t % 8), p.C + src, in);      // K-major
      cp_async16(sB + j * 128 + (t / 8) * (N * 16) + 16 * (t % 8), p.B + src, in);  // MN-major
    }
  };
  auto load_x = [&](int64_t t0) {
    const int rows = (int)min((int64_t)kQ, p.L - t0);
    constexpr int kPieces = kQ * kP / 8;
#pragma unroll
    for (int i = 0; i < kPieces / kThreads; i++) {
      const int q = tid + i * kThreads;
      const int t = (q % 8) + 8 * (q / (8 * (kP / 8))), j = (q / 8) % (kP / 8);
      const bool in = t < rows;
      const int64_t src = (b * p.L + t0 + (in ? t : 0)) * p.d_inner + (int64_t)h * kP + 8 * j;
      cp_async16(sX + j * 128 + (t / 8) * 1024 + 16 * (t % 8), p.x + src, in);  // MN-major
    }
  };

  load_bc(t_begin);
  load_x(t_begin);
  cp_async_commit();
  float2 dt_raw = make_float2(0.f, 0.f);
  if (warp == 0) {
    chunk_decays(p, h, t_begin, load_dt_pair(p, b, h, t_begin, lane), lane, sDt, sS, sW);
    if (t_begin + kQ < t_end) dt_raw = load_dt_pair(p, b, h, t_begin + kQ, lane);
  }
  bool ok = true;
  if (part > 0) {
    // the state at t_begin from the part before (bounded wait; a wait that runs out records
    // code 7 and the walk goes on from what is there)
    if (tid == 0) {
      bool got = false;
      unsigned ns = 32;
      const unsigned long long want = (p.wait_tag << 8) | (unsigned long long)part;
      for (unsigned it = 0; it < p.max_polls; it++) {
        if (ld_acquire_u64(p.flags + chain) == want) {
          got = true;
          break;
        }
        __nanosleep(ns);
        ns = ns < 1024 ? 2 * ns : 1024;
      }
      if (!got) atomicMax(p.header, (p.tag << 8) | (unsigned long long)kLookbackTimeoutCode);
    }
    __syncthreads();
#pragma unroll
    for (int half = 0; half < 2; half++) {
      const int r = half ? rB : rA;
      const float* in = p.hand + (b * p.d_inner + (int64_t)h * kP + r) * N + n0;
#pragma unroll
      for (int j = 0; j < kHJ; j++) {
        const float2 v = __ldcg(reinterpret_cast<const float2*>(in + 8 * j + 2 * tq));
        H[j][2 * half] = v.x;
        H[j][2 * half + 1] = v.y;
      }
    }
    store_state();
  }
  tc_before_sync();
  __syncthreads();
  tc_after_sync();
  const uint32_t tmem = *taddr;
  const uint32_t tlane = (uint32_t)(32 * qd) << 16;

  constexpr uint32_t kIdS = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | (1u << 16) |
                            ((uint32_t)(N >> 3) << 17) | ((uint32_t)(kQ >> 4) << 24);
  constexpr uint32_t kIdYo = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kP >> 3) << 17) |
                             ((uint32_t)(kQ >> 4) << 24);
  constexpr uint32_t kIdYd = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) | ((uint32_t)(kP >> 3) << 17) |
                             ((uint32_t)(kQ >> 4) << 24);

  uint32_t phase = 0;
  int par = 0;
  for (int64_t t0 = t_begin; t0 < t_end; t0 += kQ, par ^= 1) {
    const int rows = (int)min((int64_t)kQ, p.L - t0);
    const float* cDt = sDt + par * kQ;
    const float* cS = sS + par * kQ;
    const float* cW = sW + par * kQ;
    // this thread's z pairs (rows rA, rB; channels 8 j + 2 tq), requested now
    // (this thread's outputs: rows rA, rB; channels p0 + 8 j + 2 tq (+1), j < 4)
    const int p0 = 32 * ch;
    uint32_t zr[2][4];
    const int64_t act0 = (b * p.L + t0) * p.d_inner + (int64_t)h * kP;
#pragma unroll
    for (int half = 0; half < 2; half++) {
      const int r = half ? rB : rA;
#pragma unroll
      for (int j = 0; j < 4; j++)
        zr[half][j] = (p.z && r < rows) ? __ldg(reinterpret_cast<const uint32_t*>(p.z + act0 + (int64_t)r * p.d_inner + p0 + 8 * j + 2 * tq))
                                        : 0u;
    }
    cp_async_wait_all();
    fence_async_smem();
    tc_before_sync();
    __syncthreads();  // this chunk's B, C, x and decays, and the carried state, are in shared memory
    tc_after_sync();

    // ---- first MMA group: G = C B^T (into Yd's columns) and Yo = C H^T, which need nothing computed
    if (tid == kIssuer) {
      // descriptors of the tiles' first K block; a K step advances the address field (bytes / 16)
      const uint64_t dC = smem_desc(smem_u32(sC), 1024, 128);
      const uint64_t dBk = smem_desc(smem_u32(sB), 128, N * 16);
      const uint64_t dHh = smem_desc(smem_u32(sHh), 1024, 128), dHl = smem_desc(smem_u32(sHl), 1024, 128);
      // G: M = 64 (t), N = 64 (s), K = N (n); A = C K-major, B = the B tile read K-major
      // (its rows s hold 8 consecutive states per 16 bytes: 128 bytes between state groups,
      // N * 16 between row groups)
#pragma unroll
      for (int kk = 0; kk < N / 16; kk++)
        mma_f16(tmem + kColYd, dC + kk * (2048 >> 4), dBk + kk * (256 >> 4), kIdYo, kk > 0);
      // Yo: M = 64 (t), N = 64 (p), K = N (n); A = C K-major, B = H K-major
#pragma unroll
      for (int kk = 0; kk < N / 16; kk++) {
        const uint64_t da = dC + kk * (2048 >> 4);
        mma_f16(tmem + kColYo, da, dHh + kk * (2048 >> 4), kIdYo, kk > 0);
        mma_f16(tmem + kColYo, da, dHl + kk * (2048 >> 4), kIdYo, 1);
      }
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                   ::"r"(smem_u32(bar)) : "memory");
    }
    // ---- w x as hi / lo, in x's layout (MN-major [t][p]), while the first MMA group runs
#pragma unroll
    for (int i = 0; i < kQ * kP / 8 / kThreads; i++) {
      const int q = tid + i * kThreads;
      const int t = q % kQ, pb = q / kQ;
      const int off = pb * 128 + (t / 8) * 1024 + 16 * (t % 8);
      const uint4 xv = *reinterpret_cast<const uint4*>(sX + off);
      const float w = cW[t];
      const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; e++) {
        const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&xw[e]);
        split_pair(__bfloat162float(v.x) * w, __bfloat162float(v.y) * w, hi[e], lo[e]);
      }
      *reinterpret_cast<uint4*>(sWXh + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(sWXl + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    ok = __syncthreads_and(mbar_wait(smem_u32(bar), phase)) != 0;
    phase ^= 1;
    tc_after_sync();
    if (!ok) break;  // the status word reports it below
    // ---- M = G delta_s 2^{S_t - S_s} (s <= t) as hi / lo, K-major [t][s], from this thread's
    // fragment of G: rows rA, rB, columns s = p0 + 8 j + 2 tq (+1)
    {
      uint32_t gv[16];
      tmem_ld<4>(tmem + tlane + kColYd + p0, gv);
      tmem_wait_ld();
#pragma unroll
      for (int half = 0; half < 2; half++) {
        const int r = half ? rB : rA;
        const float st = cS[r];
#pragma unroll
        for (int j = 0; j < 4; j++) {
          const int s = p0 + 8 * j + 2 * tq;
          const float2 ss = *reinterpret_cast<const float2*>(cS + s);
          const float2 dd = *reinterpret_cast<const float2*>(cDt + s);
          const float m0 = s <= r ? __uint_as_float(gv[4 * j + 2 * half]) * dd.x * ex2(st - ss.x) : 0.f;
          const float m1 = s + 1 <= r ? __uint_as_float(gv[4 * j + 2 * half + 1]) * dd.y * ex2(st - ss.y) : 0.f;
          uint32_t hi, lo;
          split_pair(m0, m1, hi, lo);
          const int off = (r / 8) * 128 + (p0 / 8 + j) * 1024 + 16 * (r % 8) + 4 * tq;
          *reinterpret_cast<uint32_t*>(sMh + off) = hi;
          *reinterpret_cast<uint32_t*>(sMl + off) = lo;
        }
      }
    }
    fence_async_smem();
    tc_before_sync();
    __syncthreads();  // M and w x are in shared memory; G has been read
    tc_after_sync();

    // ---- second MMA group: Yd = M x (over G's columns) and S = (w x)^T B
    if (tid == kIssuer) {
      const uint64_t dX = smem_desc(smem_u32(sX), 1024, 128);
      const uint64_t dMh = smem_desc(smem_u32(sMh), 1024, 128), dMl = smem_desc(smem_u32(sMl), 1024, 128);
      const uint64_t dBm = smem_desc(smem_u32(sB), N * 16, 128);
      const uint64_t dWh = smem_desc(smem_u32(sWXh), 1024, 128), dWl = smem_desc(smem_u32(sWXl), 1024, 128);
      // Yd: M = 64 (t), N = 64 (p), K = 64 (s); A = M K-major, B = x MN-major
#pragma unroll
      for (int kk = 0; kk < kQ / 16; kk++) {
        const uint64_t db = dX + kk * (2048 >> 4);
        mma_f16(tmem + kColYd, dMh + kk * (2048 >> 4), db, kIdYd, kk > 0);
        mma_f16(tmem + kColYd, dMl + kk * (2048 >> 4), db, kIdYd, 1);
      }
      // S: M = 64 (p), N = N (n), K = 64 (t); A = w x MN-major, B MN-major
#pragma unroll
      for (int kk = 0; kk < kQ / 16; kk++) {
        const uint64_t db = dBm + kk * ((2 * (N * 16)) >> 4);
        mma_f16(tmem + kColS, dWh + kk * (2048 >> 4), db, kIdS, kk > 0);
        mma_f16(tmem + kColS, dWl + kk * (2048 >> 4), db, kIdS, 1);
      }
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                   ::"r"(smem_u32(bar)) : "memory");
    }
    // the next chunk's decays while the products run
    if (warp == 0 && t0 + kQ < t_end) {
      chunk_decays(p, h, t0 + kQ, dt_raw, lane, sDt + (par ^ 1) * kQ, sS + (par ^ 1) * kQ, sW + (par ^ 1) * kQ);
      if (t0 + 2 * kQ < t_end) dt_raw = load_dt_pair(p, b, h, t0 + 2 * kQ, lane);
    }
    ok = __syncthreads_and(mbar_wait(smem_u32(bar), phase)) != 0;  // one decision for the CTA
    phase ^= 1;
    tc_after_sync();
    if (!ok) break;  // the outputs of this call are invalid; nothing is left in flight but copies
    // this thread's x pairs for the skip term; then B, C and x are free: the next chunk's rows
    // are requested now, and land while this chunk's outputs and state are worked out
    uint32_t xr[2][4];
#pragma unroll
    for (int half = 0; half < 2; half++) {
      const int r = half ? rB : rA;
#pragma unroll
      for (int j = 0; j < 4; j++)
        xr[half][j] = *reinterpret_cast<const uint32_t*>(sX + (p0 / 8 + j) * 128 + (r / 8) * 1024 + 16 * (r % 8) + 4 * tq);
    }
    __syncthreads();  // every thread has its x pairs
    if (t0 + kQ < t_end) {
      load_bc(t0 + kQ);
      load_x(t0 + kQ);
    }
    cp_async_commit();

    // ---- y = (2^{S_t} Yo + Yd + D x) silu(z), staged per row, then written as 16-byte pieces
    {
      uint32_t yo[16], yd[16];
      tmem_ld<4>(tmem + tlane + kColYo + p0, yo);
      tmem_ld<4>(tmem + tlane + kColYd + p0, yd);
      tmem_wait_ld();
#pragma unroll
      for (int half = 0; half < 2; half++) {
        const int r = half ? rB : rA;
        const float sc = ex2(cS[r]);
#pragma unroll
        for (int j = 0; j < 4; j++) {
          const int pc = p0 + 8 * j + 2 * tq;
          const __nv_bfloat162 xx = *reinterpret_cast<const __nv_bfloat162*>(&xr[half][j]);
          const float2 dd = *reinterpret_cast<const float2*>(sD + pc);
          float v0 = fmaf(sc, __uint_as_float(yo[4 * j + 2 * half]), __uint_as_float(yd[4 * j + 2 * half]));
          float v1 = fmaf(sc, __uint_as_float(yo[4 * j + 2 * half + 1]), __uint_as_float(yd[4 * j + 2 * half + 1]));
          v0 = fmaf(dd.x, __bfloat162float(xx.x), v0);
          v1 = fmaf(dd.y, __bfloat162float(xx.y), v1);
          if (p.z) {
            const __nv_bfloat162 zz = *reinterpret_cast<const __nv_bfloat162*>(&zr[half][j]);
            v0 *= silu(__bfloat162float(zz.x));
            v1 *= silu(__bfloat162float(zz.y));
          }
          *reinterpret_cast<__nv_bfloat162*>(sY + r * kStageRow + pc) = __floats2bfloat162_rn(v0, v1);
        }
      }
    }
    __syncthreads();  // staging complete
#pragma unroll
    for (int i = 0; i < kQ * kP / 8 / kThreads; i++) {
      const int q = tid + i * kThreads;
      const int t = q / 8, j = q % 8;
      if (t < rows)
        *reinterpret_cast<uint4*>(p.y + act0 + (int64_t)t * p.d_inner + 8 * j) =
            *reinterpret_cast<const uint4*>(sY + t * kStageRow + 8 * j);
    }

    // ---- H = 2^{S_last} H + S, then H (hi / lo) into shared memory for the next readout
    {
      uint32_t sv[N / 4];
      tmem_ld<N / 16>(tmem + tlane + kColS + n0, sv);
      tmem_wait_ld();
      const float decay = ex2(cS[kQ - 1]);
#pragma unroll
      for (int j = 0; j < kHJ; j++)
#pragma unroll
        for (int e = 0; e < 4; e++) H[j][e] = fmaf(decay, H[j][e], __uint_as_float(sv[4 * j + e]));
    }
    tc_before_sync();
    __syncthreads();  // every thread has read this chunk's accumulators and the staging tile
    store_state();
  }
  cp_async_wait_all();
  if (!ok && tid == 0) atomicMax(p.header, (p.tag << 8) | (unsigned long long)kLookbackTimeoutCode);

  if (t_end < p.L) {
    // hand the state over to the next part (also after a wait that ran out: the next part
    // must not wait in vain; the call's outputs are invalid then anyway)
#pragma unroll
    for (int half = 0; half < 2; half++) {
      const int r = half ? rB : rA;
      float* out = p.hand + (b * p.d_inner + (int64_t)h * kP + r) * N + n0;
#pragma unroll
      for (int j = 0; j < kHJ; j++)
        __stcg(reinterpret_cast<float2*>(out + 8 * j + 2 * tq), make_float2(H[j][2 * half], H[j][2 * half + 1]));
    }
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      st_release_u64(p.flags + chain, (p.tag << 8) | (unsigned long long)(part + 1));
    }
  } else if (ok && p.last_state) {
#pragma unroll
    for (int half = 0; half < 2; half++) {
      const int r = half ? rB : rA;
      float* out = p.last_state + (b * p.d_inner + (int64_t)h * kP + r) * N + n0;
#pragma unroll
      for (int j = 0; j < kHJ; j++)
        *reinterpret_cast<float2*>(out + 8 * j + 2 * tq) = make_float2(H[j][2 * half], H[j][2 * half + 1]);
    }
  }
  tc_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_after_sync();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols));
  }
}

template <int N>
cudaError_t launch_n(const SsdParams& p, cudaStream_t s) {
  constexpr int smem = Smem<N>::kAlloc;
  cudaError_t e = cudaFuncSetAttribute(ssd_tc_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ssd_tc_kernel<N>, kThreads, smem);
  if (e != cudaSuccess) return e;
  // time parts as for the mma.sync chain: two unless the chains spread evenly over the SMs
  const int64_t chains = p.batch * p.heads;
  const int64_t n_chunks = (p.L + kQ - 1) / kQ;
  const int64_t slots = (int64_t)std::max(1, p.sms) * std::max(1, per_sm);
  const bool even = chains % slots == 0 || (chains <= slots && chains % std::max(1, p.sms) == 0);
  int parts = even ? 1 : 2;
  if (const char* v = std::getenv("SSM_SSD_PARTS")) {
    const int f = std::atoi(v);
    if (f >= 1 && f <= 64) parts = f;
  }
  while (parts > 1 && (int64_t)parts * chains > 0x7FFFFFFF) parts--;
  const int64_t chunks_per_part = (n_chunks + parts - 1) / parts;
  parts = (int)((n_chunks + chunks_per_part - 1) / chunks_per_part);
  ssd_tc_kernel<N><<<(unsigned)(parts * chains), kThreads, smem, s>>>(p, chunks_per_part * kQ);
  return cudaGetLastError();
}

}  // namespace ssdtc

cudaError_t launch_ssd_tc(const SsdParams& p, cudaStream_t s) {
  switch (p.N) {
    case 16: return ssdtc::launch_n<16>(p, s);
    case 32: return ssdtc::launch_n<32>(p, s);
    case 64: return ssdtc::launch_n<64>(p, s);
    case 128: return ssdtc::launch_n<128>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ssm
