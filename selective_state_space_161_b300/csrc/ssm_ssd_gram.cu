// Chunk Gram matrices G = C B^T of the chunked SSD form, on the 5th-generation tensor cores.
//
// In the chunked form (youngju.dev, "Mamba: Linear-Time Sequence Modeling with Selective State
// Spaces 论文分析", section "后续研究：Mamba-2 与混合架构"; the reading is spelled out in
// ssm_ssd.cu) the intra-chunk output of every head needs G[i][j] = C_i . B_j for the steps i, j
// of a chunk.  B and C are shared by all heads (one group), so G depends only on the batch row
// and the chunk: it is computed here once and read by every head's CTA, instead of once per
// head.
//
// One CTA per (batch row, pair of consecutive chunks): the 128 rows of C and of B of the two
// chunks arrive in shared memory by TMA (cp.async.bulk.tensor, boxes of 8 states x 128 steps,
// i.e. the tensor core's canonical K-major layout without swizzle: 8-row x 16-byte core
// matrices, 16 bytes between rows, 2048 bytes between groups of 8 states); one thread issues
// d_state/16 tcgen05.mma (M = N = 128, K = 16, bf16 in, fp32 accumulate) into tensor memory;
// the four warps read their 32 rows back (tcgen05.ld) and store the two diagonal 64 x 64 blocks
// (the off-diagonal blocks pair steps of different chunks and are not needed).  Waits on the
// copy and MMA barriers are bounded: a wait that runs out leaves G unwritten, raises the call's
// status word to code 7 (read by ssm_get_status) and never hangs.

#include "ssm_device.cuh"
#include "ssm_internal.h"

#include <cuda.h>

#include <mutex>

namespace ssm {
namespace gram {

constexpr int kRows = 128;       // two chunks of 64 steps
constexpr int kThreads = 128;
constexpr unsigned kMaxPolls = 1u << 22;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Shared-memory matrix descriptor (tcgen05): start address, byte distance between core
// matrices along K (leading) and along M/N (stride), descriptor version 1, no swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46);
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (unsigned it = 0; it < kMaxPolls; it++) {
    uint32_t done;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

struct Args {
  float* G;      // [batch][chunks][64][64]
  int64_t batch, L;
  int chunks, N;
  unsigned long long* header;  // status word: (tag << 8) | code
  unsigned long long tag;
};

template <int N>
__global__ void __launch_bounds__(kThreads) gram_kernel(const __grid_constant__ CUtensorMap tmC,
                                                        const __grid_constant__ CUtensorMap tmB,
                                                        const Args a) {
  extern __shared__ __align__(1024) unsigned char smem[];
  constexpr int kTileB = kRows * N * 2;   // one operand, bf16
  unsigned char* sC = smem;
  unsigned char* sB = smem + kTileB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 2 * kTileB);  // [0] copies, [1] MMA
  uint32_t* taddr = reinterpret_cast<uint32_t*>(smem + 2 * kTileB + 16);
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int64_t b = blockIdx.y;
  const int c0 = 2 * blockIdx.x;
  const int row0 = (int)(b * a.L + (int64_t)c0 * 64);  // first global row (step) of the pair

  if (blockIdx.x == 0 && blockIdx.y == 0 && tid == 0) atomicExch(a.header, a.tag << 8);  // this call's status: ok
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bars[0])));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bars[1])));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 128;" ::"r"(smem_u32(taddr)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *taddr;

  if (tid == 0) {
    // C and B rows of the two chunks, 8 states (16 bytes) x 128 steps per box
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(&bars[0])),
                 "r"(2 * kTileB)
                 : "memory");
#pragma unroll
    for (int kg = 0; kg < N / 8; kg++) {
      asm volatile(
          "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
          ::"r"(smem_u32(sC + kg * kRows * 16)), "l"(&tmC), "r"(8 * kg), "r"(row0), "r"(smem_u32(&bars[0]))
          : "memory");
      asm volatile(
          "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
          ::"r"(smem_u32(sB + kg * kRows * 16)), "l"(&tmB), "r"(8 * kg), "r"(row0), "r"(smem_u32(&bars[0]))
          : "memory");
    }
  }
  const bool loaded = mbar_wait(smem_u32(&bars[0]), 0);

  if (tid == 0 && loaded) {
    // D (128 x 128, fp32) = C (128 x N) B^T: instruction descriptor: fp32 D, bf16 A and B, both
    // K-major, N = 128, M = 128
    const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kRows >> 3) << 17) |
                           ((uint32_t)(kRows >> 4) << 24);
    constexpr uint32_t kLbo = kRows * 16, kSbo = 128;
#pragma unroll
    for (int kk = 0; kk < N / 16; kk++) {
      const uint64_t da = smem_desc(smem_u32(sC) + kk * 2 * kLbo, kLbo, kSbo);
      const uint64_t db = smem_desc(smem_u32(sB) + kk * 2 * kLbo, kLbo, kSbo);
      asm volatile(
          "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
          ::"r"(tmem), "l"(da), "l"(db), "r"(idesc), "r"(kk > 0 ? 1u : 0u)
          : "memory");
    }
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(smem_u32(&bars[1]))
                 : "memory");
  }
  const bool done = loaded && mbar_wait(smem_u32(&bars[1]), 0);
  if (!done && tid == 0) atomicMax(a.header, (a.tag << 8) | (unsigned long long)kLookbackTimeoutCode);
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

  // Warp w reads rows 32 w .. 32 w + 31 (TMEM lanes); rows < 64 belong to chunk c0 (columns
  // 0 .. 63), the others to chunk c0 + 1 (columns 64 .. 127).
  const int r = 32 * warp + lane;
  const int half = r / 64, i = r % 64;
  const int c = c0 + half;
  if (done) {
#pragma unroll
    for (int q = 0; q < 4; q++) {
      uint32_t v[16];
      const uint32_t ta = tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)(64 * half + 16 * q);
      asm volatile(
          "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
          : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
            "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
          : "r"(ta));
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      if (c < a.chunks) {
        float4* dst = reinterpret_cast<float4*>(a.G + (((b * a.chunks + c) * 64 + i) * 64 + 16 * q));
#pragma unroll
        for (int m = 0; m < 4; m++)
          dst[m] = make_float4(__uint_as_float(v[4 * m]), __uint_as_float(v[4 * m + 1]),
                               __uint_as_float(v[4 * m + 2]), __uint_as_float(v[4 * m + 3]));
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 128;" ::"r"(tmem));
  }
}

// ---- host side: the TMA descriptors (driver entry point fetched through the runtime)

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// [rows][N] bf16, boxes of 8 columns x 128 rows; rows past the end read as zero.
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int N) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)N * 2};
  const cuuint32_t box[2] = {8, (cuuint32_t)kRows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int N>
cudaError_t launch_n(const CUtensorMap& mc, const CUtensorMap& mb, const Args& a, cudaStream_t s) {
  const int smem = 2 * kRows * N * 2 + 64;
  cudaError_t e = cudaFuncSetAttribute(gram_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)((a.chunks + 1) / 2), (unsigned)a.batch);
  gram_kernel<N><<<grid, kThreads, smem, s>>>(mc, mb, a);
  return cudaGetLastError();
}

}  // namespace gram

size_t ssd_gram_bytes(int64_t batch, int64_t L) {
  return (size_t)batch * (size_t)((L + 63) / 64) * 64 * 64 * sizeof(float);
}

cudaError_t launch_ssd_gram(const __nv_bfloat16* C, const __nv_bfloat16* B, float* G, int64_t batch,
                            int64_t L, int N, unsigned long long* header, unsigned long long tag,
                            cudaStream_t s) {
  CUtensorMap mc, mb;
  if (!gram::make_map(&mc, C, batch * L, N) || !gram::make_map(&mb, B, batch * L, N))
    return cudaErrorInvalidValue;
  gram::Args a{G, batch, L, (int)((L + 63) / 64), N, header, tag};
  switch (N) {
    case 16: return gram::launch_n<16>(mc, mb, a, s);
    case 32: return gram::launch_n<32>(mc, mb, a, s);
    case 64: return gram::launch_n<64>(mc, mb, a, s);
    case 128: return gram::launch_n<128>(mc, mb, a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ssm
