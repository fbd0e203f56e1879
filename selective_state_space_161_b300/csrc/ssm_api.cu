// C ABI of libssm (declared in include/ssm.h): argument validation, the
// chunking plan, and dispatch to the kernels on the caller's stream.

#include "ssm.h"
#include "ssm_internal.h"

#include <cuda_runtime.h>

#include <mutex>

namespace {

constexpr int kMaxState = 16;
constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices] = {0};

// SM count of the current device (cached per device), or 0 if there is no usable device.
int current_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  if (dev < kMaxDevices && g_sm_count[dev] > 0) return g_sm_count[dev];
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev < kMaxDevices) g_sm_count[dev] = sms;
  return sms;
}

bool aligned16(const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

ssm_status_t check_common(int64_t batch, int64_t L, int64_t d_inner, int d_state, ssm_dtype_t io) {
  if (io != SSM_F32 && io != SSM_BF16) return SSM_ERR_DTYPE;
  if (batch < 0 || L < 0 || d_inner < 0) return SSM_ERR_SHAPE;
  if (d_state < 1 || d_state > kMaxState) return SSM_ERR_SHAPE;
  if (d_inner % (io == SSM_BF16 ? 8 : 4) != 0) return SSM_ERR_SHAPE;
  // Keep every flat index below 2^62 and every grid below 2^31 blocks.
  const int64_t lim = (int64_t)1 << 62;
  if (batch > 0 && d_inner > 0 && (batch > lim / d_inner || (L > 0 && batch * d_inner > lim / L)))
    return SSM_ERR_SHAPE;
  if (batch * d_inner * kMaxState > lim) return SSM_ERR_SHAPE;
  return SSM_OK;
}

size_t scan_workspace_bytes(int64_t batch, int64_t L, int64_t d_inner, int d_state, int sms,
                            ssm::ScanPlan* plan) {
  ssm::plan_scan(batch, L, d_inner, sms, plan);
  if (plan->n_chunks <= 1) return 0;
  return (size_t)batch * (size_t)(plan->n_chunks - 1) * (size_t)d_inner * (size_t)(d_state + 1) *
         sizeof(float);
}

}  // namespace

extern "C" {

size_t ssm_scan_fwd_workspace_size(int64_t batch, int64_t L, int64_t d_inner, int d_state,
                                   ssm_dtype_t io) {
  if (check_common(batch, L, d_inner, d_state, io) != SSM_OK) return 0;
  const int sms = current_sm_count();
  if (sms <= 0) return 0;
  ssm::ScanPlan plan;
  return scan_workspace_bytes(batch, L, d_inner, d_state, sms, &plan);
}

}  // extern "C"

namespace {

// Optional parts of a scan call beyond ssm_scan_fwd's operands.
struct ScanExtras {
  const float* initial_state = nullptr;
  const float* conv_w = nullptr;  // non-null: conv1d + SiLU in front, u holds the block input x
  const float* conv_b = nullptr;
  int d_conv = 0;
  void* u_out = nullptr;
};

ssm_status_t scan_fwd_impl(const void* u, const void* delta, const float* A, const void* B,
                           const void* C, const float* D, const void* z, const float* delta_bias,
                           int softplus_flag, const ScanExtras& ex, void* y, float* last_state,
                           int64_t batch, int64_t L, int64_t d_inner, int d_state, ssm_dtype_t io,
                           void* workspace, size_t workspace_bytes, void* stream) {
  const float* initial_state = ex.initial_state;
  ssm_status_t st = check_common(batch, L, d_inner, d_state, io);
  if (st != SSM_OK) return st;
  const int64_t channels = batch * d_inner;
  if (channels == 0) return SSM_OK;
  if (A == nullptr) return SSM_ERR_NULL;
  if (L > 0 && (!u || !delta || !B || !C || !y)) return SSM_ERR_NULL;
  if (ex.conv_w != nullptr && (ex.d_conv < 1 || ex.d_conv > 4)) return SSM_ERR_SHAPE;
  const void* ptrs[] = {u, delta, A, B, C, D, z, delta_bias, y, last_state, workspace,
                        initial_state, ex.conv_w, ex.conv_b, ex.u_out};
  for (const void* q : ptrs)
    if (!aligned16(q)) return SSM_ERR_ALIGN;
  const int sms = current_sm_count();
  if (sms <= 0) return SSM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  if (L == 0) {
    const size_t bytes = (size_t)channels * d_state * sizeof(float);
    if (last_state && initial_state) {
      if (last_state != initial_state &&
          cudaMemcpyAsync(last_state, initial_state, bytes, cudaMemcpyDeviceToDevice, s) !=
              cudaSuccess)
        return SSM_ERR_CUDA;
    } else if (last_state && cudaMemsetAsync(last_state, 0, bytes, s) != cudaSuccess) {
      return SSM_ERR_CUDA;
    }
    return SSM_OK;
  }

  ssm::ScanParams p{};
  ssm::ScanPlan plan;
  const size_t need = scan_workspace_bytes(batch, L, d_inner, d_state, sms, &plan);
  p.chunk_len = plan.chunk_len;
  p.n_chunks = plan.n_chunks;
  p.lanes = plan.lanes;
  if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return SSM_ERR_WORKSPACE;
  const int64_t cpc = ssm::scan_channels_per_cta();
  const int64_t n_dtiles = (d_inner + cpc - 1) / cpc;
  if (n_dtiles * p.n_chunks * batch >= ((int64_t)1 << 31)) return SSM_ERR_SHAPE;
  p.u = u; p.delta = delta; p.A = A; p.B = B; p.C = C; p.D = D; p.z = z;
  p.delta_bias = delta_bias; p.softplus = softplus_flag != 0; p.y = y; p.last_state = last_state;
  p.initial_state = initial_state;
  p.conv_w = ex.conv_w; p.conv_b = ex.conv_b; p.d_conv = ex.d_conv; p.u_out = ex.u_out;
  p.batch = batch; p.L = L; p.d_inner = d_inner; p.d_state = d_state;
  if (p.n_chunks > 1) {
    p.ws_S = static_cast<float*>(workspace);
    p.ws_h = p.ws_S + (size_t)batch * (p.n_chunks - 1) * d_inner;
  }
  return ssm::launch_scan(p, io == SSM_BF16, s) == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

}  // namespace

extern "C" {

ssm_status_t ssm_scan_fwd(const void* u, const void* delta, const float* A, const void* B,
                          const void* C, const float* D, const void* z, const float* delta_bias,
                          int softplus_flag, void* y, float* last_state, int64_t batch, int64_t L,
                          int64_t d_inner, int d_state, ssm_dtype_t io, void* workspace,
                          size_t workspace_bytes, void* stream) {
  return scan_fwd_impl(u, delta, A, B, C, D, z, delta_bias, softplus_flag, ScanExtras{}, y,
                       last_state, batch, L, d_inner, d_state, io, workspace, workspace_bytes,
                       stream);
}

ssm_status_t ssm_scan_fwd_from_state(const void* u, const void* delta, const float* A,
                                     const void* B, const void* C, const float* D, const void* z,
                                     const float* delta_bias, int softplus_flag,
                                     const float* initial_state, void* y, float* last_state,
                                     int64_t batch, int64_t L, int64_t d_inner, int d_state,
                                     ssm_dtype_t io, void* workspace, size_t workspace_bytes,
                                     void* stream) {
  ScanExtras ex;
  ex.initial_state = initial_state;
  return scan_fwd_impl(u, delta, A, B, C, D, z, delta_bias, softplus_flag, ex, y, last_state,
                       batch, L, d_inner, d_state, io, workspace, workspace_bytes, stream);
}

ssm_status_t ssm_scan_fwd_conv(const void* x, const float* conv_weight, const float* conv_bias,
                               int d_conv, const void* delta, const float* A, const void* B,
                               const void* C, const float* D, const void* z,
                               const float* delta_bias, int softplus_flag,
                               const float* initial_state, void* y, float* last_state,
                               void* u_out, int64_t batch, int64_t L, int64_t d_inner,
                               int d_state, ssm_dtype_t io, void* workspace,
                               size_t workspace_bytes, void* stream) {
  if (conv_weight == nullptr && batch * d_inner > 0) return SSM_ERR_NULL;
  ScanExtras ex;
  ex.initial_state = initial_state;
  ex.conv_w = conv_weight;
  ex.conv_b = conv_bias;
  ex.d_conv = d_conv;
  ex.u_out = u_out;
  return scan_fwd_impl(x, delta, A, B, C, D, z, delta_bias, softplus_flag, ex, y, last_state,
                       batch, L, d_inner, d_state, io, workspace, workspace_bytes, stream);
}

}  // extern "C"

namespace {

ssm_status_t state_update_impl(float* state, float* conv_state, const void* u,
                               const float* conv_w, const float* conv_b, int d_conv,
                               const void* delta, const float* A, const void* B, const void* C,
                               const float* D, const void* z, void* y, const float* delta_bias,
                               int softplus_flag, int64_t batch, int64_t d_inner, int d_state,
                               ssm_dtype_t io, void* stream) {
  ssm_status_t st = check_common(batch, 1, d_inner, d_state, io);
  if (st != SSM_OK) return st;
  const int64_t channels = batch * d_inner;
  if (channels == 0) return SSM_OK;
  if (!state || !u || !delta || !A || !B || !C || !y) return SSM_ERR_NULL;
  if (conv_w != nullptr) {
    if (d_conv < 1 || d_conv > 4) return SSM_ERR_SHAPE;
    if (d_conv > 1 && conv_state == nullptr) return SSM_ERR_NULL;
  }
  const void* ptrs[] = {state, u, delta, A, B, C, D, z, y, delta_bias, conv_state, conv_w, conv_b};
  for (const void* q : ptrs)
    if (!aligned16(q)) return SSM_ERR_ALIGN;
  if (current_sm_count() <= 0) return SSM_ERR_CUDA;
  if ((channels * 4 + 255) / 256 >= ((int64_t)1 << 31)) return SSM_ERR_SHAPE;
  ssm::DecodeParams p{};
  p.state = state; p.u = u; p.delta = delta; p.A = A; p.B = B; p.C = C; p.D = D; p.z = z; p.y = y;
  p.delta_bias = delta_bias; p.softplus = softplus_flag != 0;
  p.batch = batch; p.d_inner = d_inner; p.d_state = d_state;
  p.conv_w = conv_w; p.conv_b = conv_b; p.d_conv = d_conv; p.conv_state = conv_state;
  return ssm::launch_state_update(p, io == SSM_BF16, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SSM_OK
             : SSM_ERR_CUDA;
}

}  // namespace

extern "C" {

ssm_status_t ssm_state_update(float* state, const void* u, const void* delta, const float* A,
                              const void* B, const void* C, const float* D, const void* z,
                              void* y, const float* delta_bias, int softplus_flag, int64_t batch,
                              int64_t d_inner, int d_state, ssm_dtype_t io, void* stream) {
  return state_update_impl(state, nullptr, u, nullptr, nullptr, 0, delta, A, B, C, D, z, y,
                           delta_bias, softplus_flag, batch, d_inner, d_state, io, stream);
}

ssm_status_t ssm_state_update_conv(float* state, float* conv_state, const void* x,
                                   const float* conv_weight, const float* conv_bias, int d_conv,
                                   const void* delta, const float* A, const void* B,
                                   const void* C, const float* D, const void* z, void* y,
                                   const float* delta_bias, int softplus_flag, int64_t batch,
                                   int64_t d_inner, int d_state, ssm_dtype_t io, void* stream) {
  if (conv_weight == nullptr && batch * d_inner > 0) return SSM_ERR_NULL;
  return state_update_impl(state, conv_state, x, conv_weight, conv_bias, d_conv, delta, A, B, C,
                           D, z, y, delta_bias, softplus_flag, batch, d_inner, d_state, io,
                           stream);
}

}  // extern "C"

namespace {

// Time chunking of the backward pass: the forward plan's chunks, rounded to whole tiles.
void bwd_plan(int64_t batch, int64_t L, int64_t d_inner, int sms, ssm::ScanPlan* plan) {
  ssm::plan_scan(batch, L, d_inner, sms, plan);
  plan->lanes = 1;
}

}  // namespace

extern "C" {

size_t ssm_scan_bwd_workspace_size(int64_t batch, int64_t L, int64_t d_inner, int d_state,
                                   ssm_dtype_t io) {
  if (check_common(batch, L, d_inner, d_state, io) != SSM_OK) return 0;
  const int sms = current_sm_count();
  if (sms <= 0 || batch * d_inner * L == 0) return 0;
  ssm::ScanPlan plan;
  bwd_plan(batch, L, d_inner, sms, &plan);
  return ssm::bwd_workspace_floats(batch, L, d_inner, d_state, plan.n_chunks) * sizeof(float);
}

ssm_status_t ssm_scan_bwd(const void* u, const void* delta, const float* A, const void* B,
                          const void* C, const float* D, const void* z, const float* delta_bias,
                          int softplus_flag, const float* initial_state, const void* dy,
                          const float* dlast_state, void* du, void* ddelta, float* dA, float* dB,
                          float* dC, float* dD, void* dz, float* ddelta_bias,
                          float* dinitial_state, int64_t batch, int64_t L, int64_t d_inner,
                          int d_state, ssm_dtype_t io, void* workspace, size_t workspace_bytes,
                          void* stream) {
  ssm_status_t st = check_common(batch, L, d_inner, d_state, io);
  if (st != SSM_OK) return st;
  const int64_t channels = batch * d_inner;
  if (channels == 0) return SSM_OK;
  if (!A || !dA) return SSM_ERR_NULL;
  if (L > 0 && (!u || !delta || !B || !C || !dy || !du || !ddelta || !dB || !dC)) return SSM_ERR_NULL;
  if ((D != nullptr) != (dD != nullptr) || (z != nullptr) != (dz != nullptr)) return SSM_ERR_NULL;
  const void* ptrs[] = {u, delta, A, B, C, D, z, delta_bias, initial_state, dy, dlast_state, du,
                        ddelta, dA, dB, dC, dD, dz, ddelta_bias, dinitial_state, workspace};
  for (const void* q : ptrs)
    if (!aligned16(q)) return SSM_ERR_ALIGN;
  const int sms = current_sm_count();
  if (sms <= 0) return SSM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // accumulated outputs start at zero
  if (cudaMemsetAsync(dA, 0, (size_t)d_inner * d_state * sizeof(float), s) != cudaSuccess)
    return SSM_ERR_CUDA;
  if (dD && cudaMemsetAsync(dD, 0, (size_t)d_inner * sizeof(float), s) != cudaSuccess)
    return SSM_ERR_CUDA;
  if (ddelta_bias && cudaMemsetAsync(ddelta_bias, 0, (size_t)d_inner * sizeof(float), s) != cudaSuccess)
    return SSM_ERR_CUDA;
  if (L == 0) {  // nothing flows: dinit = dlast
    const size_t bytes = (size_t)channels * d_state * sizeof(float);
    if (dinitial_state) {
      const cudaError_t e = dlast_state ? cudaMemcpyAsync(dinitial_state, dlast_state, bytes,
                                                          cudaMemcpyDeviceToDevice, s)
                                        : cudaMemsetAsync(dinitial_state, 0, bytes, s);
      if (e != cudaSuccess) return SSM_ERR_CUDA;
    }
    return SSM_OK;
  }
  const size_t bc_bytes = (size_t)batch * L * d_state * sizeof(float);
  if (cudaMemsetAsync(dB, 0, bc_bytes, s) != cudaSuccess || cudaMemsetAsync(dC, 0, bc_bytes, s) != cudaSuccess)
    return SSM_ERR_CUDA;

  ssm::ScanPlan plan;
  bwd_plan(batch, L, d_inner, sms, &plan);
  const size_t need = ssm::bwd_workspace_floats(batch, L, d_inner, d_state, plan.n_chunks) * sizeof(float);
  if (workspace == nullptr || workspace_bytes < need) return SSM_ERR_WORKSPACE;
  const int64_t tiles = (L + 15) / 16;
  if ((d_inner + 31) / 32 * tiles * batch >= ((int64_t)1 << 31)) return SSM_ERR_SHAPE;

  float* ws = static_cast<float*>(workspace);
  const int64_t ck = batch * tiles * d_inner * d_state;
  const int64_t fws = batch * (int64_t)(plan.n_chunks - 1) * d_inner;
  const int64_t rws = batch * (int64_t)plan.n_chunks * d_inner;
  ssm::BwdArgs a{};
  a.u = u; a.delta = delta; a.A = A; a.B = B; a.C = C; a.D = D; a.z = z; a.delta_bias = delta_bias;
  a.softplus = softplus_flag != 0; a.initial_state = initial_state; a.dy = dy; a.dlast = dlast_state;
  a.du = du; a.ddelta = ddelta; a.dz = dz; a.dA = dA; a.dB = dB; a.dC = dC; a.dD = dD;
  a.dbias = ddelta_bias; a.dinit = dinitial_state;
  a.batch = batch; a.L = L; a.d_inner = d_inner; a.d_state = d_state;
  a.chunk_len = plan.chunk_len; a.n_chunks = plan.n_chunks;
  a.ckpt_h = ws;
  float* fS = ws + ck;
  a.fws_S = fS;
  a.fws_h = fS + fws;
  float* rS = fS + fws * (d_state + 1);
  a.rws_S = rS;
  a.rws_m = rS + rws;

  ssm::ScanParams f{};
  f.u = u; f.delta = delta; f.A = A; f.B = B; f.C = C; f.delta_bias = delta_bias;
  f.softplus = softplus_flag != 0; f.batch = batch; f.L = L; f.d_inner = d_inner;
  f.d_state = d_state; f.chunk_len = plan.chunk_len; f.n_chunks = plan.n_chunks; f.lanes = 1;
  f.initial_state = initial_state;
  f.ws_S = fS;
  f.ws_h = fS + fws;
  return ssm::launch_scan_bwd(a, f, io == SSM_BF16, s) == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

size_t ssm_ssd_fwd_workspace_size(int64_t batch, int64_t L, int64_t d_inner, int n_heads,
                                  int d_state) {
  (void)batch; (void)L; (void)d_inner; (void)n_heads; (void)d_state;
  return 0;  // the state stays on chip: one CTA per (batch, head) walks that head's chunks
}

ssm_status_t ssm_ssd_fwd(const void* x, const void* dt, const float* A, const void* B,
                         const void* C, const float* D, const void* z, const float* dt_bias,
                         int softplus_flag, void* y, float* last_state, int64_t batch, int64_t L,
                         int64_t d_inner, int n_heads, int d_state, ssm_dtype_t io,
                         void* workspace, size_t workspace_bytes, void* stream) {
  if (io != SSM_BF16) return SSM_ERR_DTYPE;
  if (batch < 0 || L < 0 || d_inner < 0 || n_heads < 1) return SSM_ERR_SHAPE;
  if (d_state != 16 && d_state != 32 && d_state != 64 && d_state != 128) return SSM_ERR_SHAPE;
  if (d_inner != (int64_t)n_heads * ssm::ssd_head_dim()) return SSM_ERR_SHAPE;
  if (batch == 0) return SSM_OK;
  if (!A) return SSM_ERR_NULL;
  if (L > 0 && (!x || !dt || !B || !C || !y)) return SSM_ERR_NULL;
  const void* ptrs[] = {x, dt, A, B, C, D, z, dt_bias, y, last_state, workspace};
  for (const void* q : ptrs)
    if (!aligned16(q)) return SSM_ERR_ALIGN;
  if (current_sm_count() <= 0) return SSM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (L == 0) {
    if (last_state &&
        cudaMemsetAsync(last_state, 0, (size_t)batch * d_inner * d_state * sizeof(float), s) != cudaSuccess)
      return SSM_ERR_CUDA;
    return SSM_OK;
  }
  (void)workspace_bytes;  // none needed
  ssm::SsdParams p{};
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.dt = static_cast<const __nv_bfloat16*>(dt);
  p.A = A;
  p.B = static_cast<const __nv_bfloat16*>(B);
  p.C = static_cast<const __nv_bfloat16*>(C);
  p.D = D;
  p.z = static_cast<const __nv_bfloat16*>(z);
  p.dt_bias = dt_bias;
  p.softplus = softplus_flag != 0;
  p.y = static_cast<__nv_bfloat16*>(y);
  p.last_state = last_state;
  p.batch = batch; p.L = L; p.d_inner = d_inner; p.heads = n_heads; p.N = d_state;
  if (batch * n_heads >= ((int64_t)1 << 31)) return SSM_ERR_SHAPE;
  return ssm::launch_ssd(p, s) == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

const char* ssm_status_string(ssm_status_t status) {
  switch (status) {
    case SSM_OK: return "ok";
    case SSM_ERR_NULL: return "a required pointer is NULL";
    case SSM_ERR_SHAPE: return "unsupported or inconsistent sizes";
    case SSM_ERR_DTYPE: return "unknown I/O dtype";
    case SSM_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case SSM_ERR_WORKSPACE: return "workspace missing or too small";
    case SSM_ERR_CUDA: return "CUDA error (no device or launch failure)";
    case SSM_ERR_SCRATCH_LIMIT:
      return "problem needs more scratch than ssm_scan_fwd_noalloc holds (use ssm_scan_fwd)";
  }
  return "unknown status";
}

int ssm_version(void) { return 100; }

}  // extern "C"

// ---------------------------------------------------------------------------------------
// No-allocation variant of ssm_scan_fwd.  Its scratch is this file-scope device array;
// host code must not hand the symbol itself to a kernel (on the host it only names a
// host-side shadow), so its device address is looked up per device, once, below.

static __device__ __align__(256) float g_noalloc_scratch[SSM_NOALLOC_SCRATCH_BYTES / sizeof(float)];

namespace {

std::mutex g_noalloc_mutex;
float* g_noalloc_addr[kMaxDevices] = {nullptr};

// Device address of g_noalloc_scratch on the current device (looked up on first use).
float* noalloc_scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_addr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return nullptr;
    g_noalloc_addr[dev] = static_cast<float*>(ptr);
  }
  return g_noalloc_addr[dev];
}

}  // namespace

extern "C" {

ssm_status_t ssm_scan_fwd_noalloc(const void* u, const void* delta, const float* A,
                                  const void* B, const void* C, const float* D, const void* z,
                                  const float* delta_bias, int softplus_flag, void* y,
                                  float* last_state, int64_t batch, int64_t L, int64_t d_inner,
                                  int d_state, ssm_dtype_t io, void* stream) {
  ssm_status_t st = check_common(batch, L, d_inner, d_state, io);
  if (st != SSM_OK) return st;
  if (batch * d_inner == 0) return SSM_OK;
  const int sms = current_sm_count();
  if (sms <= 0) return SSM_ERR_CUDA;
  ssm::ScanPlan plan;
  const size_t need = L > 0 ? scan_workspace_bytes(batch, L, d_inner, d_state, sms, &plan) : 0;
  if (need > SSM_NOALLOC_SCRATCH_BYTES) return SSM_ERR_SCRATCH_LIMIT;
  float* scratch = nullptr;
  if (need > 0) {
    scratch = noalloc_scratch_address();
    if (scratch == nullptr) return SSM_ERR_CUDA;
  }
  return ssm_scan_fwd(u, delta, A, B, C, D, z, delta_bias, softplus_flag, y, last_state, batch, L,
                      d_inner, d_state, io, scratch, need, stream);
}

}  // extern "C"
