// C ABI of libssm (declared in include/ssm.h): argument validation, the
// chunking plan, and dispatch to the kernels on the caller's stream.

#include "ssm.h"
#include "ssm_internal.h"

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <chrono>
#include <cstdlib>
#include <mutex>
#include <random>

namespace {

constexpr int kMaxState = 16;
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];

// SM count of the current device (cached per device), or 0 if there is no usable device.
int current_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  if (dev < kMaxDevices) {
    const int c = g_sm_count[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev < kMaxDevices) g_sm_count[dev].store(sms, std::memory_order_relaxed);
  return sms;
}

// Per-call tags of the look-back records: a 54-bit counter that starts at a random value,
// so that records left in a reused workspace by earlier calls (or by another process's
// allocation) never pass for this call's.
uint64_t next_call_tag() {
  static std::atomic<uint64_t> counter{[] {
    std::random_device rd;
    const uint64_t t = (uint64_t)std::chrono::steady_clock::now().time_since_epoch().count();
    return (((uint64_t)rd() << 32) ^ (uint64_t)rd() ^ (t * 0x9E3779B97F4A7C15ull));
  }()};
  return counter.fetch_add(1, std::memory_order_relaxed) & ((1ull << 54) - 1);
}

// Look-back polls before a CTA gives up on a predecessor (about a second with the backoff).
unsigned lookback_max_polls() {
  if (const char* v = std::getenv("SSM_LOOKBACK_MAX_POLLS")) {
    const long long x = std::atoll(v);
    if (x > 0 && x < (1ll << 31)) return (unsigned)x;
  }
  return 1u << 20;
}

// Self-test of the bounded wait: with SSM_LOOKBACK_SELFTEST=1 the look-back waits for
// records of a tag that no CTA writes, so every wait runs out.
bool lookback_selftest() {
  const char* v = std::getenv("SSM_LOOKBACK_SELFTEST");
  return v != nullptr && v[0] == '1';
}

// The tag a call's waits accept: its own, or in the self-test one with bit 54 set, which no
// call ever writes (tags are 54-bit), whatever an earlier call left in a reused workspace.
uint64_t wait_tag_for(uint64_t tag) { return lookback_selftest() ? (tag | (1ull << 54)) : tag; }

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

// Workspace of a forward scan (0 for an empty problem); false if the plan cannot be made.
bool fwd_workspace(int64_t batch, int64_t L, int64_t d_inner, int d_state, bool bf16, int kind,
                   int sms, ssm::FwdPlan* plan, size_t* bytes) {
  *bytes = 0;
  if (batch * d_inner == 0 || L == 0) return true;
  if (!ssm::plan_scan_fwd(batch, L, d_inner, d_state, bf16, kind, sms, plan)) return false;
  *bytes = ssm::fwd_workspace_bytes(batch, d_inner, *plan);
  return true;
}

}  // namespace

extern "C" {

size_t ssm_scan_fwd_workspace_size(int64_t batch, int64_t L, int64_t d_inner, int d_state,
                                   ssm_dtype_t io) {
  if (check_common(batch, L, d_inner, d_state, io) != SSM_OK) return 0;
  const int sms = current_sm_count();
  if (sms <= 0) return 0;
  ssm::FwdPlan plan;
  size_t plain = 0, conv = 0;
  if (!fwd_workspace(batch, L, d_inner, d_state, io == SSM_BF16, ssm::kFwdPlain, sms, &plan, &plain) ||
      !fwd_workspace(batch, L, d_inner, d_state, io == SSM_BF16, ssm::kFwdConv, sms, &plan, &conv))
    return 0;
  return plain > conv ? plain : conv;
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

  const bool bf16 = io == SSM_BF16;
  const bool conv = ex.conv_w != nullptr;
  ssm::FwdPlan plan;
  size_t need = 0;
  if (!fwd_workspace(batch, L, d_inner, d_state, bf16, conv ? ssm::kFwdConv : ssm::kFwdPlain, sms, &plan,
                     &need))
    return SSM_ERR_CUDA;
  if (workspace == nullptr || workspace_bytes < need) return SSM_ERR_WORKSPACE;
  const int64_t n_dt = (d_inner + ssm::fwd_channels_per_cta() - 1) / ssm::fwd_channels_per_cta();
  if ((int64_t)plan.G * batch * n_dt >= ((int64_t)1 << 31)) return SSM_ERR_SHAPE;
  ssm::FwdLaunch f{};
  f.u = u; f.delta = delta; f.A = A; f.B = B; f.C = C; f.D = D; f.z = z;
  f.delta_bias = delta_bias; f.softplus = softplus_flag != 0; f.y = y; f.last_state = last_state;
  f.initial_state = initial_state;
  f.conv_w = ex.conv_w; f.conv_b = ex.conv_b; f.d_conv = ex.d_conv; f.u_out = ex.u_out;
  f.batch = batch; f.L = L; f.d_inner = d_inner; f.d_state = d_state;
  f.plan = plan;
  f.workspace = workspace;
  f.tag = next_call_tag();
  f.wait_tag = wait_tag_for(f.tag);
  f.max_polls = lookback_max_polls();
  return ssm::launch_scan_fwd(f, bf16, s) == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
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
  if ((d_inner + 63) / 64 >= ((int64_t)1 << 31)) return SSM_ERR_SHAPE;
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

// Workspace of a backward pass: the checkpoint kernel's look-back region (header first, so that
// ssm_get_status reads it), then the checkpoints and the reverse chunk summaries.
bool bwd_workspace(int64_t batch, int64_t L, int64_t d_inner, int d_state, bool bf16, int sms,
                   ssm::FwdPlan* fplan, ssm::BwdPlan* bplan, size_t* fwd_bytes, size_t* bytes) {
  ssm::plan_scan_bwd(batch, L, d_inner, sms, bplan);
  if (!fwd_workspace(batch, L, d_inner, d_state, bf16, ssm::kFwdCkpt, sms, fplan, fwd_bytes)) return false;
  *fwd_bytes = (*fwd_bytes + 255) / 256 * 256;
  *bytes = *fwd_bytes + ssm::bwd_workspace_floats(batch, L, d_inner, d_state, bplan->n_chunks) * sizeof(float);
  return true;
}

}  // namespace

extern "C" {

size_t ssm_scan_bwd_workspace_size(int64_t batch, int64_t L, int64_t d_inner, int d_state,
                                   ssm_dtype_t io) {
  if (check_common(batch, L, d_inner, d_state, io) != SSM_OK) return 0;
  const int sms = current_sm_count();
  if (sms <= 0 || batch * d_inner * L == 0) return 0;
  ssm::FwdPlan fplan;
  ssm::BwdPlan bplan;
  size_t fwd_bytes = 0, bytes = 0;
  if (!bwd_workspace(batch, L, d_inner, d_state, io == SSM_BF16, sms, &fplan, &bplan, &fwd_bytes, &bytes))
    return 0;
  return bytes;
}

int ssm_scan_bwd_launches(int64_t batch, int64_t L, int64_t d_inner, int d_state, ssm_dtype_t io) {
  if (check_common(batch, L, d_inner, d_state, io) != SSM_OK) return 0;
  const int sms = current_sm_count();
  if (sms <= 0 || batch * d_inner * L == 0) return 0;
  ssm::FwdPlan fplan;
  ssm::BwdPlan bplan;
  size_t fwd_bytes = 0, bytes = 0;
  if (!bwd_workspace(batch, L, d_inner, d_state, io == SSM_BF16, sms, &fplan, &bplan, &fwd_bytes, &bytes))
    return 0;
  return 2 + ((bplan.n_chunks > 1 && !bplan.handover) ? 1 : 0);
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

  const bool bf16 = io == SSM_BF16;
  ssm::FwdPlan fplan;
  ssm::BwdPlan bplan;
  size_t fwd_bytes = 0, need = 0;
  if (!bwd_workspace(batch, L, d_inner, d_state, bf16, sms, &fplan, &bplan, &fwd_bytes, &need))
    return SSM_ERR_CUDA;
  if (workspace == nullptr || workspace_bytes < need) return SSM_ERR_WORKSPACE;
  const int64_t n_dt = (d_inner + ssm::fwd_channels_per_cta() - 1) / ssm::fwd_channels_per_cta();
  if ((int64_t)std::max<int64_t>(fplan.G, bplan.n_chunks) * batch * ((d_inner + 31) / 32) >= ((int64_t)1 << 31))
    return SSM_ERR_SHAPE;
  (void)n_dt;

  float* ws = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) + fwd_bytes);
  const int64_t tiles = (L + ssm::kCkptSteps - 1) / ssm::kCkptSteps;
  const int64_t ck = batch * tiles * d_inner * d_state;
  const int64_t rws = batch * (int64_t)bplan.n_chunks * d_inner;
  ssm::BwdArgs a{};
  a.u = u; a.delta = delta; a.A = A; a.B = B; a.C = C; a.D = D; a.z = z; a.delta_bias = delta_bias;
  a.softplus = softplus_flag != 0; a.initial_state = initial_state; a.dy = dy; a.dlast = dlast_state;
  a.du = du; a.ddelta = ddelta; a.dz = dz; a.dA = dA; a.dB = dB; a.dC = dC; a.dD = dD;
  a.dbias = ddelta_bias; a.dinit = dinitial_state;
  a.batch = batch; a.L = L; a.d_inner = d_inner; a.d_state = d_state;
  a.chunk_len = bplan.chunk_len; a.n_chunks = bplan.n_chunks;
  a.ckpt_h = ws;
  a.rws_S = ws + ck;
  a.rws_m = ws + ck + rws;
  a.handover = bplan.handover;
  a.hflags = reinterpret_cast<unsigned long long*>(ws + ck + rws * (d_state + 1));
  a.header = reinterpret_cast<unsigned long long*>(workspace);

  ssm::FwdLaunch f{};
  f.u = u; f.delta = delta; f.A = A; f.B = B; f.C = C; f.delta_bias = delta_bias;
  f.softplus = softplus_flag != 0; f.initial_state = initial_state; f.ckpt = ws;
  f.batch = batch; f.L = L; f.d_inner = d_inner; f.d_state = d_state;
  f.plan = fplan;
  f.workspace = workspace;
  f.tag = next_call_tag();
  f.wait_tag = wait_tag_for(f.tag);
  f.max_polls = lookback_max_polls();
  a.tag = f.tag;
  a.wait_tag = f.wait_tag;
  a.max_polls = f.max_polls;
  return ssm::launch_scan_bwd(a, f, bf16, s) == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}

size_t ssm_ssd_fwd_workspace_size(int64_t batch, int64_t L, int64_t d_inner, int n_heads,
                                  int d_state) {
  (void)n_heads;
  if (batch <= 0 || L <= 0 || d_inner < 0) return 0;
  // a status word, the chunk Gram matrices C B^T (shared by every head), then one flag per
  // (batch, head) and room for the state handed from the first time half to the second
  return ssm::ssd_workspace_bytes(batch, L, d_inner, d_state);
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
  if (workspace == nullptr || workspace_bytes < ssm::ssd_workspace_bytes(batch, L, d_inner, d_state))
    return SSM_ERR_WORKSPACE;
  if (batch * L >= ((int64_t)1 << 31)) return SSM_ERR_SHAPE;  // rows of the Gram kernel's TMA maps
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
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  p.header = reinterpret_cast<unsigned long long*>(ws);
  p.tag = next_call_tag();
  p.wait_tag = wait_tag_for(p.tag);
  p.max_polls = lookback_max_polls();
  p.G = reinterpret_cast<float*>(ws + ssm::kFwdHeaderBytes);
  p.flags = reinterpret_cast<unsigned long long*>(ws + ssm::ssd_flags_offset(batch, L));
  p.hand = reinterpret_cast<float*>(ws + ssm::ssd_hand_offset(batch, L, d_inner));
  p.batch = batch; p.L = L; p.d_inner = d_inner; p.heads = n_heads; p.N = d_state;
  p.sms = current_sm_count();
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
    case SSM_ERR_LOOKBACK_TIMEOUT:
      return "a time chunk waited too long for its predecessors' records (results are invalid)";
    case SSM_ERR_SCRATCH_LIMIT:
      return "problem needs more scratch than ssm_scan_fwd_noalloc holds (use ssm_scan_fwd)";
  }
  return "unknown status";
}

int ssm_version(void) { return 200; }

}  // extern "C"

// ---------------------------------------------------------------------------------------
// No-allocation variant of ssm_scan_fwd.  Its scratch is this file-scope device array;
// host code must not hand the symbol itself to a kernel (on the host it only names a
// host-side shadow), so its device address is looked up per device and context, once,
// below.

static __device__ __align__(256) float g_noalloc_scratch[SSM_NOALLOC_SCRATCH_BYTES / sizeof(float)];

namespace {

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Process-unique id of the current CUDA context (0 if there is none or it cannot be read).
// The driver entry points are fetched through the runtime, so the library does not link
// the driver library itself.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f);
  });
  if (get_current == nullptr || get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  unsigned long long id = 0;
  return get_id(ctx, &id) == CUDA_SUCCESS ? id : 0;
}

struct ScratchSlot {
  unsigned long long ctx_id = 0;
  float* addr = nullptr;
};
std::mutex g_noalloc_mutex;
ScratchSlot g_noalloc[kMaxDevices];

// Device address of g_noalloc_scratch for the current device and context; looked up on the
// first use in a context (a device reset creates a new context, whose first use looks it up
// again).  With lookup == false, only an address already looked up is returned.
float* noalloc_scratch_address(bool lookup) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  ScratchSlot& slot = g_noalloc[dev];
  const unsigned long long id = current_context_id();
  if (slot.addr != nullptr && id != 0 && slot.ctx_id == id) return slot.addr;
  if (!lookup) return nullptr;
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return nullptr;
  slot.addr = static_cast<float*>(ptr);
  slot.ctx_id = current_context_id();  // the lookup made the device's context current
  return slot.addr;
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
  ssm::FwdPlan plan;
  size_t need = 0;
  if (!fwd_workspace(batch, L, d_inner, d_state, io == SSM_BF16, ssm::kFwdPlain, sms, &plan, &need))
    return SSM_ERR_CUDA;
  if (need > SSM_NOALLOC_SCRATCH_BYTES) return SSM_ERR_SCRATCH_LIMIT;
  float* scratch = nullptr;
  if (need > 0) {
    scratch = noalloc_scratch_address(true);
    if (scratch == nullptr) return SSM_ERR_CUDA;
  }
  return ssm_scan_fwd(u, delta, A, B, C, D, z, delta_bias, softplus_flag, y, last_state, batch, L,
                      d_inner, d_state, io, scratch, need, stream);
}

ssm_status_t ssm_get_status(const void* workspace, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return SSM_ERR_CUDA;
  const void* ws = workspace != nullptr ? workspace : noalloc_scratch_address(false);
  if (ws == nullptr) return SSM_OK;
  if (!aligned16(ws)) return SSM_ERR_ALIGN;
  unsigned long long word = 0;
  if (cudaMemcpyAsync(&word, ws, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return SSM_ERR_CUDA;
  return (word & 0xFFull) == ssm::kLookbackTimeoutCode ? SSM_ERR_LOOKBACK_TIMEOUT : SSM_OK;
}

}  // extern "C"
