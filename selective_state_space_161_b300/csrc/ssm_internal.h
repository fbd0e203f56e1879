// Internal launch interface between the C ABI layer (ssm_api.cu) and the kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssm {

struct ScanParams {
  const void* u;
  const void* delta;
  const float* A;
  const void* B;
  const void* C;
  const float* D;           // may be null
  const void* z;            // may be null
  const float* delta_bias;  // may be null
  int softplus;
  void* y;
  float* last_state;        // may be null
  const float* initial_state;  // may be null: the state before the first step is zero
  // Optional causal depthwise conv1d + SiLU in front of the scan (conv_w non-null): the
  // u operand then holds the block input x, and u = silu(conv_b + sum_k conv_w[d,k] x[t+k-(K-1)]).
  const float* conv_w;      // [d_inner][d_conv]
  const float* conv_b;      // [d_inner], may be null
  int d_conv;               // 1..4
  void* u_out;              // may be null: the conv output u, I/O dtype
  int64_t batch, L, d_inner;
  int d_state;
  // Time chunking: the sequence is cut into n_chunks chunks of chunk_len steps
  // (the last one may be shorter).  For n_chunks > 1 the workspace holds, per
  // (batch, chunk < n_chunks-1, channel), the chunk's delta sum and its end
  // state started from zero.
  int64_t chunk_len;
  int n_chunks;
  int lanes;  // 1 or 2 lanes per channel (which kernel runs)
  float* ws_S;  // [batch][n_chunks-1][d_inner]
  float* ws_h;  // [batch][n_chunks-1][d_inner][d_state]
  float* ckpt_h = nullptr;  // checkpoint pass only: [batch][ceil(L/kCkptSteps)][d_inner][d_state]
};

struct DecodeParams {
  float* state;
  const void* u;
  const void* delta;
  const float* A;
  const void* B;
  const void* C;
  const float* D;
  const void* z;
  void* y;
  const float* delta_bias;
  int softplus;
  int64_t batch, d_inner;
  int d_state;
  // Optional conv1d + SiLU on the step's input (conv_w non-null): u holds the block input x,
  // conv_state [batch][d_inner][d_conv-1] fp32 the previous inputs, shifted in place.
  const float* conv_w;
  const float* conv_b;
  int d_conv;
  float* conv_state;
};

// Arguments of the backward pass (see ssm_scan_bwd.cu and include/ssm.h).
struct BwdArgs {
  const void* u;
  const void* delta;
  const float* A;
  const void* B;
  const void* C;
  const float* D;
  const void* z;
  const float* delta_bias;
  int softplus;
  const float* initial_state;
  const void* dy;
  const float* dlast;
  void* du;
  void* ddelta;
  void* dz;
  float* dA;
  float* dB;
  float* dC;
  float* dD;
  float* dbias;
  float* dinit;
  int64_t batch, L, d_inner;
  int d_state;
  int64_t chunk_len;
  int n_chunks;
  const float* fws_S;  // forward chunk summaries (written by the forward summary kernel)
  const float* fws_h;
  float* rws_S;        // reverse chunk summaries [batch][n_chunks][d_inner] (+ [.][d_state])
  float* rws_m;
  float* ckpt_h;       // [batch][ceil(L / kCkptSteps)][d_inner][d_state]: state before every kCkptSteps steps
};


// The chunked tensor-core form for one scalar A and one step size per head (ssm_ssd.cu).
struct SsdParams {
  const __nv_bfloat16* x;   // [batch][L][d_inner]
  const __nv_bfloat16* dt;  // [batch][L][heads] (raw step size)
  const float* A;           // [heads]
  const __nv_bfloat16* B;   // [batch][L][N]
  const __nv_bfloat16* C;
  const float* D;           // [d_inner], may be null
  const __nv_bfloat16* z;   // may be null
  const float* dt_bias;     // [heads], may be null
  int softplus;
  __nv_bfloat16* y;
  float* last_state;        // [batch][d_inner][N], may be null
  float* G;                 // workspace: [batch][chunks][64][64] chunk Gram matrices C B^T
  int64_t batch, L, d_inner;
  int heads, N;
};
int ssd_head_dim();
cudaError_t launch_ssd(const SsdParams& p, cudaStream_t s);
// Chunk Gram matrices G[b][c] = C_c B_c^T (64 x 64 fp32 per batch row and chunk of 64 steps) on
// the tensor cores (tcgen05, operands by TMA); ssd_gram_bytes is the workspace they take.
size_t ssd_gram_bytes(int64_t batch, int64_t L);
cudaError_t launch_ssd_gram(const __nv_bfloat16* C, const __nv_bfloat16* B, float* G, int64_t batch,
                            int64_t L, int N, cudaStream_t s);

// ---- Single-pass forward scan with a decoupled look-back (ssm_scan_fwd.cu) ----

// Workspace header: one status word, (call tag << 8) | status code.
constexpr size_t kFwdHeaderBytes = 256;
constexpr int kCkptSteps = 8;  // backward checkpoint interval (steps)
constexpr unsigned kLookbackTimeoutCode = 7;  // SSM_ERR_LOOKBACK_TIMEOUT

// How a forward scan of given sizes runs: lanes per channel pair and states per lane (the
// kernel variant), CTA threads, and the time chunks (G; chunk 0 has len0 steps, the others
// len, the last possibly fewer).
struct FwdPlan {
  int lanes, states_per_lane, threads, G;
  int64_t len0, len;
};

struct FwdLaunch {
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
  const float* conv_w;  // non-null: conv1d + SiLU in front (u holds the block input x)
  const float* conv_b;
  int d_conv;
  void* u_out;
  int64_t batch, L, d_inner;
  int d_state;
  FwdPlan plan;
  void* workspace;                // header, flags, records (fwd_workspace_bytes)
  unsigned long long tag;         // per-call tag of the records
  unsigned long long wait_tag;    // the tag the look-back accepts (tag, except in the wait self-test)
  unsigned max_polls;             // look-back polls before giving up
};

bool plan_scan_fwd(int64_t batch, int64_t L, int64_t d_inner, int d_state, bool bf16, bool conv,
                   int sms, FwdPlan* plan);
size_t fwd_workspace_bytes(int64_t batch, int64_t d_inner, const FwdPlan& plan);
cudaError_t launch_scan_fwd(const FwdLaunch& f, bool bf16, cudaStream_t stream);
int fwd_channels_per_cta();

// ---- Two-pass chunked scan kernels (ssm_scan.cu), used by the backward pass ----

// Channels handled by one CTA of the scan kernels.
int scan_channels_per_cta();

// How a scan of these sizes runs on a device with `sms` SMs: the kernel (lanes per
// channel) and the time chunking.
struct ScanPlan {
  int lanes;
  int64_t chunk_len;
  int n_chunks;
};
void plan_scan(int64_t batch, int64_t L, int64_t d_inner, int sms, ScanPlan* plan);

cudaError_t launch_scan(const ScanParams& p, bool bf16, cudaStream_t stream);
// Only the forward summary pass (one lane per channel) of a chunked scan plan.
cudaError_t launch_scan_summary(const ScanParams& p, bool bf16, cudaStream_t stream);
// The main pass's states from initial_state and the chunk summaries, with no output: the state
// before every kCkptSteps steps into p.ckpt_h (one lane per channel).
cudaError_t launch_scan_ckpt(const ScanParams& p, bool bf16, cudaStream_t stream);
// Floats of scratch the backward pass needs for n_chunks time chunks.
size_t bwd_workspace_floats(int64_t batch, int64_t L, int64_t d_inner, int d_state, int n_chunks);
cudaError_t launch_scan_bwd(const BwdArgs& a, const ScanParams& fwd, bool bf16, cudaStream_t s);
cudaError_t launch_state_update(const DecodeParams& p, bool bf16, cudaStream_t stream);

}  // namespace ssm
