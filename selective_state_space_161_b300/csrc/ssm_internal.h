// Internal launch interface between the C ABI layer (ssm_api.cu) and the kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssm {

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
  float* rws_S;        // reverse chunk summaries [batch][n_chunks][d_inner] (+ [.][d_state])
  float* rws_m;        // (hand-over plans: the carry each chunk hands to the one before it)
  int handover;        // 1: chunks run as a chain from the last back to the first, no summaries
  unsigned long long* hflags;  // [batch][n_chunks][64-channel tiles] hand-over tags
  unsigned long long* header;  // workspace status word (a hand-over wait that runs out: code 7)
  unsigned long long tag, wait_tag;
  unsigned max_polls;
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
  unsigned long long* header;  // workspace status word: (tag << 8) | code (code 7: a wait ran out)
  unsigned long long tag;      // this call's tag
  unsigned long long wait_tag; // the tag the second time half waits for (== tag but in a self-test)
  unsigned max_polls;          // polls of that wait before it gives up
  unsigned long long* flags;   // workspace: [batch][heads] the first half's "state is out" tag
  float* hand;                 // workspace: [batch][d_inner][N] the state at the end of the first half
  int64_t batch, L, d_inner;
  int heads, N;
  int sms;                     // SMs of the device (the launch picks the number of time parts)
};
int ssd_head_dim();
// Workspace of ssm_ssd_fwd: status word, chunk Gram matrices, the time parts' flags and hand-over
// states.
size_t ssd_workspace_bytes(int64_t batch, int64_t L, int64_t d_inner, int N);
size_t ssd_flags_offset(int64_t batch, int64_t L);
size_t ssd_hand_offset(int64_t batch, int64_t L, int64_t d_inner);
cudaError_t launch_ssd(const SsdParams& p, cudaStream_t s);
// The per-head chain on tcgen05 (ssm_ssd_tc.cu); G must hold the chunk Gram matrices.
cudaError_t launch_ssd_tc(const SsdParams& p, cudaStream_t s);
// Chunk Gram matrices G[b][c] = C_c B_c^T (64 x 64 fp32 per batch row and chunk of 64 steps) on
// the tensor cores (tcgen05, operands by TMA); ssd_gram_bytes is the workspace they take.
size_t ssd_gram_bytes(int64_t batch, int64_t L);
// The status word at `header` is set to (tag << 8) by the launch and raised to (tag << 8) | 7 if
// a wait on the copies or the MMA runs out.
cudaError_t launch_ssd_gram(const __nv_bfloat16* C, const __nv_bfloat16* B, float* G, int64_t batch,
                            int64_t L, int N, unsigned long long* header, unsigned long long tag,
                            cudaStream_t s);

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
  int chain;  // 1: no aggregate passes; each chunk continues from the end state of the one before
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
  float* ckpt;  // non-null: the backward's checkpoint kernel (no outputs; states every kCkptSteps)
  int64_t batch, L, d_inner;
  int d_state;
  FwdPlan plan;
  void* workspace;                // header, flags, records (fwd_workspace_bytes)
  unsigned long long tag;         // per-call tag of the records
  unsigned long long wait_tag;    // the tag the look-back accepts (tag, except in the wait self-test)
  unsigned max_polls;             // look-back polls before giving up
};

// Kernel kinds: the scan, the scan with the conv1d in front, the backward's checkpoints.
constexpr int kFwdPlain = 0, kFwdConv = 1, kFwdCkpt = 2;
bool plan_scan_fwd(int64_t batch, int64_t L, int64_t d_inner, int d_state, bool bf16, int kind,
                   int sms, FwdPlan* plan);
size_t fwd_workspace_bytes(int64_t batch, int64_t d_inner, const FwdPlan& plan);
cudaError_t launch_scan_fwd(const FwdLaunch& f, bool bf16, cudaStream_t stream);
int fwd_channels_per_cta();

// ---- Backward pass (ssm_scan_bwd.cu) ----

// Time chunks of the backward's gradient kernel (chunk_len a multiple of 32 steps).
struct BwdPlan {
  int64_t chunk_len;
  int n_chunks;
  int handover;  // chunks as a chain handing the adjoint carry back (no reverse summaries)
};
void plan_scan_bwd(int64_t batch, int64_t L, int64_t d_inner, int sms, BwdPlan* plan);
// Floats of scratch the backward's checkpoints and reverse summaries take for n_chunks chunks
// (after the checkpoint kernel's look-back region at the start of the workspace).
size_t bwd_workspace_floats(int64_t batch, int64_t L, int64_t d_inner, int d_state, int n_chunks);
// ckpt: the checkpoint kernel's launch (its ckpt pointer set); a: the gradient kernels'.
cudaError_t launch_scan_bwd(const BwdArgs& a, const FwdLaunch& ckpt, bool bf16, cudaStream_t s);
cudaError_t launch_state_update(const DecodeParams& p, bool bf16, cudaStream_t stream);

}  // namespace ssm
