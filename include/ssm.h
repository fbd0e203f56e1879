/*
 * ssm.h -- C ABI of libssm: the Mamba selective-scan forward pass and its
 * single-token decode step, as CUDA kernels for NVIDIA B300 (sm_103a).
 *
 * The operation (citations are page title + section):
 *   delta_t = softplus(delta_raw_t + delta_bias)          (or without softplus)
 *   dA_t    = exp(delta_t * A)                             per (channel, state)
 *   dBu_t   = delta_t * B_t * u_t
 *   h_t     = dA_t * h_{t-1} + dBu_t,  h_{-1} = 0
 *   y_t     = (sum_n C_{t,n} h_{t,n} + D * u_t) * silu(z_t)
 * - discretisation, recurrence and readout: youngju.dev, "Mamba: Linear-Time
 *   Sequence Modeling with Selective State Spaces 论文分析", section
 *   "解决方案：Kernel Fusion + Recomputation" (selective_scan concept code);
 *   ai-lab.club "机器学习基础算法", section "状态空间模型：连续系统的离散化"
 *   (h_k = Abar h_{k-1} + Bbar x_k, y_k = C h_k + D x_k);
 * - selection (B, C, delta per token): youngju.dev, section
 *   "Mamba 的解决方案：Selection Mechanism";
 * - gate y * silu(z) and the biased delta projection: youngju.dev, section
 *   "Mamba 模块架构";
 * - the single-step (decode) form: ai-lab.club, section "核心优势"
 *   (constant work per generated token, like an RNN).
 *
 * Conventions shared by every entry point
 * - All tensor pointers are DEVICE pointers owned by the caller; the library
 *   never allocates, frees or keeps them.  Every call is asynchronous on
 *   `stream` (a cudaStream_t; NULL = the legacy default stream).
 * - Layouts are row-major, channels (d_inner) innermost:
 *     u, delta, z, y  [batch][L][d_inner]      (I/O dtype)
 *     B, C            [batch][L][d_state]      (I/O dtype)
 *     A               [d_inner][d_state]       fp32
 *     D, delta_bias   [d_inner]                fp32
 *     last_state      [batch][d_inner][d_state] fp32
 *   The I/O dtype (`io`) is fp32 or bf16; the state and all arithmetic are
 *   fp32, bf16 outputs are rounded to nearest even.
 * - Requirements: every non-NULL pointer 16-byte aligned; d_inner a multiple
 *   of 8 (bf16) or 4 (fp32); 1 <= d_state <= 16; batch, L, d_inner >= 0.
 *   Outputs must not overlap inputs.
 * - The return value reports argument validation and launch errors only.  The one
 *   device-side failure mode is a time chunk of a scan that waits too long for the
 *   records of the chunks before it (see ssm_scan_fwd); ssm_get_status reports it.
 * - Calls on different streams are independent if their outputs and
 *   workspaces are distinct.
 */
#ifndef SSM_H
#define SSM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SSM_API __attribute__((visibility("default")))
#else
#define SSM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { SSM_F32 = 0, SSM_BF16 = 1 } ssm_dtype_t;

typedef enum {
  SSM_OK = 0,
  SSM_ERR_NULL = 1,       /* a required pointer is NULL */
  SSM_ERR_SHAPE = 2,      /* negative size, d_state outside 1..16, bad d_inner multiple */
  SSM_ERR_DTYPE = 3,      /* io is neither SSM_F32 nor SSM_BF16 */
  SSM_ERR_ALIGN = 4,      /* a pointer is not 16-byte aligned */
  SSM_ERR_WORKSPACE = 5,  /* workspace NULL or smaller than the size query says */
  SSM_ERR_CUDA = 6,       /* no usable CUDA device, a launch failed, or a CUDA error is pending */
  SSM_ERR_LOOKBACK_TIMEOUT = 7, /* (ssm_get_status) a bounded wait in a kernel ran out: a time
                                   chunk waiting for its predecessors' records, or an SSD kernel
                                   waiting for its copies or tensor-core products; that call's
                                   outputs are invalid */
  SSM_ERR_SCRATCH_LIMIT = 8 /* ssm_scan_fwd_noalloc: the problem needs more scratch than it holds */
} ssm_status_t;

/*
 * Bytes of workspace the forward scans (ssm_scan_fwd, ssm_scan_fwd_from_state,
 * ssm_scan_fwd_conv) need for these sizes on the current device; 0 only for an empty
 * problem (batch * L * d_inner == 0).  The workspace holds a status word (read by
 * ssm_get_status) and, when the sequence is cut into time chunks, one record per chunk
 * and channel tile: the chunk's aggregate (sum of delta, end state from zero) and its
 * inclusive prefix (the true state at its end), each with a flag.  Records carry a tag
 * unique to the call, so the contents need no initialisation and are dead after the call
 * completes, except the status word.
 */
SSM_API size_t ssm_scan_fwd_workspace_size(int64_t batch, int64_t L, int64_t d_inner, int d_state,
                                   ssm_dtype_t io);

/*
 * Selective-scan forward over whole sequences.
 *   u, delta, B, C : inputs (io dtype), required when batch*L*d_inner > 0.
 *   A              : fp32 [d_inner][d_state], required.
 *   D, z, delta_bias: optional (NULL = no skip term / no gate / zero bias).
 *   softplus_flag  : nonzero -> delta = softplus(delta_raw + bias), else delta_raw + bias.
 *   y              : output (io dtype), required when batch*L*d_inner > 0.
 *   last_state     : optional fp32 output, h after the last step (before D and the gate);
 *                    zeros when L == 0.
 *   workspace      : device scratch of workspace_bytes >= ssm_scan_fwd_workspace_size(...);
 *                    may be NULL when that size is 0.  Calls that overlap on the GPU need
 *                    distinct workspaces.
 *
 * Time chunks.  When batch * d_inner channels cannot fill the GPU, the sequence is cut
 * into chunks processed at the same time, joined by a decoupled look-back: a chunk
 * publishes its aggregate, then folds its predecessors' aggregates until it finds an
 * inclusive prefix, publishes its own and produces its outputs (the recurrence is
 * associative: "看懂Mamba，Transformer最强竞争者（一）…", section "3. 状态空间"; the parallel scan
 * of "Mamba一作最新大發長文！", section "(3) 訓練效率").  When the channels alone fill about
 * one wave of CTAs but spread unevenly over the SMs, the plan uses two or three chunks with no
 * aggregate at all, each continuing from its predecessor's end state (a finer division of the
 * same work).  Every wait is bounded; a chunk that gives up records SSM_ERR_LOOKBACK_TIMEOUT
 * for ssm_get_status and finishes (its outputs are then invalid) instead of hanging.
 */
SSM_API ssm_status_t ssm_scan_fwd(const void* u, const void* delta, const float* A, const void* B,
                          const void* C, const float* D, const void* z, const float* delta_bias,
                          int softplus_flag, void* y, float* last_state, int64_t batch, int64_t L,
                          int64_t d_inner, int d_state, ssm_dtype_t io, void* workspace,
                          size_t workspace_bytes, void* stream);

/*
 * ssm_scan_fwd continuing from a given state instead of zero: h_{-1} = initial_state
 * ([batch][d_inner][d_state] fp32, device; NULL = zero, i.e. exactly ssm_scan_fwd).
 * Loading a state saved from an earlier sequence and continuing from it is the "state
 * swapping" of d9bl.com, "Mamba 深度解读", section "状态交换作为一种新的提示范式"; it also
 * chains a long sequence processed in segments: running L1 steps, then the rest from the
 * returned last_state, gives the same y and last_state as one call.  initial_state must not
 * overlap last_state (except that with L == 0 the two may be the same buffer); workspace
 * as for ssm_scan_fwd.  With L == 0, last_state receives initial_state.
 */
SSM_API ssm_status_t ssm_scan_fwd_from_state(const void* u, const void* delta, const float* A,
                                             const void* B, const void* C, const float* D,
                                             const void* z, const float* delta_bias,
                                             int softplus_flag, const float* initial_state,
                                             void* y, float* last_state, int64_t batch, int64_t L,
                                             int64_t d_inner, int d_state, ssm_dtype_t io,
                                             void* workspace, size_t workspace_bytes,
                                             void* stream);

/*
 * The block's input path fused in front of the scan: u = silu(conv1d(x)), a causal
 * depthwise convolution of the block input x with d_conv taps and optional bias, then
 * SiLU (youngju.dev, "Mamba 模块架构": Conv1d with groups = d_inner, padding d_conv - 1,
 * truncated to the sequence length, then F.silu), followed by ssm_scan_fwd_from_state on u:
 *   u[b,t,d] = silu(conv_bias[d] + sum_{k<d_conv} conv_weight[d][k] * x[b, t+k-(d_conv-1), d])
 * with x = 0 before t = 0.  u never goes to HBM unless u_out (nullable, io dtype,
 * [batch][L][d_inner]) asks for it.  conv_weight [d_inner][d_conv] fp32 (required),
 * conv_bias [d_inner] fp32 (nullable), 1 <= d_conv <= 4.  Other operands, the workspace and
 * initial_state as for ssm_scan_fwd_from_state.
 */
SSM_API ssm_status_t ssm_scan_fwd_conv(const void* x, const float* conv_weight,
                                       const float* conv_bias, int d_conv, const void* delta,
                                       const float* A, const void* B, const void* C,
                                       const float* D, const void* z, const float* delta_bias,
                                       int softplus_flag, const float* initial_state, void* y,
                                       float* last_state, void* u_out, int64_t batch, int64_t L,
                                       int64_t d_inner, int d_state, ssm_dtype_t io,
                                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * One decode step on a carried state, in place:
 *   state [batch][d_inner][d_state] fp32 (read, then overwritten with h_t);
 *   u, delta, z, y [batch][d_inner] (io dtype); B, C [batch][d_state] (io dtype);
 *   A [d_inner][d_state], D, delta_bias [d_inner] fp32.
 * D, z, delta_bias are optional (NULL); softplus_flag as for ssm_scan_fwd.
 * L calls from a zero state reproduce ssm_scan_fwd's y and last_state.
 */
SSM_API ssm_status_t ssm_state_update(float* state, const void* u, const void* delta, const float* A,
                              const void* B, const void* C, const float* D, const void* z,
                              void* y, const float* delta_bias, int softplus_flag, int64_t batch,
                              int64_t d_inner, int d_state, ssm_dtype_t io, void* stream);

/*
 * ssm_scan_fwd without a caller-supplied workspace, for callers that cannot allocate
 * device memory at the point of the call: code that runs under an allocator it does not
 * own (a framework plugin or custom operator whose host forbids allocations while it
 * executes), latency-critical loops where a cudaMalloc/cudaFree would synchronise the
 * device, or embedded callers held to a fixed memory budget.  (The pages have no
 * counterpart to this entry point; it exists for such callers only.)
 *
 * Same arguments, results and requirements as ssm_scan_fwd, minus the workspace.  The
 * scratch it needs (the status word and the time chunks' look-back records) comes from an
 * array of SSM_NOALLOC_SCRATCH_BYTES (8 MiB) that the library places in device memory at
 * load time; every GPU that loads the library keeps that array until the process exits.
 * Problems whose scratch need exceeds it return SSM_ERR_SCRATCH_LIMIT without launching
 * anything.  The need is bounded by one wave of resident CTAs (a few MiB on B300), so
 * only time-chunk counts forced above the default plan reach the limit.
 * - The first call on each device (and after a device reset, in each new context) looks
 *   up the array's device address with that device current and caches it; make that
 *   first call before any stream capture.
 * - All calls share the one array: calls whose executions overlap on the GPU (on
 *   different streams, or from different threads) race on it and give wrong results.
 *   Serialise them.  The array needs no clearing: a call reads only records tagged by
 *   itself.  ssm_get_status(NULL, stream) reports on the latest call.
 * - It allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 */
#define SSM_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
SSM_API ssm_status_t ssm_scan_fwd_noalloc(const void* u, const void* delta, const float* A,
                                          const void* B, const void* C, const float* D,
                                          const void* z, const float* delta_bias,
                                          int softplus_flag, void* y, float* last_state,
                                          int64_t batch, int64_t L, int64_t d_inner,
                                          int d_state, ssm_dtype_t io, void* stream);

/*
 * One decode step with the block's conv1d + SiLU in front (the single-token form of
 * ssm_scan_fwd_conv): x [batch][d_inner] is the block input; conv_state
 * [batch][d_inner][d_conv-1] fp32 holds the previous d_conv-1 inputs (oldest first) and is
 * shifted in place (x appended); u = silu(conv_bias + conv_weight . (conv_state, x)) feeds
 * the step exactly as ssm_state_update's u.  conv_state may be NULL only when d_conv == 1.
 * L calls from zero states reproduce ssm_scan_fwd_conv's y and last_state.
 */
SSM_API ssm_status_t ssm_state_update_conv(float* state, float* conv_state, const void* x,
                                           const float* conv_weight, const float* conv_bias,
                                           int d_conv, const void* delta, const float* A,
                                           const void* B, const void* C, const float* D,
                                           const void* z, void* y, const float* delta_bias,
                                           int softplus_flag, int64_t batch, int64_t d_inner,
                                           int d_state, ssm_dtype_t io, void* stream);

/*
 * Backward pass of ssm_scan_fwd_from_state (gradients for training).  Given dy = dL/dy
 * ([batch][L][d_inner], io dtype) and optionally dlast_state = dL/dlast_state
 * ([batch][d_inner][d_state] fp32, NULL = 0), writes
 *   du, ddelta (gradient w.r.t. delta_raw), dz (NULL iff z is NULL): io dtype, like u;
 *   dA [d_inner][d_state], dB, dC [batch][L][d_state], dD (NULL iff D is NULL),
 *   ddelta_bias (NULL: not computed), dinitial_state (NULL: not computed): fp32.
 * dA, dB, dC, dD, ddelta_bias are sums over batch/time/channels; they are overwritten.
 * The forward inputs (u, delta, A, B, C, D, z, delta_bias, softplus_flag, initial_state)
 * are the ones the forward call used; no forward output is needed.  The intermediate
 * states are recomputed, not stored by the forward (youngju.dev, "Mamba: Linear-Time
 * Sequence Modeling with Selective State Spaces 论文分析", section "解决方案：Kernel
 * Fusion + Recomputation"): the pass keeps one state per 8 steps and per channel in the
 * workspace (ssm_scan_bwd_workspace_size bytes: a status word and the look-back records of
 * the forward recompute, as for ssm_scan_fwd, then about batch * L * d_inner * d_state / 2
 * bytes of states, the per-chunk summaries (or handed-over carries) of the reverse pass and
 * one 8-byte tag per (batch, chunk, 64 channels); not initialised by the caller: every record
 * carries a per-call tag).  The forward recompute waits on its time chunks like ssm_scan_fwd,
 * and when the gradient CTAs run as a chain of time chunks (each handing its adjoint carry to
 * the chunk before it) each waits for the one after it; all waits are bounded, and
 * ssm_get_status(workspace, stream) reports a wait that ran out.  dB and dC are
 * accumulated with atomic additions, so their last bits may vary from run to run.
 */
SSM_API size_t ssm_scan_bwd_workspace_size(int64_t batch, int64_t L, int64_t d_inner,
                                           int d_state, ssm_dtype_t io);
/* Kernels one ssm_scan_bwd call launches for these sizes on the current device: the forward
 * recompute and the gradient kernel, plus the reverse-summary kernel when the plan joins its
 * time chunks by summaries (2 or 3; the zeroing of the accumulated outputs is done by
 * cudaMemsetAsync and not counted).  0 for invalid arguments, an empty problem or no device. */
SSM_API int ssm_scan_bwd_launches(int64_t batch, int64_t L, int64_t d_inner, int d_state,
                                  ssm_dtype_t io);
SSM_API ssm_status_t ssm_scan_bwd(const void* u, const void* delta, const float* A, const void* B,
                                  const void* C, const float* D, const void* z,
                                  const float* delta_bias, int softplus_flag,
                                  const float* initial_state, const void* dy,
                                  const float* dlast_state, void* du, void* ddelta, float* dA,
                                  float* dB, float* dC, float* dD, void* dz, float* ddelta_bias,
                                  float* dinitial_state, int64_t batch, int64_t L,
                                  int64_t d_inner, int d_state, ssm_dtype_t io, void* workspace,
                                  size_t workspace_bytes, void* stream);

/*
 * The chunked tensor-core ("state space duality", Mamba-2) form, for the case of one scalar
 * A and one step size per head: youngju.dev, section "后续研究：Mamba-2 与混合架构" names
 * State Space Duality (the recurrence as attention-like matrix products) without equations.
 * It computes exactly ssm_scan_fwd with A[d][n] = A_head[h] and delta[b][t][d] = dt[b][t][h]
 * for the head's channels d = h * 64 .. h * 64 + 63, every state n (and delta_bias per head):
 * per chunk of 64 steps, the products C B^T (masked by the decays), (.) x, x^T B and C H^T
 * run on the tensor cores (bf16 operands, computed operands split into bf16 hi + lo parts,
 * fp32 accumulation); the fp32 state is carried from chunk to chunk on chip.
 *   x, z, y [batch][L][d_inner]; dt [batch][L][n_heads]; B, C [batch][L][d_state]: bf16;
 *   A_head, dt_bias [n_heads], D [d_inner], last_state [batch][d_inner][d_state]: fp32.
 * Requirements: io == SSM_BF16; d_inner == 64 * n_heads (head dimension 64); d_state in
 * {16, 32, 64, 128}; D, z, dt_bias, last_state nullable; batch * L < 2^31.
 * The chunks' Gram matrices G = C B^T do not depend on the head (B and C are shared by all
 * heads): a first tensor-core kernel (tcgen05.mma with operands brought in by TMA) computes
 * them once per batch row and chunk into the workspace, and every head reads them.  When the
 * (batch, head) chains would not spread evenly over the SMs, each chain is run as two time
 * halves of whole chunks: the first hands its end state to the second through the workspace.
 * Workspace (ssm_ssd_fwd_workspace_size bytes, caller-owned, no initialisation needed: every
 * record carries a per-call tag): a 256-byte status word; batch * ceil(L / 64) * 64 * 64 fp32
 * Gram matrices; one 8-byte flag per (batch, head), padded to a multiple of 256 bytes;
 * batch * d_inner * d_state fp32 for the handed-over states.  The kernels' waits (on their
 * copies, their tensor-core products, and the second half's wait for the first half's state)
 * are bounded: a wait that runs out makes ssm_get_status(workspace, stream) return
 * SSM_ERR_LOOKBACK_TIMEOUT (the outputs are then invalid), never a hang.
 */
SSM_API size_t ssm_ssd_fwd_workspace_size(int64_t batch, int64_t L, int64_t d_inner, int n_heads,
                                          int d_state);
SSM_API ssm_status_t ssm_ssd_fwd(const void* x, const void* dt, const float* A_head,
                                 const void* B, const void* C, const float* D, const void* z,
                                 const float* dt_bias, int softplus_flag, void* y,
                                 float* last_state, int64_t batch, int64_t L, int64_t d_inner,
                                 int n_heads, int d_state, ssm_dtype_t io, void* workspace,
                                 size_t workspace_bytes, void* stream);

/*
 * Device-side status of the most recent forward scan, backward pass (whose forward
 * recompute runs the same chunked kernel) or chunked SSD call that used `workspace`: waits
 * for `stream` (a cudaStream_t, NULL = legacy default stream) to finish, then returns
 *   SSM_ERR_CUDA             if the stream reports a CUDA error (asynchronous or sticky),
 *   SSM_ERR_LOOKBACK_TIMEOUT if a wait of that call ran out: a time chunk waiting for its
 *                            predecessors' records, or an SSD kernel waiting for its copies,
 *                            its tensor-core products or the state of the first time half
 *                            (the outputs are invalid),
 *   SSM_OK                   otherwise.
 * workspace == NULL checks the scratch of ssm_scan_fwd_noalloc on the current device (if
 * it has been used), or only the stream when it has not.  The workspace must have been
 * passed to such a call with a non-empty problem before (its status word is written by
 * every such call).  Synchronises, so it cannot be captured in a CUDA graph.
 */
SSM_API ssm_status_t ssm_get_status(const void* workspace, void* stream);

/* Human-readable name of a status code (static string). */
SSM_API const char* ssm_status_string(ssm_status_t status);

/* Library ABI version (major * 100 + minor): 200. */
SSM_API int ssm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SSM_H */
