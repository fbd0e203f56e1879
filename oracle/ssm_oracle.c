/*
 * ssm_oracle.c -- plain, sequential float64 reference for the Mamba selective
 * scan and its single-token decode step.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this library; the product path never does.  It shares
 * no code with the CUDA path.  Every input is taken as the exact (already
 * rounded) value the GPU reads, widened to double; everything is computed in
 * double, in the order the equations are written, one channel at a time.
 *
 * What is computed, and where the pages state it:
 *  - Discretisation: dA = exp(delta * A), dBu = delta * B * u
 *      youngju.dev, "Mamba: Linear-Time Sequence Modeling with Selective State
 *      Spaces 论文分析", section "解决方案：Kernel Fusion + Recomputation"
 *      (selective_scan concept code: deltaA, deltaB_x); ai-lab.club
 *      "机器学习基础算法", section "状态空间模型：连续系统的离散化".
 *  - Recurrence h_t = dA_t * h_{t-1} + dBu_t from h = 0, readout with the
 *      updated state y_t = sum_n C_{t,n} h_{t,n}: same concept code.
 *  - Skip term D * u: d9bl.com "Mamba 深度解读", equation (1b) and section
 *      "理解 SSM 矩阵"; ai-lab.club, discrete equations (y_k = C h_k + D x_k).
 *  - Gate y * silu(z): youngju.dev, section "Mamba 模块架构" (the block's
 *      forward multiplies the SSM output by F.silu(z)).
 *  - delta = softplus(delta_raw + bias) when softplus_flag is set, else
 *      delta_raw + bias: the pages show a biased delta projection (youngju.dev,
 *      "Mamba 模块架构", dt_proj with bias=True) but no positivity map; the
 *      softplus reading is the workload's statement of the problem.
 *  - Decode: one step of the same recurrence on a carried state (ai-lab.club,
 *      "核心优势": constant work per generated token).
 *  - Starting from a saved state instead of zero: d9bl.com, section
 *      "状态交换作为一种新的提示范式" (a state computed on one text is loaded
 *      into the model and the sequence continues from it).
 * Readings where the pages are silent: D and the gate act on the output only
 * (last_state is the pre-readout h); B and C are per (batch, time) and shared
 * by every channel (concept code B.unsqueeze(2)); the state starts at zero
 * unless an initial state is given.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* softplus(x) = log(1 + e^x), written so that neither branch overflows. */
double oracle_softplus(double x) {
  if (x > 0.0) return x + log1p(exp(-x));
  return log1p(exp(x));
}

/* silu(z) = z * sigmoid(z) = z / (1 + e^-z). */
static double oracle_silu(double z) { return z / (1.0 + exp(-z)); }

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Step size for one element. */
static double step_size(double delta_raw, const double* delta_bias, int64_t d, int softplus_flag) {
  double x = delta_raw + (delta_bias ? delta_bias[d] : 0.0);
  return softplus_flag ? oracle_softplus(x) : x;
}

/*
 * Full-sequence forward from a given state.
 * u, delta, z, y: [batch][L][d_inner]; B, C: [batch][L][d_state];
 * A: [d_inner][d_state]; D, delta_bias: [d_inner];
 * initial_state, last_state: [batch][d_inner][d_state].
 * D, z, delta_bias, last_state may be NULL (no skip term, no gate, zero bias, not returned);
 * initial_state NULL means h starts at zero.
 * Returns 0, or -1 for a bad argument.
 */
int oracle_scan_fwd_from_state(const double* u, const double* delta, const double* A,
                               const double* B, const double* C, const double* D,
                               const double* z, const double* delta_bias, int softplus_flag,
                               const double* initial_state, double* y, double* last_state,
                               int64_t batch, int64_t L, int64_t d_inner, int64_t d_state,
                               int nthreads) {
  if (batch < 0 || L < 0 || d_inner < 0 || d_state < 1) return -1;
  if ((L > 0 && (!u || !delta || !B || !C || !y)) || !A) return -1;
  if (nthreads < 1) nthreads = 1;
  int64_t channels = batch * d_inner;
  int bad = 0;
#pragma omp parallel num_threads(nthreads)
  {
    double* h = (double*)malloc(sizeof(double) * (size_t)d_state);
    if (!h) {
#pragma omp atomic write
      bad = 1;
    }
#pragma omp for schedule(dynamic, 1)
    for (int64_t ch = 0; ch < channels; ch++) {
      if (!h) continue;
      int64_t b = ch / d_inner, d = ch % d_inner;
      for (int64_t n = 0; n < d_state; n++)
        h[n] = initial_state ? initial_state[(b * d_inner + d) * d_state + n] : 0.0;
      for (int64_t t = 0; t < L; t++) {
        int64_t e = (b * L + t) * d_inner + d;        /* element (b, t, d) */
        const double* Bt = B + (b * L + t) * d_state;  /* row B[b, t, :] */
        const double* Ct = C + (b * L + t) * d_state;
        double dt = step_size(delta[e], delta_bias, d, softplus_flag);
        double s = 0.0;
        for (int64_t n = 0; n < d_state; n++) {
          double dA = exp(dt * A[d * d_state + n]);
          double dBu = dt * Bt[n] * u[e];
          h[n] = dA * h[n] + dBu;
          s += Ct[n] * h[n];
        }
        if (D) s += D[d] * u[e];
        if (z) s *= oracle_silu(z[e]);
        y[e] = s;
      }
      if (last_state)
        for (int64_t n = 0; n < d_state; n++) last_state[(b * d_inner + d) * d_state + n] = h[n];
    }
    free(h);
  }
  return bad ? -1 : 0;
}

/* Full-sequence forward from zero: the state before the first step is 0. */
int oracle_scan_fwd(const double* u, const double* delta, const double* A, const double* B,
                    const double* C, const double* D, const double* z,
                    const double* delta_bias, int softplus_flag, double* y, double* last_state,
                    int64_t batch, int64_t L, int64_t d_inner, int64_t d_state, int nthreads) {
  return oracle_scan_fwd_from_state(u, delta, A, B, C, D, z, delta_bias, softplus_flag, NULL, y,
                                    last_state, batch, L, d_inner, d_state, nthreads);
}

/*
 * Causal depthwise convolution followed by SiLU, the block's input path before the scan:
 * youngju.dev, section "Mamba 模块架构" (a Conv1d with groups = d_inner, kernel d_conv and
 * padding d_conv - 1, truncated to the sequence length, then F.silu).  With the padding on
 * the left only, output t sees inputs t - (d_conv - 1) .. t:
 *   u[b,t,d] = silu(bias[d] + sum_{k=0}^{d_conv-1} w[d,k] * x[b, t + k - (d_conv - 1), d]),
 * x outside the sequence being zero.  x_prev ([batch][d_inner][d_conv-1], may be NULL =
 * zeros) supplies the inputs before t = 0 (x_prev[.., j] is x at time j - (d_conv - 1)).
 * x, u: [batch][L][d_inner]; w: [d_inner][d_conv]; bias: [d_inner] or NULL.
 */
int oracle_conv1d_silu(const double* x, const double* w, const double* bias,
                       const double* x_prev, double* u, int64_t batch, int64_t L,
                       int64_t d_inner, int64_t d_conv) {
  if (batch < 0 || L < 0 || d_inner < 0 || d_conv < 1) return -1;
  for (int64_t b = 0; b < batch; b++)
    for (int64_t t = 0; t < L; t++)
      for (int64_t d = 0; d < d_inner; d++) {
        double acc = bias ? bias[d] : 0.0;
        for (int64_t k = 0; k < d_conv; k++) {
          const int64_t s = t + k - (d_conv - 1);
          double xv = 0.0;
          if (s >= 0) xv = x[(b * L + s) * d_inner + d];
          else if (x_prev) xv = x_prev[(b * d_inner + d) * (d_conv - 1) + (s + d_conv - 1)];
          acc += w[d * d_conv + k] * xv;
        }
        u[(b * L + t) * d_inner + d] = oracle_silu(acc);
      }
  return 0;
}

/* sigmoid(x) = 1 / (1 + e^-x): the derivative of softplus. */
static double oracle_sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/*
 * Gradients of the forward scan (reverse mode), for a loss L whose gradients with respect
 * to y (dy, [batch][L][d_inner]) and, optionally, to last_state (dlast,
 * [batch][d_inner][d_state], NULL = 0) are given.  The pages prescribe this pass only as
 * "recompute the intermediate states in the backward pass" (youngju.dev, section
 * "解决方案：Kernel Fusion + Recomputation"); the arithmetic is the chain rule through the
 * forward of oracle_scan_fwd_from_state, written out step by step:
 *   s_t = sum_n C_t,n h_t,n + D u_t,   y_t = s_t g_t,  g_t = silu(z_t)
 *   ds_t = dy_t g_t,  dz_t = dy_t s_t silu'(z_t),  silu'(z) = sig(z) (1 + z (1 - sig(z)))
 *   lambda_t = ds_t C_t + dA_{t+1} lambda_{t+1}   (lambda_{L-1} gets dlast added)
 *   dC_t,n = ds_t h_t,n;  dD += ds_t u_t;  du_t = ds_t D + delta_t sum_n lambda_t,n B_t,n
 *   ddelta_t = sum_n lambda_t,n (h_{t-1},n dA_t,n A_n + B_t,n u_t)
 *   dA_n += lambda_t,n h_{t-1},n dA_t,n delta_t;  dB_t,n = lambda_t,n delta_t u_t
 *   ddelta_raw_t = ddelta_t softplus'(x_t) (= sigmoid(x_t)), or ddelta_t without softplus;
 *   dbias += ddelta_raw_t;  dinitial_state = dA_0 lambda_0.
 * Outputs (all required unless noted): du, ddelta, dz (NULL iff z is NULL): [batch][L][d_inner];
 * dB, dC: [batch][L][d_state]; dA: [d_inner][d_state]; dD, dbias: [d_inner] (dD NULL iff D is
 * NULL, dbias may be NULL); dinit: [batch][d_inner][d_state] or NULL.  Accumulated outputs
 * are overwritten, not added to.  Serial over channels (dB, dC sum over channels).
 */
int oracle_scan_bwd(const double* u, const double* delta, const double* A, const double* B,
                    const double* C, const double* D, const double* z, const double* delta_bias,
                    int softplus_flag, const double* initial_state, const double* dy,
                    const double* dlast, double* du, double* ddelta, double* dA, double* dB,
                    double* dC, double* dD, double* dz, double* dbias, double* dinit,
                    int64_t batch, int64_t L, int64_t d_inner, int64_t d_state) {
  if (batch < 0 || L < 0 || d_inner < 0 || d_state < 1) return -1;
  const int64_t N = d_state;
  for (int64_t i = 0; i < d_inner * N; i++) dA[i] = 0.0;
  for (int64_t i = 0; i < batch * L * N; i++) { dB[i] = 0.0; dC[i] = 0.0; }
  for (int64_t d = 0; d < d_inner; d++) {
    if (dD) dD[d] = 0.0;
    if (dbias) dbias[d] = 0.0;
  }
  double* hs = (double*)malloc(sizeof(double) * (size_t)((L + 1) * N));  /* h_{-1} .. h_{L-1} */
  double* lam = (double*)malloc(sizeof(double) * (size_t)N);
  if (!hs || !lam) { free(hs); free(lam); return -1; }
  for (int64_t b = 0; b < batch; b++)
    for (int64_t d = 0; d < d_inner; d++) {
      /* forward, keeping every state (this is the oracle, not the fast path) */
      for (int64_t n = 0; n < N; n++)
        hs[n] = initial_state ? initial_state[(b * d_inner + d) * N + n] : 0.0;
      for (int64_t t = 0; t < L; t++) {
        const int64_t e = (b * L + t) * d_inner + d;
        const double dt = step_size(delta[e], delta_bias, d, softplus_flag);
        for (int64_t n = 0; n < N; n++)
          hs[(t + 1) * N + n] = exp(dt * A[d * N + n]) * hs[t * N + n] +
                                dt * B[(b * L + t) * N + n] * u[e];
      }
      /* reverse */
      for (int64_t n = 0; n < N; n++) lam[n] = dlast ? dlast[(b * d_inner + d) * N + n] : 0.0;
      for (int64_t t = L - 1; t >= 0; t--) {
        const int64_t e = (b * L + t) * d_inner + d;
        const double x = delta[e] + (delta_bias ? delta_bias[d] : 0.0);
        const double dt = softplus_flag ? oracle_softplus(x) : x;
        const double* Bt = B + (b * L + t) * N;
        const double* Ct = C + (b * L + t) * N;
        const double* h = hs + (t + 1) * N;      /* h_t */
        const double* hp = hs + t * N;           /* h_{t-1} */
        double s = 0.0;
        for (int64_t n = 0; n < N; n++) s += Ct[n] * h[n];
        if (D) s += D[d] * u[e];
        double g = 1.0;
        if (z) {
          g = oracle_silu(z[e]);
          const double sg = oracle_sigmoid(z[e]);
          dz[e] = dy[e] * s * sg * (1.0 + z[e] * (1.0 - sg));
        }
        const double ds = dy[e] * g;
        double ddt = 0.0, du_e = D ? ds * D[d] : 0.0;
        if (D) dD[d] += ds * u[e];
        for (int64_t n = 0; n < N; n++) {
          lam[n] += ds * Ct[n];                  /* lambda_t */
          const double dAn = exp(dt * A[d * N + n]);
          dC[(b * L + t) * N + n] += ds * h[n];
          dB[(b * L + t) * N + n] += lam[n] * dt * u[e];
          du_e += lam[n] * dt * Bt[n];
          ddt += lam[n] * (hp[n] * dAn * A[d * N + n] + Bt[n] * u[e]);
          dA[d * N + n] += lam[n] * hp[n] * dAn * dt;
          lam[n] *= dAn;                         /* carry dA_t lambda_t to step t-1 */
        }
        du[e] = du_e;
        const double dx = softplus_flag ? ddt * oracle_sigmoid(x) : ddt;
        ddelta[e] = dx;
        if (dbias) dbias[d] += dx;
      }
      if (dinit)
        for (int64_t n = 0; n < N; n++) dinit[(b * d_inner + d) * N + n] = lam[n];
    }
  free(hs);
  free(lam);
  return 0;
}

/*
 * One decode step on a carried state, updated in place.
 * state: [batch][d_inner][d_state]; u, delta, z, y: [batch][d_inner];
 * B, C: [batch][d_state]; A: [d_inner][d_state]; D, delta_bias: [d_inner].
 */
int oracle_state_update(double* state, const double* u, const double* delta, const double* A,
                        const double* B, const double* C, const double* D, const double* z,
                        double* y, const double* delta_bias, int softplus_flag, int64_t batch,
                        int64_t d_inner, int64_t d_state, int nthreads) {
  if (batch < 0 || d_inner < 0 || d_state < 1) return -1;
  if (batch * d_inner > 0 && (!state || !u || !delta || !A || !B || !C || !y)) return -1;
  if (nthreads < 1) nthreads = 1;
  int64_t channels = batch * d_inner;
#pragma omp parallel for num_threads(nthreads) schedule(static)
  for (int64_t ch = 0; ch < channels; ch++) {
    int64_t b = ch / d_inner, d = ch % d_inner;
    double* h = state + ch * d_state;
    const double* Bb = B + b * d_state;
    const double* Cb = C + b * d_state;
    double dt = step_size(delta[ch], delta_bias, d, softplus_flag);
    double s = 0.0;
    for (int64_t n = 0; n < d_state; n++) {
      double dA = exp(dt * A[d * d_state + n]);
      double dBu = dt * Bb[n] * u[ch];
      h[n] = dA * h[n] + dBu;
      s += Cb[n] * h[n];
    }
    if (D) s += D[d] * u[ch];
    if (z) s *= oracle_silu(z[ch]);
    y[ch] = s;
  }
  return 0;
}
