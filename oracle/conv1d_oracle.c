/*
 * Causal depthwise conv1d + SiLU oracle: a plain, slow, f64 CPU implementation.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark load this library.  The product path never
 * links, imports or calls it, and this file shares no code, header or
 * constant with that path.
 *
 * What it computes (the convolution in front of the selective scan in a
 * Mamba block; K taps per channel, causal, depthwise):
 *   inputs   x : [B][L][D]     w : [D][K]     bias : [D]
 *            state0 : [B][D][K-1]  the K-1 inputs before t = 0, oldest first
 *                                  (optional: zeros)
 *   let xx(t) = x[b][t][d] for t >= 0 and state0[b][d][K-1+t] for -(K-1) <= t < 0
 *   forward  pre[b,t,d] = bias[d] + sum_{k=0..K-1} w[d][k] * xx(t - (K-1) + k)
 *            out[b,t,d] = pre * sigmoid(pre)                     (SiLU)
 *            state_last[b][d][j] = xx(L - (K-1) + j), j = 0..K-2 (the last K-1 inputs)
 *   step     one time step from a state: pre = bias + sum_{k<K-1} w[k]*state[k]
 *            + w[K-1]*x_t; out = SiLU(pre); the state shifts by one and takes x_t.
 *   backward (loss = sum dout * out; chain rule, pinned by finite differences):
 *            s = sigmoid(pre);  dpre = dout * s * (1 + pre * (1 - s))
 *            dx[b,t,d]      = sum_k w[d][k] * dpre[b, t + (K-1) - k, d]   (terms with 0 <= t+(K-1)-k < L)
 *            dw[d][k]       = sum_{b,t} dpre[b,t,d] * xx(t - (K-1) + k)
 *            dbias[d]       = sum_{b,t} dpre[b,t,d]
 *            dstate0[b][d][j] = sum_k w[d][k] * dpre[b, j - k, d]          (terms with 0 <= j-k < L)
 * Sums over (b,t) for dw and dbias run in ascending b, then t.
 *
 * Sources: the mamba-rs kernels.rs page registers "Single-step depthwise
 * conv1d forward with SiLU", "Single-step depthwise conv1d backward",
 * "Multi-step conv1d forward with state saves for backward" and "Multi-step
 * conv1d backward", and "SiLU forward: x * sigmoid(x)"; the
 * deterministic_backward.py page runs the causal conv1d with the SiLU
 * activation and sums its weight and bias gradients batch by batch in a fixed
 * order (ordered_conv).  Neither page prints the formulas: the window
 * convention above (output t reads inputs t-K+1 .. t, tap k on input
 * t-(K-1)+k) is the causal convolution's, pinned in tests by an impulse
 * response and by numpy.convolve.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

static double c1o_sigmoid(double v) { return 1.0 / (1.0 + exp(-v)); }

/* xx(t) of the definition above */
static double c1o_in(const double *x, const double *state0, int64_t L, int64_t D, int64_t K,
                     int64_t b, int64_t t, int64_t d) {
  if (t >= 0) return x[(b * L + t) * D + d];
  if (!state0) return 0.0;
  return state0[(b * D + d) * (K - 1) + (K - 1 + t)];
}

static double c1o_pre(const double *x, const double *w, const double *bias, const double *state0,
                      int64_t L, int64_t D, int64_t K, int64_t b, int64_t t, int64_t d) {
  double pre = bias[d];
  for (int64_t k = 0; k < K; ++k) pre += w[d * K + k] * c1o_in(x, state0, L, D, K, b, t - (K - 1) + k, d);
  return pre;
}

int c1o_fwd(int64_t B, int64_t L, int64_t D, int64_t K, const double *x, const double *w,
            const double *bias, const double *state0, double *out, double *state_last) {
  if (B < 0 || L < 0 || D < 0 || K < 1) return 1;
  for (int64_t b = 0; b < B; ++b)
    for (int64_t t = 0; t < L; ++t)
      for (int64_t d = 0; d < D; ++d) {
        const double pre = c1o_pre(x, w, bias, state0, L, D, K, b, t, d);
        out[(b * L + t) * D + d] = pre * c1o_sigmoid(pre);
      }
  if (state_last)
    for (int64_t b = 0; b < B; ++b)
      for (int64_t d = 0; d < D; ++d)
        for (int64_t j = 0; j < K - 1; ++j)
          state_last[(b * D + d) * (K - 1) + j] = c1o_in(x, state0, L, D, K, b, L - (K - 1) + j, d);
  return 0;
}

int c1o_step(int64_t B, int64_t D, int64_t K, const double *x_t, const double *w, const double *bias,
             double *state, double *out) {
  if (B < 0 || D < 0 || K < 1) return 1;
  for (int64_t b = 0; b < B; ++b)
    for (int64_t d = 0; d < D; ++d) {
      double *st = state + (b * D + d) * (K - 1);
      const double xv = x_t[b * D + d];
      double pre = bias[d];
      for (int64_t k = 0; k < K - 1; ++k) pre += w[d * K + k] * st[k];
      pre += w[d * K + K - 1] * xv;
      out[b * D + d] = pre * c1o_sigmoid(pre);
      for (int64_t k = 0; k + 1 < K - 1; ++k) st[k] = st[k + 1];
      if (K > 1) st[K - 2] = xv;
    }
  return 0;
}

int c1o_bwd(int64_t B, int64_t L, int64_t D, int64_t K, const double *x, const double *w,
            const double *bias, const double *state0, const double *dout, double *dx, double *dw,
            double *dbias, double *dstate0) {
  if (B < 0 || L < 0 || D < 0 || K < 1) return 1;
  double *dpre = (double *)malloc(sizeof(double) * (size_t)(B * L * D > 0 ? B * L * D : 1));
  if (!dpre) return 2;
  for (int64_t b = 0; b < B; ++b)
    for (int64_t t = 0; t < L; ++t)
      for (int64_t d = 0; d < D; ++d) {
        const double pre = c1o_pre(x, w, bias, state0, L, D, K, b, t, d);
        const double s = c1o_sigmoid(pre);
        dpre[(b * L + t) * D + d] = dout[(b * L + t) * D + d] * s * (1.0 + pre * (1.0 - s));
      }
  for (int64_t b = 0; b < B; ++b)
    for (int64_t t = 0; t < L; ++t)
      for (int64_t d = 0; d < D; ++d) {
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) {
          const int64_t to = t + (K - 1) - k;
          if (to < L) acc += w[d * K + k] * dpre[(b * L + to) * D + d];
        }
        dx[(b * L + t) * D + d] = acc;
      }
  for (int64_t d = 0; d < D; ++d) {
    for (int64_t k = 0; k < K; ++k) dw[d * K + k] = 0.0;
    dbias[d] = 0.0;
  }
  for (int64_t b = 0; b < B; ++b)
    for (int64_t t = 0; t < L; ++t)
      for (int64_t d = 0; d < D; ++d) {
        const double g = dpre[(b * L + t) * D + d];
        for (int64_t k = 0; k < K; ++k) dw[d * K + k] += g * c1o_in(x, state0, L, D, K, b, t - (K - 1) + k, d);
        dbias[d] += g;
      }
  if (dstate0)
    for (int64_t b = 0; b < B; ++b)
      for (int64_t d = 0; d < D; ++d)
        for (int64_t j = 0; j < K - 1; ++j) {
          double acc = 0.0;
          for (int64_t k = 0; k < K; ++k) {
            const int64_t to = j - k;
            if (to >= 0 && to < L) acc += w[d * K + k] * dpre[(b * L + to) * D + d];
          }
          dstate0[(b * D + d) * (K - 1) + j] = acc;
        }
  free(dpre);
  return 0;
}
