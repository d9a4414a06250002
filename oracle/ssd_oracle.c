/*
 * Mamba-2 SSD (scalar A per head) oracle: a plain, slow, f64 CPU implementation.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark load this library.  The product path never
 * links, imports or calls it, and this file shares no code, header or
 * constant with that path.
 *
 * What it computes (the selective state-space recurrence with one scalar
 * decay per head, evaluated step by step -- the definition, not the chunked
 * algorithm a GPU uses to reach the same numbers):
 *   inputs   x : [B][L][H][P]        dt_raw : [B][L][H]
 *            Bm, Cm : [B][L][G][N]   (head h reads group g = h / (H / G))
 *            dt_bias, A_log, Dp : [H]  h0 : [B][H][N][P] (optional: zeros)
 *            dt_min <= dt_max: the limit on delta (0 and +inf: none)
 *   per (b, h), t = 0 .. L-1:
 *            delta = min(max(softplus(dt_raw[b,t,h] + dt_bias[h]), dt_min), dt_max)
 *            a     = exp(delta * A_h),  A_h = -exp(A_log[h])
 *            S[n][p] = a * S[n][p] + delta * Bm[b,t,g,n] * x[b,t,h,p]
 *            y[b,t,h,p] = sum_n Cm[b,t,g,n] * S[n][p] + Dp[h] * x[b,t,h,p]
 *   outputs  y : [B][L][H][P];  h_last : [B][H][N][P] = S after the last step
 *
 * Sources: the deterministic_backward.py page patches the Mamba-2 SSD
 * kernels (ssd_combined with its chunk_cumsum, chunk_state, state_passing,
 * bmm and chunk_scan stages) and passes dt per (batch, step, head) with one
 * scalar A and one dt_bias per head, dt_softplus and dt_limit; the
 * mamba3_preprocess_backward.slang page clamps softplus(dt) to [dt_min,
 * dt_max].  Neither page writes the recurrence out; the one above is the S6
 * recurrence of the other pages with A[d][n] = A_h shared by the head's P
 * channels and N states and B/C shared by the heads of a group -- pinned in
 * tests against the S6 oracle (that reduction), a closed form and the
 * chunked matmul form written independently in numpy.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double ssdo_softplus(double s) { return s > 0.0 ? s + log1p(exp(-s)) : log1p(exp(s)); }

int ssdo_fwd(int64_t B, int64_t L, int64_t H, int64_t P, int64_t G, int64_t N, const double *x,
             const double *dt_raw, const double *dt_bias, const double *A_log, const double *Bm,
             const double *Cm, const double *Dp, const double *h0, double dt_min, double dt_max,
             double *y, double *h_last) {
  if (B < 0 || L < 0 || H < 1 || P < 1 || G < 1 || N < 1 || H % G != 0 || !(dt_min <= dt_max)) return -1;
  const int64_t hpg = H / G;
  double *S = (double *)malloc(sizeof(double) * (size_t)(N * P));
  if (!S) return -2;
  for (int64_t b = 0; b < B; ++b)
    for (int64_t h = 0; h < H; ++h) {
      const int64_t g = h / hpg;
      const double A = -exp(A_log[h]);
      if (h0)
        memcpy(S, h0 + (b * H + h) * N * P, sizeof(double) * (size_t)(N * P));
      else
        memset(S, 0, sizeof(double) * (size_t)(N * P));
      for (int64_t t = 0; t < L; ++t) {
        double delta = ssdo_softplus(dt_raw[(b * L + t) * H + h] + dt_bias[h]);
        if (delta < dt_min) delta = dt_min;
        if (delta > dt_max) delta = dt_max;
        const double a = exp(delta * A);
        const double *xt = x + ((b * L + t) * H + h) * P;
        const double *Bt = Bm + ((b * L + t) * G + g) * N;
        const double *Ct = Cm + ((b * L + t) * G + g) * N;
        for (int64_t n = 0; n < N; ++n)
          for (int64_t p = 0; p < P; ++p) S[n * P + p] = a * S[n * P + p] + delta * Bt[n] * xt[p];
        double *yt = y + ((b * L + t) * H + h) * P;
        for (int64_t p = 0; p < P; ++p) {
          double acc = 0.0;
          for (int64_t n = 0; n < N; ++n) acc += Ct[n] * S[n * P + p];
          yt[p] = acc + Dp[h] * xt[p];
        }
      }
      if (h_last) memcpy(h_last + (b * H + h) * N * P, S, sizeof(double) * (size_t)(N * P));
    }
  free(S);
  return 0;
}
