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
 * and the backward of loss = sum(dy * y) + sum(dh_last * h_last) by the chain
 * rule through that recurrence, walking t = L-1 .. 0 with Gr = dloss/dS_t
 * (from dh_last, zeros when absent) and the states recomputed forward:
 *            Gr      += C_t dy_t^T              (step t's readout)
 *            dCm_t   += S_t dy_t   (sum over p; heads of a group add up)
 *            dDp_h   += dy_t . x_t
 *            dx_t     = Dp_h dy_t + delta_t Gr^T B_t
 *            dBm_t   += delta_t Gr x_t   (sum over p; heads of a group add up)
 *            ddelta   = sum(Gr o (A_h a_t S_{t-1} + B_t x_t^T))
 *            dA_h    += delta_t a_t sum(Gr o S_{t-1})
 *            Gr       = a_t Gr                  (on to S_{t-1})
 *            ddt_raw  = ddelta * sigmoid(s) * [dt_min <= softplus(s) <= dt_max],
 *                       s = dt_raw + dt_bias (softplus' = sigmoid; the limit's
 *                       mask is inclusive at both ends)
 *            ddt_bias_h += ddt_raw
 *   then dh0 = Gr and dA_log_h = dA_h * A_h (A = -exp(A_log)).
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

static double ssdo_sigmoid(double s) { return 1.0 / (1.0 + exp(-s)); }

int ssdo_bwd(int64_t B, int64_t L, int64_t H, int64_t P, int64_t G, int64_t N, const double *x,
             const double *dt_raw, const double *dt_bias, const double *A_log, const double *Bm,
             const double *Cm, const double *Dp, const double *h0, const double *dy, const double *dh_last,
             double dt_min, double dt_max, double *dx, double *ddt_raw, double *ddt_bias, double *dA_log,
             double *dBm, double *dCm, double *dDp, double *dh0) {
  if (B < 0 || L < 0 || H < 1 || P < 1 || G < 1 || N < 1 || H % G != 0 || !(dt_min <= dt_max)) return -1;
  const int64_t per = H / G, NP = N * P;
  double *St = (double *)malloc(sizeof(double) * (size_t)((L + 1) * NP)); /* S_{-1} .. S_{L-1} */
  double *Gr = (double *)malloc(sizeof(double) * (size_t)NP);
  if (!St || !Gr) {
    free(St);
    free(Gr);
    return -2;
  }
  memset(dBm, 0, sizeof(double) * (size_t)(B * L * G * N));
  memset(dCm, 0, sizeof(double) * (size_t)(B * L * G * N));
  memset(ddt_bias, 0, sizeof(double) * (size_t)H);
  memset(dA_log, 0, sizeof(double) * (size_t)H);
  memset(dDp, 0, sizeof(double) * (size_t)H);
  for (int64_t b = 0; b < B; ++b)
    for (int64_t h = 0; h < H; ++h) {
      const int64_t grp = h / per;
      const double Ah = -exp(A_log[h]);
      /* the states, step by step (St + (t + 1) * NP holds S_t) */
      if (h0)
        memcpy(St, h0 + (b * H + h) * NP, sizeof(double) * (size_t)NP);
      else
        memset(St, 0, sizeof(double) * (size_t)NP);
      for (int64_t t = 0; t < L; ++t) {
        const int64_t it = (b * L + t) * H + h;
        double dl = ssdo_softplus(dt_raw[it] + dt_bias[h]);
        dl = dl < dt_min ? dt_min : (dl > dt_max ? dt_max : dl);
        const double at = exp(dl * Ah);
        const double *xv = x + ((b * L + t) * H + h) * P, *bv = Bm + ((b * L + t) * G + grp) * N;
        const double *prev = St + t * NP;
        double *next = St + (t + 1) * NP;
        for (int64_t n = 0; n < N; ++n)
          for (int64_t p = 0; p < P; ++p) next[n * P + p] = at * prev[n * P + p] + dl * bv[n] * xv[p];
      }
      /* backward in time */
      if (dh_last)
        memcpy(Gr, dh_last + (b * H + h) * NP, sizeof(double) * (size_t)NP);
      else
        memset(Gr, 0, sizeof(double) * (size_t)NP);
      double dAh = 0.0;
      for (int64_t t = L - 1; t >= 0; --t) {
        const int64_t it = (b * L + t) * H + h;
        const double sarg = dt_raw[it] + dt_bias[h];
        const double sp = ssdo_softplus(sarg);
        const double dl = sp < dt_min ? dt_min : (sp > dt_max ? dt_max : sp);
        const double at = exp(dl * Ah);
        const double *xv = x + ((b * L + t) * H + h) * P, *gy = dy + ((b * L + t) * H + h) * P;
        const double *bv = Bm + ((b * L + t) * G + grp) * N, *cv = Cm + ((b * L + t) * G + grp) * N;
        const double *Scur = St + (t + 1) * NP, *Sprev = St + t * NP;
        double *dbv = dBm + ((b * L + t) * G + grp) * N, *dcv = dCm + ((b * L + t) * G + grp) * N;
        double *dxv = dx + ((b * L + t) * H + h) * P;
        for (int64_t n = 0; n < N; ++n)
          for (int64_t p = 0; p < P; ++p) Gr[n * P + p] += cv[n] * gy[p];
        for (int64_t n = 0; n < N; ++n) {
          double sc = 0.0, sb = 0.0;
          for (int64_t p = 0; p < P; ++p) {
            sc += Scur[n * P + p] * gy[p];
            sb += Gr[n * P + p] * xv[p];
          }
          dcv[n] += sc;
          dbv[n] += dl * sb;
        }
        for (int64_t p = 0; p < P; ++p) {
          double sg = 0.0;
          for (int64_t n = 0; n < N; ++n) sg += Gr[n * P + p] * bv[n];
          dxv[p] = Dp[h] * gy[p] + dl * sg;
          dDp[h] += gy[p] * xv[p];
        }
        double gs = 0.0, gbx = 0.0;
        for (int64_t n = 0; n < N; ++n)
          for (int64_t p = 0; p < P; ++p) {
            gs += Gr[n * P + p] * Sprev[n * P + p];
            gbx += Gr[n * P + p] * bv[n] * xv[p];
          }
        const double ddl = Ah * at * gs + gbx;
        dAh += dl * at * gs;
        for (int64_t i = 0; i < NP; ++i) Gr[i] *= at;
        const double g_raw = (sp >= dt_min && sp <= dt_max) ? ddl * ssdo_sigmoid(sarg) : 0.0;
        ddt_raw[it] = g_raw;
        ddt_bias[h] += g_raw;
      }
      memcpy(dh0 + (b * H + h) * NP, Gr, sizeof(double) * (size_t)NP);
      dA_log[h] += dAh * Ah;
    }
  free(St);
  free(Gr);
  return 0;
}
