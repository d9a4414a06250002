/*
 * S6 selective-scan oracle: a plain, slow, f64 CPU implementation.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark load this library.  The product path (the
 * CUDA library and its Python binding) never links, imports or calls it, and
 * this file shares no code, header or constant with that path.
 *
 * What it computes (names follow the Mamba S6 notation):
 *   inputs   u, delta_raw, z : [B][L][D]      Bm, Cm : [B][L][N]
 *            A_log : [D][N]   Dp, delta_bias : [D]   h0 : [B][D][N] (optional)
 *   forward  s     = delta_raw[b,t,d] + delta_bias[d]
 *            delta = softplus(s) = log(1 + e^s)
 *            A     = -exp(A_log[d,n])
 *            a     = exp(delta * A)                      (zero-order-hold Abar)
 *            h_t   = a * h_{t-1} + delta * Bm[b,t,n] * u   (h_{-1} = h0 or 0)
 *            y     = sum_n Cm[b,t,n] * h_t + Dp[d] * u
 *            out   = y * z * sigmoid(z)                  (out = y when z is absent)
 *   optional Δ limit [dt_min, dt_max] (no limit: 0 and +inf):
 *            delta = min(max(softplus(s), dt_min), dt_max)
 *            and in the backward d_delta_raw is multiplied by the mask
 *            [dt_min <= softplus(s) <= dt_max] (both ends inclusive): the
 *            clamped steps pass no gradient to delta_raw and delta_bias.
 *            Source: the mamba3_preprocess_backward.slang page (oarust crate)
 *            clamps softplus(raw dt + bias) to [dt_min, dt_max] and masks the
 *            raw-dt gradient with that inclusive test; the
 *            deterministic_backward.py page passes dt_limit = (0, inf) as the
 *            default of the same clamp.
 *   Sources: the recurrence, discretisation and readout are the ones the final
 *   selective_scan_kernel on the POPCORNBENCH page (transcript
 *   FW-GLM-5-1__l2_p30) computes: A as minus the exponential of A_log, the
 *   decay as the exponential of delta times A, the state scaled by the decay
 *   plus delta times B times the input, and the output as the sum over n of
 *   C times the state plus D times the input.  The softplus on delta, the
 *   exp_negate of A_log, the SiLU gate and gating_backward are the kernels the
 *   mamba-rs kernels.rs page registers (MambaKernels, "SSM recurrence",
 *   "Activations" and "Elementwise" groups).
 *
 *   backward (loss = sum dout*out + sum dh_last*h_last; derived by the chain
 *   rule, since no page writes it out; pinned by finite differences in tests):
 *            sz  = sigmoid(z);  dy = dout * z * sz
 *            dz  = dout * y * sz * (1 + z * (1 - sz))
 *            g_t = dy_t * Cm_t + a_{t+1} * g_{t+1},  g at t = L-1 starts from dh_last
 *            du  = Dp * dy + delta * sum_n g * Bm
 *            ddelta = sum_n g * (A * a * h_{t-1} + Bm * u)
 *            d_delta_raw = ddelta * sigmoid(s) * mask   (softplus' = sigmoid)
 *            dBm[b,t,n] = sum_d g * delta * u           dCm[b,t,n] = sum_d dy * h_t
 *            dDp[d] = sum_{b,t} dy * u                  d_delta_bias[d] = sum_{b,t} d_delta_raw
 *            dA_log[d,n] = A * sum_{b,t} g * delta * a * h_{t-1}   (dA/dA_log = A)
 *            dh0 = a_0 * g_0
 *
 * Sums over (b,t) for the parameter gradients run in ascending b, then t.
 * Sums over d for dBm/dCm run in ascending d inside fixed blocks of 16
 * channels, the block partials then added in ascending block order; the
 * result does not depend on the thread count.  Threads (pthreads) only split
 * independent channels; every (b,d) scan is the plain sequential loop below.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define S6O_DBLOCK 16

typedef struct {
  int64_t B, L, D, N;
  const double *u, *delta_raw, *z, *Bm, *Cm, *A_log, *Dp, *delta_bias, *h0;
  double dt_min, dt_max; /* the limit on delta (0 and +inf: none) */
} s6o_problem;

/* softplus(s) = log(1 + e^s), written so that neither branch overflows. */
static double s6o_softplus(double s) {
  return s > 0.0 ? s + log1p(exp(-s)) : log1p(exp(s));
}

/* delta = softplus(s) clamped to [dt_min, dt_max] */
static double s6o_delta(const s6o_problem *p, double sp) {
  if (sp < p->dt_min) return p->dt_min;
  if (sp > p->dt_max) return p->dt_max;
  return sp;
}

/* logistic sigmoid; for x -> -inf exp(-x) overflows to inf and the result is 0. */
static double s6o_sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* Index helpers for the row-major layouts listed in the header comment. */
static inline int64_t ix_bld(const s6o_problem *p, int64_t b, int64_t t, int64_t d) {
  return (b * p->L + t) * p->D + d;
}
static inline int64_t ix_bln(const s6o_problem *p, int64_t b, int64_t t, int64_t n) {
  return (b * p->L + t) * p->N + n;
}

/*
 * Sequential forward scan of one (b,d) channel over t = 0..L-1.
 *   h      : [N] state, holds h_{-1} on entry and h_{L-1} on return
 *   out    : [B][L][D] gated output (written at (b,:,d)); may be NULL
 *   hist_h : [L][N] h_t for every t, or NULL
 *   hist_a : [L][N] a_t for every t, or NULL
 *   hist_y : [L] pre-gate y_t, or NULL
 * The single-step call (ssm_step) is this same function with L = 1.
 */
static void s6o_scan_channel(const s6o_problem *p, int64_t b, int64_t d, double *h,
                             double *out, double *hist_h, double *hist_a,
                             double *hist_y) {
  const int64_t N = p->N;
  for (int64_t t = 0; t < p->L; ++t) {
    const double u = p->u[ix_bld(p, b, t, d)];
    const double s = p->delta_raw[ix_bld(p, b, t, d)] + p->delta_bias[d];
    const double delta = s6o_delta(p, s6o_softplus(s));
    double y = 0.0;
    for (int64_t n = 0; n < N; ++n) {
      const double A = -exp(p->A_log[d * N + n]);
      const double a = exp(delta * A);
      const double bt = delta * p->Bm[ix_bln(p, b, t, n)] * u;
      h[n] = a * h[n] + bt;
      y += p->Cm[ix_bln(p, b, t, n)] * h[n];
      if (hist_h) hist_h[t * N + n] = h[n];
      if (hist_a) hist_a[t * N + n] = a;
    }
    y += p->Dp[d] * u;
    if (hist_y) hist_y[t] = y;
    if (out) {
      double o = y;
      if (p->z) {
        const double z = p->z[ix_bld(p, b, t, d)];
        o = y * z * s6o_sigmoid(z);
      }
      out[ix_bld(p, b, t, d)] = o;
    }
  }
}

/* ------------------------------------------------------------------ forward */

typedef struct {
  const s6o_problem *p;
  int64_t b0, b1, d0, d1;
  double *out, *h_last;
  int64_t next_d; /* work counter, guarded by mu */
  pthread_mutex_t mu;
} s6o_fwd_job;

static void *s6o_fwd_worker(void *arg) {
  s6o_fwd_job *job = (s6o_fwd_job *)arg;
  const s6o_problem *p = job->p;
  double *h = (double *)malloc(sizeof(double) * (size_t)(p->N > 0 ? p->N : 1));
  for (;;) {
    pthread_mutex_lock(&job->mu);
    const int64_t d = job->next_d++;
    pthread_mutex_unlock(&job->mu);
    if (d >= job->d1) break;
    for (int64_t b = job->b0; b < job->b1; ++b) {
      for (int64_t n = 0; n < p->N; ++n) h[n] = p->h0 ? p->h0[(b * p->D + d) * p->N + n] : 0.0;
      s6o_scan_channel(p, b, d, h, job->out, NULL, NULL, NULL);
      if (job->h_last)
        for (int64_t n = 0; n < p->N; ++n) job->h_last[(b * p->D + d) * p->N + n] = h[n];
    }
  }
  free(h);
  return NULL;
}

static int s6o_nthreads(int requested, int64_t work) {
  int nt = requested > 0 ? requested : 1;
  if (nt > 256) nt = 256;
  if (work < nt) nt = work > 0 ? (int)work : 1;
  return nt;
}

/*
 * Forward over channels d in [d0,d1) of batches b in [b0,b1).  Outputs are
 * full-size arrays; only the selected (b,d) entries are written.
 * Returns 0, or -1 on a bad range.
 */
int s6o_fwd(int64_t B, int64_t L, int64_t D, int64_t N, const double *u,
            const double *delta_raw, const double *z, const double *Bm, const double *Cm,
            const double *A_log, const double *Dp, const double *delta_bias,
            const double *h0, double *out, double *h_last, int64_t b0, int64_t b1,
            int64_t d0, int64_t d1, int nthreads, double dt_min, double dt_max) {
  if (B < 0 || L < 0 || D < 0 || N < 0 || b0 < 0 || b1 > B || b0 > b1 || d0 < 0 || d1 > D ||
      d0 > d1 || !(dt_min <= dt_max))
    return -1;
  s6o_problem p = {B, L, D, N, u, delta_raw, z, Bm, Cm, A_log, Dp, delta_bias, h0, dt_min, dt_max};
  s6o_fwd_job job;
  job.p = &p;
  job.b0 = b0; job.b1 = b1; job.d0 = d0; job.d1 = d1;
  job.out = out; job.h_last = h_last;
  job.next_d = d0;
  pthread_mutex_init(&job.mu, NULL);
  const int nt = s6o_nthreads(nthreads, d1 - d0);
  pthread_t th[256];
  for (int i = 1; i < nt; ++i) pthread_create(&th[i], NULL, s6o_fwd_worker, &job);
  s6o_fwd_worker(&job);
  for (int i = 1; i < nt; ++i) pthread_join(th[i], NULL);
  pthread_mutex_destroy(&job.mu);
  return 0;
}

/*
 * Single decode step: s6o_fwd's channel scan with L = 1.  u, delta_raw, z are
 * [B][D], Bm, Cm are [B][N], h is the [B][D][N] state (read, then overwritten
 * with the new state), out is [B][D].
 */
int s6o_step(int64_t B, int64_t D, int64_t N, const double *u, const double *delta_raw,
             const double *z, const double *Bm, const double *Cm, const double *A_log,
             const double *Dp, const double *delta_bias, double *h, double *out, double dt_min,
             double dt_max) {
  if (B < 0 || D < 0 || N < 0 || !(dt_min <= dt_max)) return -1;
  s6o_problem p = {B, 1, D, N, u, delta_raw, z, Bm, Cm, A_log, Dp, delta_bias, NULL, dt_min, dt_max};
  for (int64_t b = 0; b < B; ++b)
    for (int64_t d = 0; d < D; ++d) s6o_scan_channel(&p, b, d, h + (b * D + d) * N, out, NULL, NULL, NULL);
  return 0;
}

/* ----------------------------------------------------------------- backward */

typedef struct {
  const s6o_problem *p;
  const double *dout, *dh_last;
  int64_t b0, b1, d0, d1;
  double *du, *d_delta_raw, *dz, *dA_log, *dDp, *d_delta_bias, *dh0;
  double *part_dB, *part_dC; /* [nblk][B][L][N] block partials over d */
  int64_t nblk, next_blk;
  pthread_mutex_t mu;
} s6o_bwd_job;

/* Backward of one (b,d) channel; adds its dBm/dCm terms into pdB/pdC ([L][N]
 * slices of the block partials) and its parameter terms into the per-d sums. */
static void s6o_bwd_channel(s6o_bwd_job *job, int64_t b, int64_t d, double *hist_h,
                            double *hist_a, double *hist_y, double *h, double *g,
                            double *pdB, double *pdC, double *acc_dA, double *acc_dD,
                            double *acc_dbias) {
  const s6o_problem *p = job->p;
  const int64_t N = p->N, L = p->L;
  for (int64_t n = 0; n < N; ++n) h[n] = p->h0 ? p->h0[(b * p->D + d) * N + n] : 0.0;
  s6o_scan_channel(p, b, d, h, NULL, hist_h, hist_a, hist_y);

  /* g holds the carry a_{t+1} * g_{t+1}; at t = L-1 that is dh_last. */
  for (int64_t n = 0; n < N; ++n) g[n] = job->dh_last ? job->dh_last[(b * p->D + d) * N + n] : 0.0;

  for (int64_t t = L - 1; t >= 0; --t) {
    const int64_t i = ix_bld(p, b, t, d);
    const double u = p->u[i];
    const double s = p->delta_raw[i] + p->delta_bias[d];
    const double sp = s6o_softplus(s);
    const double delta = s6o_delta(p, sp);
    const double mask = (sp >= p->dt_min && sp <= p->dt_max) ? 1.0 : 0.0;
    const double y = hist_y[t];
    const double dout = job->dout[i];
    double dy;
    if (p->z) {
      const double z = p->z[i];
      const double sz = s6o_sigmoid(z);
      dy = dout * z * sz;
      if (job->dz) job->dz[i] = dout * y * sz * (1.0 + z * (1.0 - sz));
    } else {
      dy = dout;
    }
    double sum_gB = 0.0, sum_dh_ddelta = 0.0;
    for (int64_t n = 0; n < N; ++n) {
      const double A = -exp(p->A_log[d * N + n]);
      const double a = hist_a[t * N + n];
      const double h_prev = t > 0 ? hist_h[(t - 1) * N + n]
                                  : (p->h0 ? p->h0[(b * p->D + d) * N + n] : 0.0);
      const double Bn = p->Bm[ix_bln(p, b, t, n)];
      const double Cn = p->Cm[ix_bln(p, b, t, n)];
      const double gt = dy * Cn + g[n];
      sum_gB += gt * Bn;
      sum_dh_ddelta += gt * (A * a * h_prev + Bn * u);
      pdB[t * N + n] += gt * delta * u;
      pdC[t * N + n] += dy * hist_h[t * N + n];
      acc_dA[n] += gt * delta * a * h_prev;
      g[n] = a * gt; /* carry for step t-1 */
    }
    if (job->du) job->du[i] = p->Dp[d] * dy + delta * sum_gB;
    const double d_raw = sum_dh_ddelta * s6o_sigmoid(s) * mask;
    if (job->d_delta_raw) job->d_delta_raw[i] = d_raw;
    *acc_dD += dy * u;
    *acc_dbias += d_raw;
  }
  if (job->dh0)
    for (int64_t n = 0; n < N; ++n) job->dh0[(b * p->D + d) * N + n] = g[n];
}

static void *s6o_bwd_worker(void *arg) {
  s6o_bwd_job *job = (s6o_bwd_job *)arg;
  const s6o_problem *p = job->p;
  const int64_t N = p->N, L = p->L;
  const size_t nl = (size_t)(L > 0 ? L : 1), nn = (size_t)(N > 0 ? N : 1);
  double *hist_h = (double *)malloc(sizeof(double) * nl * nn);
  double *hist_a = (double *)malloc(sizeof(double) * nl * nn);
  double *hist_y = (double *)malloc(sizeof(double) * nl);
  double *h = (double *)malloc(sizeof(double) * nn);
  double *g = (double *)malloc(sizeof(double) * nn);
  double *acc_dA = (double *)malloc(sizeof(double) * nn);
  for (;;) {
    pthread_mutex_lock(&job->mu);
    const int64_t blk = job->next_blk++;
    pthread_mutex_unlock(&job->mu);
    if (blk >= job->nblk) break;
    const int64_t da = job->d0 + blk * S6O_DBLOCK;
    const int64_t db = da + S6O_DBLOCK < job->d1 ? da + S6O_DBLOCK : job->d1;
    for (int64_t d = da; d < db; ++d) {
      double acc_dD = 0.0, acc_dbias = 0.0;
      for (int64_t n = 0; n < N; ++n) acc_dA[n] = 0.0;
      for (int64_t b = job->b0; b < job->b1; ++b) {
        double *pdB = job->part_dB + ((blk * p->B + b) * L) * N;
        double *pdC = job->part_dC + ((blk * p->B + b) * L) * N;
        s6o_bwd_channel(job, b, d, hist_h, hist_a, hist_y, h, g, pdB, pdC, acc_dA, &acc_dD,
                        &acc_dbias);
      }
      if (job->dA_log)
        for (int64_t n = 0; n < N; ++n) job->dA_log[d * N + n] = -exp(p->A_log[d * N + n]) * acc_dA[n];
      if (job->dDp) job->dDp[d] = acc_dD;
      if (job->d_delta_bias) job->d_delta_bias[d] = acc_dbias;
    }
  }
  free(hist_h); free(hist_a); free(hist_y); free(h); free(g); free(acc_dA);
  return NULL;
}

/*
 * Backward over channels d in [d0,d1) of batches b in [b0,b1).
 * dBm/dCm ([B][L][N]) receive the sum over the selected channels only, and
 * dA_log/dDp/d_delta_bias the sum over the selected batches only; the full
 * gradients are the case d0 = 0, d1 = D, b0 = 0, b1 = B.  Any output pointer
 * may be NULL.  Returns 0, -1 on a bad range, -2 when out of memory.
 */
int s6o_bwd(int64_t B, int64_t L, int64_t D, int64_t N, const double *u,
            const double *delta_raw, const double *z, const double *Bm, const double *Cm,
            const double *A_log, const double *Dp, const double *delta_bias,
            const double *h0, const double *dout, const double *dh_last, double *du,
            double *d_delta_raw, double *dz, double *dBm, double *dCm, double *dA_log,
            double *dDp, double *d_delta_bias, double *dh0, int64_t b0, int64_t b1,
            int64_t d0, int64_t d1, int nthreads, double dt_min, double dt_max) {
  if (B < 0 || L < 0 || D < 0 || N < 0 || b0 < 0 || b1 > B || b0 > b1 || d0 < 0 || d1 > D ||
      d0 > d1 || !(dt_min <= dt_max))
    return -1;
  s6o_problem p = {B, L, D, N, u, delta_raw, z, Bm, Cm, A_log, Dp, delta_bias, h0, dt_min, dt_max};
  s6o_bwd_job job;
  memset(&job, 0, sizeof(job));
  job.p = &p;
  job.dout = dout; job.dh_last = dh_last;
  job.b0 = b0; job.b1 = b1; job.d0 = d0; job.d1 = d1;
  job.du = du; job.d_delta_raw = d_delta_raw; job.dz = dz;
  job.dA_log = dA_log; job.dDp = dDp; job.d_delta_bias = d_delta_bias; job.dh0 = dh0;
  job.nblk = (d1 - d0 + S6O_DBLOCK - 1) / S6O_DBLOCK;
  const size_t slab = (size_t)B * (size_t)L * (size_t)N;
  const size_t cnt = (size_t)(job.nblk > 0 ? job.nblk : 1) * (slab > 0 ? slab : 1);
  job.part_dB = (double *)calloc(cnt, sizeof(double));
  job.part_dC = (double *)calloc(cnt, sizeof(double));
  if (!job.part_dB || !job.part_dC) {
    free(job.part_dB); free(job.part_dC);
    return -2;
  }
  pthread_mutex_init(&job.mu, NULL);
  const int nt = s6o_nthreads(nthreads, job.nblk);
  pthread_t th[256];
  for (int i = 1; i < nt; ++i) pthread_create(&th[i], NULL, s6o_bwd_worker, &job);
  s6o_bwd_worker(&job);
  for (int i = 1; i < nt; ++i) pthread_join(th[i], NULL);
  pthread_mutex_destroy(&job.mu);

  /* Block partials summed in ascending block order (fixed, thread-independent). */
  for (size_t j = 0; j < slab; ++j) {
    double sb = 0.0, sc = 0.0;
    for (int64_t k = 0; k < job.nblk; ++k) {
      sb += job.part_dB[(size_t)k * slab + j];
      sc += job.part_dC[(size_t)k * slab + j];
    }
    if (dBm) dBm[j] = sb;
    if (dCm) dCm[j] = sc;
  }
  free(job.part_dB); free(job.part_dC);
  return 0;
}
