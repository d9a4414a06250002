/*
 * ssm_scan.h — C ABI of the GB300 (sm_103a) S6 selective-scan library.
 *
 * The operation (Mamba S6, "selective state space"): for every batch b,
 * channel d and state n,
 *     s      = delta_raw[b,t,d] + delta_bias[d]
 *     delta  = softplus(s)
 *     Abar   = exp(delta * A[d,n]),   A = -exp(A_log[d,n])
 *     h_t    = Abar * h_{t-1} + delta * Bm[b,t,n] * u[b,t,d]      (h_{-1} = h0, or 0)
 *     y      = sum_n Cm[b,t,n] * h_t + Dp[d] * u[b,t,d]
 *     out    = y * silu(z[b,t,d])                                  (out = y when z is NULL)
 * This is the recurrence, discretisation and readout of the final
 * selective_scan_kernel on the POPCORNBENCH transcript page (FW-GLM-5-1__l2_p30),
 * with the softplus / exp_negate / SiLU-gate steps and the "SSM recurrence"
 * entry points (single-step forward, multi-step forward with and without
 * activation saves, local backward plus dB/dC/dD/dA_log reductions) of the
 * mamba-rs kernels.rs page (MambaKernels).
 *
 * Entry points: the scan (forward with and without saves, backward, its two
 * halves, a no-allocation backward, the decode step), their _ex variants with
 * a limit on delta, the causal depthwise conv1d + SiLU in front of the scan
 * (forward, backward, step), and the Mamba-2 SSD forward (with and without
 * state saves) and backward.
 *
 * Conventions shared by every entry point
 *   - Shapes: B = batch, L = seqlen, D = dim (d_inner), N = dstate, 1 <= N <= 16.
 *   - Layouts are dense row-major, last index contiguous:
 *       u, delta_raw, z, dout, du, d_delta_raw, dz : [B][L][D]   (activation dtype)
 *       Bm, Cm, dBm, dCm                            : [B][L][N]   (activation dtype)
 *       A_log, dA_log : [D][N] f32;  Dp, dDp, delta_bias, d_delta_bias : [D] f32
 *       h0, h_last, dh0, dh_last, h (step)          : [B][D][N] f32
 *       chunk_states : [B][ssm_num_chunks(L)][D][N] f32
 *   - The activation dtype `act` is SSM_F32 or SSM_BF16; parameters, states
 *     and parameter gradients are always f32; arithmetic is f32.
 *   - All tensor pointers are DEVICE pointers owned by the caller, aligned
 *     to their element size; outputs must not overlap inputs (except `h` of
 *     ssm_step, which is updated in place).  Pointers marked "nullable" may
 *     be NULL.  The library never allocates or frees device memory; scratch
 *     space is the caller's `ws` buffer.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call
 *     only enqueues work on it and returns; errors found while enqueueing are
 *     returned, errors of the asynchronous work surface at the caller's next
 *     synchronisation.
 *   - Gradients overwrite their outputs (no accumulation).
 *   - Results are deterministic: the same inputs give bit-identical outputs
 *     on every call (fixed-order reductions, no floating-point atomics).
 *   - Return value: SSM_OK (0) or an ssm_status error code; on error nothing
 *     has been enqueued unless the code is SSM_ERR_CUDA.  ssm_last_error()
 *     returns a message for the calling thread's last error.
 */
#ifndef SSM_SCAN_H
#define SSM_SCAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SSM_OK = 0,
  SSM_ERR_INVALID_ARG = 1, /* bad shape, NULL required pointer, misaligned pointer */
  SSM_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. N > 16) */
  SSM_ERR_WORKSPACE = 3,   /* ws NULL or ws_bytes below the required size */
  SSM_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
  SSM_ERR_TIMEOUT = 5,     /* a bounded device-side wait gave up */
  SSM_ERR_INTERNAL = 6     /* a device-side consistency check failed */
} ssm_status;

typedef enum { SSM_F32 = 0, SSM_BF16 = 1 } ssm_dtype;

/* Steps between saved chunk states (the forward's checkpoints for the backward). */
#define SSM_CHUNK_LEN 32
/* Largest supported state size N. */
#define SSM_MAX_DSTATE 16

/* Human-readable name of a status code.  Never NULL. */
const char *ssm_status_string(int status);

/* Message describing the calling thread's most recent error ("" if none). */
const char *ssm_last_error(void);

/* Library version as major*10000 + minor*100 + patch. */
int ssm_version(void);

/* Synchronises `stream`, then reads and clears the library's device status
 * word on the current device.  Returns SSM_ERR_TIMEOUT if a kernel's bounded
 * pipeline wait gave up since the last check (its outputs are then invalid),
 * SSM_ERR_INTERNAL if a kernel found its shared-memory layout unusable and
 * skipped its work (outputs invalid), SSM_ERR_CUDA if the stream reports an
 * error, else SSM_OK. */
int ssm_check_device_status(void *stream);

/* Self-test of the give-up path (no counterpart on the pages): enqueues on
 * `stream` one tiny kernel whose single thread waits on an mbarrier that
 * nothing arrives at; the bounded wait gives up after about 2 s and sets the
 * timeout bit, so the next ssm_check_device_status() returns SSM_ERR_TIMEOUT
 * (and clears it).  Nothing faults and the context stays usable.  Returns
 * SSM_OK, or SSM_ERR_CUDA if the launch fails. */
int ssm_selftest_wait_timeout(void *stream);

/* Number of saved chunk states: ceil(seqlen / SSM_CHUNK_LEN); 0 for seqlen <= 0. */
int64_t ssm_num_chunks(int64_t seqlen);

/* Scratch bytes ssm_scan_fwd / ssm_scan_fwd_nosave need in `ws` for this
 * shape; -1 for an invalid shape.  May be 0, in which case ws may be NULL. */
int64_t ssm_fwd_workspace_bytes(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, int act);

/* Scratch bytes ssm_scan_bwd needs in `ws` (per-tile partial sums of dBm/dCm
 * and per-batch partial sums of the parameter gradients); -1 if invalid. */
int64_t ssm_bwd_workspace_bytes(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, int act);

/* The time-segment plans of the forward and the backward scan for this shape
 * (the chunked parallel scan of the kernels.rs page's "parallel scan" entry
 * point), on the TMA path (dstate 4, 8 or 16; 16-byte aligned tensors); a
 * function of the shape only.
 *   *fwd_segments: 1 = one sequential pass per channel; n > 1 = per-segment
 *     aggregates, a carry pass, then the n segments at once.
 *   *bwd_segments: the backward splits the (batch, 64-channel tile)
 *     sequences over 152 equal ranges of 64-step chunks, one CTA each.  1 =
 *     no aggregate pass (no sequence cut, or every cut sequence hands its
 *     carry from CTA to CTA within the launch); n > 1 = up to n pieces per
 *     sequence, with piece aggregates and a carry pass first.
 * Each pointer nullable; returns SSM_OK, or SSM_ERR_INVALID_ARG for an invalid
 * shape. */
int ssm_plan_segments(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, int act,
                      int *fwd_segments, int *bwd_segments);

/* Number of calls since the library was loaded (all threads and devices)
 * whose plan's cooperative mode -- the forward's stream mode, the backward's
 * hand-over mode -- could not be resident at once on the GPU (another SM
 * count or shared-memory size than the plans assume) and that ran in the
 * non-cooperative form instead: same results, bit for bit, but slower.
 * Host-only; never fails. */
int64_t ssm_plan_fallbacks(void);

/*
 * Forward scan with saves for the backward (mamba-rs kernels.rs page:
 * MambaKernels "Multi-step SSM forward with activation saves for backward").
 *   inputs : u, delta_raw, Bm, Cm, A_log, Dp, delta_bias;  z nullable (no gate);
 *            h0 nullable (zero initial state)
 *   outputs: out [B][L][D];  h_last nullable (final state h_{L-1});
 *            chunk_states [B][nc][D][N] = state before step c*SSM_CHUNK_LEN
 *            (chunk 0 holds h0); it is what ssm_scan_bwd reads.
 *   ws/ws_bytes: scratch of ssm_fwd_workspace_bytes() bytes (nullable when 0).
 *     Long sequences over few channels are split into time segments that run
 *     in parallel (a chunked parallel scan: per-segment decay products and
 *     end states, composed in segment order); ws holds those aggregates.  The
 *     plan is a function of the shape alone, so results are deterministic.
 */
int ssm_scan_fwd(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, int act,
                 const void *u, const void *delta_raw, const void *z, const void *Bm,
                 const void *Cm, const float *A_log, const float *Dp, const float *delta_bias,
                 const float *h0, void *out, float *h_last, float *chunk_states, void *ws,
                 size_t ws_bytes, void *stream);

/*
 * Forward scan without saves (kernels.rs page: "Multi-step SSM forward
 * without activation saves (target network)").  Same as ssm_scan_fwd without
 * the chunk_states output.
 */
int ssm_scan_fwd_nosave(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, int act,
                        const void *u, const void *delta_raw, const void *z, const void *Bm,
                        const void *Cm, const float *A_log, const float *Dp,
                        const float *delta_bias, const float *h0, void *out, float *h_last,
                        void *ws, size_t ws_bytes, void *stream);

/*
 * Backward of  loss = sum(dout * out) + sum(dh_last * h_last)  (kernels.rs
 * page: "Per-(b,t,d,n) local SSM backward" and the dB / dC / dD / d_a_log
 * reductions; no page writes the equations, which follow from the chain rule):
 *   inputs : the forward's inputs (same pointers/values), chunk_states from
 *            ssm_scan_fwd on those inputs, dout [B][L][D]; dh_last nullable.
 *   outputs: du, d_delta_raw [B][L][D]; dz [B][L][D] (required iff z != NULL);
 *            dBm, dCm [B][L][N]; dA_log [D][N]; dDp, d_delta_bias [D];
 *            dh0 nullable ([B][D][N], gradient w.r.t. h0).
 *   d_delta_raw is the gradient w.r.t. delta_raw (softplus' already applied);
 *   d_delta_bias is its sum over (b, t).  Reductions over channels (dBm, dCm)
 *   and over (b, t) (dA_log, dDp, d_delta_bias) use fixed summation trees, so
 *   repeated calls are bit-identical (the determinism policy of the
 *   deterministic_backward.py page: single writer, fixed order, no atomics).
 *   ws/ws_bytes: at least ssm_bwd_workspace_bytes() bytes.
 */
int ssm_scan_bwd(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, int act,
                 const void *u, const void *delta_raw, const void *z, const void *Bm,
                 const void *Cm, const float *A_log, const float *Dp, const float *delta_bias,
                 const float *h0, const float *chunk_states, const void *dout,
                 const float *dh_last, void *du, void *d_delta_raw, void *dz, void *dBm,
                 void *dCm, float *dA_log, float *dDp, float *d_delta_bias, float *dh0,
                 void *ws, size_t ws_bytes, void *stream);

/*
 * The two halves of ssm_scan_bwd, for callers that want to schedule (or time)
 * them separately; ssm_scan_bwd is exactly ssm_scan_bwd_partials followed by
 * ssm_scan_bwd_finalize on the same stream with the same ws.
 *   ssm_scan_bwd_partials: the backward scan.  Writes du, d_delta_raw, dz and
 *     dh0 (same meaning as above) and leaves the per-tile / per-batch partial
 *     sums of dBm, dCm, dA_log, dDp, d_delta_bias in ws.
 *   ssm_scan_bwd_finalize: adds those partials in fixed order into dBm, dCm
 *     ([B][L][N], act dtype), dA_log, dDp, d_delta_bias (f32).  It reads only
 *     ws, so the shape must match the partials call.
 */
int ssm_scan_bwd_partials(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, int act,
                          const void *u, const void *delta_raw, const void *z, const void *Bm,
                          const void *Cm, const float *A_log, const float *Dp,
                          const float *delta_bias, const float *chunk_states, const void *dout,
                          const float *dh_last, void *du, void *d_delta_raw, void *dz,
                          float *dh0, void *ws, size_t ws_bytes, void *stream);

int ssm_scan_bwd_finalize(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, int act,
                          void *dBm, void *dCm, float *dA_log, float *dDp, float *d_delta_bias,
                          const void *ws, size_t ws_bytes, void *stream);

/*
 * ssm_scan_bwd for callers that cannot allocate device memory.  (The pages
 * have no counterpart of this entry point; it is a deployment convenience.)
 * Same arguments and results as ssm_scan_bwd, minus ws/ws_bytes: the scratch
 * for the partial sums is a fixed array of ssm_noalloc_scratch_bytes()
 * (16 MiB) inside the library, reserved on every GPU that loads it until the
 * process exits.  Meant for callers that must not call cudaMalloc: hosts whose
 * framework owns the device allocator, plugin interfaces that pass only input
 * and output pointers, loops that must not allocate or synchronise.
 *   - Shapes needing more scratch than that (ssm_bwd_workspace_bytes() >
 *     ssm_noalloc_scratch_bytes()) are rejected with SSM_ERR_UNSUPPORTED.
 *   - The first call on a device looks the array's device address up with
 *     cudaGetSymbolAddress (that device current), and so does the first call
 *     after that device's context was reset (cudaDeviceReset: the array may
 *     then sit elsewhere); make those calls before any stream capture.
 *   - All calls on a device share the array and it keeps the last call's
 *     contents; calls whose GPU work may overlap race on it and must be
 *     ordered by the caller (same stream, or events).
 *   - Allocates and frees nothing.
 */
size_t ssm_noalloc_scratch_bytes(void);

int ssm_scan_bwd_noalloc(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, int act,
                         const void *u, const void *delta_raw, const void *z, const void *Bm,
                         const void *Cm, const float *A_log, const float *Dp,
                         const float *delta_bias, const float *h0, const float *chunk_states,
                         const void *dout, const float *dh_last, void *du, void *d_delta_raw,
                         void *dz, void *dBm, void *dCm, float *dA_log, float *dDp,
                         float *d_delta_bias, float *dh0, void *stream);

/*
 * One decode step, T = 1 (kernels.rs page: "Single-step SSM forward (T=1
 * inference)").  u, delta_raw, z [B][D] (z nullable), Bm, Cm [B][N], h
 * [B][D][N] f32 read and overwritten in place with the new state, out [B][D].
 * Calling it L times on the slices t = 0..L-1 equals ssm_scan_fwd from h0 = h.
 */
int ssm_step(int64_t batch, int64_t dim, int64_t dstate, int act, const void *u,
             const void *delta_raw, const void *z, const void *Bm, const void *Cm,
             const float *A_log, const float *Dp, const float *delta_bias, float *h, void *out,
             void *stream);

/* ---------------------------------------------------------------------------
 * Limit on delta (dt_limit).  The _ex entry points below are the ones above
 * with one more argument, `opts` (NULL: the defaults, identical to the plain
 * calls).  With opts->dt_min / dt_max the discretisation step is clamped,
 *   delta = min(max(softplus(s), dt_min), dt_max)
 * (mamba3_preprocess_backward.slang page: dt = clamp(softplus, dt_min,
 * dt_max)), and the backward passes no gradient to delta_raw / delta_bias
 * through a clamped step (that page's dt mask).  The forward, the backward
 * and the step of one problem must be given the same limit.  0 <= dt_min <=
 * dt_max (dt_max may be +inf), else SSM_ERR_INVALID_ARG.  Defaults: 0, +inf
 * (no limit).  At a step whose softplus falls exactly on a bound the mask
 * may take either value.
 */
typedef struct ssm_scan_options {
  float dt_min;
  float dt_max;
} ssm_scan_options;

/* ssm_scan_fwd with options; chunk_states nullable (no saves, as
 * ssm_scan_fwd_nosave). */
int ssm_scan_fwd_ex(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, int act,
                    const void *u, const void *delta_raw, const void *z, const void *Bm,
                    const void *Cm, const float *A_log, const float *Dp, const float *delta_bias,
                    const float *h0, void *out, float *h_last, float *chunk_states, void *ws,
                    size_t ws_bytes, void *stream, const ssm_scan_options *opts);

int ssm_scan_bwd_ex(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, int act,
                    const void *u, const void *delta_raw, const void *z, const void *Bm,
                    const void *Cm, const float *A_log, const float *Dp, const float *delta_bias,
                    const float *h0, const float *chunk_states, const void *dout,
                    const float *dh_last, void *du, void *d_delta_raw, void *dz, void *dBm,
                    void *dCm, float *dA_log, float *dDp, float *d_delta_bias, float *dh0,
                    void *ws, size_t ws_bytes, void *stream, const ssm_scan_options *opts);

int ssm_scan_bwd_partials_ex(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, int act,
                             const void *u, const void *delta_raw, const void *z, const void *Bm,
                             const void *Cm, const float *A_log, const float *Dp,
                             const float *delta_bias, const float *chunk_states, const void *dout,
                             const float *dh_last, void *du, void *d_delta_raw, void *dz,
                             float *dh0, void *ws, size_t ws_bytes, void *stream,
                             const ssm_scan_options *opts);

int ssm_step_ex(int64_t batch, int64_t dim, int64_t dstate, int act, const void *u,
                const void *delta_raw, const void *z, const void *Bm, const void *Cm,
                const float *A_log, const float *Dp, const float *delta_bias, float *h, void *out,
                void *stream, const ssm_scan_options *opts);

/* ---------------------------------------------------------------------------
 * Mamba-2 SSD forward: the scan with one scalar decay per head (the
 * deterministic_backward.py page's ssd_combined kernels: dt per (batch, step,
 * head), one A and one dt_bias per head, softplus and dt_limit).  For each
 * (b, h), t = 0 .. L-1, with g = h / (H / G) the head's group:
 *   delta = min(max(softplus(dt_raw[b,t,h] + dt_bias[h]), dt_min), dt_max)
 *   S[n][p] = exp(-exp(A_log[h]) * delta) * S[n][p] + delta * Bm[b,t,g,n] * x[b,t,h,p]
 *   y[b,t,h,p] = sum_n Cm[b,t,g,n] * S[n][p] + Dp[h] * x[b,t,h,p]
 * evaluated in its chunked matrix form (64-step chunks, tensor cores).
 *   x, y [B][L][H][P]; dt_raw [B][L][H]; Bm, Cm [B][L][G][N] (act dtype);
 *   dt_bias, A_log, Dp [H] f32; h0 (nullable: zeros), h_last (nullable)
 *   [B][H][N][P] f32; h0 and h_last may be the same buffer (the state
 *   updated in place).  opts: the limit on delta (NULL: none).
 * Supported: act = SSM_BF16, P = headdim in {32, 64, 128, 192, 256}, N =
 * dstate in {64, 128}, H % G == 0; x, dt_raw, Bm, Cm, y 16-byte aligned.  (A
 * head of P = 64 m columns runs as m sub-heads of 64 columns sharing the
 * head's dt, A, Dp and the group's Bm, Cm: the columns of S evolve
 * independently.  A head of 32 columns runs as 64 whose last 32 are zero,
 * which adds exact zeros to every sum; nothing is written past column 32.)
 * Other shapes return SSM_ERR_UNSUPPORTED.  Asynchronous on `stream`;
 * allocates nothing.
 */
int ssm_ssd_fwd(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim, int64_t ngroups,
                int64_t dstate, int act, const void *x, const void *dt_raw, const float *dt_bias,
                const float *A_log, const void *Bm, const void *Cm, const float *Dp, const float *h0,
                void *y, float *h_last, const ssm_scan_options *opts, void *stream);

/* Steps per chunk of the SSD's chunked form (and between its saved states). */
#define SSM_SSD_CHUNK_LEN 64

/*
 * ssm_ssd_fwd that also saves, for the backward, the state entering every
 * chunk: chunk_states [B][H][ceil(L/64)][N][P] bf16 (device, caller-owned,
 * 16-byte aligned), chunk c holding the state before step 64c as the bf16
 * copy the chunk's readout uses (chunk 0: h0, or zeros).  Otherwise the same
 * as ssm_ssd_fwd (same results, bit for bit).
 */
int ssm_ssd_fwd_save(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim, int64_t ngroups,
                     int64_t dstate, int act, const void *x, const void *dt_raw, const float *dt_bias,
                     const float *A_log, const void *Bm, const void *Cm, const float *Dp, const float *h0,
                     void *y, float *h_last, void *chunk_states, const ssm_scan_options *opts, void *stream);

/* Scratch bytes ssm_ssd_bwd needs in `ws` (per-head dBm / dCm terms,
 * per-(batch, head) parameter sums, and the flags and state gradients that
 * CTAs hand over when sequences outnumber the SMs); -1 for an invalid or
 * unsupported shape. */
int64_t ssm_ssd_bwd_workspace_bytes(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
                                    int64_t ngroups, int64_t dstate, int act);

/*
 * Mamba-2 SSD backward (deterministic_backward.py page: the backward of the
 * ssd_combined kernels -- dx, dB, dC, the dt and A gradients -- by single
 * writers with every sum in a fixed order, no float atomics).  The gradient of
 *   loss = sum(dy * y) + sum(dh_last * h_last)
 * through the recurrence of ssm_ssd_fwd (same shapes, same limit `opts`):
 *   inputs : the forward's inputs; chunk_states from ssm_ssd_fwd_save on
 *            them; dy [B][L][H][P]; dh_last nullable (zeros) [B][H][N][P] f32
 *   outputs: dx [B][L][H][P]; ddt_raw [B][L][H] (the gradient w.r.t. dt_raw,
 *            softplus' applied, zero where the limit clamped delta; the mask
 *            is inclusive at both bounds); dBm, dCm [B][L][G][N] (summed over
 *            the heads of a group in ascending head order) -- act dtype;
 *            ddt_bias, dA_log, dDp [H] f32 (summed over batch and steps in a
 *            fixed order); dh0 nullable [B][H][N][P] f32.
 *   ws/ws_bytes: at least ssm_ssd_bwd_workspace_bytes() bytes, 256-byte
 *            aligned.
 * Evaluated per chunk of 64 steps, last chunk first, in the chunked matrix
 * form on the tensor cores (bf16 operands, f32 accumulation; the state's
 * gradient in f32).  With more (batch, head) sequences than SMs, one range of
 * chunks per SM, launched cooperatively (all resident; where the GPU cannot
 * hold them, one CTA per sequence, same per-sequence results).  Supported: as ssm_ssd_fwd (bf16, P in {32, 64, 128, 192,
 * 256}, N in {64, 128}); dy, dx, dh_last, dh0, chunk_states 16-byte aligned.  Results are
 * bit-identical from call to call.  Asynchronous on `stream`.
 */
int ssm_ssd_bwd(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim, int64_t ngroups,
                int64_t dstate, int act, const void *x, const void *dt_raw, const float *dt_bias,
                const float *A_log, const void *Bm, const void *Cm, const float *Dp,
                const void *chunk_states, const void *dy, const float *dh_last, void *dx, void *ddt_raw,
                float *ddt_bias, float *dA_log, void *dBm, void *dCm, float *dDp, float *dh0, void *ws,
                size_t ws_bytes, const ssm_scan_options *opts, void *stream);

/* ---------------------------------------------------------------------------
 * Causal depthwise conv1d + SiLU, the convolution in front of the scan in a
 * Mamba block (kernels.rs page: "Multi-step conv1d forward with state saves
 * for backward", "Multi-step conv1d backward", "Single-step depthwise conv1d
 * forward with SiLU"; deterministic_backward.py page: weight and bias
 * gradients summed in a fixed order).  K = width taps per channel, 1..8:
 *   pre[b,t,d] = bias[d] + sum_{k<K} w[d][k] * xx(b, t-(K-1)+k, d)
 *   out[b,t,d] = pre * sigmoid(pre)
 * where xx(b,t,d) = x[b][t][d] for t >= 0 and state0[b][d][K-1+t] for t < 0
 * (the K-1 inputs before the first step, oldest first; zeros when state0 is
 * NULL).  Layouts: x, out, dout, dx [B][L][D] (act dtype); w [D][K], bias
 * [D] f32; states [B][D][K-1] in the act dtype; dstate0 [B][D][K-1] f32.
 * Same pointer and error rules as the scan entry points.
 */
#define SSM_MAX_CONV_WIDTH 8

/* Forward.  state_last (nullable) receives the last K-1 inputs (the state to
 * continue from: a second call on the next steps with state0 = state_last
 * equals one call on the whole sequence, bit for bit). */
int ssm_conv1d_fwd(int64_t batch, int64_t seqlen, int64_t dim, int64_t width, int act,
                   const void *x, const float *w, const float *bias, const void *state0, void *out,
                   void *state_last, void *stream);

/* Scratch bytes ssm_conv1d_bwd needs in `ws` (per-run partial sums of dw and
 * dbias); -1 for an invalid shape. */
int64_t ssm_conv1d_bwd_workspace_bytes(int64_t batch, int64_t seqlen, int64_t dim, int64_t width, int act);

/* Backward of loss = sum dout * out: dx (act), dw, dbias (f32, overwritten;
 * sums over (b, t) in a fixed order, bit-identical from call to call), and
 * dstate0 (nullable, f32) = the gradient of the initial state. */
int ssm_conv1d_bwd(int64_t batch, int64_t seqlen, int64_t dim, int64_t width, int act,
                   const void *x, const float *w, const float *bias, const void *state0,
                   const void *dout, void *dx, float *dw, float *dbias, float *dstate0, void *ws,
                   size_t ws_bytes, void *stream);

/* One step: x [B][D], state [B][D][K-1] read and shifted in place (it takes
 * x as its newest entry), out [B][D].  Steps in a row equal ssm_conv1d_fwd. */
int ssm_conv1d_step(int64_t batch, int64_t dim, int64_t width, int act, const void *x,
                    const float *w, const float *bias, void *state, void *out, void *stream);

/* Which kernels a conv1d call with these shapes and pointers runs (host-only
 * query, no launch): SSM_CONV_PATH_TILE (TMA tiles of 64 steps x 128
 * channels: D*elem a multiple of 16 bytes, x and dout 16-byte aligned),
 * SSM_CONV_PATH_VECTOR (4 channels per thread: D % 4 == 0, 8-byte (bf16) or
 * 16-byte (f32) aligned) or SSM_CONV_PATH_SCALAR; dout NULL asks about the
 * forward (y = out), else the backward (y = dx).  All three give the same
 * results within rounding.  Negative status on an invalid shape. */
#define SSM_CONV_PATH_SCALAR 0
#define SSM_CONV_PATH_VECTOR 1
#define SSM_CONV_PATH_TILE 2
int ssm_conv1d_path(int64_t batch, int64_t seqlen, int64_t dim, int64_t width, int act,
                    const void *x, const void *dout, const void *y);

#ifdef __cplusplus
}
#endif

#endif /* SSM_SCAN_H */
