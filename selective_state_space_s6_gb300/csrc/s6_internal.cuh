// Internal declarations shared by the S6 kernels and the C-ABI host code.
// Not part of the public interface (that is include/ssm_scan.h).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "ssm_scan.h"

namespace s6 {

constexpr int kChunk = SSM_CHUNK_LEN;  // steps between saved chunk states
constexpr int kDTile = 64;             // channels per CTA in the forward scan kernels
constexpr int kBwdTile = 128;          // channels per CTA (and per sequence) in the TMA backward
constexpr int kThreadsPerChannel = 2;  // each channel's N states are split over 2 lanes
constexpr int kScanThreads = kDTile * kThreadsPerChannel;
constexpr int kSub = 8;                // backward: steps kept in registers per sub-chunk
constexpr unsigned int kStatusWaitTimeoutBit = 1u;  // same bit as kStatusWaitTimeout
constexpr unsigned int kStatusLayoutBit = 2u;       // same bit as kStatusLayout

// ---------------------------------------------------------------- params

// Work plan of a persistent scan: the (batch, channel tile) sequences, each
// of nch chunks, are laid out as U = nseq * nch chunk units (sequence
// s = b * ndt + j) and cut into P ranges, one per persistent CTA.  A range
// covers pieces of one or more sequences; a sequence cut by range
// boundaries has K > 1 pieces, numbered in time order.  The plan is a
// function of the shape only.  Two layouts:
//   contiguous (H == 0): unit s * nch + c, P equal ranges
//     (range w = [bound(w), bound(w + 1)), bound(w) = floor(w * U / P));
//   split (H > 0, backward only, when there are fewer sequences than
//     ranges): every sequence is a head of its first H chunks, which is
//     range s by itself, and a tail of the other T = nch - H chunks; the
//     tails, laid end to end after the heads (unit nseq * H + s * T + c - H),
//     are cut into the other P - nseq ranges equally.  H = ceil(U / P), so
//     no range is longer than in the contiguous layout, and the later pieces
//     -- the ones the aggregate pass walks -- are as short as a cut of every
//     sequence allows.
//   Backward (128-channel tiles): piece k > 0 needs the adjoint carry of the
//   pieces after it -- handed over between CTAs, or composed from piece
//   aggregates (the chunked parallel scan); piece k of sequence (b, j) owns
//   row b * maxp + k of the parameter partials.
//   Forward (128/TPC-channel tiles, contiguous, unit s * nch + (nch - 1 - c)):
//   a range starts with a sequence's first piece and ends with another's
//   last, whose start state the CTA holding the first piece hands over.
struct ScanPlan {
  long long U;  // chunk units
  int P;        // worker CTAs (ranges), 1 <= P <= U
  int nch;      // chunks per sequence
  int ndt;      // 64-channel tiles
  int maxp;     // most pieces any sequence has
  int H;        // split layout: head chunks per sequence (0: contiguous layout)
  // carries handed from CTA to CTA (no aggregate pass): every sequence in at
  // most two pieces and no range shorter than a sequence
  bool handover;
};

// M units (sequences of len units end to end) cut into R equal ranges
struct PlanCut {
  long long M, R;
  int len;
};
__host__ __device__ inline long long cut_bound(const PlanCut& c, long long w) { return w * c.M / c.R; }
// number of w in [0, R] with cut_bound(w) <= X, for 0 <= X < M
__host__ __device__ inline long long cut_count_le(const PlanCut& c, long long X) { return ((X + 1) * c.R + c.M - 1) / c.M; }
__host__ __device__ inline int cut_pieces(const PlanCut& c, long long s) {
  const long long S0 = s * c.len, S1 = S0 + c.len;
  return (int)(cut_count_le(c, S1 - 1) - cut_count_le(c, S0)) + 1;
}
__host__ __device__ inline void cut_piece_range(const PlanCut& c, long long s, int k, int& lo, int& hi) {
  const long long S0 = s * c.len;
  const long long wa = cut_count_le(c, S0);  // first range boundary after the sequence start
  const int K = cut_pieces(c, s);
  lo = k == 0 ? 0 : (int)(cut_bound(c, wa + k - 1) - S0);
  hi = k == K - 1 ? c.len : (int)(cut_bound(c, wa + k) - S0);
}

__host__ __device__ inline long long plan_nseq(const ScanPlan& pl) { return pl.nch > 0 ? pl.U / pl.nch : 0; }
// the cut of the contiguous layout, or of the split layout's tails
__host__ __device__ inline PlanCut plan_cut(const ScanPlan& pl) {
  PlanCut c;
  if (pl.H == 0) {
    c.M = pl.U;
    c.R = pl.P;
    c.len = pl.nch;
  } else {
    const long long ns = plan_nseq(pl);
    c.len = pl.nch - pl.H;
    c.M = ns * c.len;
    c.R = pl.P - ns;
  }
  return c;
}
__host__ __device__ inline long long plan_bound(const ScanPlan& pl, long long w) {
  if (pl.H == 0) return w * pl.U / pl.P;
  const long long ns = plan_nseq(pl);
  return w <= ns ? w * pl.H : ns * pl.H + cut_bound(plan_cut(pl), w - ns);
}
// pieces of sequence s
__host__ __device__ inline int plan_pieces(const ScanPlan& pl, long long s) {
  return (pl.H == 0 ? 0 : 1) + cut_pieces(plan_cut(pl), s);
}
// chunk range [c_lo, c_hi) of piece k of sequence s
__host__ __device__ inline void plan_piece_range(const ScanPlan& pl, long long s, int k, int& c_lo, int& c_hi) {
  if (pl.H == 0) {
    cut_piece_range(plan_cut(pl), s, k, c_lo, c_hi);
  } else if (k == 0) {
    c_lo = 0;
    c_hi = pl.H;
  } else {
    cut_piece_range(plan_cut(pl), s, k - 1, c_lo, c_hi);
    c_lo += pl.H;
    c_hi += pl.H;
  }
}
// The item of a range that starts at unit u (range end u_end): sequence sq,
// its chunks [c_lo, c_hi), piece index k, and the unit after the item.
__host__ __device__ inline void plan_item(const ScanPlan& pl, long long u, long long u_end, long long& sq, int& c_lo,
                                          int& c_hi, int& k, long long& next) {
  const long long heads = pl.H == 0 ? 0 : plan_nseq(pl) * pl.H;
  if (u < heads) {  // a whole head
    sq = u / pl.H;
    next = (sq + 1) * pl.H < u_end ? (sq + 1) * pl.H : u_end;
    c_lo = (int)(u - sq * pl.H);
    c_hi = (int)(next - sq * pl.H);
    k = 0;
    return;
  }
  const PlanCut c = plan_cut(pl);
  const long long v = u - heads, S0 = (v / c.len) * c.len;
  sq = v / c.len;
  next = heads + (S0 + c.len < u_end - heads ? S0 + c.len : u_end - heads);
  c_lo = pl.H + (int)(v - S0);
  c_hi = pl.H + (int)(next - heads - S0);
  k = (pl.H == 0 ? 0 : 1) + (int)(cut_count_le(c, v) - cut_count_le(c, S0));
}

using BwdPlan = ScanPlan;
using FwdPlan = ScanPlan;

// The backward's aggregate pass works on sub-pieces of at most kAggSub
// chunks of the later pieces (k >= 1) of each sequence, so that its longest
// sequential walk is kAggSub chunks.  Sub-piece (k, j) of a sequence has
// slot floor(start chunk / kAggSub) + k (contiguous layout), or
// floor((start chunk - H) / kAggSub) + k - 1 (split layout: only the tails
// are aggregated) -- unique and increasing in time.
constexpr int kAggSub = 8;
__host__ __device__ inline int agg_slot_of(const ScanPlan& pl, int chunk, int k) {
  return pl.H == 0 ? chunk / kAggSub + k : (chunk - pl.H) / kAggSub + k - 1;
}
__host__ __device__ inline int agg_slots(const ScanPlan& pl) {
  return pl.H == 0 ? (pl.nch + kAggSub - 1) / kAggSub + pl.maxp
                   : (pl.nch - pl.H + kAggSub - 1) / kAggSub + pl.maxp - 1;
}
// slots [z0, z1] of piece k of sequence s
__host__ __device__ inline void agg_piece_slots(const ScanPlan& pl, long long s, int k, int& z0, int& z1) {
  int lo, hi;
  plan_piece_range(pl, s, k, lo, hi);
  z0 = agg_slot_of(pl, lo, k);
  z1 = agg_slot_of(pl, hi - 1, k);
}
// the sub-piece in slot z of sequence s: piece k >= 1, chunks [cs, ce); false if none
__host__ __device__ inline bool agg_slot(const ScanPlan& pl, long long s, int z, int& k, int& cs, int& ce) {
  const int K = plan_pieces(pl, s);
  for (int kk = 1; kk < K; ++kk) {
    int z0, z1, lo, hi;
    plan_piece_range(pl, s, kk, lo, hi);
    z0 = agg_slot_of(pl, lo, kk);
    z1 = agg_slot_of(pl, hi - 1, kk);
    if (z >= z0 && z <= z1) {
      k = kk;
      // sub-piece boundaries: multiples of kAggSub from the aggregated region's origin
      const int org = pl.H;
      const int j = z - z0 + (lo - org) / kAggSub;  // sub-block index from the origin
      cs = lo > org + j * kAggSub ? lo : org + j * kAggSub;
      ce = hi < org + (j + 1) * kAggSub ? hi : org + (j + 1) * kAggSub;
      return cs < ce;
    }
  }
  return false;
}

struct FwdParams {
  const void* u;
  const void* delta_raw;
  const void* z;  // nullable
  const void* Bm;
  const void* Cm;
  const float* A_log;
  const float* Dp;
  const float* delta_bias;
  const float* h0;      // nullable
  void* out;
  float* h_last;        // nullable (may alias h0 for the decode step)
  float* chunk_states;  // nullable (nosave)
  unsigned int* status;  // device status word (bounded waits report here)
  float dt_min, dt_max;   // limit on delta = softplus(s); 0 and +inf: none
  // Time segments (long sequences): the steps are split into nseg segments
  // of seg_len steps (a multiple of kChunk), run in parallel.  seg_agg
  // ([B][nseg][D][N][2] f32: decay product and zero-start end state of each
  // segment) is written by the aggregate pass, seg_start ([B][nseg][D][N]
  // f32: state before each segment's first step) by the carry kernel.
  int seg_len, nseg;
  float* seg_agg;
  float* seg_start;
  // Stream mode (plan.handover, cooperative launch of plan.P CTAs): the CTA
  // walking a sequence's first piece stores the state it ends with in
  // seq_carry [nseq][128/TPC][N] and raises seq_flag[sequence]; the CTA
  // walking the last piece waits for it.  nullptr = grid mode.
  FwdPlan plan;
  int* seq_flag;
  float* seq_carry;
  int B, L, D, N, nchunks;
};

struct BwdParams {
  const void* u;
  const void* delta_raw;
  const void* z;  // nullable
  const void* Bm;
  const void* Cm;
  const float* A_log;
  const float* Dp;
  const float* delta_bias;
  const float* chunk_states;
  const void* dout;
  const float* dh_last;  // nullable
  void* du;
  void* d_delta_raw;
  void* dz;    // non-null iff z non-null
  float* dh0;  // nullable
  float* ws_dbc;    // [ndt][B][L][2][N] per-channel-tile sums of the dBm / dCm terms
  int* ws_ndt;      // the number ndt of those tile rows, written by the kernel that fills them
  float* ws_param;  // [B][nseg][D][N+2] per-(batch, segment) sums: A*sum(...), dDp, d_delta_bias
  unsigned int* status;  // device status word (bounded waits report here)
  float dt_min, dt_max;   // limit on delta = softplus(s); 0 and +inf: none
  // Pieces (chunked parallel scan): nseg = plan.maxp rows per batch;
  // seg_agg [B][nslot][D][N][2] holds each aggregate sub-piece's decay
  // product and zero-carry adjoint carry-out (slots: agg_slot), seg_carry
  // [B][nseg][D][N] the adjoint carry entering each piece's last step.  The
  // generic kernel uses row 0 only.
  BwdPlan plan;
  int nseg, nslot;
  float* seg_agg;
  float* seg_carry;
  // Hand-over mode (cooperative launch, every sequence in at most two
  // pieces): instead of aggregates, the CTA holding a sequence's last piece
  // walks it first, writes the carry it ends with to seg_carry row 0 and
  // raises seq_flag[sequence]; the CTA holding the first piece, which it
  // walks last, waits for the flag.  nullptr = aggregate mode.
  int* seq_flag;
  int B, L, D, N, nchunks;
};

// Causal depthwise conv1d + SiLU (s6_conv1d.cu).  For the step, x is x_t
// [B][D], state_last is the state [B][D][K-1] read and updated in place.
struct ConvParams {
  const void* x;
  const float* w;        // [D][K]
  const float* bias;     // [D]
  const void* state0;    // [B][D][K-1] nullable (zeros)
  void* out;
  void* state_last;      // [B][D][K-1] nullable
  const void* dout;
  void* dx;
  float* dw;
  float* dbias;
  float* dstate0;        // nullable
  float* ws;             // backward partial sums
  unsigned int* status;  // device status word (bounded waits report here)
  int B, L, D, K;
};

// ---------------------------------------------------------------- launchers
// Each returns the cudaError_t of its launch(es).

cudaError_t launch_fwd(const FwdParams& p, int act, cudaStream_t stream);
bool fwd_tma_supported(const FwdParams& p, int act);
cudaError_t launch_fwd_tma(const FwdParams& p, int act, cudaStream_t stream);
bool step_supported(const FwdParams& p, int act);
cudaError_t launch_step(const FwdParams& p, int act, cudaStream_t stream);
// Segment count the TMA forward uses for this shape on a GPU with `sms` SMs (1 = none).
int fwd_segments(int B, int L, int D, int N, int sms);
// Device address of the library's status word on the current device (nullptr on error).
unsigned int* device_status_word();
// The calling thread's current CUDA context (driver handle), or nullptr.
void* current_context();
// Device addresses of a __device__ variable, one per device, looked up with
// cudaGetSymbolAddress (the device current) on first use and again whenever
// the device's context has changed since (e.g. after cudaDeviceReset, which
// reloads the module: the variable may then sit at another address).
struct SymbolCache {
  static constexpr int kMaxDevices = 64;
  std::mutex mu;
  void* addr[kMaxDevices] = {nullptr};
  void* ctx[kMaxDevices] = {nullptr};
};
cudaError_t symbol_address(SymbolCache& cache, const void* symbol, void** out);
// SM count of the current device, queried once per device (0 on error).
int device_sm_count();
// Counts a call whose planned cooperative mode (forward stream mode, backward
// hand-over mode) could not be resident on this GPU and ran in its
// non-cooperative form instead (same results, slower); ssm_plan_fallbacks().
void note_plan_fallback();
long long plan_fallbacks();
// Sets the calling thread's ssm_last_error() message; returns `code`.
int report_error(int code, const char* fmt, ...);
cudaError_t launch_bwd(const BwdParams& p, int act, cudaStream_t stream);
bool bwd_tma_supported(const BwdParams& p, int act);
cudaError_t launch_bwd_tma(const BwdParams& p, int act, cudaStream_t stream);
size_t conv1d_bwd_workspace_bytes(int B, int L, int D, int K);
cudaError_t launch_conv1d(const ConvParams& p, int act, bool bwd, cudaStream_t stream);
// SSM_CONV_PATH_* that launch_conv1d would take for these parameters
int conv1d_path(const ConvParams& p, int act, bool bwd);

// Mamba-2 SSD forward (s6_ssd.cu)
struct SsdArgs {
  const void* x;       // [B][L][H][P] act
  const void* dt_raw;  // [B][L][H] act
  const void* Bm;      // [B][L][G][N] act
  const void* Cm;
  const float* dt_bias;  // [H]
  const float* A_log;    // [H]
  const float* Dp;       // [H]
  const float* h0;       // [B][H][N][P] or null
  void* y;               // [B][L][H][P] act
  float* h_last;         // [B][H][N][P] or null
  void* chunk_states;    // [B][H][ceil(L/64)][N][P] bf16 or null (forward: written; backward: read)
  unsigned int* status;
  float dt_min, dt_max;
  int B, L, H, G, N;
  // sub-heads per head: P / 64.  A head of P = 64 m columns is m sub-heads of
  // 64 columns sharing the head's dt, A, D and the group's Bm, Cm (the p
  // columns of the SSD recurrence evolve independently); the kernels walk
  // sub-heads, x / y / dx / dy being [B][L][H m][64] in memory.  P = 32: m = 1
  // and w = 32 (the sub-head's columns in memory; else w = 64)
  int m, w;
};
// Mamba-2 SSD backward (s6_ssd_bwd.cu); the forward's SsdArgs plus these
struct SsdBwdArgs {
  SsdArgs f;             // the forward's inputs; f.chunk_states read, f.y unused
  const void* dy;        // [B][L][H][P] act
  const float* dh_last;  // [B][H][N][P] or null
  void* dx;              // [B][L][H][P] act
  void* ddt_raw;         // [B][L][H] act
  void* dBm;             // [B][L][G][N] act
  void* dCm;
  float* dA_log;         // [H]
  float* ddt_bias;       // [H]
  float* dDp;            // [H]
  float* dh0;            // [B][H][N][P] or null
  float* ws;             // scratch: per-sub-head dBm/dCm terms, per-(batch, sub-head) scalars,
                         // per-sub-head ddt_raw terms (m > 1)
};
// H heads of m sub-heads (headdim 64 m)
size_t ssd_bwd_workspace_bytes(int B, int L, int H, int m, int G, int N);
cudaError_t launch_ssd_bwd(const SsdBwdArgs& a, cudaStream_t stream);
bool ssd_supported(int act, int P, int N);
cudaError_t launch_ssd_fwd(const SsdArgs& a, cudaStream_t stream);
// the tensor map of an x-shaped [B][L][H][P] bf16 tensor (x, dy) for the SSD
// kernels' [64 steps][64 columns] boxes of one sub-head: 3D over
// [B][L][H m * 64] when w = 64; 4D over [B][L][H][32] when w = 32, the box's
// columns 32..63 past the tensor's inner extent (filled with zeros)
bool ssd_encode_x_map(void* map, const void* base, const SsdArgs& a);
cudaError_t launch_conv1d_step(const ConvParams& p, int act, cudaStream_t stream);
// The TMA backward's work plan for this shape with `sms` worker CTAs.
BwdPlan bwd_plan(int B, int L, int D, int N, int sms);
// The TMA forward's stream plan (three CTAs on each of `sms` SMs); handover
// is false when the grid mode is kept.
FwdPlan fwd_stream_plan(int B, int L, int D, int N, int act, int sms);
// ndt: the device int the partials kernel wrote (how many tile rows ws_dbc holds)
cudaError_t launch_reduce_dbc(const float* ws_dbc, const int* ndt, int B, int L, int N, void* dBm,
                              void* dCm, int act, cudaStream_t stream);
cudaError_t launch_reduce_params(const float* ws_param, int B, int D, int N, float* dA_log,
                                 float* dDp, float* d_delta_bias, cudaStream_t stream);
// (B here is the number of partial rows: batches x segments.)

// ---------------------------------------------------------------- device helpers

template <typename T>
__device__ __forceinline__ float ld_act(const T* p);
template <>
__device__ __forceinline__ float ld_act<float>(const float* p) {
  return __ldg(p);
}
template <>
__device__ __forceinline__ float ld_act<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(__ldg(p));
}

template <typename T>
__device__ __forceinline__ void st_act(T* p, float v);
template <>
__device__ __forceinline__ void st_act<float>(float* p, float v) {
  *p = v;
}
template <>
__device__ __forceinline__ void st_act<__nv_bfloat16>(__nv_bfloat16* p, float v) {
  *p = __float2bfloat16_rn(v);
}

// softplus(s) = log(1 + e^s); above 20 it equals s to within 2e-9 relative
// (the threshold the POPCORNBENCH kernel's softplus uses).
__device__ __forceinline__ float softplus_f(float s) { return s > 20.f ? s : log1pf(expf(s)); }

// delta limited to [lo, hi] (the dt_limit clamp; lo = 0, hi = +inf leaves
// every softplus value as it is)
__device__ __forceinline__ float clamp_dt(float sp, float lo, float hi) { return fminf(fmaxf(sp, lo), hi); }

__device__ __forceinline__ float sigmoid_f(float x) { return 1.f / (1.f + expf(-x)); }

}  // namespace s6
