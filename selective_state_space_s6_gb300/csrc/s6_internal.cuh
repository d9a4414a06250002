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
// of nch chunks, are laid end to end as U = nseq * nch chunk units
// (sequence s = b * ndt + j) and cut into P equal ranges, one per persistent
// CTA (range w = [bound(w), bound(w + 1)), bound(w) = floor(w * U / P)).  A
// range covers pieces of one or more sequences; a sequence cut by range
// boundaries has K > 1 pieces, numbered in time order.  The plan is a
// function of the shape only.
//   Backward (128-channel tiles, unit s * nch + c): piece k > 0 needs the
//   adjoint carry of the pieces after it -- handed over between CTAs, or
//   composed from piece aggregates (the chunked parallel scan); piece k of
//   sequence (b, j) owns row b * maxp + k of the parameter partials.
//   Forward (128/TPC-channel tiles, unit s * nch + (nch - 1 - c)): a range
//   starts with a sequence's first piece and ends with another's last, whose
//   start state the CTA holding the first piece hands over.
struct ScanPlan {
  long long U;  // chunk units
  int P;        // worker CTAs (ranges), 1 <= P <= U
  int nch;      // chunks per sequence
  int ndt;      // 64-channel tiles
  int maxp;     // most pieces any sequence has
  // carries handed from CTA to CTA (no aggregate pass): every sequence in at
  // most two pieces and no range shorter than a sequence
  bool handover;
};

__host__ __device__ inline long long plan_bound(const ScanPlan& pl, long long w) { return w * pl.U / pl.P; }
// number of w in [0, P] with plan_bound(w) <= X, for 0 <= X < U
__host__ __device__ inline long long plan_count_le(const ScanPlan& pl, long long X) {
  return ((X + 1) * pl.P + pl.U - 1) / pl.U;
}
// pieces of sequence s
__host__ __device__ inline int plan_pieces(const ScanPlan& pl, long long s) {
  const long long S0 = s * pl.nch, S1 = S0 + pl.nch;
  return (int)(plan_count_le(pl, S1 - 1) - plan_count_le(pl, S0)) + 1;
}
// chunk range [c_lo, c_hi) of piece k of sequence s
__host__ __device__ inline void plan_piece_range(const ScanPlan& pl, long long s, int k, int& c_lo, int& c_hi) {
  const long long S0 = s * pl.nch;
  const long long wa = plan_count_le(pl, S0);  // first range boundary after the sequence start
  const int K = plan_pieces(pl, s);
  c_lo = k == 0 ? 0 : (int)(plan_bound(pl, wa + k - 1) - S0);
  c_hi = k == K - 1 ? pl.nch : (int)(plan_bound(pl, wa + k) - S0);
}

using BwdPlan = ScanPlan;
using FwdPlan = ScanPlan;

// The backward's aggregate pass works on sub-pieces of at most kAggSub
// chunks of the later pieces (k >= 1) of each sequence, so that its longest
// sequential walk is kAggSub chunks; sub-piece (k, j) of a sequence has slot
// floor(start chunk / kAggSub) + k, unique and increasing in time.
constexpr int kAggSub = 8;
__host__ __device__ inline int agg_slots(const ScanPlan& pl) { return (pl.nch + kAggSub - 1) / kAggSub + pl.maxp; }
// slots [z0, z1] of piece k of sequence s
__host__ __device__ inline void agg_piece_slots(const ScanPlan& pl, long long s, int k, int& z0, int& z1) {
  int lo, hi;
  plan_piece_range(pl, s, k, lo, hi);
  z0 = lo / kAggSub + k;
  z1 = (hi - 1) / kAggSub + k;
}
// the sub-piece in slot z of sequence s: piece k >= 1, chunks [cs, ce); false if none
__host__ __device__ inline bool agg_slot(const ScanPlan& pl, long long s, int z, int& k, int& cs, int& ce) {
  const int K = plan_pieces(pl, s);
  for (int kk = 1; kk < K; ++kk) {
    int lo, hi;
    plan_piece_range(pl, s, kk, lo, hi);
    const int z0 = lo / kAggSub + kk, z1 = (hi - 1) / kAggSub + kk;
    if (z >= z0 && z <= z1) {
      k = kk;
      cs = lo > (z - kk) * kAggSub ? lo : (z - kk) * kAggSub;
      ce = hi < (z - kk + 1) * kAggSub ? hi : (z - kk + 1) * kAggSub;
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
  float* ws;             // scratch: per-head dBm/dCm terms, per-(batch, head) scalars
};
size_t ssd_bwd_workspace_bytes(int B, int L, int H, int G, int N);
cudaError_t launch_ssd_bwd(const SsdBwdArgs& a, cudaStream_t stream);
bool ssd_supported(int act, int P, int N);
cudaError_t launch_ssd_fwd(const SsdArgs& a, cudaStream_t stream);
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
