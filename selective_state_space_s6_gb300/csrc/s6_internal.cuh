// Internal declarations shared by the S6 kernels and the C-ABI host code.
// Not part of the public interface (that is include/ssm_scan.h).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ssm_scan.h"

namespace s6 {

constexpr int kChunk = SSM_CHUNK_LEN;  // steps between saved chunk states
constexpr int kDTile = 64;             // channels per CTA in the scan kernels
constexpr int kThreadsPerChannel = 2;  // each channel's N states are split over 2 lanes
constexpr int kScanThreads = kDTile * kThreadsPerChannel;
constexpr int kSub = 8;                // backward: steps kept in registers per sub-chunk
constexpr unsigned int kStatusWaitTimeoutBit = 1u;  // same bit as kStatusWaitTimeout
constexpr unsigned int kStatusLayoutBit = 2u;       // same bit as kStatusLayout

// ---------------------------------------------------------------- params

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
  // Time segments (long sequences): the steps are split into nseg segments
  // of seg_len steps (a multiple of kChunk), run in parallel.  seg_agg
  // ([B][nseg][D][N][2] f32: decay product and zero-start end state of each
  // segment) is written by the aggregate pass, seg_start ([B][nseg][D][N]
  // f32: state before each segment's first step) by the carry kernel.
  int seg_len, nseg;
  float* seg_agg;
  float* seg_start;
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
  float* ws_dbc;    // [ndt][B][L][2][N] per-CTA sums of the dBm / dCm terms
  float* ws_param;  // [B][nseg][D][N+2] per-(batch, segment) sums: A*sum(...), dDp, d_delta_bias
  unsigned int* status;  // device status word (bounded waits report here)
  // Time segments (chunked parallel scan, as in FwdParams): seg_len steps
  // (a multiple of kChunk) each; seg_agg [B][nseg][D][N][2] holds each
  // segment's decay product and zero-carry adjoint carry-out, seg_carry
  // [B][nseg][D][N] the adjoint carry entering each segment's last step.
  int seg_len, nseg;
  float* seg_agg;
  float* seg_carry;
  int B, L, D, N, nchunks;
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
// Sets the calling thread's ssm_last_error() message; returns `code`.
int report_error(int code, const char* fmt, ...);
cudaError_t launch_bwd(const BwdParams& p, int act, cudaStream_t stream);
bool bwd_tma_supported(const BwdParams& p, int act);
cudaError_t launch_bwd_tma(const BwdParams& p, int act, cudaStream_t stream);
// Segment count the TMA backward uses for this shape on a GPU with `sms` SMs (1 = none).
int bwd_segments(int B, int L, int D, int N, int sms);
cudaError_t launch_reduce_dbc(const float* ws_dbc, int ndt, int B, int L, int N, void* dBm,
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

__device__ __forceinline__ float sigmoid_f(float x) { return 1.f / (1.f + expf(-x)); }

}  // namespace s6
