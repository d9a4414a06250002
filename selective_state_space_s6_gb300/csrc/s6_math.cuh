// Device math shared by the scan, step and conv1d kernels: the activation
// loads from shared memory, softplus and its derivative, SiLU and the decay
// of a pair of states.  "fast" variants run on the special-function unit
// (ex2 / lg2 / rcp approximations; the bf16 paths, whose rounding dwarfs
// their error); the others use expf / log1pf and IEEE division.
#pragma once

#include <cuda_bf16.h>

#include "s6_internal.cuh"
#include "s6_tma.cuh"

namespace s6 {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <typename Act>
__device__ __forceinline__ float lds_act(const Act* p);
template <>
__device__ __forceinline__ float lds_act<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float lds_act<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}

// softplus(s) = max(s, 0) + log1p(e^-|s|) on the special-function unit; the
// series e - e^2/2 + e^3/3 covers e < 2^-6, where log2(1 + e) loses relative
// precision.
__device__ __forceinline__ float softplus_fast(float s) {
  const float e = ex2_approx(-fabsf(s) * kLog2e);
  const float lg = lg2_approx(1.f + e) * kLn2;
  const float ser = e * fmaf(e, fmaf(e, 1.f / 3.f, -0.5f), 1.f);
  return fmaxf(s, 0.f) + (e < 0.015625f ? ser : lg);
}

// sigmoid(s) written through delta = softplus(s): sigmoid(s) = 1 - e^{-delta}
// (the identity the oarust Slang page uses for its dt gradient), with a
// series for small delta where 1 - e^{-delta} would cancel.
__device__ __forceinline__ float dsoftplus_fast(float delta) {
  const float em = ex2_approx(-delta * kLog2e);
  const float ser = delta * fmaf(delta, fmaf(delta, 1.f / 6.f, -0.5f), 1.f);
  return delta < 0.03125f ? ser : 1.f - em;
}

__device__ __forceinline__ float sigmoid_fast(float z) { return rcp_approx(1.f + ex2_approx(-z * kLog2e)); }

__device__ __forceinline__ float silu_fast(float z) { return z * sigmoid_fast(z); }

template <bool kFast>
__device__ __forceinline__ float softplus_k(float s) {
  return kFast ? softplus_fast(s) : softplus_f(s);
}
template <bool kFast>
__device__ __forceinline__ float silu_k(float z) {
  return kFast ? silu_fast(z) : z * sigmoid_f(z);
}

// Abar for a pair of states: fast path 2^(delta * A*log2e) on the SFU,
// accurate path expf(delta * A).
template <bool kFast>
__device__ __forceinline__ float2 decay2(float2 dd, float2 A) {
  const float2 x = fmul2(dd, A);
  if (kFast) return make_float2(ex2_approx(x.x), ex2_approx(x.y));
  return make_float2(expf(x.x), expf(x.y));
}

}  // namespace s6
