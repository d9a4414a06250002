// Causal depthwise conv1d + SiLU (the convolution in front of the selective
// scan in a Mamba block; mamba-rs kernels.rs page: "Multi-step conv1d forward
// with state saves", "Multi-step conv1d backward", "Single-step depthwise
// conv1d forward with SiLU"; deterministic_backward.py page: ordered weight
// and bias sums).  With K taps per channel and the K-1 inputs before t = 0
// taken from state0 (zeros if absent):
//   pre[b,t,d] = bias[d] + sum_k w[d][k] * x[b, t-(K-1)+k, d],  out = pre * sigmoid(pre)
//
// All three kernels are bound by HBM.  A thread owns V consecutive channels
// (V = 4, one vector access, where the layout allows it, else V = 1) and
// walks a run of consecutive time steps, keeping the last K
// input rows (and in the backward the last K pre-activation gradients) in
// registers, so every row is read once per run; neighbouring threads read
// neighbouring vectors of the same row (coalesced).
//
// Backward: a run of kRun steps computes dpre for its steps and the K-1 after
// it, dx for its steps, and its partial sums of dw and dbias (fixed order),
// which a second kernel adds over (batch, run) in ascending order: no float
// atomics, bit-identical results from run to run.
#include <algorithm>
#include <type_traits>

#include "s6_internal.cuh"
#include "s6_tma.cuh"

namespace s6 {

namespace {

constexpr int kConvThreads = 256;
constexpr int kRun = 64;  // backward: time steps per thread

template <typename Act, int V>
struct Vec;  // V consecutive activations, loaded / stored as one access
template <>
struct Vec<float, 1> {
  static __device__ __forceinline__ void load(const float* p, float* v) { v[0] = __ldg(p); }
  static __device__ __forceinline__ void store(float* p, const float* v) { *p = v[0]; }
};
template <>
struct Vec<float, 4> {
  static __device__ __forceinline__ void load(const float* p, float* v) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p));
    v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w;
  }
  static __device__ __forceinline__ void store(float* p, const float* v) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
};
template <>
struct Vec<__nv_bfloat16, 1> {
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, float* v) { v[0] = __bfloat162float(p[0]); }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, const float* v) { p[0] = __float2bfloat16_rn(v[0]); }
};
template <>
struct Vec<__nv_bfloat16, 4> {
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, float* v) {
    const uint2 a = __ldg(reinterpret_cast<const uint2*>(p));
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&a);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      v[2 * i] = f.x, v[2 * i + 1] = f.y;
    }
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, const float* v) {
    uint2 a;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&a);
#pragma unroll
    for (int i = 0; i < 2; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    *reinterpret_cast<uint2*>(p) = a;
  }
};
// sigmoid: on the SFU (ex2, rcp approximations) for bf16 activations, whose
// rounding dwarfs their error; expf and an IEEE division for f32
template <typename Act>
__device__ __forceinline__ float sig(float v) {
  if constexpr (std::is_same<Act, __nv_bfloat16>::value)
    return rcp_approx(1.f + ex2_approx(-v * 1.4426950408889634f));
  else
    return sigmoid_f(v);
}

// x row t (t >= 0) or, for t < 0, the state entries of the same V channels
template <typename Act, int V>
__device__ __forceinline__ void load_in(const Act* x, const Act* state0, int L, int D, int K, int b, int t,
                                        int d, float* v) {
  if (t >= 0) {
    Vec<Act, V>::load(x + ((size_t)b * L + t) * D + d, v);
  } else {
#pragma unroll
    for (int i = 0; i < V; ++i)
      v[i] = state0 ? ld_act(state0 + ((size_t)b * D + d + i) * (K - 1) + (K - 1 + t)) : 0.f;
  }
}

// Forward: a thread walks kRun steps of V channels.
template <typename Act, int V, int K>
__global__ void __launch_bounds__(kConvThreads) s6_conv1d_fwd_kernel(const Act* __restrict__ x,
                                                                     const float* __restrict__ w,
                                                                     const float* __restrict__ bias,
                                                                     const Act* __restrict__ state0,
                                                                     Act* __restrict__ out, int B, int L, int D) {
  const int nvec = D / V;
  const int nrun = (L + kRun - 1) / kRun;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)B * nrun * nvec) return;
  const int dv = (int)(idx % nvec);
  const int run = (int)((idx / nvec) % nrun);
  const int b = (int)(idx / ((long long)nvec * nrun));
  const int d = dv * V;
  float wk[K][V], bs[V];
#pragma unroll
  for (int i = 0; i < V; ++i) {
    bs[i] = bias[d + i];
#pragma unroll
    for (int k = 0; k < K; ++k) wk[k][i] = w[(size_t)(d + i) * K + k];
  }
  const int t0 = run * kRun, t1 = min(L, t0 + kRun);
  float win[K][V];  // win[k] = input t - (K-1) + k
#pragma unroll
  for (int k = 0; k < K - 1; ++k) load_in<Act, V>(x, state0, L, D, K, b, t0 - (K - 1) + k, d, win[k]);
#pragma unroll 4
  for (int t = t0; t < t1; ++t) {
    Vec<Act, V>::load(x + ((size_t)b * L + t) * D + d, win[K - 1]);
    float o[V];
#pragma unroll
    for (int i = 0; i < V; ++i) {
      float pre = bs[i];
#pragma unroll
      for (int k = 0; k < K; ++k) pre += wk[k][i] * win[k][i];
      o[i] = pre * sig<Act>(pre);
    }
    Vec<Act, V>::store(out + ((size_t)b * L + t) * D + d, o);
#pragma unroll
    for (int k = 0; k < K - 1; ++k)
#pragma unroll
      for (int i = 0; i < V; ++i) win[k][i] = win[k + 1][i];
  }
}

// state_last[b][d][j] = input L-(K-1)+j (from x, or from state0 when L < K-1)
template <typename Act>
__global__ void s6_conv1d_state_kernel(const Act* x, const Act* state0, Act* state_last, int B, int L, int D,
                                       int K) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long total = (long long)B * D * (K - 1);
  if (idx >= total) return;
  const int j = (int)(idx % (K - 1));
  const int d = (int)((idx / (K - 1)) % D);
  const int b = (int)(idx / ((long long)(K - 1) * D));
  const int t = L - (K - 1) + j;
  float v;
  load_in<Act, 1>(x, state0, L, D, K, b, t, d, &v);
  st_act(state_last + idx, v);
}

// Backward: a thread walks kRun steps of V channels from the last to the
// first.  xw[k] = input t-(K-1)+k (one new row per step) and gw[k] =
// dpre[t+k] slide down with t; dx[t] = sum_k w[k] * dpre[t+(K-1)-k]; the dw
// and dbias terms of its own steps are summed in step order (last first).
template <typename Act, int V, int K>
__global__ void __launch_bounds__(kConvThreads) s6_conv1d_bwd_kernel(
    const Act* __restrict__ x, const float* __restrict__ w, const float* __restrict__ bias,
    const Act* __restrict__ state0, const Act* __restrict__ dout, Act* __restrict__ dx,
    float* __restrict__ dstate0, float* __restrict__ part, int B, int L, int D) {
  const int nvec = D / V;
  const int nrun = (L + kRun - 1) / kRun;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)B * nrun * nvec) return;
  const int dv = (int)(idx % nvec);
  const int run = (int)((idx / nvec) % nrun);
  const int b = (int)(idx / ((long long)nvec * nrun));
  const int d = dv * V;
  float wk[K][V], bs[V];
#pragma unroll
  for (int i = 0; i < V; ++i) {
    bs[i] = bias[d + i];
#pragma unroll
    for (int k = 0; k < K; ++k) wk[k][i] = w[(size_t)(d + i) * K + k];
  }
  const int t0 = run * kRun, t1 = min(L, t0 + kRun);
  // dpre of step t from its inputs in[k] = input t-(K-1)+k (0 for t >= L)
  auto dpre_from = [&](int t, float (&in)[K][V], float* g) {
    if (t >= L) {
#pragma unroll
      for (int i = 0; i < V; ++i) g[i] = 0.f;
      return;
    }
    float go[V];
    Vec<Act, V>::load(dout + ((size_t)b * L + t) * D + d, go);
#pragma unroll
    for (int i = 0; i < V; ++i) {
      float pre = bs[i];
#pragma unroll
      for (int k = 0; k < K; ++k) pre += wk[k][i] * in[k][i];
      const float s = sig<Act>(pre);
      g[i] = go[i] * s * fmaf(pre, 1.f - s, 1.f);
    }
  };
  auto dpre_at = [&](int t, float* g) {
    float in[K][V];
    if (t < L) {
#pragma unroll
      for (int k = 0; k < K; ++k) load_in<Act, V>(x, state0, L, D, K, b, t - (K - 1) + k, d, in[k]);
    }
    dpre_from(t, in, g);
  };
  float gw[K][V];  // gw[k] = dpre[t + k]
#pragma unroll
  for (int k = 1; k < K; ++k) dpre_at(t1 - 1 + k, gw[k]);
  float xw[K][V];  // xw[k] = input t - (K-1) + k
#pragma unroll
  for (int k = 1; k < K; ++k) load_in<Act, V>(x, state0, L, D, K, b, t1 - 1 - (K - 1) + k, d, xw[k]);
  float aw[K][V], ab[V];  // this run's sums of the dw[k] and dbias terms
#pragma unroll
  for (int i = 0; i < V; ++i) {
    ab[i] = 0.f;
#pragma unroll
    for (int k = 0; k < K; ++k) aw[k][i] = 0.f;
  }
#pragma unroll 4
  for (int t = t1 - 1; t >= t0; --t) {
    load_in<Act, V>(x, state0, L, D, K, b, t - (K - 1), d, xw[0]);
    dpre_from(t, xw, gw[0]);
    float o[V];
#pragma unroll
    for (int i = 0; i < V; ++i) {
      float acc = 0.f;
#pragma unroll
      for (int k = 0; k < K; ++k) acc += wk[k][i] * gw[K - 1 - k][i];
      o[i] = acc;
      ab[i] += gw[0][i];
#pragma unroll
      for (int k = 0; k < K; ++k) aw[k][i] += gw[0][i] * xw[k][i];
    }
    Vec<Act, V>::store(dx + ((size_t)b * L + t) * D + d, o);
    // slide down one step
#pragma unroll
    for (int k = K - 1; k > 0; --k)
#pragma unroll
      for (int i = 0; i < V; ++i) {
        gw[k][i] = gw[k - 1][i];
        xw[k][i] = xw[k - 1][i];
      }
  }
  // the first run also owns the state's gradient: dstate0[j] = sum_{k<=j} w[k] * dpre[j - k]
  if (run == 0 && dstate0 && K > 1) {
    float g0[K][V];  // dpre[0 .. K-2] (0 past L)
#pragma unroll
    for (int m = 0; m < K - 1; ++m) dpre_at(m, g0[m]);
#pragma unroll
    for (int j = 0; j < K - 1; ++j)
#pragma unroll
      for (int i = 0; i < V; ++i) {
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k <= j; ++k) acc += wk[k][i] * g0[j - k][i];
        dstate0[((size_t)b * D + d + i) * (K - 1) + j] = acc;
      }
  }
  // partials [b][run][d][K+1]: dw terms k = 0..K-1, then dbias
  float* pp = part + (((size_t)b * nrun + run) * D + d) * (K + 1);
#pragma unroll
  for (int i = 0; i < V; ++i) {
#pragma unroll
    for (int k = 0; k < K; ++k) pp[i * (K + 1) + k] = aw[k][i];
    pp[i * (K + 1) + K] = ab[i];
  }
}

// dw[d][k], dbias[d] = sum over (b, run), ascending, of the partials
__global__ void s6_conv1d_reduce_kernel(const float* part, int R, int D, int K, float* dw, float* dbias) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;  // (d, k) with k = K meaning the bias
  if (e >= D * (K + 1)) return;
  const int d = e / (K + 1), k = e % (K + 1);
  float s = 0.f;
  for (int r = 0; r < R; ++r) s += part[((size_t)r * D + d) * (K + 1) + k];
  if (k < K)
    dw[(size_t)d * K + k] = s;
  else
    dbias[d] = s;
}

// One step: state [B][D][K-1] (oldest first) and x_t give out_t; the state
// shifts by one and takes x_t.
template <typename Act, int K>
__global__ void s6_conv1d_step_kernel(const Act* x, const float* w, const float* bias, Act* state, Act* out,
                                      int B, int D) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)B * D) return;
  const int d = (int)(idx % D);
  Act* st = state + idx * (K - 1);
  const float xv = ld_act(x + idx);
  float in[K];
#pragma unroll
  for (int k = 0; k < K - 1; ++k) in[k] = ld_act(st + k);
  in[K - 1] = xv;
  float pre = bias[d];
#pragma unroll
  for (int k = 0; k < K; ++k) pre += w[(size_t)d * K + k] * in[k];
  st_act(out + idx, pre * sig<Act>(pre));
#pragma unroll
  for (int k = 0; k < K - 1; ++k) st_act(st + k, in[k + 1]);
}

template <typename Act, int V, int K>
cudaError_t fwd_vk(const ConvParams& p, cudaStream_t stream) {
  const int nrun = (p.L + kRun - 1) / kRun;
  const long long threads = (long long)p.B * nrun * (p.D / V);
  if (threads > 0)
    s6_conv1d_fwd_kernel<Act, V, K><<<(unsigned)((threads + kConvThreads - 1) / kConvThreads), kConvThreads, 0,
                                       stream>>>(static_cast<const Act*>(p.x), p.w, p.bias,
                                                 static_cast<const Act*>(p.state0), static_cast<Act*>(p.out),
                                                 p.B, p.L, p.D);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || !p.state_last || K == 1) return e;
  const long long n = (long long)p.B * p.D * (K - 1);
  s6_conv1d_state_kernel<Act><<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(
      static_cast<const Act*>(p.x), static_cast<const Act*>(p.state0), static_cast<Act*>(p.state_last), p.B, p.L,
      p.D, K);
  return cudaGetLastError();
}

template <typename Act, int V, int K>
cudaError_t bwd_vk(const ConvParams& p, cudaStream_t stream) {
  const int nrun = (p.L + kRun - 1) / kRun;
  const long long threads = (long long)p.B * nrun * (p.D / V);
  if (threads > 0)
    s6_conv1d_bwd_kernel<Act, V, K><<<(unsigned)((threads + kConvThreads - 1) / kConvThreads), kConvThreads, 0,
                                       stream>>>(
        static_cast<const Act*>(p.x), p.w, p.bias, static_cast<const Act*>(p.state0),
        static_cast<const Act*>(p.dout), static_cast<Act*>(p.dx), p.dstate0, p.ws, p.B, p.L, p.D);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int n = p.D * (K + 1);
  s6_conv1d_reduce_kernel<<<(n + 255) / 256, 256, 0, stream>>>(p.ws, p.B * nrun, p.D, K, p.dw, p.dbias);
  return cudaGetLastError();
}

template <typename Act, int V>
cudaError_t dispatch_k(const ConvParams& p, bool bwd, cudaStream_t stream) {
  switch (p.K) {
#define S6_CONV_K(KK) \
  case KK:            \
    return bwd ? bwd_vk<Act, V, KK>(p, stream) : fwd_vk<Act, V, KK>(p, stream);
    S6_CONV_K(1)
    S6_CONV_K(2)
    S6_CONV_K(3)
    S6_CONV_K(4)
    S6_CONV_K(5)
    S6_CONV_K(6)
    S6_CONV_K(7)
    S6_CONV_K(8)
#undef S6_CONV_K
    default:
      return cudaErrorInvalidValue;
  }
}

// Vector path: 4 channels per thread (16 bytes of f32, 8 of bf16; four keep
// the backward's windows in registers at full occupancy).
bool vec_ok(const ConvParams& p, int act) {
  constexpr int V = 4;
  const uintptr_t mask = act == SSM_BF16 ? 7 : 15;
  if (p.D % V != 0) return false;
  const void* ptrs[] = {p.x, p.out, p.dout, p.dx};
  for (const void* q : ptrs)
    if (q && (reinterpret_cast<uintptr_t>(q) & mask)) return false;
  return true;
}

template <typename Act, int K>
cudaError_t step_k(const ConvParams& p, cudaStream_t stream) {
  const long long n = (long long)p.B * p.D;
  if (n > 0)
    s6_conv1d_step_kernel<Act, K><<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(
        static_cast<const Act*>(p.x), p.w, p.bias, static_cast<Act*>(p.state_last), static_cast<Act*>(p.out), p.B,
        p.D);
  return cudaGetLastError();
}

template <typename Act>
cudaError_t step_dispatch(const ConvParams& p, cudaStream_t stream) {
  switch (p.K) {
#define S6_CONV_K(KK) \
  case KK:            \
    return step_k<Act, KK>(p, stream);
    S6_CONV_K(1)
    S6_CONV_K(2)
    S6_CONV_K(3)
    S6_CONV_K(4)
    S6_CONV_K(5)
    S6_CONV_K(6)
    S6_CONV_K(7)
    S6_CONV_K(8)
#undef S6_CONV_K
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace

size_t conv1d_bwd_workspace_bytes(int B, int L, int D, int K) {
  const size_t nrun = (size_t)(L + kRun - 1) / kRun;
  return (size_t)B * nrun * D * (K + 1) * sizeof(float);
}

cudaError_t launch_conv1d(const ConvParams& p, int act, bool bwd, cudaStream_t stream) {
  const bool vec = vec_ok(p, act);
  if (act == SSM_BF16)
    return vec ? dispatch_k<__nv_bfloat16, 4>(p, bwd, stream) : dispatch_k<__nv_bfloat16, 1>(p, bwd, stream);
  return vec ? dispatch_k<float, 4>(p, bwd, stream) : dispatch_k<float, 1>(p, bwd, stream);
}

cudaError_t launch_conv1d_step(const ConvParams& p, int act, cudaStream_t stream) {
  return act == SSM_BF16 ? step_dispatch<__nv_bfloat16>(p, stream) : step_dispatch<float>(p, stream);
}

}  // namespace s6
