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
#include "s6_math.cuh"
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
  static __device__ __forceinline__ void lds(const float* p, float* v) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w;
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
  static __device__ __forceinline__ void lds(const __nv_bfloat16* p, float* v) {
    const uint2 a = *reinterpret_cast<const uint2*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&a);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      v[2 * i] = f.x, v[2 * i + 1] = f.y;
    }
  }
};
// sigmoid: on the SFU (ex2, rcp approximations) for bf16 activations, whose
// rounding dwarfs their error; expf and an IEEE division for f32
template <typename Act>
__device__ __forceinline__ float sig(float v) {
  if constexpr (std::is_same<Act, __nv_bfloat16>::value)
    return sigmoid_fast(v);
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

// ---------------------------------------------------------------- TMA tiles
// A CTA of kTileWarps warps owns kTileT steps x kTileCh channels of one batch
// row.  One TMA load per tensor brings the tile's inputs into shared memory
// (forward: x for its steps and the K-1 before; backward: x for its steps
// and the K-1 on either side, dout for its steps and the K-1 after), so a
// CTA has its whole tile in flight whatever its register count, and the
// copy engine rather than the threads carries the halo rows.  Warp w then
// walks steps w*16 .. w*16+15 of the tile from shared memory, lane l on
// channels 4l .. 4l+3 (one 8- or 16-byte access per row: conflict-free).
// Rows outside [0, L) and channels past D arrive as zeros (the bounds of the
// 3D tensor map [B][L][D]): that is the causal padding when there is no
// state0, and it makes dpre = 0 for steps past the end; with state0 the
// inputs before t = 0 are read from it.
constexpr int kTileT = kRun;                   // steps per CTA (one partial-sum row)
constexpr int kTileWarps = 4;
constexpr int kTileSeg = kTileT / kTileWarps;  // steps per warp
constexpr int kTileCh = 128;                   // channels per CTA: 32 lanes x 4
static_assert(kTileSeg >= SSM_MAX_CONV_WIDTH - 1, "a warp's segment must hold the state gradient's steps");

struct ConvTileParams {
  CUtensorMap map_x, map_dout;
  ConvParams p;
};

template <typename Act>
constexpr size_t tile_rows_bytes(int rows) {
  return ((size_t)rows * kTileCh * sizeof(Act) + 127) / 128 * 128;
}

template <typename Act, int K>
constexpr size_t fwd_tile_smem() {
  return tile_rows_bytes<Act>(kTileT + K - 1) + 16;
}

template <typename Act, int K>
constexpr size_t bwd_tile_smem() {
  return tile_rows_bytes<Act>(kTileT + 2 * (K - 1)) + tile_rows_bytes<Act>(kTileT + K - 1) +
         (size_t)kTileWarps * kTileCh * (K + 1) * 4 + 16;
}

// weights and bias of channels d .. d+3 (zeros past D)
template <int K>
__device__ __forceinline__ void load_weights(const ConvParams& p, int d, bool cv, float (&wk)[K][4], float (&bs)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    bs[i] = cv ? __ldg(p.bias + d + i) : 0.f;
#pragma unroll
    for (int k = 0; k < K; ++k) wk[k][i] = cv ? __ldg(p.w + (size_t)(d + i) * K + k) : 0.f;
  }
}

// thread 0 sets up the barrier; all threads see it before anyone waits
__device__ __forceinline__ void tile_barrier_init(uint64_t* bar) {
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
}

template <typename Act, int K>
__global__ void __launch_bounds__(kTileWarps * 32) s6_conv1d_fwd_tile_kernel(const __grid_constant__ ConvTileParams P) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int kRows = kTileT + K - 1;  // smem row r holds input t0 - (K-1) + r
  const ConvParams& p = P.p;
  Act* xs = reinterpret_cast<Act*>(smem);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + tile_rows_bytes<Act>(kRows));
  const int c0 = blockIdx.x * kTileCh, t0 = blockIdx.y * kTileT, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  tile_barrier_init(bar);
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(bar, (uint32_t)(kRows * kTileCh * sizeof(Act)));
    tma_load_3d(xs, &P.map_x, bar, c0, t0 - (K - 1), b);
  }
  const int d = c0 + 4 * lane;
  const bool cv = d < p.D;
  float wk[K][4], bs[4];
  load_weights<K>(p, d, cv, wk, bs);
  const Act* __restrict__ s0 = static_cast<const Act*>(p.state0);
  const int ts = t0 + warp * kTileSeg;
  float win[K][4];  // win[k] = input t - (K-1) + k
  // the window's first K-1 inputs: from state0 before t = 0, if given (then
  // ts = 0 and input ts-(K-1)+k is state entry k), else from the tile
#pragma unroll
  for (int k = 0; k < K - 1; ++k)
    if (s0 && ts - (K - 1) + k < 0) {
#pragma unroll
      for (int i = 0; i < 4; ++i) win[k][i] = cv ? ld_act(s0 + ((size_t)b * p.D + d + i) * (K - 1) + k) : 0.f;
    }
  if (!mbar_wait(bar, 0, p.status)) return;
  if (ts >= p.L) return;
#pragma unroll
  for (int k = 0; k < K - 1; ++k)
    if (!(s0 && ts - (K - 1) + k < 0)) Vec<Act, 4>::lds(xs + (warp * kTileSeg + k) * kTileCh + 4 * lane, win[k]);
  Act* __restrict__ out = static_cast<Act*>(p.out) + ((size_t)b * p.L + ts) * p.D + d;
  const int nt = min(kTileSeg, p.L - ts);  // steps of this segment inside [0, L)
#pragma unroll 4
  for (int i = 0; i < kTileSeg; ++i) {
    Vec<Act, 4>::lds(xs + (warp * kTileSeg + i + K - 1) * kTileCh + 4 * lane, win[K - 1]);
    float o[4];
    if constexpr (std::is_same<Act, __nv_bfloat16>::value) {
      // two channels per packed op; per channel the same operations in the
      // same order as the scalar form (the other paths and the step), so the
      // results are the same bit for bit
#pragma unroll
      for (int jp = 0; jp < 2; ++jp) {
        float2 pre = make_float2(bs[2 * jp], bs[2 * jp + 1]);
#pragma unroll
        for (int k = 0; k < K; ++k)
          pre = ffma2(make_float2(wk[k][2 * jp], wk[k][2 * jp + 1]), make_float2(win[k][2 * jp], win[k][2 * jp + 1]), pre);
        const float2 x = fmul2(pre, make_float2(-kLog2e, -kLog2e));
        const float2 den = fadd2(make_float2(1.f, 1.f), make_float2(ex2_approx(x.x), ex2_approx(x.y)));
        const float2 r = fmul2(pre, make_float2(rcp_approx(den.x), rcp_approx(den.y)));
        o[2 * jp] = r.x;
        o[2 * jp + 1] = r.y;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float pre = bs[j];
#pragma unroll
        for (int k = 0; k < K; ++k) pre += wk[k][j] * win[k][j];
        o[j] = pre * sig<Act>(pre);
      }
    }
    if (cv && i < nt) Vec<Act, 4>::store(out, o);
    out += p.D;
#pragma unroll
    for (int k = 0; k < K - 1; ++k)
#pragma unroll
      for (int j = 0; j < 4; ++j) win[k][j] = win[k + 1][j];
  }
}

template <typename Act, int K>
__global__ void __launch_bounds__(kTileWarps * 32) s6_conv1d_bwd_tile_kernel(const __grid_constant__ ConvTileParams P) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int kXRows = kTileT + 2 * (K - 1);  // xs row r: input t0 - (K-1) + r
  constexpr int kGRows = kTileT + K - 1;        // gs row r: dout of step t0 + r
  const ConvParams& p = P.p;
  Act* xs = reinterpret_cast<Act*>(smem);
  Act* gs = reinterpret_cast<Act*>(smem + tile_rows_bytes<Act>(kXRows));
  float* red = reinterpret_cast<float*>(smem + tile_rows_bytes<Act>(kXRows) + tile_rows_bytes<Act>(kGRows));
  uint64_t* bar = reinterpret_cast<uint64_t*>(red + kTileWarps * kTileCh * (K + 1));
  const int c0 = blockIdx.x * kTileCh, t0 = blockIdx.y * kTileT, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  tile_barrier_init(bar);
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(bar, (uint32_t)((kXRows + kGRows) * kTileCh * sizeof(Act)));
    tma_load_3d(xs, &P.map_x, bar, c0, t0 - (K - 1), b);
    tma_load_3d(gs, &P.map_dout, bar, c0, t0, b);
  }
  const int d = c0 + 4 * lane;
  const bool cv = d < p.D;
  float wk[K][4], bs[4];
  load_weights<K>(p, d, cv, wk, bs);
  const Act* __restrict__ s0 = static_cast<const Act*>(p.state0);
  const bool ok = mbar_wait(bar, 0, p.status);
  const int ts = t0 + warp * kTileSeg;
  // input tau of this thread's channels
  auto xin = [&](int tau, float* v) {
    if (tau < 0 && s0) {
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = cv ? ld_act(s0 + ((size_t)b * p.D + d + i) * (K - 1) + (K - 1 + tau)) : 0.f;
    } else {
      Vec<Act, 4>::lds(xs + (tau - t0 + K - 1) * kTileCh + 4 * lane, v);
    }
  };
  // dpre of step t from its inputs in[k] = input t-(K-1)+k (0 past L: dout is 0 there)
  auto dpre_from = [&](int t, const float (&in)[K][4], float* g) {
    float go[4];
    Vec<Act, 4>::lds(gs + (t - t0) * kTileCh + 4 * lane, go);
    if constexpr (std::is_same<Act, __nv_bfloat16>::value) {
      // two channels per packed op, per channel the scalar form's operations
      // in its order (bit-identical to the other paths)
#pragma unroll
      for (int jp = 0; jp < 2; ++jp) {
        float2 pre = make_float2(bs[2 * jp], bs[2 * jp + 1]);
#pragma unroll
        for (int k = 0; k < K; ++k)
          pre = ffma2(make_float2(wk[k][2 * jp], wk[k][2 * jp + 1]), make_float2(in[k][2 * jp], in[k][2 * jp + 1]), pre);
        const float2 x = fmul2(pre, make_float2(-kLog2e, -kLog2e));
        const float2 den = fadd2(make_float2(1.f, 1.f), make_float2(ex2_approx(x.x), ex2_approx(x.y)));
        const float2 s = make_float2(rcp_approx(den.x), rcp_approx(den.y));
        const float2 f = ffma2(pre, fadd2(make_float2(1.f, 1.f), make_float2(-s.x, -s.y)), make_float2(1.f, 1.f));
        const float2 gg = fmul2(fmul2(make_float2(go[2 * jp], go[2 * jp + 1]), s), f);
        g[2 * jp] = gg.x;
        g[2 * jp + 1] = gg.y;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float pre = bs[i];
#pragma unroll
        for (int k = 0; k < K; ++k) pre += wk[k][i] * in[k][i];
        const float s = sig<Act>(pre);
        g[i] = go[i] * s * fmaf(pre, 1.f - s, 1.f);
      }
    }
  };
  float aw[K][4], ab[4];  // this warp's sums of the dw[k] and dbias terms
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    ab[i] = 0.f;
#pragma unroll
    for (int k = 0; k < K; ++k) aw[k][i] = 0.f;
  }
  if (ok && ts < p.L) {
    float gw[K][4];  // gw[k] = dpre[t + k]
#pragma unroll
    for (int k = 1; k < K; ++k) {
      const int t = ts + kTileSeg - 1 + k;
      float in[K][4];
#pragma unroll
      for (int j = 0; j < K; ++j) xin(t - (K - 1) + j, in[j]);
      dpre_from(t, in, gw[k]);
    }
    float xw[K][4];  // xw[k] = input t - (K-1) + k
#pragma unroll
    for (int k = 1; k < K; ++k) xin(ts + kTileSeg - 1 - (K - 1) + k, xw[k]);
    Act* __restrict__ dx = static_cast<Act*>(p.dx);
#pragma unroll
    for (int i = kTileSeg - 1; i >= 0; --i) {
      const int t = ts + i;
      xin(t - (K - 1), xw[0]);
      dpre_from(t, xw, gw[0]);
      float o[4];
#pragma unroll
      for (int jp = 0; jp < 2; ++jp) {
        const int j0 = 2 * jp, j1 = 2 * jp + 1;
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < K; ++k)
          acc = ffma2(make_float2(wk[k][j0], wk[k][j1]), make_float2(gw[K - 1 - k][j0], gw[K - 1 - k][j1]), acc);
        o[j0] = acc.x;
        o[j1] = acc.y;
        const float2 g0 = make_float2(gw[0][j0], gw[0][j1]);
        const float2 sb = fadd2(make_float2(ab[j0], ab[j1]), g0);
        ab[j0] = sb.x;
        ab[j1] = sb.y;
#pragma unroll
        for (int k = 0; k < K; ++k) {
          const float2 sw = ffma2(g0, make_float2(xw[k][j0], xw[k][j1]), make_float2(aw[k][j0], aw[k][j1]));
          aw[k][j0] = sw.x;
          aw[k][j1] = sw.y;
        }
      }
      if (cv && t < p.L) Vec<Act, 4>::store(dx + ((size_t)b * p.L + t) * p.D + d, o);
#pragma unroll
      for (int k = K - 1; k > 0; --k)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          gw[k][j] = gw[k - 1][j];
          xw[k][j] = xw[k - 1][j];
        }
    }
    // the first warp of the first tile owns the state's gradient; here
    // gw[m + 1] = dpre[m]: dstate0[j] = sum_{k<=j} w[k] * dpre[j - k]
    if (ts == 0 && p.dstate0 && K > 1 && cv) {
#pragma unroll
      for (int j = 0; j < K - 1; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float acc = 0.f;
#pragma unroll
          for (int k = 0; k <= j; ++k) acc += wk[k][i] * gw[j - k + 1][i];
          p.dstate0[((size_t)b * p.D + d + i) * (K - 1) + j] = acc;
        }
    }
  }
  // the tile's partial sums: warps added in order 0..3 (fixed), written as
  // row (b, tile) of partials [b][tile][d][K+1]
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float* r = red + ((size_t)warp * kTileCh + 4 * lane + i) * (K + 1);
#pragma unroll
    for (int k = 0; k < K; ++k) r[k] = aw[k][i];
    r[K] = ab[i];
  }
  __syncthreads();
  if (!ok) return;
  const int nrun = (p.L + kTileT - 1) / kTileT;
  const int nvalid = min(kTileCh, p.D - c0) * (K + 1);
  float* pp = p.ws + (((size_t)b * nrun + blockIdx.y) * p.D + c0) * (K + 1);
  for (int e = threadIdx.x; e < nvalid; e += kTileWarps * 32) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kTileWarps; ++w) s += red[w * kTileCh * (K + 1) + e];
    pp[e] = s;
  }
}

// dw[d][k], dbias[d] = sum of the partial rows r = 0 .. R-1 (one per batch
// row and run): a block covers kRedCols columns (d, k), k = K meaning the
// bias; its kRedGroups warps sum the rows r = g (mod kRedGroups), each in
// ascending r, and the group sums are added in ascending g.  A fixed order,
// so the result does not depend on timing.
constexpr int kRedCols = 32, kRedGroups = 8;

__global__ void __launch_bounds__(kRedCols * kRedGroups) s6_conv1d_reduce_kernel(const float* __restrict__ part, int R,
                                                                                int D, int K, float* dw,
                                                                                float* dbias) {
  __shared__ float gsum[kRedGroups][kRedCols];
  const int col = threadIdx.x % kRedCols, g = threadIdx.x / kRedCols;
  const int ncol = D * (K + 1);
  const int e = blockIdx.x * kRedCols + col;
  float s = 0.f;
  if (e < ncol) {
#pragma unroll 8
    for (int r = g; r < R; r += kRedGroups) s += __ldg(part + (size_t)r * ncol + e);
  }
  gsum[g][col] = s;
  __syncthreads();
  if (g != 0 || e >= ncol) return;
  float t = gsum[0][col];
#pragma unroll
  for (int j = 1; j < kRedGroups; ++j) t += gsum[j][col];
  const int d = e / (K + 1), k = e % (K + 1);
  if (k < K)
    dw[(size_t)d * K + k] = t;
  else
    dbias[d] = t;
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

// state_last (K > 1 and asked for): the last K-1 inputs
template <typename Act>
cudaError_t launch_state(const ConvParams& p, cudaStream_t stream) {
  if (!p.state_last || p.K == 1) return cudaSuccess;
  const long long n = (long long)p.B * p.D * (p.K - 1);
  s6_conv1d_state_kernel<Act><<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(
      static_cast<const Act*>(p.x), static_cast<const Act*>(p.state0), static_cast<Act*>(p.state_last), p.B, p.L,
      p.D, p.K);
  return cudaGetLastError();
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
  if (e != cudaSuccess) return e;
  return launch_state<Act>(p, stream);
}

cudaError_t launch_reduce(const ConvParams& p, int nrun, cudaStream_t stream) {
  const int n = p.D * (p.K + 1);
  s6_conv1d_reduce_kernel<<<(n + kRedCols - 1) / kRedCols, kRedCols * kRedGroups, 0, stream>>>(
      p.ws, p.B * nrun, p.D, p.K, p.dw, p.dbias);
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
  return launch_reduce(p, nrun, stream);
}

template <typename Act, int K>
cudaError_t tile_k(const ConvTileParams& P, bool bwd, cudaStream_t stream) {
  const ConvParams& p = P.p;
  const dim3 grid((p.D + kTileCh - 1) / kTileCh, (p.L + kTileT - 1) / kTileT, p.B);
  if (!bwd) {
    auto kern = s6_conv1d_fwd_tile_kernel<Act, K>;
    constexpr size_t smem = fwd_tile_smem<Act, K>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kTileWarps * 32, smem, stream>>>(P);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_state<Act>(p, stream);
  }
  auto kern = s6_conv1d_bwd_tile_kernel<Act, K>;
  constexpr size_t smem = bwd_tile_smem<Act, K>();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kTileWarps * 32, smem, stream>>>(P);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_reduce(p, (p.L + kTileT - 1) / kTileT, stream);
}

template <typename Act>
cudaError_t tile_dispatch(const ConvTileParams& P, bool bwd, cudaStream_t stream) {
  switch (P.p.K) {
#define S6_CONV_K(KK) \
  case KK:            \
    return tile_k<Act, KK>(P, bwd, stream);
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

// Tile path: the vector path's conditions, rows of a whole number of 16-byte
// units (what a tensor map's strides need), 16-byte aligned TMA sources, the
// grid within its limits, and tensor maps the driver accepts.
bool tile_maps(const ConvParams& p, int act, bool bwd, ConvTileParams* P) {
  if (!vec_ok(p, act) || p.L < 1 || p.B < 1 || p.D < 1) return false;
  const uint64_t e = act == SSM_BF16 ? 2 : 4;
  if ((p.D * e) % 16 != 0) return false;
  if (reinterpret_cast<uintptr_t>(p.x) & 15) return false;
  if (bwd && (reinterpret_cast<uintptr_t>(p.dout) & 15)) return false;
  if ((p.L + kTileT - 1) / kTileT > 65535 || p.B > 65535) return false;
  const uint64_t dims[3] = {(uint64_t)p.D, (uint64_t)p.L, (uint64_t)p.B};
  const uint64_t strides[2] = {p.D * e, (uint64_t)p.L * p.D * e};
  const uint32_t box_x[3] = {kTileCh, (uint32_t)(kTileT + (bwd ? 2 : 1) * (p.K - 1)), 1};
  if (!encode_tile_map(&P->map_x, p.x, act == SSM_BF16, 3, dims, strides, box_x)) return false;
  if (bwd) {
    const uint32_t box_g[3] = {kTileCh, (uint32_t)(kTileT + p.K - 1), 1};
    if (!encode_tile_map(&P->map_dout, p.dout, act == SSM_BF16, 3, dims, strides, box_g)) return false;
  } else {
    P->map_dout = P->map_x;
  }
  P->p = p;
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

int conv1d_path(const ConvParams& p, int act, bool bwd) {
  ConvTileParams P;
  if (tile_maps(p, act, bwd, &P)) return SSM_CONV_PATH_TILE;
  return vec_ok(p, act) ? SSM_CONV_PATH_VECTOR : SSM_CONV_PATH_SCALAR;
}

cudaError_t launch_conv1d(const ConvParams& p, int act, bool bwd, cudaStream_t stream) {
  ConvTileParams P;
  if (tile_maps(p, act, bwd, &P))
    return act == SSM_BF16 ? tile_dispatch<__nv_bfloat16>(P, bwd, stream) : tile_dispatch<float>(P, bwd, stream);
  const bool vec = vec_ok(p, act);
  if (act == SSM_BF16)
    return vec ? dispatch_k<__nv_bfloat16, 4>(p, bwd, stream) : dispatch_k<__nv_bfloat16, 1>(p, bwd, stream);
  return vec ? dispatch_k<float, 4>(p, bwd, stream) : dispatch_k<float, 1>(p, bwd, stream);
}

cudaError_t launch_conv1d_step(const ConvParams& p, int act, cudaStream_t stream) {
  return act == SSM_BF16 ? step_dispatch<__nv_bfloat16>(p, stream) : step_dispatch<float>(p, stream);
}

}  // namespace s6
