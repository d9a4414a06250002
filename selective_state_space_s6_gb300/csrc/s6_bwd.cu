// S6 selective-scan backward.
//
// Same work split as the forward: one CTA per (64-channel tile, batch), a
// lane pair per channel, each lane owning NG states in registers.  The lane
// walks its chunks (kChunk steps, restarted from the forward's saved chunk
// states) from last to first:
//   pass A: recompute h forward over the chunk, keeping the state at every
//           kSub-th step in shared memory;
//   pass B: for each kSub-step sub-chunk, last first: recompute its kSub
//           states into registers, then step backward through it with the
//           adjoint recurrence g_t = dy_t*C_t + Abar_{t+1}*g_{t+1}.
// Per step, the channel-sums of the dBm and dCm terms are taken over the
// CTA's 64 channels in shared memory in a fixed order and stored as one
// partial per CTA; the parameter-gradient sums over t stay in registers and
// are stored as one partial per batch.  Two small kernels then add the
// partials in ascending tile / batch order.  No floating-point atomics
// anywhere, so results are bit-identical from run to run (the single-writer,
// fixed-order policy of the deterministic_backward.py page, ordered_cumsum).
#include "s6_internal.cuh"

namespace s6 {

// Shared-memory layout of the per-step channel reduction: for each of the
// two quantities (dBm, dCm), the 64 channels are stored in 4 groups of 16,
// each group padded by 8 floats so that the reading lanes of one warp fall
// into distinct banks.
template <int NP>
struct RedLayout {
  static constexpr int kGroup = 16 * NP + 8;
  static constexpr int kQ = 4 * kGroup;
  static constexpr int kBuf = 2 * kQ;
  __device__ static int at(int q, int d, int n) { return q * kQ + (d >> 4) * kGroup + (d & 15) * NP + n; }
};

// sum += x with a running compensation term (Kahan); plain IEEE ops, no reassociation.
__device__ __forceinline__ void kahan_add(float& sum, float& comp, float x) {
  const float y = __fsub_rn(x, comp);
  const float t = __fadd_rn(sum, y);
  comp = __fsub_rn(__fsub_rn(t, sum), y);
  sum = t;
}

template <typename Act, int NG>
__global__ void __launch_bounds__(kScanThreads)
    s6_bwd_kernel(const BwdParams p) {
  constexpr int NP = 2 * NG;  // padded state count of a channel
  using RL = RedLayout<NP>;
  extern __shared__ float smem[];
  float* ckpt = smem;                                      // [kChunk/kSub][kScanThreads][NG]
  float* red = smem + (kChunk / kSub) * kScanThreads * NG;  // [2][RL::kBuf]

  const int tid = threadIdx.x;
  const int half = tid & 1;
  const int dl = tid >> 1;
  const int d = blockIdx.x * kDTile + dl;
  const int b = blockIdx.y;
  if (blockIdx.x == 0 && b == 0 && tid == 0) *p.ws_ndt = gridDim.x;  // tile rows of ws_dbc, for the finalize
  const bool dvalid = d < p.D;
  const int dc = dvalid ? d : p.D - 1;
  const int L = p.L, D = p.D, N = p.N;

  // Parameter-gradient sums over t: each chunk sums its kChunk terms in
  // registers (accA, accD, accBias), and the chunk sums are added into the
  // totals with a compensated (Kahan) add, so long sequences keep f32 accuracy.
  float A[NG], g[NG], accA[NG], totA[NG], cmpA[NG];
#pragma unroll
  for (int i = 0; i < NG; ++i) {
    const int n = half * NG + i;
    const bool nv = n < N;
    A[i] = nv ? -expf(p.A_log[dc * N + n]) : 0.f;
    g[i] = (nv && p.dh_last && dvalid) ? p.dh_last[((size_t)b * D + d) * N + n] : 0.f;
    totA[i] = 0.f;
    cmpA[i] = 0.f;
  }
  const float bias = p.delta_bias[dc];
  const float Dd = p.Dp[dc];
  float totD = 0.f, cmpD = 0.f, totBias = 0.f, cmpBias = 0.f;

  const size_t row0 = (size_t)b * L * D + dc;
  const Act* up = static_cast<const Act*>(p.u) + row0;
  const Act* rp = static_cast<const Act*>(p.delta_raw) + row0;
  const Act* zp = p.z ? static_cast<const Act*>(p.z) + row0 : nullptr;
  const Act* gp = static_cast<const Act*>(p.dout) + row0;
  Act* dup = static_cast<Act*>(p.du) + row0;
  Act* drp = static_cast<Act*>(p.d_delta_raw) + row0;
  Act* dzp = p.z ? static_cast<Act*>(p.dz) + row0 : nullptr;
  const Act* Bp = static_cast<const Act*>(p.Bm) + (size_t)b * L * N + half * NG;
  const Act* Cp = static_cast<const Act*>(p.Cm) + (size_t)b * L * N + half * NG;

  // reducer role in the per-step channel sum: output o = (q, n), channel quarter r
  const int red_o = tid >> 2, red_r = tid & 3;
  const int red_q = red_o / NP, red_n = red_o % NP;
  const bool red_active = red_o < 2 * NP;

  int step_parity = 0;
  for (int c = p.nchunks - 1; c >= 0; --c) {
    const int t0 = c * kChunk;
    const int t1 = min(t0 + kChunk, L);
    float accD = 0.f, accBias = 0.f;
#pragma unroll
    for (int i = 0; i < NG; ++i) accA[i] = 0.f;
    // ---- pass A: forward recompute from the chunk state, checkpoint every kSub steps
    float h[NG];
    {
      const float* cs = p.chunk_states + (((size_t)b * p.nchunks + c) * D + dc) * N + half * NG;
#pragma unroll
      for (int i = 0; i < NG; ++i) h[i] = (half * NG + i < N) ? cs[i] : 0.f;
    }
    for (int t = t0; t < t1; ++t) {
      if (((t - t0) % kSub) == 0) {
        float* ck = ckpt + (((t - t0) / kSub) * kScanThreads + tid) * NG;
#pragma unroll
        for (int i = 0; i < NG; ++i) ck[i] = h[i];
      }
      const size_t o = (size_t)t * D;
      const float delta = clamp_dt(softplus_f(ld_act(rp + o) + bias), p.dt_min, p.dt_max);
      const float du = delta * ld_act(up + o);
#pragma unroll
      for (int i = 0; i < NG; ++i) {
        const float Bn = (half * NG + i < N) ? ld_act(Bp + (size_t)t * N + i) : 0.f;
        h[i] = fmaf(expf(delta * A[i]), h[i], du * Bn);
      }
    }
    // ---- pass B: sub-chunks in reverse
    const int nsub = (t1 - t0 + kSub - 1) / kSub;
    for (int j = nsub - 1; j >= 0; --j) {
      const int ts = t0 + j * kSub;
      const int cnt = min(kSub, t1 - ts);
      float hs[kSub][NG];
      float hstart[NG];
      {
        const float* ck = ckpt + (j * kScanThreads + tid) * NG;
#pragma unroll
        for (int i = 0; i < NG; ++i) hstart[i] = ck[i];
      }
#pragma unroll
      for (int k = 0; k < kSub; ++k) {
        if (k < cnt) {
          const int t = ts + k;
          const size_t o = (size_t)t * D;
          const float delta = clamp_dt(softplus_f(ld_act(rp + o) + bias), p.dt_min, p.dt_max);
          const float du = delta * ld_act(up + o);
#pragma unroll
          for (int i = 0; i < NG; ++i) {
            const float hp = k == 0 ? hstart[i] : hs[k > 0 ? k - 1 : 0][i];
            const float Bn = (half * NG + i < N) ? ld_act(Bp + (size_t)t * N + i) : 0.f;
            hs[k][i] = fmaf(expf(delta * A[i]), hp, du * Bn);
          }
        }
      }
#pragma unroll
      for (int k = kSub - 1; k >= 0; --k) {
        if (k < cnt) {
          const int t = ts + k;
          const size_t o = (size_t)t * D;
          const float u = ld_act(up + o);
          const float s = ld_act(rp + o) + bias;
          const float sp = softplus_f(s);
          const float delta = clamp_dt(sp, p.dt_min, p.dt_max);
          // softplus' = sigmoid, masked where the limit clamps (both ends inclusive)
          const float sig_s = (sp >= p.dt_min && sp <= p.dt_max) ? sigmoid_f(s) : 0.f;
          const float dout = ld_act(gp + o);
          float Bn[NG], Cn[NG];
          float ypart = 0.f;
#pragma unroll
          for (int i = 0; i < NG; ++i) {
            const bool nv = half * NG + i < N;
            Bn[i] = nv ? ld_act(Bp + (size_t)t * N + i) : 0.f;
            Cn[i] = nv ? ld_act(Cp + (size_t)t * N + i) : 0.f;
            ypart = fmaf(Cn[i], hs[k][i], ypart);
          }
          const float y = ypart + __shfl_xor_sync(0xffffffffu, ypart, 1) + Dd * u;
          float dy = dout, dzv = 0.f;
          if (zp) {
            const float zz = ld_act(zp + o);
            const float sz = sigmoid_f(zz);
            dy = dout * zz * sz;
            dzv = dout * y * sz * (1.f + zz * (1.f - sz));
          }
          const float du_ = delta * u;
          float sgB = 0.f, sAp = 0.f;
          float* rb = red + step_parity * RL::kBuf;
#pragma unroll
          for (int i = 0; i < NG; ++i) {
            const float a = expf(delta * A[i]);
            const float hp = k == 0 ? hstart[i] : hs[k > 0 ? k - 1 : 0][i];
            const float gt = fmaf(dy, Cn[i], g[i]);
            const float ah = a * hp;
            sgB = fmaf(gt, Bn[i], sgB);
            sAp = fmaf(A[i] * ah, gt, sAp);
            accA[i] = fmaf(delta * ah, gt, accA[i]);
            rb[RL::at(0, dl, half * NG + i)] = dvalid ? gt * du_ : 0.f;
            rb[RL::at(1, dl, half * NG + i)] = dvalid ? dy * hs[k][i] : 0.f;
            g[i] = a * gt;
          }
          sgB += __shfl_xor_sync(0xffffffffu, sgB, 1);
          sAp += __shfl_xor_sync(0xffffffffu, sAp, 1);
          if (half == 0 && dvalid) {
            const float dd = fmaf(u, sgB, sAp);
            const float draw = dd * sig_s;
            st_act(dup + o, fmaf(Dd, dy, delta * sgB));
            st_act(drp + o, draw);
            if (zp) st_act(dzp + o, dzv);
            accD = fmaf(dy, u, accD);
            accBias += draw;
          }
          __syncthreads();
          // fixed-order channel sum: 16 channels per lane, then ((r0+r1)+(r2+r3))
          float v = 0.f;
          if (red_active) {
#pragma unroll 4
            for (int k2 = 0; k2 < 16; ++k2) v += rb[RL::at(red_q, red_r * 16 + k2, red_n)];
          }
          v += __shfl_down_sync(0xffffffffu, v, 1);
          v += __shfl_down_sync(0xffffffffu, v, 2);
          if (red_active && red_r == 0 && red_n < N)
            p.ws_dbc[((((size_t)blockIdx.x * p.B + b) * L + t) * 2 + red_q) * N + red_n] = v;
          step_parity ^= 1;
        }
      }
    }
#pragma unroll
    for (int i = 0; i < NG; ++i) kahan_add(totA[i], cmpA[i], accA[i]);
    kahan_add(totD, cmpD, accD);
    kahan_add(totBias, cmpBias, accBias);
  }
  // ---- per-batch parameter-gradient partials and dh0
  if (dvalid) {
    float* wp = p.ws_param + ((size_t)b * p.nseg * D + d) * (N + 2);  // segment row 0
#pragma unroll
    for (int i = 0; i < NG; ++i) {
      const int n = half * NG + i;
      if (n < N) {
        wp[n] = A[i] * totA[i];
        if (p.dh0) p.dh0[((size_t)b * D + d) * N + n] = g[i];
      }
    }
    if (half == 0) {
      wp[N] = totD;
      wp[N + 1] = totBias;
    }
  }
}

// dBm/dCm[b,t,n] = sum over channel tiles k (ascending) of ws_dbc[k][b][t][q][n]
template <typename Act>
__global__ void s6_reduce_dbc_kernel(const float* __restrict__ ws, const int* __restrict__ ndt_ptr, int B, int L,
                                     int N, Act* __restrict__ dBm, Act* __restrict__ dCm) {
  const size_t per = (size_t)B * L * 2 * N;
  const int ndt = *ndt_ptr;
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < per;
       e += (size_t)gridDim.x * blockDim.x) {
    float s = 0.f;
    for (int k = 0; k < ndt; ++k) s += ws[(size_t)k * per + e];
    const int n = (int)(e % N);
    const size_t btq = e / N;
    const int q = (int)(btq % 2);
    const size_t bt = btq / 2;
    Act* dst = q == 0 ? dBm : dCm;
    st_act(dst + bt * N + n, s);
  }
}

// dA_log[d,n], dDp[d], d_delta_bias[d] = sum over b (ascending) of ws_param[b][d][.]
__global__ void s6_reduce_params_kernel(const float* __restrict__ ws, int B, int D, int N,
                                        float* __restrict__ dA_log, float* __restrict__ dDp,
                                        float* __restrict__ d_delta_bias) {
  const int W = N + 2;
  const size_t per = (size_t)D * W;
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < per;
       e += (size_t)gridDim.x * blockDim.x) {
    float s = 0.f;
    for (int k = 0; k < B; ++k) s += ws[(size_t)k * per + e];
    const int d = (int)(e / W), j = (int)(e % W);
    if (j < N)
      dA_log[(size_t)d * N + j] = s;
    else if (j == N)
      dDp[d] = s;
    else
      d_delta_bias[d] = s;
  }
}

template <typename Act, int NG>
static cudaError_t launch_bwd_ng(const BwdParams& p, cudaStream_t stream) {
  constexpr int NP = 2 * NG;
  const size_t smem = sizeof(float) * ((kChunk / kSub) * kScanThreads * NG + 2 * RedLayout<NP>::kBuf);
  cudaError_t e = cudaFuncSetAttribute(s6_bwd_kernel<Act, NG>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const dim3 grid((p.D + kDTile - 1) / kDTile, p.B);
  s6_bwd_kernel<Act, NG><<<grid, kScanThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

template <typename Act>
static cudaError_t launch_bwd_t(const BwdParams& p, cudaStream_t stream) {
  const int ng = (p.N + 1) / 2;
  if (ng <= 1) return launch_bwd_ng<Act, 1>(p, stream);
  if (ng <= 2) return launch_bwd_ng<Act, 2>(p, stream);
  if (ng <= 4) return launch_bwd_ng<Act, 4>(p, stream);
  return launch_bwd_ng<Act, 8>(p, stream);
}

cudaError_t launch_bwd(const BwdParams& p, int act, cudaStream_t stream) {
  return act == SSM_BF16 ? launch_bwd_t<__nv_bfloat16>(p, stream) : launch_bwd_t<float>(p, stream);
}

cudaError_t launch_reduce_dbc(const float* ws_dbc, const int* ndt, int B, int L, int N, void* dBm,
                              void* dCm, int act, cudaStream_t stream) {
  const size_t per = (size_t)B * L * 2 * N;
  if (per == 0) return cudaSuccess;
  const int threads = 256;
  const int blocks = (int)((per + threads - 1) / threads < 152 * 16 ? (per + threads - 1) / threads : 152 * 16);
  if (act == SSM_BF16)
    s6_reduce_dbc_kernel<__nv_bfloat16><<<blocks, threads, 0, stream>>>(
        ws_dbc, ndt, B, L, N, static_cast<__nv_bfloat16*>(dBm), static_cast<__nv_bfloat16*>(dCm));
  else
    s6_reduce_dbc_kernel<float><<<blocks, threads, 0, stream>>>(
        ws_dbc, ndt, B, L, N, static_cast<float*>(dBm), static_cast<float*>(dCm));
  return cudaGetLastError();
}

cudaError_t launch_reduce_params(const float* ws_param, int B, int D, int N, float* dA_log,
                                 float* dDp, float* d_delta_bias, cudaStream_t stream) {
  const size_t per = (size_t)D * (N + 2);
  if (per == 0) return cudaSuccess;
  const int threads = 256;
  const int blocks = (int)((per + threads - 1) / threads);
  s6_reduce_params_kernel<<<blocks, threads, 0, stream>>>(ws_param, B, D, N, dA_log, dDp,
                                                           d_delta_bias);
  return cudaGetLastError();
}

}  // namespace s6
