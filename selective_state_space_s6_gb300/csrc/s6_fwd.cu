// S6 selective-scan forward (with and without chunk-state saves).
//
// Work split: one CTA per (64-channel tile, batch); each channel's N states
// are held in registers by a pair of adjacent lanes (NG = ceil(N/2) states
// each), so the readout sum over n is one xor-shuffle.  Every lane walks the
// whole sequence in order: h_t = Abar*h_{t-1} + delta*B_t*u_t, the state never
// leaves registers, and every kChunk steps the state is stored as the
// checkpoint the backward restarts from (the "activation saves" of the
// kernels.rs page's multi-step forward).
#include "s6_internal.cuh"

namespace s6 {

template <typename Act, int NG, bool kSave>
__global__ void __launch_bounds__(kScanThreads)
    s6_fwd_kernel(const FwdParams p) {
  const int tid = threadIdx.x;
  const int half = tid & 1;
  const int d = blockIdx.x * kDTile + (tid >> 1);
  const int b = blockIdx.y;
  const bool dvalid = d < p.D;
  const int dc = dvalid ? d : p.D - 1;  // clamped channel for loads of idle lanes
  const int L = p.L, D = p.D, N = p.N;

  float A[NG], h[NG];
#pragma unroll
  for (int i = 0; i < NG; ++i) {
    const int n = half * NG + i;
    const bool nv = n < N;
    A[i] = nv ? -expf(p.A_log[dc * N + n]) : 0.f;
    h[i] = (nv && p.h0) ? p.h0[((size_t)b * D + dc) * N + n] : 0.f;
  }
  const float bias = p.delta_bias[dc];
  const float Dd = p.Dp[dc];

  const size_t row0 = (size_t)b * L * D + dc;
  const Act* up = static_cast<const Act*>(p.u) + row0;
  const Act* rp = static_cast<const Act*>(p.delta_raw) + row0;
  const Act* zp = p.z ? static_cast<const Act*>(p.z) + row0 : nullptr;
  Act* op = static_cast<Act*>(p.out) + row0;
  const Act* Bp = static_cast<const Act*>(p.Bm) + (size_t)b * L * N + half * NG;
  const Act* Cp = static_cast<const Act*>(p.Cm) + (size_t)b * L * N + half * NG;

  for (int t = 0; t < L; ++t) {
    if (kSave && (t % kChunk) == 0 && dvalid) {
      float* cs = p.chunk_states + (((size_t)b * p.nchunks + t / kChunk) * D + d) * N + half * NG;
#pragma unroll
      for (int i = 0; i < NG; ++i)
        if (half * NG + i < N) cs[i] = h[i];
    }
    const size_t o = (size_t)t * D;
    const float u = ld_act(up + o);
    const float delta = clamp_dt(softplus_f(ld_act(rp + o) + bias), p.dt_min, p.dt_max);
    const float du = delta * u;
    float y = 0.f;
#pragma unroll
    for (int i = 0; i < NG; ++i) {
      const bool nv = half * NG + i < N;
      const float Bn = nv ? ld_act(Bp + (size_t)t * N + i) : 0.f;
      const float Cn = nv ? ld_act(Cp + (size_t)t * N + i) : 0.f;
      const float a = expf(delta * A[i]);
      h[i] = fmaf(a, h[i], du * Bn);
      y = fmaf(Cn, h[i], y);
    }
    y += __shfl_xor_sync(0xffffffffu, y, 1);
    if (half == 0 && dvalid) {
      float outv = fmaf(Dd, u, y);
      if (zp) {
        const float zz = ld_act(zp + o);
        outv *= zz * sigmoid_f(zz);
      }
      st_act(op + o, outv);
    }
  }
  if (p.h_last && dvalid) {
    float* hl = p.h_last + ((size_t)b * D + d) * N + half * NG;
#pragma unroll
    for (int i = 0; i < NG; ++i)
      if (half * NG + i < N) hl[i] = h[i];
  }
}

template <typename Act, bool kSave>
static cudaError_t launch_fwd_t(const FwdParams& p, cudaStream_t stream) {
  const dim3 grid((p.D + kDTile - 1) / kDTile, p.B);
  const dim3 block(kScanThreads);
  const int ng = (p.N + 1) / 2;
  if (ng <= 1)
    s6_fwd_kernel<Act, 1, kSave><<<grid, block, 0, stream>>>(p);
  else if (ng <= 2)
    s6_fwd_kernel<Act, 2, kSave><<<grid, block, 0, stream>>>(p);
  else if (ng <= 4)
    s6_fwd_kernel<Act, 4, kSave><<<grid, block, 0, stream>>>(p);
  else
    s6_fwd_kernel<Act, 8, kSave><<<grid, block, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_fwd(const FwdParams& p, int act, cudaStream_t stream) {
  const bool save = p.chunk_states != nullptr;
  if (act == SSM_BF16)
    return save ? launch_fwd_t<__nv_bfloat16, true>(p, stream)
                : launch_fwd_t<__nv_bfloat16, false>(p, stream);
  return save ? launch_fwd_t<float, true>(p, stream) : launch_fwd_t<float, false>(p, stream);
}

}  // namespace s6
