// Decode step of the S6 scan (T = 1; mamba-rs kernels.rs page: "Single-step
// SSM forward (T=1 inference)"): h [B][D][N] read and written in place.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <type_traits>

#include "s6_internal.cuh"
#include "s6_math.cuh"
#include "s6_tma.cuh"

namespace s6 {

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// One decode step (T = 1), streamed.  A CTA owns one tile of kCh = 256/TPC
// channels and walks a range of batch rows, TPC rows per stage.  A producer
// warp brings a stage's states (box [TPC rows][kCh channels][N] of h, 16 KB),
// its u, delta_raw and z boxes [TPC][kCh] and its Bm, Cm boxes [TPC][N]
// into a kStepStages-deep shared-memory ring with one TMA copy per tensor,
// so that each CTA keeps all its rows' copies in flight at once; the copy
// engine handles the ragged edges (channels past D, rows past B arrive as
// zeros and are not stored).  Consumer thread (c, q) owns states 4q..4q+3 of
// channel c for the stage's TPC rows (TPC = N/4 lanes per channel).  Work
// that depends only on (b, d) -- softplus of delta with its limit, silu of
// the gate -- is done once per (b, d), by lane j for row j of the stage, and
// passed round with shuffles; A = -exp(A_log) once per thread.  The
// arithmetic per row is the scan kernel's, in the same order (softplus,
// limit, decays, state update, per-lane readout, the channel's lanes added
// in lane order, skip, gate), so that L steps equal one L-step scan bit for
// bit.  Bound by HBM: every state is read and written once.
constexpr int kStepConsumers = 256;
constexpr int kStepStages = 3;

template <typename Act, int TPC>
struct StepTile {
  static constexpr int N = 4 * TPC;
  static constexpr int R = TPC;                      // batch rows per stage
  static constexpr int kCh = kStepConsumers / TPC;   // channels per tile
  static constexpr int kH = R * kCh * N * 4;         // [R][kCh][N] f32
  static constexpr int kV = R * kCh * (int)sizeof(Act);  // [R][kCh] act
  static constexpr int kBC = R * N * (int)sizeof(Act);   // [R][N] act
  // every box lands on a 128-byte boundary (a TMA tensor copy's shared-memory
  // destination must be 128-byte aligned)
  static constexpr int kBCr = (kBC + 127) / 128 * 128;
  static constexpr int kOffU = kH, kOffR = kH + kV, kOffZ = kH + 2 * kV, kOffB = kH + 3 * kV,
                       kOffC = kOffB + kBCr;
  static constexpr int kStage = kOffC + kBCr;
  static_assert(kH % 128 == 0 && kV % 128 == 0 && kOffB % 128 == 0 && kOffC % 128 == 0 && kStage % 128 == 0,
                "TMA destinations must be 128-byte aligned");
};

template <typename Act, int TPC>
constexpr size_t step_smem_bytes() {
  return (size_t)kStepStages * StepTile<Act, TPC>::kStage + 2 * kStepStages * 8;
}

struct StepTmaParams {
  CUtensorMap map_h, map_u, map_r, map_z, map_B, map_C;  // 64-byte aligned members first
  FwdParams p;
  int ndt;     // channel tiles
  int groups;  // batch-row groups (CTAs = ndt * groups)
};

// 4 consecutive activations from shared memory
__device__ __forceinline__ float4 lds4_act(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 lds4_act(const __nv_bfloat16* p) {
  const uint2 v = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

template <typename Act, int TPC, bool kFast, bool kGate>
__global__ void __launch_bounds__(kStepConsumers + 32) s6_step_kernel(const __grid_constant__ StepTmaParams P) {
  using T = StepTile<Act, TPC>;
  constexpr int N = T::N, R = T::R;
  const FwdParams& p = P.p;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStepStages * T::kStage);
  uint64_t* empty = full + kStepStages;
  const int dt = blockIdx.x % P.ndt, grp = blockIdx.x / P.ndt;
  // this CTA's rows: whole blocks of R rows [blk_lo, blk_hi), the last block ragged at B
  const int nblk = (p.B + R - 1) / R;
  const int blk_lo = (int)((long long)grp * nblk / P.groups), blk_hi = (int)((long long)(grp + 1) * nblk / P.groups);
  const int nst = blk_hi - blk_lo;  // stages to walk
  const int d0 = dt * T::kCh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStepStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kStepConsumers / 32);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kStepConsumers / 32) {
    // producer: one lane issues stage i's copies once the consumers have
    // released the stage's previous use
    if (lane == 0) {
      tma_prefetch_desc(&P.map_h);
      constexpr uint32_t tx = T::kH + (kGate ? 3u : 2u) * T::kV + 2u * T::kBC;
      for (int i = 0; i < nst; ++i) {
        const int s = i % kStepStages;
        if (i >= kStepStages && !mbar_wait(&empty[s], ((i / kStepStages) - 1) & 1, p.status)) break;
        unsigned char* st = smem + (size_t)s * T::kStage;
        const int b0 = (blk_lo + i) * R;
        mbar_arrive_expect_tx(&full[s], tx);
        tma_load_3d(st, &P.map_h, &full[s], 0, d0, b0);
        tma_load_2d(st + T::kOffU, &P.map_u, &full[s], d0, b0);
        tma_load_2d(st + T::kOffR, &P.map_r, &full[s], d0, b0);
        if (kGate) tma_load_2d(st + T::kOffZ, &P.map_z, &full[s], d0, b0);
        tma_load_2d(st + T::kOffB, &P.map_B, &full[s], 0, b0);
        tma_load_2d(st + T::kOffC, &P.map_C, &full[s], 0, b0);
      }
    }
    return;
  }

  const int c = threadIdx.x / TPC, q = threadIdx.x % TPC;
  const int d = min(d0 + c, p.D - 1);  // lanes past D repeat the last channel (they still shuffle)
  const bool cv = d0 + c < p.D;
  const int lead = lane - q;  // lane 0 of this channel
  const float4 al = __ldg(reinterpret_cast<const float4*>(p.A_log + (size_t)d * N + 4 * q));
  float2 A2[2];
  {
    const float a0 = -expf(al.x), a1 = -expf(al.y), a2 = -expf(al.z), a3 = -expf(al.w);
    A2[0] = kFast ? make_float2(a0 * kLog2e, a1 * kLog2e) : make_float2(a0, a1);
    A2[1] = kFast ? make_float2(a2 * kLog2e, a3 * kLog2e) : make_float2(a2, a3);
  }
  const float bias = p.delta_bias[d];
  const float Dd = p.Dp[d];
  for (int i = 0; i < nst; ++i) {
    const int s = i % kStepStages;
    if (!mbar_wait(&full[s], (i / kStepStages) & 1, p.status)) break;
    const unsigned char* st = smem + (size_t)s * T::kStage;
    const Act* su = reinterpret_cast<const Act*>(st + T::kOffU);
    // this lane's row q of the stage: delta (with its limit) and the gate factor
    const float sp_q = clamp_dt(softplus_k<kFast>(lds_act(reinterpret_cast<const Act*>(st + T::kOffR) + q * T::kCh + c) + bias),
                                p.dt_min, p.dt_max);
    const float sl_q = kGate ? silu_k<kFast>(lds_act(reinterpret_cast<const Act*>(st + T::kOffZ) + q * T::kCh + c)) : 1.f;
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const int b = (blk_lo + i) * R + j;
      const float sp = __shfl_sync(0xffffffffu, sp_q, lead + j);
      const float sl = __shfl_sync(0xffffffffu, sl_q, lead + j);
      const float u = lds_act(su + j * T::kCh + c);
      const float4 hv = *reinterpret_cast<const float4*>(st + (size_t)((j * T::kCh + c) * N + 4 * q) * 4);
      const float4 bb = lds4_act(reinterpret_cast<const Act*>(st + T::kOffB) + j * N + 4 * q);
      const float4 cb = lds4_act(reinterpret_cast<const Act*>(st + T::kOffC) + j * N + 4 * q);
      float2 h[2] = {make_float2(hv.x, hv.y), make_float2(hv.z, hv.w)};
      const float2 Bv[2] = {make_float2(bb.x, bb.y), make_float2(bb.z, bb.w)};
      const float2 Cv[2] = {make_float2(cb.x, cb.y), make_float2(cb.z, cb.w)};
      const float du = sp * u;
      const float2 dd = make_float2(sp, sp), uu = make_float2(du, du);
      const float2 a0 = decay2<kFast>(dd, A2[0]);
      const float2 a1 = decay2<kFast>(dd, A2[1]);
      h[0] = ffma2(a0, h[0], fmul2(uu, Bv[0]));
      h[1] = ffma2(a1, h[1], fmul2(uu, Bv[1]));
      const float2 y2 = ffma2(Cv[1], h[1], fmul2(Cv[0], h[0]));
      const float part = y2.x + y2.y;
      // the channel's partial readouts, added in lane order
      float y = __shfl_sync(0xffffffffu, part, lead);
#pragma unroll
      for (int r = 1; r < TPC; ++r) y += __shfl_sync(0xffffffffu, part, lead + r);
      if (cv && b < p.B) {
        const size_t bd = (size_t)b * p.D + d;
        *reinterpret_cast<float4*>(p.h_last + bd * N + 4 * q) = make_float4(h[0].x, h[0].y, h[1].x, h[1].y);
        if (q == j) {
          float o = fmaf(Dd, u, y);
          if (kGate) o *= sl;
          st_act(static_cast<Act*>(p.out) + bd, o);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);  // this warp is done with the stage
  }
}

template <typename Act, int TPC, bool kFast>
cudaError_t launch_step_tpc(const FwdParams& p, cudaStream_t stream) {
  using T = StepTile<Act, TPC>;
  StepTmaParams P;
  memset(&P, 0, sizeof(P));
  P.p = p;
  const bool bf = std::is_same<Act, __nv_bfloat16>::value;
  const uint64_t e = sizeof(Act);
  {
    const uint64_t dims[3] = {(uint64_t)T::N, (uint64_t)p.D, (uint64_t)p.B};
    const uint64_t strides[2] = {(uint64_t)T::N * 4, (uint64_t)p.D * T::N * 4};
    const uint32_t box[3] = {(uint32_t)T::N, (uint32_t)T::kCh, (uint32_t)T::R};
    if (!encode_tile_map(&P.map_h, p.h0, false, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[2] = {(uint64_t)p.D, (uint64_t)p.B};
    const uint64_t strides[1] = {(uint64_t)p.D * e};
    const uint32_t box[2] = {(uint32_t)T::kCh, (uint32_t)T::R};
    if (!encode_tile_map(&P.map_u, p.u, bf, 2, dims, strides, box) ||
        !encode_tile_map(&P.map_r, p.delta_raw, bf, 2, dims, strides, box))
      return cudaErrorInvalidValue;
    if (p.z && !encode_tile_map(&P.map_z, p.z, bf, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[2] = {(uint64_t)T::N, (uint64_t)p.B};
    const uint64_t strides[1] = {(uint64_t)T::N * e};
    const uint32_t box[2] = {(uint32_t)T::N, (uint32_t)T::R};
    if (!encode_tile_map(&P.map_B, p.Bm, bf, 2, dims, strides, box) ||
        !encode_tile_map(&P.map_C, p.Cm, bf, 2, dims, strides, box))
      return cudaErrorInvalidValue;
  }
  constexpr size_t smem = step_smem_bytes<Act, TPC>();
  auto kern = p.z ? s6_step_kernel<Act, TPC, kFast, true> : s6_step_kernel<Act, TPC, kFast, false>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  int per_sm = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kStepConsumers + 32, smem);
  if (err != cudaSuccess) return err;
  const int sms = device_sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  // channel tiles x batch-row groups, all resident at once
  P.ndt = (p.D + T::kCh - 1) / T::kCh;
  const int nblk = (p.B + T::R - 1) / T::R;
  P.groups = std::max(1, std::min(nblk, std::max(1, per_sm) * sms / P.ndt));
  const long long blocks = (long long)P.ndt * P.groups;
  if (blocks > INT32_MAX) return cudaErrorInvalidValue;
  kern<<<(unsigned)blocks, kStepConsumers + 32, smem, stream>>>(P);
  return cudaGetLastError();
}

}  // namespace

// The step kernel takes the shapes of the TMA scan, whose arithmetic it
// repeats: N in {4, 8, 16}, rows of whole 16-byte units and 16-byte aligned
// tensors (its tensor maps need the same), plus 16-byte aligned h and A_log;
// other shapes take one step of the generic scan.
bool step_supported(const FwdParams& p, int act) {
  if (!(p.N == 4 || p.N == 8 || p.N == 16)) return false;
  if (act == SSM_BF16 && p.N == 4) return false;  // the TMA scan's rule for bf16
  if (!aligned16(p.A_log) || !aligned16(p.h0) || !aligned16(p.h_last)) return false;
  if ((long long)p.B * p.D * (p.N / 4) >= (1LL << 40)) return false;
  // bit-identity with the scan needs the scan of the same shape to take the TMA path
  return fwd_tma_supported(p, act);
}

cudaError_t launch_step(const FwdParams& p, int act, cudaStream_t stream) {
  const int tpc = p.N / 4;
  if (act == SSM_BF16) {
    if (tpc == 4) return launch_step_tpc<__nv_bfloat16, 4, true>(p, stream);
    if (tpc == 2) return launch_step_tpc<__nv_bfloat16, 2, true>(p, stream);
    return cudaErrorInvalidValue;
  }
  if (tpc == 4) return launch_step_tpc<float, 4, false>(p, stream);
  if (tpc == 2) return launch_step_tpc<float, 2, false>(p, stream);
  if (tpc == 1) return launch_step_tpc<float, 1, false>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace s6
