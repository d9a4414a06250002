// S6 forward, TMA-pipelined (sm_103a).
//
// CTA = (channel tile, batch); 5 warps:
//   warps 0-3  consumers: each channel's N states are split over TPC = N/4
//              lanes, 4 states per lane in registers (the tile is 128/TPC
//              channels); every lane walks the sequence in order;
//   warp 4     producer: one lane streams [TT x 64] tiles of u, delta_raw, z and
//              [TT x N] tiles of Bm, Cm into an S-stage shared-memory ring with
//              cp.async.bulk.tensor (TMA), completion tracked by mbarriers.
// A lane reads the Bm and Cm values of its 4 states straight from the tiles:
// 16 bytes each in f32, 8 bytes in bf16, widened in registers (exact).  (The
// 8-byte reads take half the shared-memory wavefronts of 16-byte reads of an
// f32 copy; the recurrence's step is bound in part by those wavefronts.)
// A consumer handles a 32-step tile in three phases, so that only the state
// update is carried from step to step and everything else has independent
// work to overlap:
//   1. softplus: each lane computes (delta, delta*u) for the steps it owns
//      (step k belongs to lane k mod TPC of the channel) into shared memory;
//   2. recurrence: per step, for its 4 states, x = delta*A*log2(e),
//      Abar = 2^x, h = Abar*h + (delta*u)*B, y += C*h with packed f32x2
//      multiplies / FMAs (one instruction covers two states); the lane's
//      partial readout goes to shared memory;
//   3. output: for its owned steps a lane adds the channel's TPC partial
//      readouts in fixed order, adds Dp*u, gates with silu(z) and stores.
// Every SSM_CHUNK_LEN steps the state is stored as a chunk state (the
// activation saves of the kernels.rs page's multi-step forward).
//
// All pipeline waits are bounded (s6_tma.cuh); nothing else spins.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "s6_internal.cuh"
#include "s6_math.cuh"
#include "s6_tma.cuh"

namespace s6 {

namespace {

constexpr int kTT = 32;          // steps per pipeline stage
constexpr int kFwdWarps = 5;     // 4 consumers + producer

template <typename Act>
struct FwdCfg {
  // bf16: two stages keep a CTA at ~42 KB of shared memory, four CTAs per SM
  // (a tile takes microseconds of compute, well above the copy latency)
  static constexpr int kStages = std::is_same<Act, float>::value ? 3 : 2;
  // one stage: u, delta_raw, z tiles [kTT][128/TPC] and Bm, Cm tiles [kTT][N],
  // rounded up to 1024 bytes so that every stage's tiles start on the
  // swizzle's alignment
  template <int TPC>
  static constexpr int stage_bytes() {
    return ((3 * kTT * (kScanThreads / TPC) + 2 * kTT * 4 * TPC) * (int)sizeof(Act) + 1023) / 1024 * 1024;
  }
};

struct FwdTmaParams {
  CUtensorMap map_u, map_raw, map_z, map_B, map_C;  // 64-byte aligned members first
  FwdParams p;
};

// TPC lanes per channel, 4 states per lane (N = 4 * TPC); 128 consumer lanes
// cover kCh = 128 / TPC channels.  grid.z = time segment.  kAgg: the
// aggregate pass of the chunked parallel scan -- from a zero state, run the
// segment and store its end state and its decay product exp(A * sum(delta))
// (no readout, no output; z and Cm are not loaded).
template <typename Act, int TPC, bool kSave, bool kFast, bool kGate, bool kAgg = false, bool kStream = false>
__global__ void __launch_bounds__(kFwdWarps * 32) s6_fwd_tma_kernel(const __grid_constant__ FwdTmaParams P) {
  constexpr int N = 4 * TPC;
  constexpr int kCh = kScanThreads / TPC;  // channels per CTA
  constexpr int S = FwdCfg<Act>::kStages;
  constexpr int kTile = kTT * kCh;        // elements of a [TT x kCh] tile
  constexpr int kBC = kTT * N;            // elements of a [TT x N] tile
  constexpr bool kBf16 = std::is_same<Act, __nv_bfloat16>::value;
  constexpr int kStageBytes = FwdCfg<Act>::template stage_bytes<TPC>();
  constexpr int kOwn = kTT / TPC;          // steps whose (t, d) work a lane owns
  constexpr int kPer = 8 / TPC;            // owned steps per 8 rows (the swizzle period)
  constexpr int kPrepRow = kCh + 4;        // float2 row stride of prep (see below)
  constexpr int kYRow = kScanThreads + 1;  // float row stride of ypart (see below)
  using AT = SwzTile<Act, kCh, kTT>;  // u, delta_raw, z tiles

  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* stages = smem;
  // (delta, delta*u) per (step, channel); rows padded by 32 bytes so that the
  // 64-bit accesses of a half-warp (4 rows x 4 channels) fill the banks once
  float2* prep = reinterpret_cast<float2*>(smem + (size_t)S * kStageBytes);  // [TT][kPrepRow]
  // per-lane partial readouts; rows padded by one float so that the TPC lanes
  // of a channel, reading rows k, k+1, .. at once, hit different banks
  float* ypart = reinterpret_cast<float*>(prep + kTT * kPrepRow);  // [TT][kYRow]
  uint64_t* full = reinterpret_cast<uint64_t*>(ypart + kTT * kYRow);
  uint64_t* empty = full + S;

  const FwdParams& p = P.p;
  // the swizzled tiles need 1024-byte aligned stages (uniform: the whole CTA leaves)
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.status, kStatusLayout);
    return;
  }
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int L = p.L, D = p.D;
  // Work items, walked in the same order by every role.  Grid mode: one item,
  // (channel tile blockIdx.x, batch blockIdx.y, time segment blockIdx.z).
  // Stream mode (kStream): the CTA's range of the plan's chunk units, laid
  // out sequence by sequence with time running backwards inside a sequence,
  // so that a range starts with the first piece (in time) of a sequence and
  // ends with the last piece of another; item = (sequence, its chunks).
  const FwdPlan& pl = p.plan;
  const int u_begin = kStream ? (int)plan_bound(pl, blockIdx.x) : 0;
  const int u_end = kStream ? (int)plan_bound(pl, blockIdx.x + 1) : 1;
  struct Item {
    int b, d0, t_begin, t_end, next, sq;
    bool first, last;  // the item starts / ends its sequence
  };
  auto item_at = [&](int u) {
    Item it;
    if (kStream) {
      const int sq = u / pl.nch, S0 = sq * pl.nch;
      it.next = min(S0 + pl.nch, u_end);
      const int c_lo = pl.nch - (it.next - S0), c_hi = pl.nch - (u - S0);
      it.sq = sq;
      it.b = sq / pl.ndt;
      it.d0 = (sq % pl.ndt) * kCh;
      it.t_begin = c_lo * kChunk;
      it.t_end = min(L, c_hi * kChunk);
      it.first = c_lo == 0;
      it.last = c_hi == pl.nch;
    } else {
      const int seg = blockIdx.z;
      it.next = 1;
      it.sq = 0;
      it.b = blockIdx.y;
      it.d0 = blockIdx.x * kCh;
      it.t_begin = seg * p.seg_len;
      it.t_end = min(L, it.t_begin + p.seg_len);
      it.first = seg == 0;
      it.last = seg == (int)gridDim.z - 1;
    }
    return it;
  };

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 4);
    }
    fence_mbar_init();
  }
  __syncthreads();

  auto tile_u = [&](int s) { return reinterpret_cast<Act*>(stages + (size_t)s * kStageBytes); };
  auto tile_raw = [&](int s) { return tile_u(s) + kTile; };
  auto tile_z = [&](int s) { return tile_u(s) + 2 * kTile; };
  auto tile_B = [&](int s) { return tile_u(s) + 3 * kTile; };
  auto tile_C = [&](int s) { return tile_u(s) + 3 * kTile + kBC; };
  // activation tile: kNBox boxes of kChBox channels side by side
  auto load_act = [&](Act* dst, const CUtensorMap* m, uint64_t* bar, int d0, int row) {
#pragma unroll
    for (int bx = 0; bx < AT::kNBox; ++bx)
      tma_load_2d(reinterpret_cast<unsigned char*>(dst) + bx * (kTT * AT::kRowB), m, bar, d0 + bx * AT::kChBox, row);
  };

  if (warp == 4) {
    // ---------------- producer
    if (lane == 0) {
      tma_prefetch_desc(&P.map_u);
      tma_prefetch_desc(&P.map_raw);
      if (kGate) tma_prefetch_desc(&P.map_z);
      tma_prefetch_desc(&P.map_B);
      tma_prefetch_desc(&P.map_C);
      constexpr bool kZ = kGate && !kAgg;
      const uint32_t bytes = (uint32_t)(((kZ ? 3 : 2) * kTile + (kAgg ? 1 : 2) * kBC) * sizeof(Act));
      int issued = 0;  // tiles issued over all items
      bool ok = true;
      for (int u = u_begin; u < u_end && ok;) {
        const Item it = item_at(u);
        u = it.next;
        const int ntiles = (it.t_end - it.t_begin + kTT - 1) / kTT;
        for (int k = 0; k < ntiles; ++k) {
          const int s = issued % S;
          const uint32_t use = (uint32_t)(issued / S);
          if (issued >= S && !mbar_wait(&empty[s], (use - 1) & 1, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], bytes);
          const int row = it.b * L + it.t_begin + k * kTT;
          load_act(tile_u(s), &P.map_u, &full[s], it.d0, row);
          load_act(tile_raw(s), &P.map_raw, &full[s], it.d0, row);
          if (kZ) load_act(tile_z(s), &P.map_z, &full[s], it.d0, row);
          tma_load_2d(tile_B(s), &P.map_B, &full[s], 0, row);
          if (!kAgg) tma_load_2d(tile_C(s), &P.map_C, &full[s], 0, row);
          ++issued;
        }
      }
      // never leave with copies in flight: wait for the last use of every stage
      for (int s = 0; s < S && s < issued; ++s) {
        const int k_last = s + S * ((issued - 1 - s) / S);
        mbar_wait(&full[s], (uint32_t)(k_last / S) & 1, p.status);
      }
    }
    return;
  }
  // ---------------- consumers
  const int q = tid % TPC;    // state group: states 4q .. 4q+3
  const int cl = tid / TPC;   // channel within the tile
  // swizzled offsets of this lane's channel in the rows of its owned steps
  // (minus the row's own offset; the pattern repeats every 8 rows)
  int colo[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) colo[j] = AT::col(j * TPC + q, cl);

  // A wait that gives up marks the CTA failed (status word set); the
  // consumers then skip every later wait but keep the same control flow, so
  // that every named barrier is still reached by all of them.
  int kt = 0;  // tiles over all items
  bool failed = false;
  for (int u = u_begin; u < u_end;) {
  const Item it = item_at(u);
  u = it.next;
  const int b = it.b, t_begin = it.t_begin, t_end = it.t_end;
  const int ntiles = (t_end - t_begin + kTT - 1) / kTT;
  const int d = it.d0 + cl;
  const bool dvalid = d < D;
  const int dc = dvalid ? d : D - 1;
  const float* hin;  // initial state: zero (aggregate pass), handed over, the composed segment start, or h0
  if (kAgg) {
    hin = nullptr;
  } else if (kStream && !it.first) {
    // stream mode: the state at t_begin comes from the CTA walking the sequence's first piece
    if (lane == 0 && !failed) failed = !flag_wait(p.seq_flag + it.sq, p.status);
    failed = __shfl_sync(0xffffffffu, failed, 0);
    __syncwarp();
    hin = p.seq_carry + ((size_t)it.sq * kCh + cl) * N;
  } else if (!kStream && p.nseg > 1) {
    hin = p.seg_start + (((size_t)b * p.nseg + blockIdx.z) * D + dc) * N;
  } else {
    hin = p.h0 ? p.h0 + ((size_t)b * D + dc) * N : nullptr;
  }
  float2 A2[2], h[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int n = 4 * q + 2 * i;
    const float a0 = -expf(p.A_log[dc * N + n]);
    const float a1 = -expf(p.A_log[dc * N + n + 1]);
    A2[i] = kFast ? make_float2(a0 * kLog2e, a1 * kLog2e) : make_float2(a0, a1);
    h[i] = hin ? make_float2(__ldcg(hin + n), __ldcg(hin + n + 1)) : make_float2(0.f, 0.f);
  }
  const float bias = p.delta_bias[dc];
  const float Dd = p.Dp[dc];
  Act* outp = static_cast<Act*>(p.out) + (size_t)b * L * D + d;
  float dsum = 0.f;  // aggregate pass: sum of delta over the segment (per-tile partials added)

  for (int k = 0; k < ntiles; ++k, ++kt) {
    const int s = kt % S;
    const uint32_t par = (uint32_t)(kt / S) & 1;
    if (!failed) failed = !mbar_wait(&full[s], par, p.status);
    const int tbase = t_begin + k * kTT;
    const int cnt = min(kTT, t_end - tbase);
    if (kSave && !kAgg && (tbase % kChunk) == 0 && dvalid) {
      float* cs = p.chunk_states + (((size_t)b * p.nchunks + tbase / kChunk) * D + d) * N + 4 * q;
      *reinterpret_cast<float4*>(cs) = make_float4(h[0].x, h[0].y, h[1].x, h[1].y);
    }
    const unsigned char* su = reinterpret_cast<const unsigned char*>(tile_u(s));
    const unsigned char* sr = reinterpret_cast<const unsigned char*>(tile_raw(s));
    const unsigned char* sz = reinterpret_cast<const unsigned char*>(tile_z(s));
    // activation at (tile row kr, this lane's channel); i = owned-step index when kr is that step
    auto act_at = [&](const unsigned char* t, int kr, int i, bool exact) {
      const int o = exact ? kr * AT::kRowB + colo[i % kPer] : AT::off(kr, cl);
      return lds_act(reinterpret_cast<const Act*>(t + o));
    };
    // Bm / Cm of the lane's 4 states in step kk: one 16-byte (f32) or 8-byte
    // (bf16, widened exactly) shared-memory read
    const Act* Bt = tile_B(s) + 4 * q;
    const Act* Ct = tile_C(s) + 4 * q;
    auto ld4 = [&](const Act* row) -> float4 {
      if constexpr (kBf16) {
        const uint2 r = *reinterpret_cast<const uint2*>(row);
        return make_float4(__uint_as_float(r.x << 16), __uint_as_float(r.x & 0xffff0000u),
                           __uint_as_float(r.y << 16), __uint_as_float(r.y & 0xffff0000u));
      } else {
        return *reinterpret_cast<const float4*>(row);
      }
    };

    // one recurrence step for this lane's 4 states; the partial readout goes to ypart
    float tsum = 0.f;
    auto step = [&](int kk) {
      const float2 dv = prep[kk * kPrepRow + cl];
      const float2 dd = make_float2(dv.x, dv.x);
      const float2 uu = make_float2(dv.y, dv.y);
      const float4 Bv = ld4(Bt + kk * N);
      const float2 a0 = decay2<kFast>(dd, A2[0]);
      const float2 a1 = decay2<kFast>(dd, A2[1]);
      h[0] = ffma2(a0, h[0], fmul2(uu, make_float2(Bv.x, Bv.y)));
      h[1] = ffma2(a1, h[1], fmul2(uu, make_float2(Bv.z, Bv.w)));
      if (kAgg) {
        tsum += dv.x;
      } else {
        const float4 Cv = ld4(Ct + kk * N);
        const float2 y2 = ffma2(make_float2(Cv.z, Cv.w), h[1], fmul2(make_float2(Cv.x, Cv.y), h[0]));
        ypart[kk * kYRow + tid] = y2.x + y2.y;
      }
    };
    // One tile in three phases.  kFull (all kTT steps valid, the common case)
    // has no data-dependent branches, so the independent iterations of each
    // phase overlap; the last, partial tile takes the guarded version.
    auto run_tile = [&](auto full_tag) {
      constexpr bool kFull = decltype(full_tag)::value;
      const int n_valid = kFull ? kTT : cnt;
      // phase 1: (delta, delta*u) of the owned steps (k % TPC == q); steps past
      // the end get (0, 0), which leaves the state unchanged (Abar = 1, input 0)
      float2 pv[kOwn];
#pragma unroll
      for (int i = 0; i < kOwn; ++i) {
        const int km = i * TPC + q;
        const int kr = kFull ? km : min(km, n_valid - 1);
        const float sp = clamp_dt(softplus_k<kFast>(act_at(sr, kr, i, kFull) + bias), p.dt_min, p.dt_max);
        pv[i] = make_float2(sp, sp * act_at(su, kr, i, kFull));
        if (!kFull && km >= n_valid) pv[i] = make_float2(0.f, 0.f);
      }
#pragma unroll
      for (int i = 0; i < kOwn; ++i) prep[(i * TPC + q) * kPrepRow + cl] = pv[i];
      __syncwarp();
      // phase 2: the recurrence; only h is carried from step to step
      if (kFull) {
#pragma unroll
        for (int kk = 0; kk < kTT; ++kk) step(kk);
      } else {
        for (int kk = 0; kk < n_valid; ++kk) step(kk);
      }
      if (kAgg) return;
      __syncwarp();
      // phase 3: complete the readout of the owned steps (fixed order over the
      // channel's TPC lanes), add Dp*u, gate with silu(z), store
      float ov[kOwn];
#pragma unroll
      for (int i = 0; i < kOwn; ++i) {
        const int km = i * TPC + q;
        const int kr = kFull ? km : min(km, n_valid - 1);
        const float* yp = ypart + kr * kYRow + cl * TPC;
        float y = yp[0];
#pragma unroll
        for (int r = 1; r < TPC; ++r) y += yp[r];
        float o = fmaf(Dd, act_at(su, kr, i, kFull), y);
        if (kGate) o *= silu_k<kFast>(act_at(sz, kr, i, kFull));
        ov[i] = o;
      }
#pragma unroll
      for (int i = 0; i < kOwn; ++i) {
        const int km = i * TPC + q;
        if (dvalid && (kFull || km < n_valid)) st_act(outp + (size_t)(tbase + km) * D, ov[i]);
      }
    };
    if (cnt == kTT)
      run_tile(std::true_type{});
    else
      run_tile(std::false_type{});
    dsum += tsum;
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  if (kAgg) {
    if (dvalid) {
      // decay product over the segment, exp(A * sum(delta)), and the end state from zero
      float* ag = p.seg_agg + ((((size_t)b * p.nseg + blockIdx.z) * D + d) * N + 4 * q) * 2;
      const float2 x0 = fmul2(make_float2(dsum, dsum), A2[0]);
      const float2 x1 = fmul2(make_float2(dsum, dsum), A2[1]);
      const float P0 = kFast ? ex2_approx(x0.x) : expf(x0.x), P1 = kFast ? ex2_approx(x0.y) : expf(x0.y);
      const float P2 = kFast ? ex2_approx(x1.x) : expf(x1.x), P3 = kFast ? ex2_approx(x1.y) : expf(x1.y);
      reinterpret_cast<float4*>(ag)[0] = make_float4(P0, h[0].x, P1, h[0].y);
      reinterpret_cast<float4*>(ag)[1] = make_float4(P2, h[1].x, P3, h[1].y);
    }
  } else if (p.h_last && dvalid && it.last) {
    float* hl = p.h_last + ((size_t)b * D + d) * N + 4 * q;
    *reinterpret_cast<float4*>(hl) = make_float4(h[0].x, h[0].y, h[1].x, h[1].y);
  }
  if (kStream && !it.last) {
    // stream mode, the sequence's first piece: hand the state at t_end over
    float* co = p.seq_carry + ((size_t)it.sq * kCh + cl) * N + 4 * q;
    __stcg(co, h[0].x);
    __stcg(co + 1, h[0].y);
    __stcg(co + 2, h[1].x);
    __stcg(co + 3, h[1].y);
    __threadfence();
    named_bar_sync(1, kScanThreads);
    if (tid == 0) st_release_gpu(p.seq_flag + it.sq, 1);
  }
  }  // items
}

// Carry pass of the chunked parallel scan: per (b, d, n), in segment order,
// seg_start[s] = state before segment s, seg_start[s+1] = P_s * seg_start[s] + hloc_s.
__global__ void s6_fwd_seg_carry_kernel(const FwdParams p) {
  const size_t per = (size_t)p.D * p.N;
  const size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int b = blockIdx.y;
  if (e >= per) return;
  float h = p.h0 ? p.h0[(size_t)b * per + e] : 0.f;
  for (int sg = 0; sg < p.nseg; ++sg) {
    p.seg_start[((size_t)b * p.nseg + sg) * per + e] = h;
    if (sg + 1 < p.nseg) {
      const float* ag = p.seg_agg + (((size_t)b * p.nseg + sg) * per + e) * 2;
      h = fmaf(ag[0], h, ag[1]);
    }
  }
}

// ---------------------------------------------------------------- host side

// 2D map over a row-major [rows][cols] tensor, box [box_rows][box_cols].
bool make_map(CUtensorMap* m, const void* base, int act, uint64_t rows, uint64_t cols, uint32_t box_rows,
              uint32_t box_cols, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE) {
  const uint64_t e = act == SSM_BF16 ? 2 : 4;
  const uint64_t dims[2] = {cols, rows};
  const uint64_t strides[1] = {cols * e};
  const uint32_t box[2] = {box_cols, box_rows};
  return encode_tile_map(m, base, act == SSM_BF16, 2, dims, strides, box, swizzle);
}

template <typename Act, int TPC>
constexpr size_t fwd_smem_bytes() {
  constexpr int kCh = kScanThreads / TPC, S = FwdCfg<Act>::kStages;
  return (size_t)S * FwdCfg<Act>::template stage_bytes<TPC>() + (size_t)kTT * (kCh + 4) * 8 +
         (size_t)kTT * (kScanThreads + 1) * 4 + 2 * S * 8;
}

template <typename Act, int TPC, bool kSave, bool kFast, bool kGate, bool kAgg>
cudaError_t launch_kernel(const FwdTmaParams& P, int nz, cudaStream_t stream) {
  auto kern = s6_fwd_tma_kernel<Act, TPC, kSave, kFast, kGate, kAgg>;
  constexpr size_t smem = fwd_smem_bytes<Act, TPC>();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  constexpr int kCh = kScanThreads / TPC;
  const dim3 grid((P.p.D + kCh - 1) / kCh, P.p.B, nz);
  kern<<<grid, kFwdWarps * 32, smem, stream>>>(P);
  return cudaGetLastError();
}

// Stream mode: the plan's P CTAs, exactly three per SM (the shared memory
// request is raised so that a fourth does not fit), launched cooperatively so
// that all are resident while they hand states over.  Returns
// cudaErrorCooperativeLaunchTooLarge when this GPU cannot hold them.
constexpr size_t kStreamSmemFloor = 60 * 1024;
template <typename Act, int TPC, bool kSave, bool kFast, bool kGate>
cudaError_t launch_stream(const FwdTmaParams& P, cudaStream_t stream) {
  auto kern = s6_fwd_tma_kernel<Act, TPC, kSave, kFast, kGate, false, true>;
  const size_t smem = std::max<size_t>(fwd_smem_bytes<Act, TPC>(), kStreamSmemFloor);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kFwdWarps * 32, smem);
  if (e != cudaSuccess) return e;
  const int sms = device_sm_count();
  if (per_sm != 3 || (long long)per_sm * sms < P.p.plan.P) return cudaErrorCooperativeLaunchTooLarge;
  e = cudaMemsetAsync(P.p.seq_flag, 0, sizeof(int) * (size_t)P.p.B * P.p.plan.ndt, stream);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)P.p.plan.P);
  cfg.blockDim = dim3(kFwdWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, P);
}

template <typename Act, int TPC, bool kSave, bool kFast, bool kGate>
cudaError_t launch_one(const FwdTmaParams& P, cudaStream_t stream) {
  if (P.p.plan.handover && P.p.seq_flag) {
    const cudaError_t e = launch_stream<Act, TPC, kSave, kFast, kGate>(P, stream);
    if (e != cudaErrorCooperativeLaunchTooLarge) return e;
    (void)cudaGetLastError();  // not three resident per SM here: the grid mode gives the same result
    note_plan_fallback();
  }
  if (P.p.nseg > 1) {
    // chunked parallel scan: segment aggregates -> carries -> all segments at once
    cudaError_t e = launch_kernel<Act, TPC, false, kFast, kGate, true>(P, P.p.nseg - 1, stream);
    if (e != cudaSuccess) return e;
    const dim3 cgrid((unsigned)(((size_t)P.p.D * P.p.N + 255) / 256), P.p.B);
    s6_fwd_seg_carry_kernel<<<cgrid, 256, 0, stream>>>(P.p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return launch_kernel<Act, TPC, kSave, kFast, kGate, false>(P, P.p.nseg, stream);
}

template <typename Act, int TPC, bool kFast>
cudaError_t launch_tpc(const FwdTmaParams& P, cudaStream_t stream) {
  const bool save = P.p.chunk_states != nullptr, gate = P.p.z != nullptr;
  if (save)
    return gate ? launch_one<Act, TPC, true, kFast, true>(P, stream) : launch_one<Act, TPC, true, kFast, false>(P, stream);
  return gate ? launch_one<Act, TPC, false, kFast, true>(P, stream) : launch_one<Act, TPC, false, kFast, false>(P, stream);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace


// Stream plan: 3 * sms equal ranges of chunk units over the (batch,
// 128/TPC-channel tile) sequences.  Taken when some sequence is cut, none
// more than once, and no range is shorter than a sequence (so the first
// piece of a cut sequence is done before its last piece is reached); the
// grid mode's tail wave (sequences not a multiple of the resident CTAs) then
// disappears.
FwdPlan fwd_stream_plan(int B, int L, int D, int N, int act, int sms) {
  FwdPlan pl;
  pl.handover = false;
  pl.maxp = 1;
  pl.H = 0;  // contiguous layout
  pl.P = 1;
  pl.U = 1;
  pl.nch = L > 0 ? (L + kChunk - 1) / kChunk : 0;
  if (!(N == 4 || N == 8 || N == 16) || (act == SSM_BF16 && N == 4) || B <= 0 || D <= 0 || pl.nch == 0) return pl;
  const int kch = kScanThreads / (N / 4);
  pl.ndt = (D + kch - 1) / kch;
  const long long U = (long long)B * pl.ndt * pl.nch;
  const int P = 3 * sms;
  if (U < P || U >= (1LL << 31)) return pl;
  pl.U = U;
  pl.P = P;
  const long long nseq = (long long)B * pl.ndt;
  for (long long sq = 0; sq < nseq; ++sq) pl.maxp = std::max(pl.maxp, plan_pieces(pl, sq));
  pl.handover = pl.maxp == 2 && (long long)pl.nch <= pl.U / pl.P;
  // only worth it when the grid mode has a tail wave: sequences not a
  // multiple of the four resident CTAs per SM
  if (nseq % (4LL * sms) == 0) pl.handover = false;
  return pl;
}

// Segments are used when the (batch x channel-tile) grid alone would leave
// most SMs idle: enough segments for about three CTAs per SM, each at least
// 512 steps long (a multiple of the chunk length).
int fwd_segments(int B, int L, int D, int N, int sms) {
  if (!(N == 4 || N == 8 || N == 16) || L < 1024 || B <= 0 || D <= 0) return 1;
  const int kch = kScanThreads / (N / 4);
  const long ctas = (long)B * ((D + kch - 1) / kch);
  const long want = 3L * sms;
  if (ctas * 2 >= want) return 1;
  long nseg = (want + ctas - 1) / ctas;
  nseg = std::min<long>(nseg, L / 512);
  if (nseg < 2) return 1;
  const int seg_len = (int)((((long)L + nseg - 1) / nseg + kChunk - 1) / kChunk * kChunk);
  return (L + seg_len - 1) / seg_len;
}

// The TMA path covers N in {4, 8, 16} with N*e and D*e multiples of 16 bytes
// and 16-byte aligned activation pointers; everything else takes the generic
// kernel.  bf16 activations use the SFU exp/log (ex2/lg2.approx); f32
// activations keep expf/log1pf.
bool fwd_tma_supported(const FwdParams& p, int act) {
  const int e = act == SSM_BF16 ? 2 : 4;
  if (!(p.N == 4 || p.N == 8 || p.N == 16)) return false;
  if ((p.N * e) % 16 != 0 || (p.D * e) % 16 != 0) return false;
  if (!aligned16(p.u) || !aligned16(p.delta_raw) || !aligned16(p.Bm) || !aligned16(p.Cm)) return false;
  if (p.z && !aligned16(p.z)) return false;
  if (p.chunk_states && !aligned16(p.chunk_states)) return false;
  if (p.h_last && !aligned16(p.h_last)) return false;
  if (p.h0 && (reinterpret_cast<uintptr_t>(p.h0) & 7)) return false;
  return tensor_map_encoder() != nullptr;
}

cudaError_t launch_fwd_tma(const FwdParams& p, int act, cudaStream_t stream) {
  FwdTmaParams P;
  memset(&P, 0, sizeof(P));
  P.p = p;
  const int tpc = p.N / 4;
  const uint32_t kch = (uint32_t)(kScanThreads / tpc);
  const uint64_t rows = (uint64_t)p.B * p.L;
  // activation boxes: rows of min(kch * e, 128) bytes with the swizzle of that width
  const uint32_t e = act == SSM_BF16 ? 2 : 4;
  const uint32_t row_b = std::min<uint32_t>(kch * e, 128);
  const uint32_t abox = row_b / e;
  const CUtensorMapSwizzle sw = swizzle_for_row_bytes((int)row_b);
  bool ok = make_map(&P.map_u, p.u, act, rows, p.D, kTT, abox, sw) &&
            make_map(&P.map_raw, p.delta_raw, act, rows, p.D, kTT, abox, sw) &&
            make_map(&P.map_B, p.Bm, act, rows, p.N, kTT, p.N) &&
            make_map(&P.map_C, p.Cm, act, rows, p.N, kTT, p.N);
  if (p.z) ok = ok && make_map(&P.map_z, p.z, act, rows, p.D, kTT, abox, sw);
  if (!ok) return cudaErrorInvalidValue;
  if (act == SSM_BF16) {
    if (tpc == 4) return launch_tpc<__nv_bfloat16, 4, true>(P, stream);
    if (tpc == 2) return launch_tpc<__nv_bfloat16, 2, true>(P, stream);
    return cudaErrorInvalidValue;
  }
  if (tpc == 4) return launch_tpc<float, 4, false>(P, stream);
  if (tpc == 2) return launch_tpc<float, 2, false>(P, stream);
  if (tpc == 1) return launch_tpc<float, 1, false>(P, stream);
  return cudaErrorInvalidValue;
}

}  // namespace s6
