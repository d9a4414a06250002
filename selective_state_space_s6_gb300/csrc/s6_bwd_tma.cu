// S6 backward, TMA-pipelined (sm_103a).
//
// CTA = (64-channel tile, batch, time segment), 2*TPC + 3 warps: 2*TPC
// consumer warps (TPC = N/4 lanes per channel, 4 states per lane), a TMA
// producer warp, a converter warp (bf16: Bm/Cm tiles widened to f32 once per
// tile) and a reducer warp (cross-warp sums of the dBm/dCm terms).
//
// Each lane walks its chunks (SSM_CHUNK_LEN = 64 steps, restarted from the
// forward's chunk states) from last to first.  The producer streams each
// chunk twice through an S-stage ring of 32-step tiles:
//   pass A (tiles in forward order; delta_raw, u, Bm): recompute h from the
//     chunk state, store (delta, delta*u) in shared memory for the chunk and
//     every state of the chunk in tensor memory (TMEM: 64 steps x 4 states
//     per lane, 8 steps per 32-column store);
//   pass B (tiles in reverse order; all inputs): for each 8-step sub-chunk,
//     last first, load its 8 states from TMEM into registers, then step
//     backward with the adjoint g_t = dy_t*C_t + Abar_{t+1}*g_{t+1}, producing
//     du, d_delta_raw, dz and the dBm/dCm/dA_log/dDp/d_delta_bias terms.
// (The second read of a chunk's tiles comes from L2.)
//
// Per step, the channel sums of the dBm and dCm terms over the CTA's 64
// channels are taken in shared memory in a fixed order (within a warp: 4
// channels per lane with packed adds, then an xor butterfly over the lane
// groups; then the warps in ascending order) and stored as one partial per
// CTA; the sums over t of the parameter terms stay in registers per chunk
// and are added into per-lane totals with a compensated (Kahan) add.  A small
// kernel adds the partials in ascending tile / batch order (s6_bwd.cu).  No
// floating-point atomics: results are bit-identical from run to run (the
// single-writer, fixed-order policy of deterministic_backward.py).
//
// Work that depends only on (t, d) -- softplus, the gate's sigmoid, dy, the
// softplus derivative, the outputs du / d_delta_raw / dz -- is done for step
// k by lane k % TPC of the channel and shared through shared memory.
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

constexpr int kTT = 32;           // steps per tile
constexpr int kAggWarps = 6;  // aggregate pass: 4 consumer warps + producer + converter
template <typename Act>
struct BwdStages {
  static constexpr int value = std::is_same<Act, float>::value ? 2 : 3;
};
// Warp-local reduction scratch of one step: two blocks (dBm terms, dCm terms),
// each holding one 16-byte chunk (a lane's 4 states) per lane in lane order,
// padded to 144 floats so that the 64-bit reads of a half-warp hit distinct
// banks.  Two step slots per warp.
constexpr int kRedBlock = 32 * 4 + 16;
constexpr int kRedSlot = 2 * kRedBlock;
constexpr int kRedSlots = 2;

struct BwdTmaParams {
  CUtensorMap map_u, map_raw, map_z, map_dout, map_B, map_C;
  BwdParams p;
};

__device__ __forceinline__ void kahan_add(float& sum, float& comp, float x) {
  const float y = __fsub_rn(x, comp);
  const float t = __fadd_rn(sum, y);
  comp = __fsub_rn(__fsub_rn(t, sum), y);
  sum = t;
}

// Row stride (float2) of the per-step channel arrays dbuf / bprep: 64 + 4, so
// that consecutive rows (read at once by the lanes of a channel, which own
// consecutive steps) start 32 bytes apart in the banks: a half-warp's 64-bit
// accesses (4 channels x 4 rows) then fill the 32 banks once.
constexpr int kRow = kDTile + 4;

// activation at a byte offset of a (swizzled) tile
template <typename Act>
__device__ __forceinline__ float lds_at(const Act* tile, int byte_off) {
  return lds_act(reinterpret_cast<const Act*>(reinterpret_cast<const unsigned char*>(tile) + byte_off));
}

// TPC lanes per channel, 4 states per lane (N = 4 * TPC); a CTA covers 64
// channels with 64 * TPC consumer threads (2 * TPC warps), plus a producer
// and a converter warp.  kLimit: delta is clamped to [dt_min, dt_max] (a
// separate instance, so the unlimited scan pays nothing for it).
template <typename Act, int TPC, bool kFast, bool kGate, bool kLimit>
__global__ void __launch_bounds__((2 * TPC + 3) * 32, 1) s6_bwd_tma_kernel(const __grid_constant__ BwdTmaParams P) {
  constexpr int N = 4 * TPC;
  constexpr int kLanes = kDTile * TPC;  // consumer threads
  constexpr int kCW = kLanes / 32;      // consumer warps
  constexpr int kTile = kTT * kDTile;
  constexpr int kBC = kTT * N;
  constexpr bool kBf16 = std::is_same<Act, __nv_bfloat16>::value;
  constexpr int kStageElems = 4 * kTile + 2 * kBC;
  constexpr int S = BwdStages<Act>::value;
  constexpr int kBst = kBf16 ? 2 * N : N;  // f32 row stride of the B (and C) rows
  constexpr int kOwnA = kTT / TPC;         // pass-A steps a lane owns per tile
  constexpr int kOwnB = kSub / TPC;        // pass-B steps a lane owns per sub-chunk
  // per-step rows of the lanes' partial sums, one float4 of padding: the TPC
  // lanes of a channel read rows k, k+1, .. at once, 16 bytes apart in the banks
  constexpr int kPartRow = kLanes + 1;
  constexpr uint32_t kTmemCols = 512;
  static_assert(kCW <= 8, "two consumer warps per TMEM lane quarter at most");
  using AT = SwzTile<Act, kDTile, kTT>;  // u, delta_raw, z, dout tiles (128-byte rows)
  constexpr int kRB = AT::kRowB;

  extern __shared__ __align__(1024) unsigned char smem[];
  Act* stages = reinterpret_cast<Act*>(smem);
  float* bcf = reinterpret_cast<float*>(smem + (size_t)S * kStageElems * sizeof(Act));  // [S][TT][2][N] (bf16)
  float2* dbuf = reinterpret_cast<float2*>(bcf + (kBf16 ? S * kTT * 2 * N : 0));       // [kChunk][kRow] (delta, delta*u)
  float4* hc0 = reinterpret_cast<float4*>(dbuf + kChunk * kRow);   // [kLanes] state at the chunk start
  float* redw = reinterpret_cast<float*>(hc0 + kLanes);            // [kCW][kRedSlots][kRedSlot]
  float* wpart = redw + kCW * kRedSlots * kRedSlot;                // [2][kSub][kCW][32]
  float4* part = reinterpret_cast<float4*>(wpart + 2 * kSub * kCW * 32);  // [kSub][kPartRow] (y, gB, Ap, -)
  float2* bprep = reinterpret_cast<float2*>(part + kSub * kPartRow);      // [kSub][kRow] (dy, dz factor)
  float* tot = reinterpret_cast<float*>(bprep + kSub * kRow);             // [2 (sum, comp)][kLanes][6]
  uint64_t* full = reinterpret_cast<uint64_t*>(tot + 2 * kLanes * 6);
  uint64_t* conv = full + S;
  uint64_t* empty = conv + S;
  uint64_t* wfull = empty + S;  // [2] wpart slot written by every consumer warp
  uint64_t* wempty = wfull + 2; // [2] wpart slot summed by the reducer warp
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(wempty + 2);

  const BwdParams& p = P.p;
  // the swizzled tiles need 1024-byte aligned stages (uniform: the whole CTA leaves)
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.status, kStatusLayout);
    return;
  }
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int L = p.L, D = p.D;
  const int nchunks = p.nchunks;
  // this CTA's range of chunk units; every role walks its pieces in unit
  // order: piece = sequence sq (batch sq / ndt, channel tile sq % ndt),
  // chunks [c_lo, c_hi)
  const BwdPlan& pl = p.plan;
  // (the plan keeps U below 2^31, so unit indices fit an int)
  const int u_begin = (int)plan_bound(pl, blockIdx.x), u_end = (int)plan_bound(pl, blockIdx.x + 1);

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&conv[s], 32);
      mbar_init(&empty[s], kCW);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&wfull[i], kCW);
      mbar_init(&wempty[i], 1);
    }
    fence_mbar_init();
  }
  // TMEM holds every state of the chunk being processed: per consumer warp
  // 256 columns (64 steps x 4 states) of its 32 lanes; warps w and w + 4
  // share a lane quarter and take columns 0..255 / 256..511
  if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();

  auto tile_u = [&](int s) { return stages + (size_t)s * kStageElems; };
  auto tile_raw = [&](int s) { return stages + (size_t)s * kStageElems + kTile; };
  auto tile_z = [&](int s) { return stages + (size_t)s * kStageElems + 2 * kTile; };
  auto tile_g = [&](int s) { return stages + (size_t)s * kStageElems + 3 * kTile; };
  auto tile_B = [&](int s) { return stages + (size_t)s * kStageElems + 4 * kTile; };
  auto tile_C = [&](int s) { return stages + (size_t)s * kStageElems + 4 * kTile + kBC; };

  // activation tile: AT::kNBox boxes of AT::kChBox channels side by side
  auto load_act = [&](Act* dst, const CUtensorMap* m, uint64_t* bar, int d0, int row) {
#pragma unroll
    for (int bx = 0; bx < AT::kNBox; ++bx)
      tma_load_2d(reinterpret_cast<unsigned char*>(dst) + bx * AT::kBoxBytes, m, bar, d0 + bx * AT::kChBox, row);
  };

  // The item sequence every role walks: for each piece, for chunk c =
  // last..first of the piece, with ntl tiles: pass A tiles 0..ntl-1, then
  // pass B tiles ntl-1..0.
  auto chunk_tiles = [&](int c) { return (min(kChunk, L - c * kChunk) + kTT - 1) / kTT; };
  auto piece_at = [&](int u, int& b, int& d0, int& c_lo, int& c_hi, int& next) {
    const int sq = u / pl.nch, S0 = sq * pl.nch;
    next = min(S0 + pl.nch, u_end);
    b = sq / pl.ndt;
    d0 = (sq % pl.ndt) * kDTile;
    c_lo = u - S0;
    c_hi = next - S0;
  };

  if (warp == kCW) {
    // ---------------- producer
    if (lane == 0) {
      tma_prefetch_desc(&P.map_u);
      tma_prefetch_desc(&P.map_raw);
      tma_prefetch_desc(&P.map_dout);
      if (kGate) tma_prefetch_desc(&P.map_z);
      tma_prefetch_desc(&P.map_B);
      tma_prefetch_desc(&P.map_C);
      const uint32_t bytesA = (uint32_t)((2 * kTile + kBC) * sizeof(Act));
      const uint32_t bytesB = (uint32_t)(((kGate ? 4 : 3) * kTile + 2 * kBC) * sizeof(Act));
      int item = 0;
      bool ok = true;
      for (int u = u_begin, next; u < u_end && ok; u = next) {
        int b, d0, c_lo, c_hi;
        piece_at(u, b, d0, c_lo, c_hi, next);
        for (int c = c_hi - 1; c >= c_lo && ok; --c) {
          const int ntl = chunk_tiles(c);
          for (int it = 0; it < 2 * ntl; ++it, ++item) {
            const bool passA = it < ntl;
            const int j = passA ? it : 2 * ntl - 1 - it;
            const int s = item % S;
            const uint32_t use = (uint32_t)(item / S);
            if (item >= S && !mbar_wait(&empty[s], (use - 1) & 1, p.status)) {
              ok = false;
              break;
            }
            const int row = b * L + c * kChunk + j * kTT;
            mbar_arrive_expect_tx(&full[s], passA ? bytesA : bytesB);
            load_act(tile_u(s), &P.map_u, &full[s], d0, row);
            load_act(tile_raw(s), &P.map_raw, &full[s], d0, row);
            tma_load_2d(tile_B(s), &P.map_B, &full[s], 0, row);
            if (!passA) {
              if (kGate) load_act(tile_z(s), &P.map_z, &full[s], d0, row);
              load_act(tile_g(s), &P.map_dout, &full[s], d0, row);
              tma_load_2d(tile_C(s), &P.map_C, &full[s], 0, row);
            }
          }
        }
      }
      // never leave with copies in flight: wait for the last use of every stage
      for (int s = 0; s < S && s < item; ++s) {
        const int k_last = s + S * ((item - 1 - s) / S);
        mbar_wait(&full[s], (uint32_t)(k_last / S) & 1, p.status);
      }
    }
    return;
  }
  if (warp == kCW + 1) {
    // ---------------- converter (bf16): Bm (and Cm in pass B) -> f32
    if (kBf16) {
      int item = 0;
      bool ok = true;
      for (int u = u_begin, next; u < u_end; u = next) {
        int b, d0, c_lo, c_hi;
        piece_at(u, b, d0, c_lo, c_hi, next);
        for (int c = c_hi - 1; c >= c_lo; --c) {
          const int ntl = chunk_tiles(c);
          for (int it = 0; it < 2 * ntl; ++it, ++item) {
            const bool passA = it < ntl;
            const int s = item % S;
            if (ok) ok = mbar_wait(&full[s], (uint32_t)(item / S) & 1, p.status);
            const __nv_bfloat162* tb = reinterpret_cast<const __nv_bfloat162*>(tile_B(s));
            const __nv_bfloat162* tc = reinterpret_cast<const __nv_bfloat162*>(tile_C(s));
            float* dst = bcf + (size_t)s * kTT * 2 * N;
            for (int e = lane; e < kBC / 2; e += 32) {
              const int t = (2 * e) / N, n = (2 * e) % N;
              *reinterpret_cast<float2*>(dst + (t * 2 + 0) * N + n) = __bfloat1622float2(tb[e]);
              if (!passA) *reinterpret_cast<float2*>(dst + (t * 2 + 1) * N + n) = __bfloat1622float2(tc[e]);
            }
            mbar_arrive(&conv[s]);
          }
        }
      }
    }
    return;
  }

  if (warp == kCW + 2) {
    // ---------------- reducer: cross-warp sums of each sub-chunk's dBm/dCm
    // partials (fixed warp order) -> this CTA's partial row in ws_dbc
    int n = 0;
    bool ok = true;
    for (int u = u_begin, next; u < u_end; u = next) {
      int b, d0, c_lo, c_hi;
      piece_at(u, b, d0, c_lo, c_hi, next);
      float* ws_dbc_r = p.ws_dbc + ((size_t)(d0 / kDTile) * p.B + b) * (size_t)L * 2 * N;
      for (int c = c_hi - 1; c >= c_lo; --c) {
        const int clen = min(kChunk, L - c * kChunk);
        for (int j = chunk_tiles(c) - 1; j >= 0; --j) {
          const int cnt = min(kTT, clen - j * kTT);
          for (int sc = (cnt + kSub - 1) / kSub - 1; sc >= 0; --sc, ++n) {
            const int cnt8 = min(kSub, cnt - sc * kSub);
            const int slot = n & 1;
            if (ok) ok = mbar_wait(&wfull[slot], (uint32_t)(n >> 1) & 1, p.status);
            const float* wp = wpart + slot * (kSub * kCW * 32);
            float* dst = ws_dbc_r + (size_t)(c * kChunk + j * kTT + sc * kSub) * 2 * N;
            for (int idx = lane; idx < cnt8 * 2 * N; idx += 32) {
              const int k = idx / (2 * N), o = idx % (2 * N);
              const float* src = wp + k * kCW * 32 + o;
              float v = src[0];
#pragma unroll
              for (int w = 1; w < kCW; ++w) v += src[w * 32];
              dst[idx] = v;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&wempty[slot]);
          }
        }
      }
    }
    return;
  }

  // ---------------- consumers
  const int q = tid % TPC;   // state group: states 4q .. 4q+3
  const int cl = tid / TPC;  // channel within the tile
  // Lane q owns the steps k with k % TPC == q (row % 8 of owned step i of an
  // 8-step group is i*TPC + q): byte offsets of this lane's channel in those
  // rows of a swizzled tile.
  int colo[kOwnB];
#pragma unroll
  for (int i = 0; i < kOwnB; ++i) colo[i] = AT::col(i * TPC + q, cl);

  // A2 = A*log2(e) on the fast path (2^x decays), A itself otherwise; sums
  // weighted by A are taken with A2 and scaled by kAscale = A / A2 at the end.
  constexpr float kAscale = kFast ? kLn2 : 1.f;
  // this warp's TMEM region: column 32*j + 4*k + i = state i of step 8*j + k of the chunk
  const uint32_t tm = *tmem_slot + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)((warp >> 2) * 256);
  float* my_tot = tot + tid * 6;               // running totals: 4 states, dDp, d_delta_bias
  float* my_cmp = tot + kLanes * 6 + tid * 6;  // Kahan compensation

  // warp-local reducer role: output pair op = lane % N (term r_q, states r_n,
  // r_n + 1 of the channel), group r_g = lane / N of 4 channels
  const int r_op = lane % N, r_g = lane / N;
  const int r_q = r_op / (N / 2), r_n = 2 * (r_op % (N / 2));
  const int r_src = r_n / 4, r_j = r_n % 4;  // owning lane-in-channel and index in its chunk
  float* my_redw = redw + warp * kRedSlots * kRedSlot;

  bool failed = false;
  int s = 0;         // ring stage of the current item
  uint32_t par = 0;  // its phase parity
  int nsub_done = 0;  // sub-chunks handed to the reducer so far
  for (int u = u_begin, next; u < u_end; u = next) {
    int b, d0, c_lo, c_hi;
    piece_at(u, b, d0, c_lo, c_hi, next);
    // piece index in time order within its sequence, and whether it ends the sequence
    const int kp = c_lo == 0 ? 0 : (int)(plan_count_le(pl, u) - plan_count_le(pl, u - c_lo));
    const bool last_piece = c_hi == pl.nch;
    const int d = d0 + cl;
    const bool dvalid = d < D;
    const int dc = dvalid ? d : D - 1;
    const int sq = (u - c_lo) / pl.nch;  // sequence index
    if (!last_piece && p.seq_flag) {
      // hand-over mode: the carry comes from the CTA walking the sequence's last piece
      if (lane == 0 && !failed) failed = !flag_wait(p.seq_flag + sq, p.status);
      failed = __shfl_sync(0xffffffffu, failed, 0);
      __syncwarp();
    }
    float2 A2[2], carry[2];
    {
      const float* cin = !last_piece ? p.seg_carry + (((size_t)b * p.nseg + kp) * D + dc) * N
                                     : (p.dh_last ? p.dh_last + ((size_t)b * D + dc) * N : nullptr);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int n = 4 * q + 2 * i;
        const float a0 = -expf(p.A_log[dc * N + n]);
        const float a1 = -expf(p.A_log[dc * N + n + 1]);
        A2[i] = kFast ? make_float2(a0 * kLog2e, a1 * kLog2e) : make_float2(a0, a1);
        // adjoint carry entering the piece's last step: dh_last for the last
        // piece of the sequence, the composed carry of the pieces after it otherwise
        carry[i] = (cin && dvalid) ? make_float2(__ldcg(cin + n), __ldcg(cin + n + 1)) : make_float2(0.f, 0.f);
      }
    }
    const float bias = p.delta_bias[dc];
    const float Dd = p.Dp[dc];
#pragma unroll
    for (int i = 0; i < 6; ++i) {
      my_tot[i] = 0.f;
      my_cmp[i] = 0.f;
    }
    const size_t bd_off = (size_t)b * L * D + d;  // du / d_delta_raw / dz of (b, t = 0, d)
    for (int c = c_hi - 1; c >= c_lo; --c) {
      const int t0 = c * kChunk;
      const int clen = min(kChunk, L - t0);
      const int ntl = (clen + kTT - 1) / kTT;
      float2 accA[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      float accD = 0.f, accBias = 0.f;
      float2 h[2];
      {
        const float4 cs = *reinterpret_cast<const float4*>(p.chunk_states + (((size_t)b * nchunks + c) * D + dc) * N + 4 * q);
        h[0] = make_float2(cs.x, cs.y);
        h[1] = make_float2(cs.z, cs.w);
      }
      for (int it = 0; it < 2 * ntl; ++it) {
        const bool passA = it < ntl;
        const int j = passA ? it : 2 * ntl - 1 - it;
        if (!failed) failed = !mbar_wait(&full[s], par, p.status);
        if (kBf16 && !failed) failed = !mbar_wait(&conv[s], par, p.status);
        __syncwarp();
        const int tb = j * kTT;  // first step of the tile within the chunk
        const int cnt = min(kTT, clen - tb);
        const Act* su = tile_u(s);
        const Act* sr = tile_raw(s);
        const float* Bt = (kBf16 ? bcf + (size_t)s * kTT * 2 * N : reinterpret_cast<const float*>(tile_B(s))) + 4 * q;
        const float* Ct = kBf16 ? Bt + N : reinterpret_cast<const float*>(tile_C(s)) + 4 * q;
        float2* dtile = dbuf + tb * kRow;  // (delta, delta*u) rows of this tile

        if (passA) {
          // ---------- pass A: (delta, delta*u) of the owned steps, then the recurrence
          auto pass_a = [&](auto full_tag) {
            constexpr bool kFull = decltype(full_tag)::value;
            const int nv = kFull ? kTT : cnt;
#pragma unroll
            for (int i = 0; i < kOwnA; ++i) {
              const int km = i * TPC + q;
              const int kr = kFull ? km : min(km, nv - 1);
              const int o = kr * kRB + (kFull ? colo[i % kOwnB] : AT::col(kr, cl));
              const float sv = lds_at(sr, o) + bias;
              const float sp0 = kFast ? softplus_fast(sv) : softplus_f(sv);
              const float sp = kLimit ? clamp_dt(sp0, p.dt_min, p.dt_max) : sp0;
              if (kFull || km < nv) dtile[km * kRow + cl] = make_float2(sp, sp * lds_at(su, o));
            }
            __syncwarp();
            if (tb == 0) hc0[tid] = make_float4(h[0].x, h[0].y, h[1].x, h[1].y);
            // states after each step, 8 steps at a time, then to TMEM
            float hb[4 * kSub];
            auto stepA = [&](int kk) {
              const float2 dv = dtile[kk * kRow + cl];
              const float2 dd = make_float2(dv.x, dv.x), uu2 = make_float2(dv.y, dv.y);
              const float4 Bv = *reinterpret_cast<const float4*>(Bt + kk * kBst);
              h[0] = ffma2(decay2<kFast>(dd, A2[0]), h[0], fmul2(uu2, make_float2(Bv.x, Bv.y)));
              h[1] = ffma2(decay2<kFast>(dd, A2[1]), h[1], fmul2(uu2, make_float2(Bv.z, Bv.w)));
              const int r = 4 * (kk % kSub);
              hb[r] = h[0].x;
              hb[r + 1] = h[0].y;
              hb[r + 2] = h[1].x;
              hb[r + 3] = h[1].y;
            };
#pragma unroll
            for (int kk = 0; kk < kTT; ++kk) {
              if (kFull || kk < nv) stepA(kk);
              // a block with at least one valid step goes out (warp-uniform)
              if ((kk % kSub) == kSub - 1 && (kFull || kk - (kSub - 1) < nv)) tmem_st32(tm + (uint32_t)(4 * (tb + kk - (kSub - 1))), hb);
            }
          };
          if (cnt == kTT)
            pass_a(std::true_type{});
          else
            pass_a(std::false_type{});
        } else {
          // ---------- pass B: 8-step sub-chunks of this tile, last first
          const Act* sz = tile_z(s);
          const Act* sg = tile_g(s);
          const int nsub = (cnt + kSub - 1) / kSub;
          if (it == ntl) tmem_wait_st();  // the chunk's states (pass A) are in TMEM
          for (int sc = nsub - 1; sc >= 0; --sc) {
            const int ks = sc * kSub;  // first step of the sub-chunk within the tile
            const int cnt8 = min(kSub, cnt - ks);
            const int cstep = tb + ks;  // ... within the chunk
            // the state before the sub-chunk: last state of the previous block, or the chunk start
            float hq[4];
            if (cstep > 0) {
              tmem_ld4(tm + (uint32_t)(4 * cstep - 4), hq);
            } else {
              const float4 c0 = hc0[tid];
              hq[0] = c0.x, hq[1] = c0.y, hq[2] = c0.z, hq[3] = c0.w;
            }
            const float2 hstart[2] = {make_float2(hq[0], hq[1]), make_float2(hq[2], hq[3])};
            const float2* dsub = dbuf + cstep * kRow;
            // wpart slot of this sub-chunk: wait until the reducer has summed its previous use
            const int slot = nsub_done & 1;
            if (nsub_done >= 2 && !failed) failed = !mbar_wait(&wempty[slot], (uint32_t)((nsub_done >> 1) - 1) & 1, p.status);
            float* wp_sub = wpart + slot * (kSub * kCW * 32);
            auto sub = [&](auto full_tag) {
              constexpr bool kFull = decltype(full_tag)::value;
              const int nv = kFull ? kSub : cnt8;
              // B1: the sub-chunk's states from TMEM (written by pass A)
              float hv[4 * kSub];
              tmem_ld32(tm + (uint32_t)(4 * cstep), hv);
              float2 hs[kSub][2];
#pragma unroll
              for (int k = 0; k < kSub; ++k) {
                hs[k][0] = make_float2(hv[4 * k], hv[4 * k + 1]);
                hs[k][1] = make_float2(hv[4 * k + 2], hv[4 * k + 3]);
              }
              // B2: gate terms of the owned steps: dy = dout*silu(z), dz factor
#pragma unroll
              for (int i = 0; i < kOwnB; ++i) {
                const int km = i * TPC + q;
                const int kr = ks + (kFull ? km : min(km, nv - 1));
                const int o = kr * kRB + (kFull ? colo[i] : AT::col(kr, cl));
                const float gout = lds_at(sg, o);
                float2 v = make_float2(gout, 0.f);
                if (kGate) {
                  const float zz = lds_at(sz, o);
                  const float sgz = kFast ? sigmoid_fast(zz) : sigmoid_f(zz);
                  v.x = gout * zz * sgz;
                  v.y = gout * sgz * fmaf(zz, 1.f - sgz, 1.f);
                }
                if (!kFull && km >= nv) v = make_float2(0.f, 0.f);
                bprep[km * kRow + cl] = v;
              }
              __syncwarp();
              // B3: reverse steps in pairs; the adjoint carry is the only
              // loop-carried value.  Each step's dBm/dCm terms go to one of two
              // warp-local slots and are summed over the warp's channels after
              // each pair (fixed order) into the per-warp partial wp_sub.
#pragma unroll
              for (int gi = kSub / 2 - 1; gi >= 0; --gi) {
#pragma unroll
                for (int k = 2 * gi + 1; k >= 2 * gi; --k) {
                  if (kFull || k < nv) {
                    const float2 dv = dsub[k * kRow + cl];
                    const float dy = bprep[k * kRow + cl].x;
                    const float2 dd = make_float2(dv.x, dv.x), uu2 = make_float2(dv.y, dv.y);
                    const float2 dy2 = make_float2(dy, dy);
                    const float4 Bv4 = *reinterpret_cast<const float4*>(Bt + (ks + k) * kBst);
                    const float4 Cv4 = *reinterpret_cast<const float4*>(Ct + (ks + k) * kBst);
                    const float2 Bv[2] = {make_float2(Bv4.x, Bv4.y), make_float2(Bv4.z, Bv4.w)};
                    const float2 Cv[2] = {make_float2(Cv4.x, Cv4.y), make_float2(Cv4.z, Cv4.w)};
                    float2 ya = make_float2(0.f, 0.f), gba = make_float2(0.f, 0.f), apa = make_float2(0.f, 0.f);
                    float2 tB[2], tC[2];
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                      const float2 a = decay2<kFast>(dd, A2[i]);
                      const float2 hk = hs[k][i];
                      const float2 hp = k == 0 ? hstart[i] : hs[k > 0 ? k - 1 : 0][i];
                      const float2 g = ffma2(dy2, Cv[i], carry[i]);
                      const float2 ag = fmul2(a, g);   // adjoint carried to step k-1
                      const float2 pv = fmul2(ag, hp); // g * a * h_{k-1}
                      apa = ffma2(A2[i], pv, apa);
                      accA[i] = ffma2(dd, pv, accA[i]);
                      gba = ffma2(g, Bv[i], gba);
                      ya = ffma2(Cv[i], hk, ya);
                      tB[i] = fmul2(g, uu2);
                      tC[i] = fmul2(dy2, hk);
                      carry[i] = ag;
                    }
                    float* rb = my_redw + (k & 1) * kRedSlot;
                    // (channels past D: the tiles' zero fill makes dout and u,
                    // hence dy, g and both terms, exactly 0)
                    *reinterpret_cast<float4*>(rb + lane * 4) = make_float4(tB[0].x, tB[0].y, tB[1].x, tB[1].y);
                    *reinterpret_cast<float4*>(rb + kRedBlock + lane * 4) = make_float4(tC[0].x, tC[0].y, tC[1].x, tC[1].y);
                    part[k * kPartRow + tid] = make_float4(ya.x + ya.y, gba.x + gba.y, (apa.x + apa.y) * kAscale, 0.f);
                  }
                }
                __syncwarp();
                // channel sums of the pair's steps: 4 channels per lane, then across groups
#pragma unroll
                for (int k = 2 * gi + 1; k >= 2 * gi; --k) {
                  if (kFull || k < nv) {
                    const float* rb = my_redw + (k & 1) * kRedSlot + r_q * kRedBlock;
                    float2 v = make_float2(0.f, 0.f);
#pragma unroll
                    for (int k2 = 0; k2 < 4; ++k2) {
                      const int L2 = (r_g * 4 + k2) * TPC + r_src;
                      v = fadd2(v, *reinterpret_cast<const float2*>(rb + L2 * 4 + r_j));
                    }
#pragma unroll
                    for (int m = N; m < 32; m <<= 1)
                      v = fadd2(v, make_float2(__shfl_xor_sync(0xffffffffu, v.x, m), __shfl_xor_sync(0xffffffffu, v.y, m)));
                    // every group holds the identical sum; all store it
                    *reinterpret_cast<float2*>(wp_sub + (k * kCW + warp) * 32 + r_q * N + r_n) = v;
                  }
                }
                __syncwarp();
              }
              // B4: owned steps: combine the channel's partial sums (fixed lane
              // order), write du, d_delta_raw, dz
              float o_du[kOwnB], o_dr[kOwnB], o_dz[kOwnB];
#pragma unroll
              for (int i = 0; i < kOwnB; ++i) {
                const int km = i * TPC + q;
                const int kr = kFull ? km : min(km, nv - 1);
                float4 acc = part[kr * kPartRow + cl * TPC];
#pragma unroll
                for (int r = 1; r < TPC; ++r) {
                  const float4 o = part[kr * kPartRow + cl * TPC + r];
                  acc = make_float4(acc.x + o.x, acc.y + o.y, acc.z + o.z, 0.f);
                }
                const float2 dv = dsub[kr * kRow + cl];
                const float2 bp = bprep[kr * kRow + cl];
                const float uo = lds_at(su, (ks + kr) * kRB + (kFull ? colo[i] : AT::col(kr, cl)));
                // softplus' = sigmoid(s) = 1 - e^{-delta}; zero where the limit
                // clamped delta (delta sits on a bound: a clamped step, or a
                // softplus exactly on it, which has measure zero)
                const bool free_dt = !kLimit || ((dv.x > p.dt_min || p.dt_min <= 0.f) && dv.x < p.dt_max);
                const float dsp = free_dt ? (kFast ? dsoftplus_fast(dv.x) : -expm1f(-dv.x)) : 0.f;
                const float draw = fmaf(uo, acc.y, acc.z) * dsp;
                o_du[i] = fmaf(Dd, bp.x, dv.x * acc.y);
                o_dr[i] = draw;
                o_dz[i] = fmaf(Dd, uo, acc.x) * bp.y;
                const bool ok = kFull || km < nv;
                accD += ok ? bp.x * uo : 0.f;
                accBias += ok ? draw : 0.f;
              }
#pragma unroll
              for (int i = 0; i < kOwnB; ++i) {
                const int km = i * TPC + q;
                if (dvalid && (kFull || km < nv)) {
                  const size_t o = (size_t)(t0 + cstep + km) * D;
                  st_act(static_cast<Act*>(p.du) + bd_off + o, o_du[i]);
                  st_act(static_cast<Act*>(p.d_delta_raw) + bd_off + o, o_dr[i]);
                  if (kGate) st_act(static_cast<Act*>(p.dz) + bd_off + o, o_dz[i]);
                }
              }
            };
            if (cnt8 == kSub)
              sub(std::true_type{});
            else
              sub(std::false_type{});
            // B5: hand the sub-chunk's per-warp partials to the reducer warp
            __syncwarp();
            if (lane == 0) mbar_arrive(&wfull[slot]);
            ++nsub_done;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (++s == S) {
          s = 0;
          par ^= 1;
        }
      }
      // chunk sums -> compensated running totals (per-lane private smem)
      kahan_add(my_tot[0], my_cmp[0], accA[0].x);
      kahan_add(my_tot[1], my_cmp[1], accA[0].y);
      kahan_add(my_tot[2], my_cmp[2], accA[1].x);
      kahan_add(my_tot[3], my_cmp[3], accA[1].y);
      kahan_add(my_tot[4], my_cmp[4], accD);
      kahan_add(my_tot[5], my_cmp[5], accBias);
    }
    // ---------------- the piece's parameter partials (row b * nseg + kp) and dh0
    {
      // dDp and d_delta_bias: each lane summed its owned steps; add the channel's TPC lanes
      float tD = my_tot[4], tBs = my_tot[5];
#pragma unroll
      for (int m = 1; m < TPC; m <<= 1) {
        tD += __shfl_xor_sync(0xffffffffu, tD, m);
        tBs += __shfl_xor_sync(0xffffffffu, tBs, m);
      }
      if (dvalid) {
        float* wp = p.ws_param + (((size_t)b * p.nseg + kp) * D + d) * (N + 2);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int n = 4 * q + 2 * i;
          wp[n] = (A2[i].x * kAscale) * my_tot[2 * i];
          wp[n + 1] = (A2[i].y * kAscale) * my_tot[2 * i + 1];
          if (p.dh0 && c_lo == 0) *reinterpret_cast<float2*>(p.dh0 + ((size_t)b * D + d) * N + n) = carry[i];
        }
        if (q == 0) {
          wp[N] = tD;
          wp[N + 1] = tBs;
        }
        if (p.seq_flag) {
          // rows of pieces this sequence does not have stay zero for the finalize
          for (int k2 = plan_pieces(pl, sq); k2 < p.nseg; ++k2) {
            float* wz = p.ws_param + (((size_t)b * p.nseg + k2) * D + d) * (N + 2);
            wz[4 * q] = wz[4 * q + 1] = wz[4 * q + 2] = wz[4 * q + 3] = 0.f;
            if (q == 0) wz[N] = wz[N + 1] = 0.f;
          }
        }
      }
      if (p.seq_flag && kp > 0) {
        // hand-over mode, the sequence's last piece: its final carry enters the
        // first piece's last step; publish it and raise the flag
        if (dvalid) {
          float* co = p.seg_carry + (((size_t)b * p.nseg + kp - 1) * D + d) * N + 4 * q;
          __stcg(co, carry[0].x);
          __stcg(co + 1, carry[0].y);
          __stcg(co + 2, carry[1].x);
          __stcg(co + 3, carry[1].y);
        }
        __threadfence();
        named_bar_sync(2, kLanes);
        if (tid == 0) st_release_gpu(p.seq_flag + sq, 1);
      }
    }
  }  // pieces
  // every consumer is done with TMEM (loads waited for inline, stores before
  // the loads of the same chunk): free it
  tmem_fence_before_sync();
  named_bar_sync(1, kLanes);
  if (warp == 0) {
    tmem_fence_after_sync();
    tmem_dealloc(*tmem_slot, kTmemCols);
  }
}

// ---------------------------------------------------------------- segment aggregates
// Aggregate pass of the backward's chunked parallel scan.  For segment s >= 1
// (grid.z + 1), from a zero carry, run the adjoint recurrence
//   g_t = dy_t * C_t + carry,  carry = Abar_t * g_t
// from the segment's last step down to its first, and store per state the
// segment's decay product exp(A * sum(delta)) and the final carry.  Same warp
// roles and lane layout as the forward (TPC lanes per channel, 4 states each);
// tiles are streamed last first.
// one aggregate-pass stage: delta_raw, z, dout tiles [kTT][128/TPC] and a Cm
// tile [kTT][N], rounded up to 1024 bytes (the swizzled tiles' alignment)
template <typename Act, int TPC>
constexpr int agg_stage_bytes() {
  return ((3 * kTT * (kScanThreads / TPC) + kTT * 4 * TPC) * (int)sizeof(Act) + 1023) / 1024 * 1024;
}

template <typename Act, int TPC, bool kFast, bool kGate>
__global__ void __launch_bounds__(kAggWarps * 32) s6_bwd_agg_kernel(const __grid_constant__ BwdTmaParams P) {
  constexpr int N = 4 * TPC;
  constexpr int kCh = kScanThreads / TPC;
  constexpr int S = 3;
  constexpr int kTile = kTT * kCh;
  constexpr int kBC = kTT * N;
  constexpr bool kBf16 = std::is_same<Act, __nv_bfloat16>::value;
  constexpr int kStageBytes = agg_stage_bytes<Act, TPC>();
  constexpr int kOwn = kTT / TPC;
  constexpr int kPer = 8 / TPC;      // owned steps per 8 rows (the swizzle period)
  constexpr int kPrepRow = kCh + 4;  // float2 row stride of prep: rows 32 bytes apart in the banks
  using AT = SwzTile<Act, kCh, kTT>;  // delta_raw, z, dout tiles

  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* stages = smem;
  float* cf = reinterpret_cast<float*>(smem + (size_t)S * kStageBytes);  // [S][TT][N] (bf16)
  float2* prep = reinterpret_cast<float2*>(cf + (kBf16 ? S * kTT * N : 0));  // [TT][kPrepRow] (delta, dy)
  uint64_t* full = reinterpret_cast<uint64_t*>(prep + kTT * kPrepRow);
  uint64_t* conv = full + S;
  uint64_t* empty = conv + S;

  const BwdParams& p = P.p;
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.status, kStatusLayout);
    return;
  }
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // channels [d0, d0 + kValid) of the 64-channel tile d0 / kDTile (for
  // TPC = 1 the CTA's 128 lanes cover the tile and the next one, whose
  // lanes only load); piece seg >= 1 of the sequence (b, tile), if it has one
  constexpr int kValid = kCh < kDTile ? kCh : kDTile;
  const int b = blockIdx.y, d0 = blockIdx.x * kValid, seg = blockIdx.z + 1;
  const int L = p.L, D = p.D;
  const long long sq = (long long)b * p.plan.ndt + d0 / kDTile;
  if (seg >= plan_pieces(p.plan, sq)) return;  // the whole CTA, before any barrier or copy
  int c_lo, c_hi;
  plan_piece_range(p.plan, sq, seg, c_lo, c_hi);
  const int t_lo = c_lo * kChunk, t_hi = min(L, c_hi * kChunk);
  const int ntiles = (t_hi - t_lo + kTT - 1) / kTT;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&conv[s], 32);
      mbar_init(&empty[s], 4);
    }
    fence_mbar_init();
  }
  __syncthreads();
  auto tile_raw = [&](int s) { return reinterpret_cast<Act*>(stages + (size_t)s * kStageBytes); };
  auto tile_z = [&](int s) { return tile_raw(s) + kTile; };
  auto tile_g = [&](int s) { return tile_raw(s) + 2 * kTile; };
  auto tile_C = [&](int s) { return tile_raw(s) + 3 * kTile; };
  auto load_act = [&](Act* dst, const CUtensorMap* m, uint64_t* bar, int row) {
#pragma unroll
    for (int bx = 0; bx < AT::kNBox; ++bx)
      tma_load_2d(reinterpret_cast<unsigned char*>(dst) + bx * AT::kBoxBytes, m, bar, d0 + bx * AT::kChBox, row);
  };

  if (warp == 4) {
    if (lane == 0) {
      const uint32_t bytes = (uint32_t)(((kGate ? 3 : 2) * kTile + kBC) * sizeof(Act));
      int issued = 0;
      for (int k = 0; k < ntiles; ++k) {  // k-th tile from the end
        const int s = k % S;
        if (k >= S && !mbar_wait(&empty[s], (uint32_t)(k / S - 1) & 1, p.status)) break;
        mbar_arrive_expect_tx(&full[s], bytes);
        const int row = b * L + t_lo + (ntiles - 1 - k) * kTT;
        load_act(tile_raw(s), &P.map_raw, &full[s], row);
        if (kGate) load_act(tile_z(s), &P.map_z, &full[s], row);
        load_act(tile_g(s), &P.map_dout, &full[s], row);
        tma_load_2d(tile_C(s), &P.map_C, &full[s], 0, row);
        issued = k + 1;
      }
      for (int s = 0; s < S && s < issued; ++s) {
        const int k_last = s + S * ((issued - 1 - s) / S);
        mbar_wait(&full[s], (uint32_t)(k_last / S) & 1, p.status);
      }
    }
    return;
  }
  if (warp == 5) {
    if (kBf16) {
      for (int k = 0; k < ntiles; ++k) {
        const int s = k % S;
        if (!mbar_wait(&full[s], (uint32_t)(k / S) & 1, p.status)) break;
        const __nv_bfloat162* tc = reinterpret_cast<const __nv_bfloat162*>(tile_C(s));
        float* dst = cf + (size_t)s * kTT * N;
        for (int e = lane; e < kBC / 2; e += 32)
          *reinterpret_cast<float2*>(dst + 2 * e) = __bfloat1622float2(tc[e]);
        mbar_arrive(&conv[s]);
      }
    }
    return;
  }

  const int q = tid % TPC, cl = tid / TPC;
  const int d = d0 + cl;
  const bool dvalid = d < D && cl < kValid;
  const int dc = dvalid ? d : D - 1;
  float2 A2[2], carry[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int n = 4 * q + 2 * i;
    const float a0 = -expf(p.A_log[dc * N + n]);
    const float a1 = -expf(p.A_log[dc * N + n + 1]);
    A2[i] = kFast ? make_float2(a0 * kLog2e, a1 * kLog2e) : make_float2(a0, a1);
    carry[i] = make_float2(0.f, 0.f);
  }
  const float bias = p.delta_bias[dc];
  int colo[kPer];  // swizzled offsets of this channel in the rows of the owned steps
#pragma unroll
  for (int j = 0; j < kPer; ++j) colo[j] = AT::col(j * TPC + q, cl);
  float dsum = 0.f;
  for (int k = 0; k < ntiles; ++k) {
    const int s = k % S;
    const uint32_t par = (uint32_t)(k / S) & 1;
    if (!mbar_wait(&full[s], par, p.status)) break;
    if (kBf16 && !mbar_wait(&conv[s], par, p.status)) break;
    const int tbase = t_lo + (ntiles - 1 - k) * kTT;
    const int cnt = min(kTT, t_hi - tbase);
    const Act* sr = tile_raw(s);
    const Act* sz = tile_z(s);
    const Act* sg = tile_g(s);
    const float* Ct = (kBf16 ? cf + (size_t)s * kTT * N : reinterpret_cast<const float*>(tile_C(s))) + 4 * q;
    // phase 1: (delta, dy) of the owned steps; steps past the end get (0, 0)
    const bool full_tile = cnt == kTT;
#pragma unroll
    for (int i = 0; i < kOwn; ++i) {
      const int km = i * TPC + q;
      const int kr = min(km, cnt - 1);
      const int o = full_tile ? km * AT::kRowB + colo[i % kPer] : AT::off(kr, cl);
      const float sp = clamp_dt(kFast ? softplus_fast(lds_at(sr, o) + bias) : softplus_f(lds_at(sr, o) + bias),
                                p.dt_min, p.dt_max);
      float dy = lds_at(sg, o);
      if (kGate) {
        const float zz = lds_at(sz, o);
        dy *= zz * (kFast ? sigmoid_fast(zz) : sigmoid_f(zz));
      }
      prep[km * kPrepRow + cl] = km < cnt ? make_float2(sp, dy) : make_float2(0.f, 0.f);
    }
    __syncwarp();
    // phase 2: the adjoint recurrence, last step first; only the carry is carried
    float tsum = 0.f;
    auto rstep = [&](int kk) {
      const float2 v = prep[kk * kPrepRow + cl];
      const float2 dd = make_float2(v.x, v.x), dy2 = make_float2(v.y, v.y);
      const float4 Cv = *reinterpret_cast<const float4*>(Ct + kk * N);
      const float2 g0 = ffma2(dy2, make_float2(Cv.x, Cv.y), carry[0]);
      const float2 g1 = ffma2(dy2, make_float2(Cv.z, Cv.w), carry[1]);
      carry[0] = fmul2(decay2<kFast>(dd, A2[0]), g0);
      carry[1] = fmul2(decay2<kFast>(dd, A2[1]), g1);
      tsum += v.x;
    };
    if (cnt == kTT) {
#pragma unroll
      for (int kk = kTT - 1; kk >= 0; --kk) rstep(kk);
    } else {
      for (int kk = cnt - 1; kk >= 0; --kk) rstep(kk);
    }
    dsum += tsum;
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  if (dvalid) {
    float* ag = p.seg_agg + ((((size_t)b * p.nseg + seg) * D + d) * N + 4 * q) * 2;
    const float2 x0 = fmul2(make_float2(dsum, dsum), A2[0]);
    const float2 x1 = fmul2(make_float2(dsum, dsum), A2[1]);
    const float P0 = kFast ? ex2_approx(x0.x) : expf(x0.x), P1 = kFast ? ex2_approx(x0.y) : expf(x0.y);
    const float P2 = kFast ? ex2_approx(x1.x) : expf(x1.x), P3 = kFast ? ex2_approx(x1.y) : expf(x1.y);
    reinterpret_cast<float4*>(ag)[0] = make_float4(P0, carry[0].x, P1, carry[0].y);
    reinterpret_cast<float4*>(ag)[1] = make_float4(P2, carry[1].x, P3, carry[1].y);
  }
}

// Carry pass: per (b, d, n), over the K pieces of the sequence (b, d / 64)
// from the last to the first: seg_carry[k] = adjoint carry entering piece
// k's last step (dh_last, or 0, for the last piece); seg_carry[k - 1] =
// carry_out_k + P_k * seg_carry[k].  Also zeroes the parameter-partial rows
// k >= K of (b, d), which no piece writes.
__global__ void s6_bwd_seg_carry_kernel(const BwdParams p) {
  const size_t per = (size_t)p.D * p.N;
  const size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int b = blockIdx.y;
  if (e >= per) return;
  const int d = (int)(e / p.N), n = (int)(e % p.N);
  const int K = plan_pieces(p.plan, (long long)b * p.plan.ndt + d / kDTile);
  float chi = p.dh_last ? p.dh_last[(size_t)b * per + e] : 0.f;
  for (int k = K - 1; k >= 0; --k) {
    p.seg_carry[((size_t)b * p.nseg + k) * per + e] = chi;
    if (k > 0) {
      const float* ag = p.seg_agg + (((size_t)b * p.nseg + k) * per + e) * 2;
      chi = fmaf(ag[0], chi, ag[1]);
    }
  }
  for (int k = K; k < p.nseg; ++k) {
    float* wp = p.ws_param + (((size_t)b * p.nseg + k) * p.D + d) * (p.N + 2);
    wp[n] = 0.f;
    if (n < 2) wp[p.N + n] = 0.f;
  }
}

template <typename Act, int TPC>
size_t bwd_agg_smem_bytes() {
  constexpr int N = 4 * TPC, kCh = kScanThreads / TPC, S = 3;
  constexpr bool bf = std::is_same<Act, __nv_bfloat16>::value;
  return (size_t)S * agg_stage_bytes<Act, TPC>() + (bf ? (size_t)S * kTT * N * 4 : 0) +
         (size_t)kTT * (kCh + 4) * 8 + 3 * S * 8;
}

template <typename Act, int TPC, bool kFast, bool kGate>
cudaError_t launch_agg(const BwdTmaParams& P, cudaStream_t stream) {
  auto kern = s6_bwd_agg_kernel<Act, TPC, kFast, kGate>;
  const size_t smem = bwd_agg_smem_bytes<Act, TPC>();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  constexpr int kCh = kScanThreads / TPC;
  constexpr int kValid = kCh < kDTile ? kCh : kDTile;
  const dim3 grid((P.p.D + kValid - 1) / kValid, P.p.B, P.p.nseg - 1);
  kern<<<grid, kAggWarps * 32, smem, stream>>>(P);
  return cudaGetLastError();
}

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
size_t bwd_smem_bytes() {
  const bool bf = std::is_same<Act, __nv_bfloat16>::value;
  const int S = BwdStages<Act>::value;
  const int N = 4 * TPC, lanes = kDTile * TPC, cw = lanes / 32;
  size_t bytes = (size_t)S * (4 * kTT * kDTile + 2 * kTT * N) * sizeof(Act);
  bytes += (bf ? (size_t)S * kTT * 2 * N : 0) * 4;      // bcf
  bytes += (size_t)kChunk * kRow * 8;                    // dbuf (float2)
  bytes += (size_t)lanes * 16;                           // hc0
  bytes += (size_t)cw * kRedSlots * kRedSlot * 4;        // redw
  bytes += (size_t)2 * kSub * cw * 32 * 4;               // wpart
  bytes += (size_t)kSub * (lanes + 1) * 16;              // part (float4)
  bytes += (size_t)kSub * kRow * 8;                      // bprep
  bytes += (size_t)2 * lanes * 6 * 4;                    // tot
  bytes += (3 * S + 4) * 8 + 16;                         // barriers, TMEM address
  return bytes;
}

template <typename Act, int TPC, bool kFast, bool kGate, bool kLimit>
cudaError_t launch_one(const BwdTmaParams& P, cudaStream_t stream, bool cooperative) {
  auto kern = s6_bwd_tma_kernel<Act, TPC, kFast, kGate, kLimit>;
  const size_t smem = bwd_smem_bytes<Act, TPC>();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // persistent: one CTA per range of the plan
  if (!cooperative) {
    kern<<<P.p.plan.P, (2 * TPC + 3) * 32, smem, stream>>>(P);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)P.p.plan.P);
  cfg.blockDim = dim3((2 * TPC + 3) * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, P);
}

// the main kernel's instance for this call: gate or not, limit on delta or not
template <typename Act, int TPC, bool kFast>
cudaError_t launch_main(const BwdTmaParams& P, cudaStream_t stream, bool cooperative) {
  const bool lim = P.p.dt_min > 0.f || P.p.dt_max < INFINITY;
  if (P.p.z)
    return lim ? launch_one<Act, TPC, kFast, true, true>(P, stream, cooperative)
               : launch_one<Act, TPC, kFast, true, false>(P, stream, cooperative);
  return lim ? launch_one<Act, TPC, kFast, false, true>(P, stream, cooperative)
             : launch_one<Act, TPC, kFast, false, false>(P, stream, cooperative);
}

// TPC lanes per channel: 4 states per lane in both the main and the aggregate pass
template <typename Act, int TPC, bool kFast>
cudaError_t launch_tpc(BwdTmaParams& P, BwdTmaParams& Pagg, cudaStream_t stream) {
  const BwdPlan& pl = P.p.plan;
  if (pl.handover && P.p.seq_flag) {
    // hand-over mode: every sequence in at most two pieces and no range
    // shorter than a sequence, so the CTA holding a last piece (walked
    // first) is done with it before the CTA holding the first piece (walked
    // last) gets there; a cooperative launch keeps every CTA resident
    cudaError_t e = cudaMemsetAsync(P.p.seq_flag, 0, sizeof(int) * (size_t)P.p.B * pl.ndt, stream);
    if (e != cudaSuccess) return e;
    e = launch_main<Act, TPC, kFast>(P, stream, true);
    if (e != cudaErrorCooperativeLaunchTooLarge) return e;
    (void)cudaGetLastError();  // not resident at once on this GPU: aggregate mode
    note_plan_fallback();
  }
  P.p.seq_flag = nullptr;
  Pagg.p.seq_flag = nullptr;
  if (P.p.nseg > 1) {
    // chunked parallel scan: adjoint piece aggregates -> carries -> all pieces at once
    // (Pagg's tensor maps have the aggregate pass's 128/TPC-channel boxes)
    cudaError_t e = P.p.z ? launch_agg<Act, TPC, kFast, true>(Pagg, stream) : launch_agg<Act, TPC, kFast, false>(Pagg, stream);
    if (e != cudaSuccess) return e;
    const dim3 cgrid((unsigned)(((size_t)P.p.D * P.p.N + 255) / 256), P.p.B);
    s6_bwd_seg_carry_kernel<<<cgrid, 256, 0, stream>>>(P.p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return launch_main<Act, TPC, kFast>(P, stream, false);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

// The work plan: sms ranges of equal length over all chunk units (one
// persistent CTA per SM, no tail wave); sequences cut by a range boundary
// get aggregates for their later pieces.  N outside {4, 8, 16} never takes
// the TMA path: one piece per sequence.
BwdPlan bwd_plan(int B, int L, int D, int N, int sms) {
  BwdPlan pl;
  pl.nch = L > 0 ? (L + kChunk - 1) / kChunk : 0;
  pl.ndt = D > 0 ? (D + kDTile - 1) / kDTile : 0;
  pl.U = (long long)(B > 0 ? B : 0) * pl.ndt * pl.nch;
  pl.P = (int)std::max<long long>(1, std::min<long long>(std::max(sms, 1), pl.U));
  pl.maxp = 1;
  pl.handover = false;
  if (pl.U == 0 || !(N == 4 || N == 8 || N == 16)) {
    pl.U = std::max<long long>(pl.U, 1);
    pl.P = 1;
    return pl;
  }
  const long long nseq = (long long)B * pl.ndt;
  for (long long sq = 0; sq < nseq; ++sq) pl.maxp = std::max(pl.maxp, plan_pieces(pl, sq));
  pl.handover = pl.maxp == 2 && (long long)pl.nch <= pl.U / pl.P;
  return pl;
}

// Same shape rules as the TMA forward: N in {4, 8, 16}, N*e and D*e
// multiples of 16 bytes, 16-byte aligned tensors.
bool bwd_tma_supported(const BwdParams& p, int act) {
  const int e = act == SSM_BF16 ? 2 : 4;
  if (!(p.N == 4 || p.N == 8 || p.N == 16)) return false;
  if (act == SSM_BF16 && p.N == 4) return false;
  if ((p.N * e) % 16 != 0 || (p.D * e) % 16 != 0) return false;
  if (p.plan.U >= (1LL << 31)) return false;  // unit indices are ints in the kernel
  const void* ptrs[] = {p.u, p.delta_raw, p.Bm, p.Cm, p.dout, p.chunk_states};
  for (const void* q : ptrs)
    if (!aligned16(q)) return false;
  if (p.z && !aligned16(p.z)) return false;
  if (p.dh0 && !aligned16(p.dh0)) return false;
  if (p.dh_last && (reinterpret_cast<uintptr_t>(p.dh_last) & 7)) return false;
  return tensor_map_encoder() != nullptr;
}

cudaError_t launch_bwd_tma(const BwdParams& p, int act, cudaStream_t stream) {
  BwdTmaParams P;
  memset(&P, 0, sizeof(P));
  P.p = p;
  const uint64_t rows = (uint64_t)p.B * p.L;
  // activation tiles: 128-byte swizzled boxes of 128-byte rows (64 bf16 / 32 f32 channels)
  const uint32_t abox = act == SSM_BF16 ? kDTile : kDTile / 2;
  bool ok = make_map(&P.map_u, p.u, act, rows, p.D, kTT, abox, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_map(&P.map_raw, p.delta_raw, act, rows, p.D, kTT, abox, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_map(&P.map_dout, p.dout, act, rows, p.D, kTT, abox, CU_TENSOR_MAP_SWIZZLE_128B) &&
            make_map(&P.map_B, p.Bm, act, rows, p.N, kTT, p.N) &&
            make_map(&P.map_C, p.Cm, act, rows, p.N, kTT, p.N);
  if (p.z) ok = ok && make_map(&P.map_z, p.z, act, rows, p.D, kTT, abox, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return cudaErrorInvalidValue;
  BwdTmaParams Pagg = P;
  if (p.nseg > 1) {
    // the aggregate pass's tiles: 128/TPC channels in boxes of <= 128-byte rows, swizzled
    const uint32_t kch = (uint32_t)(kScanThreads / (p.N / 4));
    const uint32_t e = act == SSM_BF16 ? 2 : 4;
    const uint32_t row_b = std::min<uint32_t>(kch * e, 128);
    const CUtensorMapSwizzle sw = swizzle_for_row_bytes((int)row_b);
    ok = make_map(&Pagg.map_raw, p.delta_raw, act, rows, p.D, kTT, row_b / e, sw) &&
         make_map(&Pagg.map_dout, p.dout, act, rows, p.D, kTT, row_b / e, sw);
    if (p.z) ok = ok && make_map(&Pagg.map_z, p.z, act, rows, p.D, kTT, row_b / e, sw);
    if (!ok) return cudaErrorInvalidValue;
  }
  const int TPC = p.N / 4;
  if (act == SSM_BF16) {
    if (TPC == 4) return launch_tpc<__nv_bfloat16, 4, true>(P, Pagg, stream);
    if (TPC == 2) return launch_tpc<__nv_bfloat16, 2, true>(P, Pagg, stream);
    return cudaErrorInvalidValue;
  }
  if (TPC == 4) return launch_tpc<float, 4, false>(P, Pagg, stream);
  if (TPC == 2) return launch_tpc<float, 2, false>(P, Pagg, stream);
  if (TPC == 1) return launch_tpc<float, 1, false>(P, Pagg, stream);
  return cudaErrorInvalidValue;
}

}  // namespace s6
