// S6 backward, TMA-pipelined, every state of a chunk in tensor memory (sm_103a).
//
// A persistent CTA walks a range of chunk units (plan: one range per SM over
// all (batch, 128-channel tile, 32-step chunk) units, contiguous or split into
// heads and tails); each unit is one 32-step chunk of 128 channels.  Warps:
// 2*TPC consumers (TPC = N/4), a TMA producer and three reducers (the channel
// sums of the dBm and dCm terms, step halves dealt out in turn; fewer fell
// behind the consumers).  A lane reads the Bm / Cm values of its 4 states straight from
// the stage: 16 bytes each in f32, 8 bytes in bf16 widened in registers
// (exact; half the shared-memory wavefronts of an f32 copy).
//
// Consumer lane (pair cp, group q) owns channels d0 + 2cp, d0 + 2cp + 1 and
// states 4q .. 4q+3 of both: 8 cells per step, two packed f32x2 operations per
// channel for each arithmetic step.  Per chunk, last chunk of the piece first:
//   prep A: delta = softplus(delta_raw + bias) and delta*u of the lane's owned
//     steps (step k with k % TPC == q inside every 4-step group) for both
//     channels, into shared memory;
//   pass A: the recurrence h_t = Abar_t h_{t-1} + delta*u*B_t from the saved
//     chunk state, every state stored to tensor memory (8 columns per step,
//     32 columns = 4 steps per tcgen05.st);
//   pass B: 4-step sub-chunks, last first: the gate terms dy = dout*silu(z)
//     and the dz factor of the owned steps, then the adjoint
//     g_t = dy_t C_t + Abar_{t+1} g_{t+1} backwards with the states loaded from
//     tensor memory, producing every gradient term of the step, then the
//     outputs du, d_delta_raw, dz of the owned steps.
// The tile's u, delta_raw, z, dout, Bm, Cm rows stay in one shared-memory stage
// for both passes (the chunk is read from HBM once).
//
// Sums (the single-writer, fixed-order policy of deterministic_backward.py,
// with the kernels.rs page's local-backward / reduction split):
//   - over the 16 states of a channel (y, sum g*B, sum A*p): each lane adds its
//     4 in registers, the TPC lanes of the pair are added in lane order by the
//     lane that writes the step's outputs;
//   - over channels (dBm, dCm): each lane adds its 2 channels inside the FMAs;
//     bf16: the lanes' terms go to shared memory and the reducer warps add the
//     64 pairs in a fixed order (interleaved slices, then an xor butterfly);
//     f32: a 3-round xor reduce-scatter adds the warp's lanes and the
//     reducers add the warps in ascending order; either way into the tile's
//     partial row, and a small kernel adds the tiles in ascending order
//     (s6_bwd.cu);
//   - over (b, t) (dA_log, dDp, d_delta_bias): per lane per chunk, then a
//     compensated (Kahan) running total per piece, then the pieces and batches
//     in ascending order (s6_bwd.cu).
// No floating-point atomics: bit-identical results from run to run.
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

constexpr int kTT = 32;       // steps per tile (the forward's and the aggregate pass's tiles)
constexpr int kSC = 4;        // pass B: steps per sub-chunk (32 TMEM columns)
constexpr int kAggWarps = 5;  // aggregate pass: 4 consumer warps + producer
constexpr int kBS = 2;        // stages of the main kernel's ring (one chunk each)
static_assert(kChunk == kTT, "the backward's chunk is one tile");

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

// two adjacent activations at a byte offset of a (swizzled) tile
__device__ __forceinline__ float2 lds_pair(const float* tile, int byte_off) {
  return *reinterpret_cast<const float2*>(reinterpret_cast<const unsigned char*>(tile) + byte_off);
}
__device__ __forceinline__ float2 lds_pair(const __nv_bfloat16* tile, int byte_off) {
  return __bfloat1622float2(
      *reinterpret_cast<const __nv_bfloat162*>(reinterpret_cast<const unsigned char*>(tile) + byte_off));
}
// one activation at a byte offset of a (swizzled) tile
template <typename Act>
__device__ __forceinline__ float lds_at(const Act* tile, int byte_off) {
  return lds_act(reinterpret_cast<const Act*>(reinterpret_cast<const unsigned char*>(tile) + byte_off));
}
// store two adjacent outputs
__device__ __forceinline__ void st_pair(float* p, float2 v) { *reinterpret_cast<float2*>(p) = v; }
__device__ __forceinline__ void st_pair(__nv_bfloat16* p, float2 v) {
  *reinterpret_cast<__nv_bfloat162*>(p) = __float22bfloat162_rn(v);
}

// load 8 consecutive columns of this thread's lane and wait
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// issue a load of 8 consecutive columns of this thread's lane (no wait)
__device__ __forceinline__ void tmem_ld8_issue(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}
// wait for this thread's TMEM loads; the destination of the last one passes
// through the statement, so nothing reads it before the wait
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[8]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7])
               :
               : "memory");
}

template <typename Act, int TPC>
struct BwdLayout {
  static constexpr int N = 4 * TPC;
  static constexpr int kLanes = 64 * TPC;  // consumer threads: 64 channel pairs x TPC
  static constexpr int kCW = kLanes / 32;  // consumer warps
  static constexpr bool kBf16 = std::is_same<Act, __nv_bfloat16>::value;
  using AT = SwzTile<Act, kBwdTile, kTT>;  // u, delta_raw, z, dout tiles
  static constexpr int kTileB = kTT * kBwdTile * (int)sizeof(Act);
  static constexpr int kBCB = kTT * N * (int)sizeof(Act);
  // stage: u, raw, z, dout tiles, then the Bm and Cm rows; 1024-byte multiple
  static constexpr int kStageB = ((4 * kTileB + 2 * kBCB) + 1023) / 1024 * 1024;
  // Row strides, padded so that the lanes of a pair (which own different
  // steps, i.e. rows) hit different banks: pA rows of 64 float4 + 2, pY rows of
  // 64 float2 + 4, part4 / part2 rows of kLanes + 1 elements.
  // (f32: pA unpadded, to fit the larger tiles)
  static constexpr int kRA = kBf16 ? 64 + 2 : 64, kRY = 64 + 4, kRP4 = kLanes + 1, kRP2 = kLanes + 1;
  static constexpr int kPAB = kTT * kRA * 16;                    // pA [TT][kRA] float4 (delta, delta*u) x 2
  static constexpr int kPYB = kSC * kRY * 8;                     // pY [SC][kRY] float2 (dy0, dy1)
  static constexpr int kPart4B = kSC * kRP4 * 16;                // [SC][kRP4] (y0, gB0, y1, gB1)
  static constexpr int kPart2B = kSC * kRP2 * 8;                 // [SC][kRP2] (Ap0, Ap1)
  // dBm/dCm terms over the CTA's channels: bf16 -- each lane's 8 values of a
  // step in shared memory ([2 slots][SC][64 pairs][TPC groups][8] floats),
  // added by the reducer warps; f32 (less shared memory) -- a warp-level xor
  // reduce-scatter first, the warps' sums ([2 slots][SC][kCW][32]) added by
  // the reducer warps.
  // Within a pair's block the 16-byte slot j (= 2q + 0 for the dBm terms,
  // 2q + 1 for the dCm terms) sits at j ^ red_swz(pair): consecutive pairs
  // rotate through the banks, so that a warp's stores (8 pairs x 4 groups)
  // and a reducer's loads (8 slices of pairs 8 apart x 4 groups) both take
  // the minimum of four wavefronts.
  static constexpr bool kRedSmem = kBf16;
  static constexpr int kRedPair = TPC * 8;  // floats per channel pair in a step's block
  static constexpr int kRedStep = 64 * kRedPair;
  static constexpr int kRedQ = kRedPair / 4;  // 16-byte slots per pair
  __device__ static __forceinline__ int red_swz(int pair) { return (pair / (8 / kRedQ)) % kRedQ; }
  static constexpr int kDsumB = kRedSmem ? 2 * kSC * kRedStep * 4 : 2 * kSC * kCW * 32 * 4;
  static constexpr int kTotB = 2 * 12 * kLanes * 4;              // [2 (sum, comp)][12][lanes] running totals
  static constexpr int kOffPA = kBS * kStageB;
  static constexpr int kOffPY = kOffPA + kPAB;
  static constexpr int kOffPart4 = kOffPY + kPYB;
  static constexpr int kOffPart2 = kOffPart4 + kPart4B;
  static constexpr int kOffDsum = kOffPart2 + kPart2B;
  static constexpr int kOffTot = kOffDsum + kDsumB;
  static constexpr int kOffBar = kOffTot + kTotB;
  static constexpr int kBars = 2 * kBS + 4;
  static constexpr int kBytes = kOffBar + kBars * 8 + 16;
  static constexpr uint32_t kTmemCols = kCW > 4 ? 512 : 256;
  static_assert(kCW <= 8, "two consumer warps per TMEM lane quarter at most");
  static_assert(kBytes <= 227 * 1024, "shared memory");
};

// kLimit: delta is clamped to [dt_min, dt_max] (a separate instance, so the
// unlimited scan pays nothing for it).
template <typename Act, int TPC, bool kFast, bool kGate, bool kLimit>
__global__ void __launch_bounds__((2 * TPC + 4) * 32, 1) s6_bwd_tma_kernel(const __grid_constant__ BwdTmaParams P) {
  using LY = BwdLayout<Act, TPC>;
  using AT = typename LY::AT;
  constexpr int N = LY::N;
  constexpr int kLanes = LY::kLanes;
  constexpr int kCW = LY::kCW;
  constexpr bool kBf16 = LY::kBf16;
  constexpr int kRB = AT::kRowB;
  constexpr int kOwn = kSC / TPC;  // owned steps of a lane per sub-chunk
  // ln 2 on the fast path: sums weighted by A are taken with A*log2(e)
  constexpr float kAscale = kFast ? kLn2 : 1.f;

  extern __shared__ __align__(1024) unsigned char smem[];
  float4* pA = reinterpret_cast<float4*>(smem + LY::kOffPA);
  float2* pY = reinterpret_cast<float2*>(smem + LY::kOffPY);
  float4* part4 = reinterpret_cast<float4*>(smem + LY::kOffPart4);
  float2* part2 = reinterpret_cast<float2*>(smem + LY::kOffPart2);
  float* dsum = reinterpret_cast<float*>(smem + LY::kOffDsum);
  float* totS = reinterpret_cast<float*>(smem + LY::kOffTot);  // [2][12][lanes]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + LY::kOffBar);
  uint64_t* empty = full + kBS;
  uint64_t* wfull = empty + kBS;  // [2] dsum slot written by every consumer warp
  uint64_t* wempty = wfull + 2;   // [2] dsum slot summed by all three reducers
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(wempty + 2);

  const BwdParams& p = P.p;
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.status, kStatusLayout);
    return;
  }
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int L = p.L, D = p.D;
  const int nchunks = p.nchunks;
  const BwdPlan& pl = p.plan;
  const int u_begin = (int)plan_bound(pl, blockIdx.x), u_end = (int)plan_bound(pl, blockIdx.x + 1);
  if (blockIdx.x == 0 && tid == 0) *p.ws_ndt = pl.ndt;  // the finalize reads the partial-row count

  if (tid == 0) {
    for (int s = 0; s < kBS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kCW);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&wfull[i], kCW);
      mbar_init(&wempty[i], 3);  // every reducer warp
    }
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, LY::kTmemCols);
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();

  auto stage = [&](int s) { return smem + (size_t)s * LY::kStageB; };
  auto tile = [&](int s, int i) { return reinterpret_cast<Act*>(stage(s) + i * LY::kTileB); };  // 0 u 1 raw 2 z 3 dout
  auto tile_B = [&](int s) { return reinterpret_cast<Act*>(stage(s) + 4 * LY::kTileB); };
  auto tile_C = [&](int s) { return reinterpret_cast<Act*>(stage(s) + 4 * LY::kTileB + LY::kBCB); };

  // the item (a piece of one sequence) that starts at unit u of this CTA's range
  auto item_at = [&](int u, int& b, int& d0, int& c_lo, int& c_hi, int& next, int& sq, int& kp) {
    long long sq_l, next_l;
    plan_item(pl, u, u_end, sq_l, c_lo, c_hi, kp, next_l);
    sq = (int)sq_l;
    next = (int)next_l;
    b = sq / pl.ndt;
    d0 = (sq % pl.ndt) * kBwdTile;
  };
  auto piece_at = [&](int u, int& b, int& d0, int& c_lo, int& c_hi, int& next) {
    int sq, kp;
    item_at(u, b, d0, c_lo, c_hi, next, sq, kp);
  };
  auto chunk_len = [&](int c) { return min(kChunk, L - c * kChunk); };

  if (warp == kCW) {
    // ---------------- producer: one stage per chunk, chunks of each piece last first
    if (lane == 0) {
      tma_prefetch_desc(&P.map_u);
      tma_prefetch_desc(&P.map_raw);
      tma_prefetch_desc(&P.map_dout);
      if (kGate) tma_prefetch_desc(&P.map_z);
      tma_prefetch_desc(&P.map_B);
      tma_prefetch_desc(&P.map_C);
      const uint32_t bytes = (uint32_t)((kGate ? 4 : 3) * LY::kTileB + 2 * LY::kBCB);
      int item = 0;
      bool ok = true;
      for (int u = u_begin, next; u < u_end && ok; u = next) {
        int b, d0, c_lo, c_hi;
        piece_at(u, b, d0, c_lo, c_hi, next);
        for (int c = c_hi - 1; c >= c_lo; --c, ++item) {
          const int s = item % kBS;
          if (item >= kBS && !mbar_wait(&empty[s], (uint32_t)(item / kBS - 1) & 1, p.status)) {
            ok = false;
            break;
          }
          const int row = b * L + c * kChunk;
          mbar_arrive_expect_tx(&full[s], bytes);
#pragma unroll
          for (int bx = 0; bx < AT::kNBox; ++bx) {
            const int x = d0 + bx * AT::kChBox, o = bx * AT::kBoxBytes;
            tma_load_2d(reinterpret_cast<unsigned char*>(tile(s, 0)) + o, &P.map_u, &full[s], x, row);
            tma_load_2d(reinterpret_cast<unsigned char*>(tile(s, 1)) + o, &P.map_raw, &full[s], x, row);
            if (kGate) tma_load_2d(reinterpret_cast<unsigned char*>(tile(s, 2)) + o, &P.map_z, &full[s], x, row);
            tma_load_2d(reinterpret_cast<unsigned char*>(tile(s, 3)) + o, &P.map_dout, &full[s], x, row);
          }
          tma_load_2d(tile_B(s), &P.map_B, &full[s], 0, row);
          tma_load_2d(tile_C(s), &P.map_C, &full[s], 0, row);
        }
      }
      // never leave with copies in flight: wait for the last use of every stage
      for (int s = 0; s < kBS && s < item; ++s) {
        const int k_last = s + kBS * ((item - 1 - s) / kBS);
        mbar_wait(&full[s], (uint32_t)(k_last / kBS) & 1, p.status);
      }
    }
    return;
  }
  if (warp >= kCW + 1 && warp <= kCW + 3) {
    // ---------------- reducers: the consumers' per-step dBm/dCm terms summed
    // over the tile's channel pairs in a fixed order -> this tile's partial
    // row [t][2][N].  A sub-chunk's work is 2 cnt halves (step k, dBm or dCm
    // half: item 2k + half); reducer r takes the items r, r + 3, ...  (The
    // register file is allocated for 12 warps whether the CTA has 11 or 12,
    // so the third reducer is free; two alone kept the consumers waiting.)
    const int r = warp - kCW - 1;
    int n = 0;
    bool ok = true;
    for (int u = u_begin, next; u < u_end; u = next) {
      int b, d0, c_lo, c_hi;
      piece_at(u, b, d0, c_lo, c_hi, next);
      float* ws_r = p.ws_dbc + ((size_t)(d0 / kBwdTile) * p.B + b) * (size_t)L * 2 * N;
      for (int c = c_hi - 1; c >= c_lo; --c) {
        const int clen = chunk_len(c);
        for (int sc = (clen + kSC - 1) / kSC - 1; sc >= 0; --sc, ++n) {
          const int slot = n & 1;
          if (ok) ok = mbar_wait(&wfull[slot], (uint32_t)(n >> 1) & 1, p.status);
          const int cnt = min(kSC, clen - sc * kSC);
          const float* src = dsum + slot * (LY::kDsumB / 8);
          if constexpr (LY::kRedSmem) {
            // lane = slice * TPC + group: group gq = states 4gq .. 4gq+3; slice
            // sl adds pairs sl, sl + kLPG, sl + 2 kLPG, ... (so that the pairs'
            // slot rotations spread a load over the banks); slices then added
            // by an xor butterfly
            constexpr int nG = TPC, kLPG = 32 / nG, kCPL = 64 / kLPG;
            const int gq = lane % nG, sl = lane / nG;
            for (int it = r; it < 2 * cnt; it += 3) {
              const int k = it >> 1, hf = it & 1;
              const float* rp = src + k * LY::kRedStep;
              float2 a = make_float2(0.f, 0.f), b2 = make_float2(0.f, 0.f);
#pragma unroll
              for (int i = 0; i < kCPL; ++i) {
                const int pr = sl + i * kLPG;
                const int j = (2 * gq + hf) ^ LY::red_swz(pr);
                const float4 v = *reinterpret_cast<const float4*>(rp + pr * LY::kRedPair + 4 * j);
                a = fadd2(a, make_float2(v.x, v.y));
                b2 = fadd2(b2, make_float2(v.z, v.w));
              }
#pragma unroll
              for (int m = nG; m < 32; m <<= 1) {
                a = fadd2(a, make_float2(__shfl_xor_sync(0xffffffffu, a.x, m), __shfl_xor_sync(0xffffffffu, a.y, m)));
                b2 = fadd2(b2, make_float2(__shfl_xor_sync(0xffffffffu, b2.x, m), __shfl_xor_sync(0xffffffffu, b2.y, m)));
              }
              if (sl == 0)
                *reinterpret_cast<float4*>(ws_r + (size_t)(c * kChunk + sc * kSC + k) * 2 * N + hf * N + 4 * gq) =
                    make_float4(a.x, a.y, b2.x, b2.y);
            }
          } else if (lane < N) {
            for (int it = r; it < 2 * cnt; it += 3) {
              const int k = it >> 1, hf = it & 1;
              float v = src[(k * kCW) * 32 + hf * N + lane];
#pragma unroll
              for (int w = 1; w < kCW; ++w) v += src[(k * kCW + w) * 32 + hf * N + lane];
              ws_r[(size_t)(c * kChunk + sc * kSC + k) * 2 * N + hf * N + lane] = v;
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&wempty[slot]);
        }
      }
    }
    return;
  }

  // ---------------- consumers
  const int q = lane % TPC;                  // state group: states 4q .. 4q+3
  const int cp = tid / TPC;                  // channel pair in the tile: channels 2cp, 2cp+1
  const uint32_t tm = *tmem_slot + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)((warp >> 2) * 256);
  // reduce-scatter of the 8 dBm/dCm values over the warp's pairs: output of this lane
  const int rs_o = ((lane >> 4) & 1) * N + 4 * q + 2 * ((lane >> 3) & 1) + ((lane >> 2) & 1);
  const bool rs_store = (lane & (3 & ~(TPC - 1))) == 0;
  // this lane's dBm slot in a step's block of the reducers (its dCm slot: ^ 4)
  const int red_off = cp * LY::kRedPair + 4 * ((2 * q) ^ LY::red_swz(cp));
  // swizzled byte offset of the pair's channels in the rows of the lane's
  // owned steps (it depends on the row % 8 only): owned step i of a 4-step
  // sub-chunk at an even / odd sub-chunk index
  int colE[kOwn], colO[kOwn];
#pragma unroll
  for (int i = 0; i < kOwn; ++i) {
    colE[i] = AT::col(i * TPC + q, 2 * cp);
    colO[i] = AT::col(kSC + i * TPC + q, 2 * cp);
  }

  bool failed = false;
  int s = 0;         // ring stage of the current chunk
  uint32_t par = 0;  // its phase parity
  int nsub = 0;      // sub-chunks handed to the reducers so far
  for (int u = u_begin, next; u < u_end; u = next) {
    int b, d0, c_lo, c_hi, sq, kp;
    item_at(u, b, d0, c_lo, c_hi, next, sq, kp);
    const bool last_piece = c_hi == pl.nch;
    const int dA = d0 + 2 * cp;  // first channel of the pair (D is even: both valid or neither)
    const bool dvalid = dA < D;
    const int dc = dvalid ? dA : D - 2;
    if (!last_piece && p.seq_flag) {
      // hand-over mode: the carry comes from the CTA walking the sequence's last piece
      if (lane == 0 && !failed) failed = !flag_wait(p.seq_flag + sq, p.status);
      failed = __shfl_sync(0xffffffffu, failed, 0);
      __syncwarp();
    }
    // A2[c][i]: states 4q + 2i, 4q + 2i + 1 of channel dc + c
    float2 A2[2][2], carry[2][2];
    {
      const float* cin = !last_piece ? p.seg_carry + (((size_t)b * p.nseg + kp) * D + dc) * N
                                     : (p.dh_last ? p.dh_last + ((size_t)b * D + dc) * N : nullptr);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const float4 al = *reinterpret_cast<const float4*>(p.A_log + (size_t)(dc + c) * N + 4 * q);
        const float a[4] = {-expf(al.x), -expf(al.y), -expf(al.z), -expf(al.w)};
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          A2[c][i] = kFast ? make_float2(a[2 * i] * kLog2e, a[2 * i + 1] * kLog2e) : make_float2(a[2 * i], a[2 * i + 1]);
          carry[c][i] = (cin && dvalid) ? make_float2(__ldcg(cin + c * N + 4 * q + 2 * i), __ldcg(cin + c * N + 4 * q + 2 * i + 1))
                                        : make_float2(0.f, 0.f);
        }
      }
    }
    const float2 bias2 = make_float2(p.delta_bias[dc], p.delta_bias[dc + 1]);
    const float2 Dp2 = make_float2(p.Dp[dc], p.Dp[dc + 1]);
    // running totals of the piece: dA terms (8), dDp (2), d_delta_bias (2),
    // with Kahan compensation; lane-private in shared memory
    float* tot = totS + tid;
    float* cmp = totS + 12 * kLanes + tid;
#pragma unroll
    for (int i = 0; i < 12; ++i) tot[i * kLanes] = cmp[i * kLanes] = 0.f;
    const size_t bd_off = (size_t)b * L * D + dA;  // outputs of (b, t = 0, pair)
    float4 nxt[2];
    auto load_state = [&](int cs_c, float4 (&dst)[2]) {
#pragma unroll
      for (int cc = 0; cc < 2; ++cc)
        dst[cc] = dvalid ? __ldg(reinterpret_cast<const float4*>(
                               p.chunk_states + (((size_t)b * nchunks + cs_c) * D + dc + cc) * N + 4 * q))
                         : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    for (int c = c_hi - 1; c >= c_lo; --c) {
      const int t0 = c * kChunk;
      const int cnt = chunk_len(c);
      const int nsc = (cnt + kSC - 1) / kSC;
      // the chunk's saved start state (zeros for channels past D), loaded
      // during the previous chunk's pass B
      if (c == c_hi - 1) load_state(c, nxt);
      float2 h[2][2] = {{make_float2(nxt[0].x, nxt[0].y), make_float2(nxt[0].z, nxt[0].w)},
                        {make_float2(nxt[1].x, nxt[1].y), make_float2(nxt[1].z, nxt[1].w)}};
      if (!failed) failed = !mbar_wait(&full[s], par, p.status);
      __syncwarp();
      const Act* su = tile(s, 0);
      const Act* sr = tile(s, 1);
      const Act* sz = tile(s, 2);
      const Act* sg = tile(s, 3);
      // Bm / Cm of the lane's 4 states in step k: one 16-byte (f32) or 8-byte
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

      // ---------- prep A: (delta, delta*u) of the owned steps, both channels
#pragma unroll 2
      for (int j = 0; j < kTT / kSC; ++j) {
#pragma unroll
        for (int i = 0; i < kOwn; ++i) {
          const int k = j * kSC + i * TPC + q;
          if (k < cnt) {
            const int o = k * kRB + ((j & 1) ? colO[i] : colE[i]);
            const float2 sv = fadd2(lds_pair(sr, o), bias2);
            float2 sp = kFast ? make_float2(softplus_fast(sv.x), softplus_fast(sv.y))
                              : make_float2(softplus_f(sv.x), softplus_f(sv.y));
            if (kLimit) sp = make_float2(clamp_dt(sp.x, p.dt_min, p.dt_max), clamp_dt(sp.y, p.dt_min, p.dt_max));
            const float2 du2 = fmul2(sp, lds_pair(su, o));
            pA[k * LY::kRA + cp] = make_float4(sp.x, du2.x, sp.y, du2.y);
          }
        }
      }
      __syncwarp();

      // ---------- pass A: the states of the chunk into TMEM
      {
        float hb[32];
        auto stepA = [&](int k, int kk) {  // kk = k % kSC (a constant)
          const float4 v = pA[k * LY::kRA + cp];
          const float4 Bv = ld4(Bt + k * N);
          const float2 B01 = make_float2(Bv.x, Bv.y), B23 = make_float2(Bv.z, Bv.w);
          const float2 d0v = make_float2(v.x, v.x), u0v = make_float2(v.y, v.y);
          const float2 d1v = make_float2(v.z, v.z), u1v = make_float2(v.w, v.w);
          // the state before the step goes to TMEM (column block of step k)
          const int r = 8 * kk;
          hb[r] = h[0][0].x, hb[r + 1] = h[0][0].y, hb[r + 2] = h[0][1].x, hb[r + 3] = h[0][1].y;
          hb[r + 4] = h[1][0].x, hb[r + 5] = h[1][0].y, hb[r + 6] = h[1][1].x, hb[r + 7] = h[1][1].y;
          h[0][0] = ffma2(decay2<kFast>(d0v, A2[0][0]), h[0][0], fmul2(u0v, B01));
          h[0][1] = ffma2(decay2<kFast>(d0v, A2[0][1]), h[0][1], fmul2(u0v, B23));
          h[1][0] = ffma2(decay2<kFast>(d1v, A2[1][0]), h[1][0], fmul2(u1v, B01));
          h[1][1] = ffma2(decay2<kFast>(d1v, A2[1][1]), h[1][1], fmul2(u1v, B23));
        };
#pragma unroll 1
        for (int j = 0; j < nsc; ++j) {
          if (j * kSC + kSC <= cnt) {
#pragma unroll
            for (int kk = 0; kk < kSC; ++kk) stepA(j * kSC + kk, kk);
          } else {
#pragma unroll
            for (int kk = 0; kk < kSC; ++kk)
              if (j * kSC + kk < cnt) stepA(j * kSC + kk, kk);  // (warp-uniform)
          }
          tmem_st32(tm + (uint32_t)(8 * kSC * j), hb);
        }
        tmem_wait_st();
      }

      // ---------- pass B
      if (c > c_lo) load_state(c - 1, nxt);  // the next chunk's start state, in flight during pass B
      float2 accA[2][2] = {{make_float2(0.f, 0.f), make_float2(0.f, 0.f)}, {make_float2(0.f, 0.f), make_float2(0.f, 0.f)}};
      float2 accD = make_float2(0.f, 0.f), accBias = make_float2(0.f, 0.f);
      // hk: the state after the step being walked -- pass A's final state for
      // the last step, then the state TMEM holds before each step, loaded as
      // that step is walked (issued at the step's start, waited for before its
      // first use)
      float hk[8] = {h[0][0].x, h[0][0].y, h[0][1].x, h[0][1].y, h[1][0].x, h[1][0].y, h[1][1].x, h[1][1].y};
      for (int sc = nsc - 1; sc >= 0; --sc) {
        const int kb = sc * kSC;  // first step of the sub-chunk
        int colS[kOwn];
#pragma unroll
        for (int i = 0; i < kOwn; ++i) colS[i] = (sc & 1) ? colO[i] : colE[i];
        // B1: gate terms of the owned steps
        float2 dzf[kOwn];
#pragma unroll
        for (int i = 0; i < kOwn; ++i) {
          const int k = kb + i * TPC + q;
          float2 dy = make_float2(0.f, 0.f), f = make_float2(0.f, 0.f);
          if (k < cnt) {
            const int o = k * kRB + colS[i];
            const float2 g = lds_pair(sg, o);
            if (kGate) {
              const float2 zz = lds_pair(sz, o);
              const float2 sgz = kFast ? make_float2(sigmoid_fast(zz.x), sigmoid_fast(zz.y))
                                       : make_float2(sigmoid_f(zz.x), sigmoid_f(zz.y));
              dy = make_float2(g.x * zz.x * sgz.x, g.y * zz.y * sgz.y);
              f = make_float2(g.x * sgz.x * fmaf(zz.x, 1.f - sgz.x, 1.f), g.y * sgz.y * fmaf(zz.y, 1.f - sgz.y, 1.f));
            } else {
              dy = g;
            }
          }
          dzf[i] = f;
          pY[(i * TPC + q) * LY::kRY + cp] = dy;
        }
        __syncwarp();
        const int slot = nsub & 1;
        if (nsub >= 2 && !failed) failed = !mbar_wait(&wempty[slot], (uint32_t)((nsub >> 1) - 1) & 1, p.status);
        float* ds = dsum + slot * (LY::kDsumB / 8);
        // B3: reverse steps
        auto stepB = [&](int kk) {
          const int k = kb + kk;
          uint32_t hq[8];
          tmem_ld8_issue(tm + (uint32_t)(8 * k), hq);  // the state before step k
          const float4 v = pA[k * LY::kRA + cp];
          const float2 dy = pY[kk * LY::kRY + cp];
          const float4 Bv = ld4(Bt + k * N);
          const float4 Cv = ld4(Ct + k * N);
          const float2 Bp[2] = {make_float2(Bv.x, Bv.y), make_float2(Bv.z, Bv.w)};
          const float2 Cp[2] = {make_float2(Cv.x, Cv.y), make_float2(Cv.z, Cv.w)};
          const float2 dd[2] = {make_float2(v.x, v.x), make_float2(v.z, v.z)};
          const float2 uu[2] = {make_float2(v.y, v.y), make_float2(v.w, v.w)};
          const float2 yy[2] = {make_float2(dy.x, dy.x), make_float2(dy.y, dy.y)};
          float2 ya[2], gba[2], apa[2], dB[2], dC[2], agv[2][2];
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const int r = 4 * cc + 2 * i;
              const float2 h_k = make_float2(hk[r], hk[r + 1]);
              const float2 a = decay2<kFast>(dd[cc], A2[cc][i]);
              const float2 g = ffma2(yy[cc], Cp[i], carry[cc][i]);
              const float2 ag = fmul2(a, g);
              gba[cc] = i == 0 ? fmul2(g, Bp[i]) : ffma2(g, Bp[i], gba[cc]);
              ya[cc] = i == 0 ? fmul2(Cp[i], h_k) : ffma2(Cp[i], h_k, ya[cc]);
              dB[i] = cc == 0 ? fmul2(g, uu[cc]) : ffma2(g, uu[cc], dB[i]);
              dC[i] = cc == 0 ? fmul2(yy[cc], h_k) : ffma2(yy[cc], h_k, dC[i]);
              agv[cc][i] = ag;
              carry[cc][i] = ag;
            }
          }
          tmem_wait_ld(hq);
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const int r = 4 * cc + 2 * i;
              const float2 hp = make_float2(__uint_as_float(hq[r]), __uint_as_float(hq[r + 1]));
              const float2 pv = fmul2(agv[cc][i], hp);
              apa[cc] = i == 0 ? fmul2(A2[cc][i], pv) : ffma2(A2[cc][i], pv, apa[cc]);
              accA[cc][i] = ffma2(dd[cc], pv, accA[cc][i]);
            }
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) hk[j] = __uint_as_float(hq[j]);
          part4[kk * LY::kRP4 + tid] = make_float4(ya[0].x + ya[0].y, gba[0].x + gba[0].y, ya[1].x + ya[1].y, gba[1].x + gba[1].y);
          part2[kk * LY::kRP2 + tid] = make_float2(apa[0].x + apa[0].y, apa[1].x + apa[1].y);
          if constexpr (LY::kRedSmem) {
            // this lane's 8 terms (summed over its 2 channels) for the reducer warps
            float* rp = ds + kk * LY::kRedStep;
            const int off_c = red_off ^ 4;
            *reinterpret_cast<float4*>(rp + red_off) = make_float4(dB[0].x, dB[0].y, dB[1].x, dB[1].y);
            *reinterpret_cast<float4*>(rp + off_c) = make_float4(dC[0].x, dC[0].y, dC[1].x, dC[1].y);
            return;
          }
          // channel sums over the warp's pairs: xor reduce-scatter, 8 values -> 1
          const bool h16 = lane & 16, h8 = lane & 8, h4 = lane & 4;
          float r0[4];
          const float v8[8] = {dB[0].x, dB[0].y, dB[1].x, dB[1].y, dC[0].x, dC[0].y, dC[1].x, dC[1].y};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float send = h16 ? v8[i] : v8[4 + i];
            const float keep = h16 ? v8[4 + i] : v8[i];
            r0[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
          }
          float r1[2];
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const float send = h8 ? r0[i] : r0[2 + i];
            const float keep = h8 ? r0[2 + i] : r0[i];
            r1[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
          }
          float r2 = (h4 ? r1[1] : r1[0]) + __shfl_xor_sync(0xffffffffu, h4 ? r1[0] : r1[1], 4);
#pragma unroll
          for (int mk = 2; mk >= TPC; mk >>= 1) r2 += __shfl_xor_sync(0xffffffffu, r2, mk);
          if (rs_store) ds[(kk * kCW + warp) * 32 + rs_o] = r2;
        };
#pragma unroll 2
        for (int kk = min(kSC, cnt - kb) - 1; kk >= 0; --kk) stepB(kk);
        __syncwarp();
        if (lane == 0) mbar_arrive(&wfull[slot]);
        ++nsub;
        // B4: owned steps: the pair's sums over its TPC lanes (lane order), outputs
#pragma unroll
        for (int i = 0; i < kOwn; ++i) {
          const int kk = i * TPC + q, k = kb + kk;
          if (k < cnt) {
            float4 a4 = part4[kk * LY::kRP4 + cp * TPC];
            float2 a2 = part2[kk * LY::kRP2 + cp * TPC];
#pragma unroll
            for (int r = 1; r < TPC; ++r) {
              const float4 o4 = part4[kk * LY::kRP4 + cp * TPC + r];
              const float2 o2 = part2[kk * LY::kRP2 + cp * TPC + r];
              a4 = make_float4(a4.x + o4.x, a4.y + o4.y, a4.z + o4.z, a4.w + o4.w);
              a2 = make_float2(a2.x + o2.x, a2.y + o2.y);
            }
            const float4 v = pA[k * LY::kRA + cp];
            const float2 dy = pY[kk * LY::kRY + cp];
            const float2 uo = lds_pair(su, k * kRB + colS[i]);
            const float dl[2] = {v.x, v.z};
            float dsp[2];
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
              // softplus' = sigmoid(s) = 1 - e^{-delta}; zero where the limit
              // clamped delta (delta on a bound: a clamped step, or a softplus
              // exactly on it, which has measure zero)
              const bool free_dt = !kLimit || ((dl[cc] > p.dt_min || p.dt_min <= 0.f) && dl[cc] < p.dt_max);
              dsp[cc] = free_dt ? (kFast ? dsoftplus_fast(dl[cc]) : -expm1f(-dl[cc])) : 0.f;
            }
            const float2 o_du = make_float2(fmaf(Dp2.x, dy.x, dl[0] * a4.y), fmaf(Dp2.y, dy.y, dl[1] * a4.w));
            const float2 o_dr = make_float2(fmaf(uo.x, a4.y, a2.x * kAscale) * dsp[0], fmaf(uo.y, a4.w, a2.y * kAscale) * dsp[1]);
            const float2 o_dz = make_float2(fmaf(Dp2.x, uo.x, a4.x) * dzf[i].x, fmaf(Dp2.y, uo.y, a4.z) * dzf[i].y);
            accD = ffma2(dy, uo, accD);
            accBias = fadd2(accBias, o_dr);
            if (dvalid) {
              const size_t o = bd_off + (size_t)(t0 + k) * D;
              st_pair(static_cast<Act*>(p.du) + o, o_du);
              st_pair(static_cast<Act*>(p.d_delta_raw) + o, o_dr);
              if (kGate) st_pair(static_cast<Act*>(p.dz) + o, o_dz);
            }
          }
        }
        __syncwarp();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if (++s == kBS) {
        s = 0;
        par ^= 1;
      }
      // chunk sums -> compensated running totals
      {
        const float cs12[12] = {accA[0][0].x, accA[0][0].y, accA[0][1].x, accA[0][1].y,
                                accA[1][0].x, accA[1][0].y, accA[1][1].x, accA[1][1].y,
                                accD.x, accD.y, accBias.x, accBias.y};
#pragma unroll
        for (int i = 0; i < 12; ++i) {
          float sm = tot[i * kLanes], cm = cmp[i * kLanes];
          kahan_add(sm, cm, cs12[i]);
          tot[i * kLanes] = sm;
          cmp[i * kLanes] = cm;
        }
      }
    }
    // ---------------- the piece's parameter partials (row b * nseg + kp) and dh0
    {
      // dDp and d_delta_bias: each lane summed its owned steps; add the pair's TPC lanes
      float t4[4] = {tot[8 * kLanes], tot[9 * kLanes], tot[10 * kLanes], tot[11 * kLanes]};
#pragma unroll
      for (int m = 1; m < TPC; m <<= 1)
#pragma unroll
        for (int i = 0; i < 4; ++i) t4[i] += __shfl_xor_sync(0xffffffffu, t4[i], m);
      if (dvalid) {
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          float* wp = p.ws_param + (((size_t)b * p.nseg + kp) * D + dA + cc) * (N + 2);
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int n = 4 * q + 2 * i;
            wp[n] = (A2[cc][i].x * kAscale) * tot[(4 * cc + 2 * i) * kLanes];
            wp[n + 1] = (A2[cc][i].y * kAscale) * tot[(4 * cc + 2 * i + 1) * kLanes];
            if (p.dh0 && c_lo == 0)
              *reinterpret_cast<float2*>(p.dh0 + ((size_t)b * D + dA + cc) * N + n) = carry[cc][i];
          }
          if (q == 0) {
            wp[N] = t4[cc];
            wp[N + 1] = t4[2 + cc];
          }
          if (p.seq_flag) {
            // rows of pieces this sequence does not have stay zero for the finalize
            for (int k2 = plan_pieces(pl, sq); k2 < p.nseg; ++k2) {
              float* wz = p.ws_param + (((size_t)b * p.nseg + k2) * D + dA + cc) * (N + 2);
              wz[4 * q] = wz[4 * q + 1] = wz[4 * q + 2] = wz[4 * q + 3] = 0.f;
              if (q == 0) wz[N] = wz[N + 1] = 0.f;
            }
          }
        }
      }
      if (p.seq_flag && kp > 0) {
        // hand-over mode, the sequence's last piece: its final carry enters the
        // first piece's last step; publish it and raise the flag
        if (dvalid) {
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            float* co = p.seg_carry + (((size_t)b * p.nseg + kp - 1) * D + dA + cc) * N + 4 * q;
            __stcg(co, carry[cc][0].x);
            __stcg(co + 1, carry[cc][0].y);
            __stcg(co + 2, carry[cc][1].x);
            __stcg(co + 3, carry[cc][1].y);
          }
        }
        __threadfence();
        named_bar_sync(2, kLanes);
        if (tid == 0) st_release_gpu(p.seq_flag + sq, 1);
      }
    }
  }  // pieces
  // every consumer is done with TMEM (loads waited for inline, stores waited
  // for before the loads of the same chunk): free it
  tmem_fence_before_sync();
  named_bar_sync(1, kLanes);
  if (warp == 0) {
    tmem_fence_after_sync();
    tmem_dealloc(*tmem_slot, LY::kTmemCols);
  }
}

// ---------------------------------------------------------------- segment aggregates
// Aggregate pass of the backward's chunked parallel scan.  For the sub-piece
// in slot grid.z (at most kAggSub chunks of a later piece), from a zero
// carry, run the adjoint recurrence
//   g_t = dy_t * C_t + carry,  carry = Abar_t * g_t
// from the sub-piece's last step down to its first, and store per state its
// decay product exp(A * sum(delta)) and the final carry.  Same warp
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
  float2* prep = reinterpret_cast<float2*>(smem + (size_t)S * kStageBytes);  // [TT][kPrepRow] (delta, dy)
  uint64_t* full = reinterpret_cast<uint64_t*>(prep + kTT * kPrepRow);
  uint64_t* empty = full + S;

  const BwdParams& p = P.p;
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) atomicOr(p.status, kStatusLayout);
    return;
  }
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // channels [d0, d0 + kValid) of the sequence's channel tile d0 / kBwdTile
  // (for TPC = 1 the CTA's 128 lanes cover kValid = 64 channels and the next
  // 64, whose lanes only load); piece seg >= 1 of the sequence (b, tile), if
  // it has one
  constexpr int kValid = kCh < kDTile ? kCh : kDTile;
  const int b = blockIdx.y, d0 = blockIdx.x * kValid, seg = blockIdx.z;  // seg: the aggregate slot
  const int L = p.L, D = p.D;
  const long long sq = (long long)b * p.plan.ndt + d0 / kBwdTile;
  int piece, c_lo, c_hi;
  if (!agg_slot(p.plan, sq, seg, piece, c_lo, c_hi)) return;  // the whole CTA, before any barrier or copy
  const int t_lo = c_lo * kChunk, t_hi = min(L, c_hi * kChunk);
  const int ntiles = (t_hi - t_lo + kTT - 1) / kTT;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
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
    const int tbase = t_lo + (ntiles - 1 - k) * kTT;
    const int cnt = min(kTT, t_hi - tbase);
    const Act* sr = tile_raw(s);
    const Act* sz = tile_z(s);
    const Act* sg = tile_g(s);
    const Act* Ct = tile_C(s) + 4 * q;  // the Cm values of the lane's 4 states (bf16: widened exactly)
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
      float4 Cv;
      if constexpr (kBf16) {
        const uint2 r = *reinterpret_cast<const uint2*>(Ct + kk * N);
        Cv = make_float4(__uint_as_float(r.x << 16), __uint_as_float(r.x & 0xffff0000u), __uint_as_float(r.y << 16),
                         __uint_as_float(r.y & 0xffff0000u));
      } else {
        Cv = *reinterpret_cast<const float4*>(Ct + kk * N);
      }
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
    float* ag = p.seg_agg + ((((size_t)b * p.nslot + seg) * D + d) * N + 4 * q) * 2;
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
  const int K = plan_pieces(p.plan, (long long)b * p.plan.ndt + d / kBwdTile);
  const long long sq = (long long)b * p.plan.ndt + d / kBwdTile;
  float chi = p.dh_last ? p.dh_last[(size_t)b * per + e] : 0.f;
  for (int k = K - 1; k >= 0; --k) {
    p.seg_carry[((size_t)b * p.nseg + k) * per + e] = chi;
    if (k > 0) {
      // through piece k: its sub-pieces, last first
      int z0, z1;
      agg_piece_slots(p.plan, sq, k, z0, z1);
      for (int z = z1; z >= z0; --z) {
        const float* ag = p.seg_agg + (((size_t)b * p.nslot + z) * per + e) * 2;
        chi = fmaf(ag[0], chi, ag[1]);
      }
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
  constexpr int kCh = kScanThreads / TPC, S = 3;
  return (size_t)S * agg_stage_bytes<Act, TPC>() + (size_t)kTT * (kCh + 4) * 8 + 2 * S * 8;
}

template <typename Act, int TPC, bool kFast, bool kGate>
cudaError_t launch_agg(const BwdTmaParams& P, cudaStream_t stream) {
  auto kern = s6_bwd_agg_kernel<Act, TPC, kFast, kGate>;
  const size_t smem = bwd_agg_smem_bytes<Act, TPC>();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  constexpr int kCh = kScanThreads / TPC;
  constexpr int kValid = kCh < kDTile ? kCh : kDTile;
  const dim3 grid((P.p.D + kValid - 1) / kValid, P.p.B, P.p.nslot);
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

template <typename Act, int TPC, bool kFast, bool kGate, bool kLimit>
cudaError_t launch_one(const BwdTmaParams& P, cudaStream_t stream, bool cooperative) {
  auto kern = s6_bwd_tma_kernel<Act, TPC, kFast, kGate, kLimit>;
  const size_t smem = BwdLayout<Act, TPC>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // persistent: one CTA per range of the plan
  if (!cooperative) {
    kern<<<P.p.plan.P, (2 * TPC + 4) * 32, smem, stream>>>(P);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)P.p.plan.P);
  cfg.blockDim = dim3((2 * TPC + 4) * 32);
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

// The work plan: sms ranges of (near) equal length over all chunk units (one
// persistent CTA per SM, no tail wave) -- contiguous, or split into heads and
// tails when there are fewer sequences than CTAs; sequences cut by a range
// boundary get aggregates for their later pieces.  N outside {4, 8, 16} never takes
// the TMA path: one piece per sequence.
BwdPlan bwd_plan(int B, int L, int D, int N, int sms) {
  BwdPlan pl;
  pl.nch = L > 0 ? (L + kChunk - 1) / kChunk : 0;
  pl.ndt = D > 0 ? (D + kBwdTile - 1) / kBwdTile : 0;
  pl.U = (long long)(B > 0 ? B : 0) * pl.ndt * pl.nch;
  pl.P = (int)std::max<long long>(1, std::min<long long>(std::max(sms, 1), pl.U));
  pl.maxp = 1;
  pl.H = 0;
  pl.handover = false;
  if (pl.U == 0 || !(N == 4 || N == 8 || N == 16)) {
    pl.U = std::max<long long>(pl.U, 1);
    pl.P = 1;
    return pl;
  }
  const long long nseq = (long long)B * pl.ndt;
  if (nseq < pl.P) {
    // fewer sequences than CTAs: every sequence is cut.  Split layout --
    // heads of ceil(U / P) chunks, one per CTA, and short tails for the rest
    // (one sequence per CTA when the head would be the whole sequence)
    const long long H = (pl.U + pl.P - 1) / pl.P;
    if (H >= pl.nch)
      pl.P = (int)nseq;
    else
      pl.H = (int)H;
  }
  for (long long sq = 0; sq < nseq; ++sq) pl.maxp = std::max(pl.maxp, plan_pieces(pl, sq));
  pl.handover = pl.H == 0 && pl.maxp == 2 && (long long)pl.nch <= pl.U / pl.P;
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
  const uint32_t abox = act == SSM_BF16 ? 64 : 32;
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
