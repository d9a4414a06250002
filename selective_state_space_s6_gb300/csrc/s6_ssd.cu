// Mamba-2 SSD forward (scalar A per head; deterministic_backward.py page: the
// ssd_combined kernels -- chunk_cumsum, bmm, chunk_state, state_passing,
// chunk_scan -- with dt per (batch, step, head), one A and one dt_bias per
// head, dt_softplus and dt_limit):
//   delta_t = min(max(softplus(dt_raw_t + dt_bias_h), dt_min), dt_max)
//   S_t = exp(delta_t A_h) S_{t-1} + delta_t B_t x_t^T     (S: N x P per head)
//   y_t = C_t S_t + D_h x_t
// evaluated in its chunked matrix form: per chunk of Q = 64 steps, with
// cum_t the running sum of delta*A inside the chunk,
//   y = ((C B^T) o L) (delta x) + diag(e^cum) C S_in + D x,
//   L[t][s] = e^(cum_t - cum_s) for s <= t, else 0
//   S_out = e^(cum_end) S_in + B^T (w o delta x),  w_s = e^(cum_end - cum_s)
//
// A CTA owns one (batch, head) sequence and walks its chunks in order; the
// chunk's x, Bm and Cm tiles arrive by TMA (128-byte swizzled boxes of 64
// steps x 64 columns) into a two-deep ring.  All four products run on the
// 5th-generation tensor core (bf16 operands straight from the swizzled
// boxes, f32 accumulators in tensor memory, one issuing thread, completion
// on an mbarrier): G = C B^T and C S_in, then Y = M x with M = G o L o delta
// written back to shared memory as bf16, then the state update
// S = e^(cum_end) S + B^T x'.  The state S (N x 64, f32) stays in tensor
// memory for the whole sequence; its bf16 copy in shared memory feeds the
// next chunk's readout.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>

#include "s6_internal.cuh"
#include "s6_math.cuh"
#include "s6_tma.cuh"
#include "s6_umma.cuh"

namespace s6 {

namespace {

constexpr int kQ = 64;           // steps per chunk
constexpr int kP = 64;           // head dimension
constexpr int kSsdThreads = 256;  // 8 warps, two per quarter of the tensor-memory lanes
constexpr int kTileBytes = 64 * 128;  // one 64 x 64 bf16 box (128-byte rows)
constexpr int kVecSet = 320;         // floats of one chunk's decay set

struct SsdParams {
  CUtensorMap map_x, map_B, map_C;  // 64-byte aligned members first
  // H below counts sub-heads (heads x m); the per-head parameters and dt are
  // those of head h / m, and a sub-head's state is the 64 columns (h % m) * 64
  // of its head's [N][64 m] state.  w: a sub-head's columns in memory, 64, or
  // 32 for heads of 32 columns (run as 64 with columns 32..63 zero: the x / dy
  // boxes past a head's 32 columns arrive as zeros, which add exact zeros to
  // every sum, and nothing is written past column 32)
  const __nv_bfloat16* dt_raw;      // [B][L][H / m]
  const float* dt_bias;             // [H / m]
  const float* A_log;               // [H]
  const float* Dp;                  // [H]
  const float* h0;                  // [B][H][N][P] or null
  __nv_bfloat16* y;                 // [B][L][H][P]
  float* h_last;                    // [B][H][N][P] or null
  // [B][H][nch][N][P] bf16 or null: the state entering every chunk, as the
  // bf16 copy the chunk's readout uses (for the backward)
  __nv_bfloat16* chunk_states;
  unsigned int* status;
  float dt_min, dt_max;
  int B, L, H, G, N, m, w;
  // 0: one CTA per sequence, all chunks; 1: the state over chunks
  // [0, seg_chunks) only, from h0, into h_last; 2: two CTAs per sequence,
  // chunks [0, seg_chunks) from h0 and [seg_chunks, end) from h_last
  int mode, seg_chunks;
};

template <int N>
struct SsdSmem {
  static constexpr int NT = N / 64;                    // 64-column boxes of Bm / Cm
  static constexpr int kX = 0;                         // x box [64 s][64 p]
  static constexpr int kBo = kTileBytes;               // Bm boxes [NT][64 s][64 n]
  static constexpr int kCo = kBo + NT * kTileBytes;    // Cm boxes; M = (C B^T) o L o delta over box 0
  static constexpr int kBuf = kCo + NT * kTileBytes;   // one stage
  static constexpr int kXp = 2 * kBuf;                 // x' = w delta x, bf16 [64 s][64 p] (MN-major)
  static constexpr int kS = kXp + kTileBytes;          // S_in (bf16) [N n][64 p] (MN-major)
  static constexpr int kVec = kS + N * 128;            // two sets of decays (see `vec`)
  static constexpr int kBar = kVec + 2 * kVecSet * 4;  // mbarriers and the TMEM address
  static constexpr int kBytes = kBar + 128;
  static constexpr uint32_t kTx = (1 + 2 * NT) * kTileBytes;
  static_assert(kBuf % 1024 == 0 && kXp % 1024 == 0 && kS % 1024 == 0, "swizzled boxes on 1024-byte boundaries");
};

// TMEM columns of a CTA: the state S (N lanes x 64, f32), and three 64 x 64
// accumulators of the chunk: G = C B^T, Y = M x, CS = C S_in.
constexpr uint32_t kColS = 0, kColG = 64, kColY = 128, kColCS = 192, kTmemColsSsd = 256;

// instruction descriptor, kind::f16: f32 D, bf16 A and B, M x 64
__host__ __device__ constexpr uint32_t ssd_idesc(int m, bool a_mn, bool b_mn) { return umma_idesc_bf16(m, 64, a_mn, b_mn); }

template <int N, bool kStateOnly>
__global__ void __launch_bounds__(kSsdThreads) s6_ssd_fwd_kernel(const __grid_constant__ SsdParams P) {
  using SM = SsdSmem<N>;
  constexpr int NT = SM::NT;
  // this CTA's sequence and its chunks [c0, c0 + nch); chunk indices below are
  // local to that range
  const int seg = P.mode == 2 ? (int)(blockIdx.x & 1) : 0;
  const int bh = P.mode == 2 ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int c0 = seg ? P.seg_chunks : 0;
  const int c1 = (P.mode == 1 || (P.mode == 2 && seg == 0)) ? P.seg_chunks : (P.L + kQ - 1) / kQ;
  const int nch = c1 - c0;
  if (nch <= 0) return;
  const float* init = seg ? P.h_last : P.h0;  // the state entering the range
  const bool write_last = P.mode != 2 || seg == 1;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // the 128B swizzle repeats every 1024 bytes: align the base
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* smem = smem_raw + (base - raw);
  // per chunk set (two sets, by chunk parity): (cum, delta) pairs of steps
  // [0, 64) interleaved [0, 128), w*delta [128, 192), e^(cum_end) [192],
  // the blocked-decay flag [193], the blocked factors [256, 320)
  float* vec = reinterpret_cast<float*>(smem + SM::kVec);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SM::kBar);  // [2]: the stages' TMA copies
  uint64_t* bar_cs = full + 2;  // C S_in done
  uint64_t* bar_g = full + 3;   // C B^T done
  uint64_t* bar_y = full + 4;   // M x and the state update done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(full + 5);

  const int b = bh / P.H, h = bh % P.H;   // h: the sub-head
  const int Hr = P.H / P.m, hr = h / P.m;  // heads; this sub-head's head
  const int g = hr / (Hr / P.G);
  // this sub-head's state rows: [N][st_ld] f32 (or bf16 saves), from column st_c0
  const int st_ld = P.w * P.m, st_c0 = (h % P.m) * kP;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float A = -expf(P.A_log[hr]);
  const float bias = P.dt_bias[hr];
  const float Dh = P.Dp[hr];
  // Roles beside the shared row work: thread 0 issues the tensor-core
  // products (C S_in, then M x and the state update, then the next chunk's
  // C B^T, in that order on the tensor core); thread 192 issues the TMA
  // copies; warp 7 computes the decays one chunk ahead.
  constexpr int kTidMma = 0, kTidTma = 192, kWarpDecay = 7;

  if (tid == kTidMma) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    mbar_init(bar_cs, 1);
    mbar_init(bar_g, 1);
    mbar_init(bar_y, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, kTmemColsSsd);
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tquarter = tmem + ((uint32_t)(32 * (warp & 3)) << 16);  // this warp's lane quarter
  const int kq = warp >> 2;  // warps w and w + 4 share a lane quarter and split the columns
  // The 64 x 64 accumulators (M = 64) keep row r in lane (r / 16) * 32 + r % 16;
  // every thread holds 16 columns [col0, col0 + 16) of one row.
  const int row = 16 * (warp & 3) + (lane & 15);
  const int col0 = 32 * kq + 16 * (lane >> 4);
  // rows of S: N = 128 -> row n = lane of the quarter (every lane); N = 64 ->
  // the M = 64 layout; a thread holds 32 columns [sc, sc + 32)
  const bool has_srow = N == 128 || lane < 16;
  const int srow = N == 128 ? 32 * (warp & 3) + lane : row;
  const int sc = 32 * kq;
  // this thread's state columns exist in memory (w = 32: columns 32..63 are
  // the zero padding, exactly zero throughout, never read or written)
  const bool mem_s = has_srow && sc < P.w;

  auto issue = [&](int ci) {  // chunk ci's boxes into stage ci & 1 (one thread; no Cm for the state alone)
    const int s = ci & 1, c = c0 + ci;
    unsigned char* st = smem + s * SM::kBuf;
    mbar_arrive_expect_tx(&full[s], kStateOnly ? (uint32_t)((1 + NT) * kTileBytes) : SM::kTx);
    if (P.w == kP)
      tma_load_3d(st + SM::kX, &P.map_x, &full[s], h * kP, c * kQ, b);
    else  // [B][L][H][w] as 4D: the box's columns past w are zeros
      tma_load_4d(st + SM::kX, &P.map_x, &full[s], 0, h, c * kQ, b);
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      tma_load_3d(st + SM::kBo + j * kTileBytes, &P.map_B, &full[s], g * N + 64 * j, c * kQ, b);
      if (!kStateOnly) tma_load_3d(st + SM::kCo + j * kTileBytes, &P.map_C, &full[s], g * N + 64 * j, c * kQ, b);
    }
  };
  if (tid == kTidTma) {
    tma_prefetch_desc(&P.map_x);
    issue(0);
  }

  // 8 consecutive values as one 16-byte unit of a 128B-swizzled [rows][64] bf16 image
  auto put8 = [&](uint32_t off, int r, int c8, const float* v) {
    *reinterpret_cast<uint4*>(smem + off + swz(r, c8)) =
        make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]), pack_bf16(v[6], v[7]));
  };
  // this thread's 32 values of the state entering chunk c (row srow, columns
  // sc .. sc + 31) to the saved chunk states, as bf16 (the readout's copy)
  const int nch_all = (P.L + kQ - 1) / kQ;
  auto save_state = [&](int c, const float* v) {
    if (!P.chunk_states || kStateOnly || !mem_s) return;
    uint4* dst = reinterpret_cast<uint4*>(P.chunk_states + ((((size_t)b * Hr + hr) * nch_all + c) * N + srow) * st_ld + st_c0 + sc);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      dst[q] = make_uint4(pack_bf16(v[8 * q], v[8 * q + 1]), pack_bf16(v[8 * q + 2], v[8 * q + 3]),
                          pack_bf16(v[8 * q + 4], v[8 * q + 5]), pack_bf16(v[8 * q + 6], v[8 * q + 7]));
  };

  // The decay warp reads each chunk's dt one chunk ahead (two steps per
  // lane; the raw bits stay untouched until they are used, so the load's
  // latency hides behind a whole chunk) and turns them into delta, the
  // running sum of delta*A, the weights e^(cum_end - cum_s) delta_s and the
  // chunk's total decay (set ci & 1 of `vec`, ci the chunk within the CTA's range).
  const unsigned short* dt_bits = reinterpret_cast<const unsigned short*>(P.dt_raw);
  unsigned short raw_next[2] = {0, 0};
  auto load_dt = [&](int ci) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int t = min((c0 + ci) * kQ + 2 * lane + i, P.L - 1);  // past the end: any valid step, masked later
      raw_next[i] = dt_bits[((size_t)b * P.L + t) * Hr + hr];
    }
  };
  auto chunk_decays = [&](int ci) {
    float* v = vec + (ci & 1) * kVecSet;
    float d2[2], a2[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int t = (c0 + ci) * kQ + 2 * lane + i;
      const float r = __bfloat162float(__ushort_as_bfloat16(raw_next[i]));
      const float d = t < P.L ? clamp_dt(softplus_fast(r + bias), P.dt_min, P.dt_max) : 0.f;
      d2[i] = d;
      a2[i] = d * A;
    }
    float run = a2[0] + a2[1];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float u = __shfl_up_sync(0xffffffffu, run, o);
      if (lane >= o) run += u;
    }
    const float end = __shfl_sync(0xffffffffu, run, 31);
    const float c1 = run, c0 = run - a2[1];
    *reinterpret_cast<float4*>(v + 4 * lane) = make_float4(c0, d2[0], c1, d2[1]);
    v[128 + 2 * lane] = fast_exp(end - c0) * d2[0];
    v[128 + 2 * lane + 1] = fast_exp(end - c1) * d2[1];
    if (lane == 0) v[192] = fast_exp(end);
    // per step s: e^(cum_b - cum_s) delta_s with b the first step of its
    // 8-step block; usable when no block decays by more than e^64
    const float cb = __shfl_sync(0xffffffffu, c0, lane & ~3);
    v[256 + 2 * lane] = fast_exp(cb - c0) * d2[0];
    v[256 + 2 * lane + 1] = fast_exp(cb - c1) * d2[1];
    const bool blocked = __all_sync(0xffffffffu, cb - c1 < 64.f);
    if (lane == 0) v[193] = blocked ? 1.f : 0.f;
  };
  if (warp == kWarpDecay) {
    load_dt(0);
    chunk_decays(0);
    load_dt(1);
  }

  // Shared-memory matrix descriptors of the operands; the K steps add their
  // byte offset / 16 to the start-address field.
  const uint32_t st0 = base, st1 = base + SM::kBuf;
  const uint64_t dC0 = umma_desc_sw128(st0 + SM::kCo, 16u, 1024u), dC1 = umma_desc_sw128(st1 + SM::kCo, 16u, 1024u);
  const uint64_t dBk0 = umma_desc_sw128(st0 + SM::kBo, 16u, 1024u), dBk1 = umma_desc_sw128(st1 + SM::kBo, 16u, 1024u);
  const uint64_t dBmn0 = umma_desc_sw128(st0 + SM::kBo, (uint32_t)kTileBytes, 1024u),
                 dBmn1 = umma_desc_sw128(st1 + SM::kBo, (uint32_t)kTileBytes, 1024u);
  const uint64_t dX0 = umma_desc_sw128(st0 + SM::kX, (uint32_t)kTileBytes, 1024u),
                 dX1 = umma_desc_sw128(st1 + SM::kX, (uint32_t)kTileBytes, 1024u);
  // Cm / M (K-major), Bm rows as a K-major B^T, Bm as an MN-major B^T, x (MN-major) of stage s
  auto dC = [&](int s) { return s ? dC1 : dC0; };
  auto dBk = [&](int s) { return s ? dBk1 : dBk0; };
  auto dBmn = [&](int s) { return s ? dBmn1 : dBmn0; };
  auto dX = [&](int s) { return s ? dX1 : dX0; };
  const uint64_t dS = umma_desc_sw128(base + SM::kS, (uint32_t)kTileBytes, 1024u);    // S_in, MN-major
  const uint64_t dXp = umma_desc_sw128(base + SM::kXp, (uint32_t)kTileBytes, 1024u);  // x', MN-major
  constexpr uint32_t kIdG = ssd_idesc(64, false, false);  // C (K-major) x B^T (K-major rows of Bm)
  constexpr uint32_t kIdKM = ssd_idesc(64, false, true);  // K-major A x MN-major B: C S_in, M x
  constexpr uint32_t kIdS = ssd_idesc(N, true, true);     // B^T (MN-major) x x' (MN-major)
  // G = C B^T of the chunk in stage s: K = n, 16 at a time (32 bytes into a
  // 128-byte row), the next 64 n one box on; committed to bar_g
  auto issue_g = [&](int s) {
#pragma unroll
    for (int k = 0; k < N / 16; ++k) {
      const uint64_t ko = (uint64_t)(((k / 4) * kTileBytes + (k % 4) * 32) >> 4);
      umma_f16(tmem + kColG, dC(s) + ko, dBk(s) + ko, kIdG, k > 0 ? 1u : 0u);
    }
    umma_commit(bar_g);
  };

  __syncthreads();  // decays of chunk 0 published
  // the initial state: S = e^(cum_end of chunk 0) h0 in TMEM (ready for the
  // first update), h0 as bf16 for the first readout
  {
    float v[32];
    const float* h0 = (init && mem_s) ? init + (((size_t)b * Hr + hr) * N + srow) * st_ld + st_c0 + sc : nullptr;
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = h0 ? h0[i] : 0.f;
    if (!kStateOnly && has_srow)
#pragma unroll
      for (int q = 0; q < 4; ++q) put8(SM::kS, srow, 4 * kq + q, v + 8 * q);
    save_state(c0, v);
    const float dec0 = vec[192];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] *= dec0;
    __syncwarp();
    tmem_st32(tquarter + kColS + (uint32_t)sc, v);
    tmem_wait_st();
    fence_proxy_async_smem();
    tmem_fence_before_sync();
  }
  if (!kStateOnly && tid == kTidMma && mbar_wait(&full[0], 0u, P.status)) issue_g(0);
  __syncthreads();

  for (int ci = 0; ci < nch; ++ci) {
    const int s = ci & 1;
    const int t0 = (c0 + ci) * kQ;
    const uint32_t ph = (uint32_t)(ci & 1);
    const bool ok = mbar_wait(&full[s], (uint32_t)((ci >> 1) & 1), P.status);
    if (__syncthreads_or(!ok)) break;  // the copy never came: stop, uniformly
    unsigned char* st = smem + s * SM::kBuf;
    const float* cum = vec + s * kVecSet;  // cum of step t at cum[2 t], delta at cum[2 t + 1]
    const float* wd = cum + 128;

    // ---- CS = C S_in (B = S_in [n][p]: 16 rows of n per K step)
    if (!kStateOnly && tid == kTidMma) {
      tmem_fence_after_sync();
#pragma unroll
      for (int k = 0; k < N / 16; ++k) {
        const uint64_t ko = (uint64_t)(((k / 4) * kTileBytes + (k % 4) * 32) >> 4);
        umma_f16(tmem + kColCS, dC(s) + ko, dS + (uint64_t)(k * 2048 >> 4), kIdKM, k > 0 ? 1u : 0u);
      }
      umma_commit(bar_cs);
    }
    // the next chunk's boxes into the other stage (free since the last chunk)
    if (tid == kTidTma && ci + 1 < nch) issue(ci + 1);
    // ---- x' = w delta x (state-update operand)
    {
      const float w = wd[row];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int c8 = col0 / 8 + q;
        const uint4 xv = *reinterpret_cast<const uint4*>(st + SM::kX + swz(row, c8));
        const uint32_t xin[4] = {xv.x, xv.y, xv.z, xv.w};
        uint32_t xo[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 xe = unpack_bf16(xin[k]);
          xo[k] = pack_bf16(w * xe.x, w * xe.y);
        }
        *reinterpret_cast<uint4*>(smem + SM::kXp + swz(row, c8)) = make_uint4(xo[0], xo[1], xo[2], xo[3]);
      }
    }
    // the next chunk's decays; its successor's dt in flight
    if (warp == kWarpDecay && ci + 1 < nch) {
      chunk_decays(ci + 1);
      load_dt(ci + 2);
    }
    if constexpr (!kStateOnly) {
    // ---- M[t][s] = G[t][s] e^(cum_t - cum_s) delta_s for s <= t as bf16
    // over Cm box 0, once C B^T and C S_in are done with it
    mbar_wait(bar_g, ph, P.status);
    mbar_wait(bar_cs, ph, P.status);
    tmem_fence_after_sync();
    {
      float v[16];
      __syncwarp();
      tmem_ld16x2_16(tquarter + kColG + (uint32_t)(32 * kq), v);
      const float ct = cum[2 * row];
      const int s0 = col0;
      if (cum[193] != 0.f) {  // e^(cum_t - cum_s) = e^(cum_t - cum_b) e^(cum_b - cum_s), 8-step blocks b
        const float* qs = cum + 256;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int sb = s0 + 8 * k;
          const float e = fast_exp(ct - cum[2 * sb]);
          const float4 qa = *reinterpret_cast<const float4*>(qs + sb);
          const float4 qb = *reinterpret_cast<const float4*>(qs + sb + 4);
          const float qv[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
          for (int i = 0; i < 8; ++i) v[8 * k + i] = sb + i <= row ? v[8 * k + i] * e * qv[i] : 0.f;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
          const float4 cd = *reinterpret_cast<const float4*>(cum + 2 * (s0 + j));  // steps s0 + j, s0 + j + 1
          v[j] = s0 + j <= row ? v[j] * fast_exp(ct - cd.x) * cd.y : 0.f;
          v[j + 1] = s0 + j + 1 <= row ? v[j + 1] * fast_exp(ct - cd.z) * cd.w : 0.f;
        }
      }
#pragma unroll
      for (int q = 0; q < 2; ++q) put8(SM::kCo + s * SM::kBuf, row, s0 / 8 + q, v + 8 * q);
    }
    }
    fence_proxy_async_smem();
    tmem_fence_before_sync();
    __syncthreads();  // M and x' complete; decays of the next chunk published
    // ---- Y = M x and S += B^T x' (S already carries this chunk's decay)
    if (tid == kTidMma) {
      tmem_fence_after_sync();
#pragma unroll
      for (int k = 0; k < 4; ++k)  // K = s
        if (!kStateOnly)
          umma_f16(tmem + kColY, dC(s) + (uint64_t)(k * 32 >> 4), dX(s) + (uint64_t)(k * 2048 >> 4), kIdKM,
                 k > 0 ? 1u : 0u);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        umma_f16(tmem + kColS, dBmn(s) + (uint64_t)(k * 2048 >> 4), dXp + (uint64_t)(k * 2048 >> 4), kIdS, 1u);
      umma_commit(bar_y);
      // the next chunk's G, queued behind this chunk's products
      if (!kStateOnly && ci + 1 < nch && mbar_wait(&full[s ^ 1], (uint32_t)(((ci + 1) >> 1) & 1), P.status))
        issue_g(s ^ 1);
    }
    mbar_wait(bar_y, ph, P.status);
    tmem_fence_after_sync();
    // ---- y = Y + e^cum CS + D x for this thread's row and half
    if constexpr (!kStateOnly) {
      float yv[16], cv[16];
      __syncwarp();
      tmem_ld16x2_16(tquarter + kColY + (uint32_t)(32 * kq), yv);
      tmem_ld16x2_16(tquarter + kColCS + (uint32_t)(32 * kq), cv);
      const float et = fast_exp(cum[2 * row]);
      __nv_bfloat16* yrow = P.y + (((size_t)b * P.L + t0 + row) * P.H + h) * P.w;
      const bool store = t0 + row < P.L && col0 < P.w;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int c8 = col0 / 8 + q;
        const uint4 xv = *reinterpret_cast<const uint4*>(st + SM::kX + swz(row, c8));
        const uint32_t xin[4] = {xv.x, xv.y, xv.z, xv.w};
        uint32_t yo[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 xe = unpack_bf16(xin[k]);
          const int j = 8 * q + 2 * k;
          yo[k] = pack_bf16(yv[j] + et * cv[j] + Dh * xe.x, yv[j + 1] + et * cv[j + 1] + Dh * xe.y);
        }
        if (store) *reinterpret_cast<uint4*>(yrow + 8 * c8) = make_uint4(yo[0], yo[1], yo[2], yo[3]);
      }
    }
    // ---- the state after the chunk: S_in of the next readout (bf16) and,
    // scaled by the next chunk's decay, back into TMEM; or h_last
    {
      float v[32];
      __syncwarp();
      tmem_ld32(tquarter + kColS + (uint32_t)sc, v);
      if (ci + 1 < nch) {
        if (!kStateOnly && has_srow)
#pragma unroll
          for (int q = 0; q < 4; ++q) put8(SM::kS, srow, 4 * kq + q, v + 8 * q);
        save_state(c0 + ci + 1, v);
        const float dec1 = vec[(s ^ 1) * kVecSet + 192];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= dec1;
        __syncwarp();
        tmem_st32(tquarter + kColS + (uint32_t)sc, v);
        tmem_wait_st();
      } else if (write_last && P.h_last && mem_s) {
        float* hl = P.h_last + (((size_t)b * Hr + hr) * N + srow) * st_ld + st_c0 + sc;
#pragma unroll
        for (int i = 0; i < 32; i += 2) *reinterpret_cast<float2*>(hl + i) = make_float2(v[i], v[i + 1]);
      }
    }
    fence_proxy_async_smem();
    tmem_fence_before_sync();
    __syncthreads();  // S_in complete; every product on this stage done
  }
  tmem_fence_after_sync();
  if (warp == 0) tmem_dealloc(tmem, kTmemColsSsd);
}

template <int N, bool kStateOnly>
cudaError_t launch_k(const SsdParams& P, unsigned grid, cudaStream_t stream) {
  auto kern = s6_ssd_fwd_kernel<N, kStateOnly>;
  const size_t smem = SsdSmem<N>::kBytes + 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kSsdThreads, smem, stream>>>(P);
  return cudaGetLastError();
}

// With at most half as many sequences as SMs, each sequence is cut in two: a
// state-only pass over the first half writes the state at the cut into
// h_last, then one launch runs both halves at once (the second from h_last),
// every half on an SM of its own.  The state-only pass costs about half a
// full chunk per chunk, so with more sequences, where halves would share SMs,
// the cut does not pay.  Needs h_last (not overlapping h0) and four chunks
// or more.
template <int N>
cudaError_t launch_n(SsdParams P, cudaStream_t stream) {
  const int nch = (P.L + kQ - 1) / kQ;
  const int sms = device_sm_count();  // cached per device (0 on error: no cut)
  const long long seqs = (long long)P.B * P.H;
  // h0 and h_last may be one buffer (the state updated in place): then the
  // first pass would overwrite h0 before the first halves read it
  const size_t sbytes = (size_t)seqs * N * P.w * sizeof(float);
  const char *s0 = reinterpret_cast<const char*>(P.h0), *s1 = reinterpret_cast<const char*>(P.h_last);
  const bool overlap = s0 && s1 && s0 < s1 + sbytes && s1 < s0 + sbytes;
  if (P.h_last == nullptr || overlap || nch < 4 || 2 * seqs > sms) {
    P.mode = 0;
    P.seg_chunks = 0;
    return launch_k<N, false>(P, (unsigned)seqs, stream);
  }
  P.seg_chunks = nch / 2;
  P.mode = 1;
  cudaError_t e = launch_k<N, true>(P, (unsigned)seqs, stream);
  if (e != cudaSuccess) return e;
  P.mode = 2;
  return launch_k<N, false>(P, (unsigned)(2 * seqs), stream);
}

}  // namespace

// headdim P = 32 (one sub-head of 32 columns), or 64 m (m sub-heads per head;
// m <= 4 keeps every index in range of the checks made on the whole tensors)
bool ssd_supported(int act, int P, int N) {
  return act == SSM_BF16 && (P == kP / 2 || (P % kP == 0 && P >= kP && P <= 4 * kP)) && (N == 64 || N == 128);
}

bool ssd_encode_x_map(void* map, const void* base, const SsdArgs& a) {
  const uint64_t e = 2, Hs = (uint64_t)a.H * a.m;  // sub-heads
  CUtensorMap* m = static_cast<CUtensorMap*>(map);
  if (a.w == kP) {
    const uint64_t dims[3] = {Hs * kP, (uint64_t)a.L, (uint64_t)a.B};
    const uint64_t strides[2] = {Hs * kP * e, (uint64_t)a.L * Hs * kP * e};
    const uint32_t box[3] = {64, kQ, 1};
    return encode_tile_map(m, base, true, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  const uint64_t w = (uint64_t)a.w;
  const uint64_t dims[4] = {w, Hs, (uint64_t)a.L, (uint64_t)a.B};
  const uint64_t strides[3] = {w * e, Hs * w * e, (uint64_t)a.L * Hs * w * e};
  const uint32_t box[4] = {64, 1, kQ, 1};
  return encode_tile_map(m, base, true, 4, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

cudaError_t launch_ssd_fwd(const SsdArgs& a, cudaStream_t stream) {
  SsdParams P;
  memset(&P, 0, sizeof(P));
  const uint64_t e = 2;
  if (!ssd_encode_x_map(&P.map_x, a.x, a)) return cudaErrorInvalidValue;
  {
    const uint64_t dims[3] = {(uint64_t)a.G * a.N, (uint64_t)a.L, (uint64_t)a.B};
    const uint64_t strides[2] = {(uint64_t)a.G * a.N * e, (uint64_t)a.L * a.G * a.N * e};
    const uint32_t box[3] = {64, kQ, 1};
    if (!encode_tile_map(&P.map_B, a.Bm, true, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tile_map(&P.map_C, a.Cm, true, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  P.dt_raw = static_cast<const __nv_bfloat16*>(a.dt_raw);
  P.dt_bias = a.dt_bias;
  P.A_log = a.A_log;
  P.Dp = a.Dp;
  P.h0 = a.h0;
  P.y = static_cast<__nv_bfloat16*>(a.y);
  P.h_last = a.h_last;
  P.chunk_states = static_cast<__nv_bfloat16*>(a.chunk_states);
  P.status = a.status;
  P.dt_min = a.dt_min;
  P.dt_max = a.dt_max;
  P.B = a.B;
  P.L = a.L;
  P.H = a.H * a.m;
  P.m = a.m;
  P.w = a.w;
  P.G = a.G;
  P.N = a.N;
  return a.N == 128 ? launch_n<128>(P, stream) : launch_n<64>(P, stream);
}

}  // namespace s6
