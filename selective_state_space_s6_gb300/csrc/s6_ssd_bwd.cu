// Mamba-2 SSD backward (deterministic_backward.py page: the backward of the
// ssd_combined kernels -- dx, dB, dC, the dt and A gradients through
// chunk_cumsum -- with single-writer kernels and sums in a fixed order).
//
// The gradient of loss = sum(dy * y) + sum(dh_last * h_last) through the
// chunked matrix form of the forward, per chunk of Q = 64 steps, walked last
// to first with dS the gradient of the state leaving the chunk:
//   cum_t = sum_{j <= t} delta_j A,  L[t][s] = e^(cum_t - cum_s) for s <= t,
//   w_s = e^(cum_end - cum_s),  G = C B^T,  Z = dy x^T,
//   dx     = D dy + (L o G o delta_s)^T dy + diag(w delta) B dS
//   dB     = (L o Z o delta_s)^T C + diag(w delta) x dS^T
//   dC     = diag(e^cum) dy S_in^T + (L o Z o delta_s) B
//   dS_in  = e^(cum_end) dS + C^T diag(e^cum) dy
//   dcum_t = rowsum_t(F) - colsum_t(F) + e^(cum_t) dy_t . (C S_in)_t - w_t delta_t (B dS)_t . x_t
//            (+ <dS, S_out> at the chunk's last step),  F = L o G o Z o delta_s
//   ddelta_s = colsum_s(L o G o Z) + w_s (B dS)_s . x_s + A sum_{t >= s} dcum_t
//   dA     += sum_s delta_s sum_{t >= s} dcum_t
// with <dS, S_out> = e^(cum_end) <dS, S_in> + sum_s w_s delta_s (B dS)_s . x_s.
// These are the per-chunk products the oracle's backward is pinned to (its
// chunked form, written independently in numpy).
//
// A CTA owns one (batch, head) and walks its chunks backwards -- or, with
// more sequences than SMs, a range of chunks per SM that cuts a sequence at
// most once, the state gradient handed over between the two pieces (see
// SsdBwdParams); x, dy, Bm, Cm and the chunk's entering state S_in (saved by
// the forward as bf16, the copy its readout used) arrive by TMA into a
// two-deep ring of 128B-swizzled boxes.
// Every product runs on the 5th-generation tensor core (bf16 operands, f32
// accumulators in tensor memory, one issuing thread): first G, Z, C S_in,
// B dS and the state update dS <- e^(cum_end) dS + C^T dy', then -- after
// the threads have written the masked, decayed images L o G o delta and
// L o Z o delta as bf16 -- dx (accumulated on top of the scaled B dS), dB and
// dC.  dS (N x 64, f32) stays in tensor memory.  dBm/dCm are summed over the
// heads of a group by a second kernel in ascending head order, dA_log / dDp /
// ddt_bias over the batch in ascending order: no floating-point atomics.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "s6_internal.cuh"
#include "s6_math.cuh"
#include "s6_tma.cuh"
#include "s6_umma.cuh"

namespace s6 {

namespace {

constexpr int kQ = 64;              // steps per chunk
constexpr int kP = 64;              // head dimension
constexpr int kThreads = 256;       // 8 warps, two per quarter of the tensor-memory lanes
constexpr int kTileBytes = 64 * 128;  // one 64 x 64 bf16 box (128-byte rows)
constexpr int kVecSet = 6 * 64 + 8;   // floats of one chunk's decay set

struct SsdBwdParams {
  CUtensorMap map_x, map_dy, map_B, map_C, map_S;  // 64-byte aligned members first
  // H below counts sub-heads (heads x m; headdim 64 m): the per-head
  // parameters, dt and ddt_raw are those of head h / m, and a sub-head's state
  // (gradient) is the 64 columns (h % m) * 64 of its head's [N][64 m] one.
  // w: a sub-head's columns in memory, 64, or 32 for heads of 32 columns (run
  // as 64 whose columns 32..63 are zero: the x, dy and saved-state boxes past
  // column 32 arrive as zeros, so the state gradient's padding stays zero and
  // every sum over columns only gains exact zeros; nothing is written there)
  const __nv_bfloat16* dt_raw;  // [B][L][H / m]
  const float* dt_bias;         // [H / m]
  const float* A_log;           // [H]
  const float* Dp;              // [H]
  const float* dh_last;         // [B][H][N][P] or null
  __nv_bfloat16* dx;            // [B][L][H][P]
  __nv_bfloat16* ddt_raw;       // [B][L][H]
  float* dh0;                   // [B][H][N][P] or null
  float* ws_dB;                 // [B][L][H][N] per-head dBm terms
  float* ws_dC;                 // [B][L][H][N] per-head dCm terms
  float* ws_sc;                 // [B][H][2 pieces][3]: sum dA, sum dDp, sum ddt_bias
  float* ws_ddt;                // m > 1: [B][L][H] per-sub-head ddt_raw terms
  unsigned int* status;
  float dt_min, dt_max;
  int B, L, H, G, N, m, w;
  int Hr;  // heads (H / m)
  // The walk: the B H sequences (b major) of ceil(L / 64) chunks laid end to
  // end, cut into gridDim.x equal ranges, one per CTA.  gridDim.x = B H: one
  // sequence per CTA.  Fewer (one per SM, all resident: cooperative launch):
  // a range is at least a sequence long, so a sequence is cut at most once,
  // into a first piece at the end of one range and a last piece at the start
  // of the next; the CTA holding the last piece walks it first and hands the
  // state gradient it ends with (carry, [B H][N][64] f32) over through
  // seq_flag ([B H], zeroed before the launch) to the CTA holding the first
  // piece, which walks it last.
  int* seq_flag;
  float* carry;
};

template <int N>
struct BwdSmem {
  static constexpr int NT = N / 64;                     // 64-row boxes of Bm / Cm / S_in
  static constexpr int kX = 0;                          // x box [64 s][64 p]
  static constexpr int kDY = kTileBytes;                // dy box [64 t][64 p]
  static constexpr int kBo = 2 * kTileBytes;            // Bm boxes [NT][64 s][64 n]
  static constexpr int kCo = kBo + NT * kTileBytes;     // Cm boxes
  static constexpr int kSo = kCo + NT * kTileBytes;     // S_in (bf16) [N n][64 p]
  static constexpr int kBuf = kSo + NT * kTileBytes;    // one stage
  static constexpr int kDS = 2 * kBuf;                  // dS (bf16) [N n][64 p]
  static constexpr int kXw = kDS + NT * kTileBytes;     // x'' = diag(w delta) x [64 s][64 p]
  static constexpr int kDYe = kXw + kTileBytes;         // dy' = diag(e^cum) dy [64 t][64 p]
  static constexpr int kGl = kDYe + kTileBytes;         // L o G o delta_s [64 t][64 s]
  static constexpr int kZl = kGl + kTileBytes;          // L o Z o delta_s [64 t][64 s]
  static constexpr int kD2 = kZl + kTileBytes;          // f32 [64 t][65] (L o G o Z) for the column sums
  static constexpr int kRow = kD2 + 64 * 65 * 4;        // f32 [3][64 rows][4 parts]
  static constexpr int kRed = kRow + 3 * 64 * 4 * 4;    // f32 [256] block reduction scratch
  static constexpr int kVec = kRed + 256 * 4;           // two decay sets
  static constexpr int kBar = kVec + 2 * kVecSet * 4;   // mbarriers and the TMEM address
  static constexpr int kBytes = kBar + 128;
  static constexpr uint32_t kTx = (2 + 3 * NT) * kTileBytes;
  static_assert(kBuf % 1024 == 0 && kDS % 1024 == 0 && kXw % 1024 == 0 && kGl % 1024 == 0 && kZl % 1024 == 0,
                "swizzled images on 1024-byte boundaries");
};

// TMEM columns: the state gradient dS (N lanes x 64, f32); the chunk's 64-row
// accumulators G = C B^T, Z = dy x^T, CS = C S_in, X = B dS (then dx), and
// dB (N columns); dC (N columns) reuses G and Z's columns.
constexpr uint32_t kColS = 0, kColG = 64, kColZ = 128, kColCS = 192, kColX = 256, kColB = 320, kColC = 64,
                   kTmemCols = 512;

// decay set of a chunk (floats): delta [0,64), cum [64,128), e^cum [128,192),
// w = e^(cum_end - cum) [192,256), sigmoid(s) * mask [256,320), w*delta
// [320,384), e^(cum_end) [384]
//
// kCut: ranges of chunks that may cut sequences (one CTA per SM); else one
// CTA per sequence (gridDim.x = B H), whose walk is that sequence alone.
template <int N, bool kCut>
__global__ void __launch_bounds__(kThreads, 1) s6_ssd_bwd_kernel(const __grid_constant__ SsdBwdParams P) {
  using SM = BwdSmem<N>;
  constexpr int NT = SM::NT;
  const int nch = (P.L + kQ - 1) / kQ;
  // this CTA's range of chunk units [u_begin, u_end) and the n-th chunk of
  // its walk: pieces in order (the first from u_begin to its sequence's end,
  // then whole sequences, the last possibly cut short), each piece's chunks
  // last first
  const long long U = (long long)P.B * P.H * nch;
  const long long u_begin = (long long)blockIdx.x * U / gridDim.x;
  const long long u_end = (long long)(blockIdx.x + 1) * U / gridDim.x;
  const int nwalk = (int)(u_end - u_begin);
  struct WalkPos {
    int sq, c, c_lo, c_hi;  // sequence, chunk, the piece's chunks [c_lo, c_hi)
  };
  // the walk's first piece: chunks [lo0, hi0) of sequence sq0; its last
  // sequence sqz ends at chunk hiz
  const int sq0 = (int)(u_begin / nch), lo0 = (int)(u_begin - (long long)sq0 * nch);
  const int hi0 = (int)min((long long)nch, u_end - (long long)sq0 * nch);
  const int sqz = (int)((u_end - 1) / nch), hiz = (int)(u_end - (long long)sqz * nch);
  // A walker starts before the walk's first chunk; step() moves it to the
  // next chunk and says whether that chunk starts a piece.  (Every role that
  // follows the walk -- the copies, the decays, the row work -- keeps one,
  // so that no role divides per chunk.)
  auto walk_start = [&]() { return WalkPos{sq0, hi0, lo0, hi0}; };
  auto step = [&](WalkPos& w) {
    if constexpr (!kCut) return --w.c == nch - 1;  // one sequence, chunks nch-1 .. 0
    if (--w.c >= w.c_lo) return w.c == w.c_hi - 1;
    ++w.sq;
    w.c_lo = 0;
    w.c_hi = w.sq == sqz ? hiz : nch;
    w.c = w.c_hi - 1;
    return true;
  };
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* smem = smem_raw + (base - raw);
  float* vec = reinterpret_cast<float*>(smem + SM::kVec);
  float* d2 = reinterpret_cast<float*>(smem + SM::kD2);
  float* rowp = reinterpret_cast<float*>(smem + SM::kRow);
  float* red = reinterpret_cast<float*>(smem + SM::kRed);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SM::kBar);  // [2] the stages' TMA copies
  uint64_t* bar1 = full + 2;                                       // first products done
  uint64_t* bar2 = full + 3;                                       // second products done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(full + 4);

  // a sequence sq is (batch sq / H, sub-head sq % H) of head (sq % H) / m;
  // a sub-head's state-gradient rows: [N][st_ld] of its head, from column
  // (h % m) * 64
  const int Hr = P.Hr;  // heads
  const int st_ld = P.w * P.m;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Roles beside the row work: threads 0, 32 and 64 issue the tensor-core
  // products (three issuers in three warps, each accumulator written by one
  // of them; both groups complete when all three have committed); thread 192
  // issues the TMA copies; warp 7 computes the decays a chunk ahead; warps 4
  // and 5 form the log-decay gradient while the second group runs.
  constexpr int kTidMma = 0, kTidTma = 192, kWarpDecay = 7, kIssuers = 3, kTidDcum = 128;
  const bool issuer = tid < 32 * kIssuers && lane == 0;
  const int iss = tid >> 5;  // which issuer

  if (tid == kTidMma) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    mbar_init(bar1, kIssuers);
    mbar_init(bar2, kIssuers);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tquarter = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
  const int kq = warp >> 2;
  // 64-row accumulators: row r in lane (r / 16) * 32 + r % 16; this thread
  // holds 16 columns [col0, col0 + 16) of row `row`
  const int row = 16 * (warp & 3) + (lane & 15);
  const int col0 = 32 * kq + 16 * (lane >> 4);
  // rows of dS: N = 128 -> row n = lane of the quarter; N = 64 -> the 64-row
  // layout; this thread holds 32 columns [sc, sc + 32)
  const bool has_srow = N == 128 || lane < 16;
  const int srow = N == 128 ? 32 * (warp & 3) + lane : row;
  const int sc = 32 * kq;
  const bool mem_s = has_srow && sc < P.w;  // this thread's state columns exist in memory

  // the walk's chunk n into stage n & 1 (thread kTidTma, n = 0, 1, 2, ...)
  WalkPos wt = walk_start();
  int tb = sq0 / P.H, th = sq0 % P.H, thr = th / P.m, tg = thr / (Hr / P.G);
  auto issue = [&](int n) {
    if (step(wt) && kCut) tb = wt.sq / P.H, th = wt.sq % P.H, thr = th / P.m, tg = thr / (Hr / P.G);
    const int s = n & 1, c = wt.c, b = tb, h = th, hr = thr, g = tg;
    const int st_c0 = (h % P.m) * kP;
    unsigned char* st = smem + s * SM::kBuf;
    mbar_arrive_expect_tx(&full[s], SM::kTx);
    if (P.w == kP) {
      tma_load_3d(st + SM::kX, &P.map_x, &full[s], h * kP, c * kQ, b);
      tma_load_3d(st + SM::kDY, &P.map_dy, &full[s], h * kP, c * kQ, b);
    } else {  // [B][L][H][w] as 4D: the box's columns past w are zeros
      tma_load_4d(st + SM::kX, &P.map_x, &full[s], 0, h, c * kQ, b);
      tma_load_4d(st + SM::kDY, &P.map_dy, &full[s], 0, h, c * kQ, b);
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      tma_load_3d(st + SM::kBo + j * kTileBytes, &P.map_B, &full[s], g * N + 64 * j, c * kQ, b);
      tma_load_3d(st + SM::kCo + j * kTileBytes, &P.map_C, &full[s], g * N + 64 * j, c * kQ, b);
      tma_load_2d(st + SM::kSo + j * kTileBytes, &P.map_S, &full[s], st_c0, (((b * Hr + hr) * nch) + c) * N + 64 * j);
    }
  };
  if (tid == kTidTma) {
    tma_prefetch_desc(&P.map_x);
    issue(0);
  }

  auto put8 = [&](uint32_t off, int r, int c8, const float* v) {
    *reinterpret_cast<uint4*>(smem + off + swz(r, c8)) =
        make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]), pack_bf16(v[6], v[7]));
  };
  auto get8 = [&](uint32_t off, int r, int c8, float* v) {
    const uint4 u = *reinterpret_cast<const uint4*>(smem + off + swz(r, c8));
    const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 e = unpack_bf16(w4[k]);
      v[2 * k] = e.x;
      v[2 * k + 1] = e.y;
    }
  };

  // decays of the walk's chunk n into set (n & 1) (warp kWarpDecay; two steps per
  // lane).  The dt of a chunk are read one chunk ahead and kept as raw bits
  // until used, so that the load's latency hides behind a whole chunk.
  const unsigned short* dt_bits = reinterpret_cast<const unsigned short*>(P.dt_raw);
  unsigned short raw_next[2] = {0, 0};
  // the chunk's index and its head's A and dt_bias (with pieces: formed
  // when its dt is read, a chunk ahead; else the sequence's, once)
  int c_next = 0;
  WalkPos wd = walk_start();
  int db = sq0 / P.H, dhr = (sq0 % P.H) / P.m;
  float a_next = -expf(P.A_log[dhr]), bias_next = P.dt_bias[dhr];
  auto load_dt = [&](int n) {
    if (step(wd) && kCut) {
      db = wd.sq / P.H, dhr = (wd.sq % P.H) / P.m;
      a_next = -expf(P.A_log[dhr]);
      bias_next = P.dt_bias[dhr];
    }
    const int c = wd.c, b = db, hr = dhr;
    c_next = c;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int tc = min(c * kQ + 2 * lane + i, P.L - 1);  // past the end: any valid step, masked later
      raw_next[i] = dt_bits[((size_t)b * P.L + tc) * Hr + hr];
    }
  };
  auto chunk_decays = [&](int n) {
    const int c = c_next;
    const float A = a_next, bias = bias_next;
    float* v = vec + (n & 1) * kVecSet;
    float d2v[2], a2[2], sg[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int t = c * kQ + 2 * lane + i;
      const float r = __bfloat162float(__ushort_as_bfloat16(raw_next[i]));
      const float sarg = r + bias;
      const float sp = softplus_fast(sarg);
      const float d = t < P.L ? clamp_dt(sp, P.dt_min, P.dt_max) : 0.f;
      // softplus' = sigmoid(s) = 1 - e^{-softplus(s)}, zero where the limit clamped delta
      const bool free_dt = (sp >= P.dt_min) && (sp <= P.dt_max);
      sg[i] = (t < P.L && free_dt) ? dsoftplus_fast(sp) : 0.f;
      d2v[i] = d;
      a2[i] = d * A;
    }
    float run = a2[0] + a2[1];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float u = __shfl_up_sync(0xffffffffu, run, o);
      if (lane >= o) run += u;
    }
    const float end = __shfl_sync(0xffffffffu, run, 31);
    const float cm[2] = {run - a2[1], run};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int t = 2 * lane + i;
      v[t] = d2v[i];
      v[64 + t] = cm[i];
      v[128 + t] = fast_exp(cm[i]);
      v[192 + t] = fast_exp(end - cm[i]);
      v[256 + t] = sg[i];
      v[320 + t] = v[192 + t] * d2v[i];
    }
    if (lane == 0) v[384] = fast_exp(end);
  };
  if (warp == kWarpDecay) {
    load_dt(0);
    chunk_decays(0);
    if (nwalk > 1) load_dt(1);
  }

  // operand descriptors (see the forward): K-major boxes/images with 32-byte
  // K steps, MN-major ones with 16-row (2048-byte) K steps
  const uint32_t stb[2] = {base, base + SM::kBuf};
  auto kmaj = [&](uint32_t a) { return umma_desc_sw128(a, 16u, 1024u); };
  auto mnmaj = [&](uint32_t a) { return umma_desc_sw128(a, (uint32_t)kTileBytes, 1024u); };
  const uint64_t dDSk = kmaj(base + SM::kDS), dDSmn = mnmaj(base + SM::kDS);
  const uint64_t dXw = kmaj(base + SM::kXw);
  const uint64_t dDYek = kmaj(base + SM::kDYe), dDYemn = mnmaj(base + SM::kDYe);
  const uint64_t dGlmn = mnmaj(base + SM::kGl);
  const uint64_t dZlk = kmaj(base + SM::kZl), dZlmn = mnmaj(base + SM::kZl);
  constexpr uint32_t kId64kk = umma_idesc_bf16(64, 64, false, false);
  constexpr uint32_t kId64km = umma_idesc_bf16(64, 64, false, true);
  constexpr uint32_t kId64mm = umma_idesc_bf16(64, 64, true, true);
  constexpr uint32_t kIdNmm = umma_idesc_bf16(N, 64, true, true);   // M = N: the state update
  constexpr uint32_t kIdBmm = umma_idesc_bf16(64, N, true, true);   // dB first half
  constexpr uint32_t kIdBkk = umma_idesc_bf16(64, N, false, false);  // dB second half, dC first half
  constexpr uint32_t kIdCkm = umma_idesc_bf16(64, N, false, true);   // dC second half

  __syncthreads();  // decays of the first chunk published
  float accA = 0.f, accD = 0.f, accB = 0.f;  // the piece's dA, dDp, ddt_bias (thread kTidDcum)
  bool ok = true;                            // no wait gave up (uniform over the CTA)

  // a piece ends: dS is the gradient of the state entering chunk c_lo --
  // dh0, or the carry for the CTA walking the sequence's first piece
  auto piece_end = [&](const WalkPos& wp, int b, int h, int hr, int st_c0) {
    tmem_fence_after_sync();
    float v[32];
    __syncwarp();
    tmem_ld32(tquarter + kColS + (uint32_t)sc, v);
    if (wp.c_lo == 0) {
      if (P.dh0 && mem_s) {
        float* dst = P.dh0 + (((size_t)b * Hr + hr) * N + srow) * st_ld + st_c0 + sc;
#pragma unroll
        for (int i = 0; i < 32; i += 4) *reinterpret_cast<float4*>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
      }
    } else if (has_srow) {
      float* dst = P.carry + ((size_t)wp.sq * N + srow) * kP + sc;
#pragma unroll
      for (int i = 0; i < 32; i += 4) __stcg(reinterpret_cast<float4*>(dst + i), make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]));
    }
    if (tid == kTidDcum) {
      // the piece's sums: row 0 for the first piece (or the whole sequence), 1 for the last
      float* w6 = P.ws_sc + ((size_t)b * P.H + h) * 6;
      float* w3 = w6 + (wp.c_lo == 0 ? 0 : 3);
      w3[0] = accA;
      w3[1] = accD;
      w3[2] = accB;
      if (wp.c_lo == 0 && wp.c_hi == nch) w6[3] = w6[4] = w6[5] = 0.f;  // not cut
      accA = accD = accB = 0.f;
    }
    if (wp.c_lo > 0) {
      __threadfence();
      __syncthreads();
      if (tid == 0) st_release_gpu(P.seq_flag + wp.sq, 1);
    }
  };
  // the walk's position, advanced chunk by chunk (divisions only when the
  // sequence changes): chunk c of the piece [c_lo, c_hi) of sequence sq =
  // (batch b, sub-head h of head hr)
  WalkPos wp = walk_start();
  int b = sq0 / P.H, h = sq0 % P.H, hr = h / P.m, st_c0 = (h % P.m) * kP;
  float A = -expf(P.A_log[hr]), Dh = P.Dp[hr];
  for (int n = 0; n < nwalk; ++n) {
    const bool piece_start = step(wp);
    const int c = wp.c;
    if (piece_start) {
      if constexpr (kCut) {
        b = wp.sq / P.H, h = wp.sq % P.H, hr = h / P.m;
        st_c0 = (h % P.m) * kP;
        A = -expf(P.A_log[hr]);
        Dh = P.Dp[hr];
      }
      // a piece starts: dS = dh_last (or 0) into TMEM, or, for the first piece
      // of a cut sequence, the carry that the CTA walking its last piece hands over
      const bool handed = wp.c_hi < nch;
      const bool came = !(handed && tid == 0) || flag_wait(P.seq_flag + wp.sq, P.status);
      if (__syncthreads_or(!came)) {  // (bounded wait; the status word says so)
        ok = false;
        break;
      }
      float v[32];
      if (handed) {
        const float* src = P.carry + ((size_t)wp.sq * N + srow) * kP + sc;
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = has_srow ? __ldcg(src + i) : 0.f;
      } else {
        const float* src =
            (P.dh_last && mem_s) ? P.dh_last + (((size_t)b * Hr + hr) * N + srow) * st_ld + st_c0 + sc : nullptr;
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = src ? src[i] : 0.f;
      }
      __syncwarp();
      tmem_st32(tquarter + kColS + (uint32_t)sc, v);
      tmem_wait_st();
    }
    const int s = n & 1;
    const int t0 = c * kQ;
    const uint32_t ph = (uint32_t)(n & 1);
    const bool got = mbar_wait(&full[s], (uint32_t)((n >> 1) & 1), P.status);
    if (__syncthreads_or(!got)) {  // the copy never came: stop, uniformly
      ok = false;
      break;
    }
    unsigned char* st = smem + s * SM::kBuf;
    const float* vc = vec + s * kVecSet;
    // the next chunk's boxes into the other stage (free since the last chunk)
    if (tid == kTidTma && n + 1 < nwalk) issue(n + 1);

    // ---- 1: dS as a bf16 image, <dS, S_in>, dS scaled by e^(cum_end) for the
    // update; x'' = diag(w delta) x and dy' = diag(e^cum) dy; dy . x
    float part_dss = 0.f, part_dyx = 0.f;
    {
      float v[32];
      tmem_fence_after_sync();
      __syncwarp();
      tmem_ld32(tquarter + kColS + (uint32_t)sc, v);
      if (has_srow) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          put8(SM::kDS, srow, 4 * kq + q, v + 8 * q);
          float sv[8];
          get8(SM::kSo + s * SM::kBuf, srow, 4 * kq + q, sv);
#pragma unroll
          for (int i = 0; i < 8; ++i) part_dss = fmaf(v[8 * q + i], sv[i], part_dss);
        }
      }
      const float ecend = vc[384];
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] *= ecend;
      __syncwarp();
      tmem_st32(tquarter + kColS + (uint32_t)sc, v);
      tmem_wait_st();
    }
    {
      const float wd = vc[320 + row], ec = vc[128 + row];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int c8 = col0 / 8 + q;
        float xv[8], yv[8], o[8];
        get8(SM::kX + s * SM::kBuf, row, c8, xv);
        get8(SM::kDY + s * SM::kBuf, row, c8, yv);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          part_dyx = fmaf(yv[i], xv[i], part_dyx);
          o[i] = wd * xv[i];
        }
        put8(SM::kXw, row, c8, o);
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = ec * yv[i];
        put8(SM::kDYe, row, c8, o);
      }
    }
    fence_proxy_async_smem();
    tmem_fence_before_sync();
    __syncthreads();

    // ---- 2: G = C B^T and Z = dy x^T (issuer 0), CS = C S_in and the update
    // dS += C^T dy' (issuer 1), X = B dS (issuer 2)
    if (issuer) {
      tmem_fence_after_sync();
      const uint64_t dCk = kmaj(stb[s] + SM::kCo), dBk = kmaj(stb[s] + SM::kBo), dCmn = mnmaj(stb[s] + SM::kCo);
      const uint64_t dDYk = kmaj(stb[s] + SM::kDY), dXk = kmaj(stb[s] + SM::kX), dSmn = mnmaj(stb[s] + SM::kSo);
      if (iss == 0) {
#pragma unroll
        for (int k = 0; k < N / 16; ++k) {  // K = n
          const uint64_t ko = (uint64_t)(((k / 4) * kTileBytes + (k % 4) * 32) >> 4);
          umma_f16(tmem + kColG, dCk + ko, dBk + ko, kId64kk, k > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)  // K = p
          umma_f16(tmem + kColZ, dDYk + (uint64_t)(2 * k), dXk + (uint64_t)(2 * k), kId64kk, k > 0 ? 1u : 0u);
      } else if (iss == 1) {
#pragma unroll
        for (int k = 0; k < N / 16; ++k) {
          const uint64_t ko = (uint64_t)(((k / 4) * kTileBytes + (k % 4) * 32) >> 4);
          umma_f16(tmem + kColCS, dCk + ko, dSmn + (uint64_t)(k * 128), kId64km, k > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)  // K = t
          umma_f16(tmem + kColS, dCmn + (uint64_t)(k * 128), dDYemn + (uint64_t)(k * 128), kIdNmm, 1u);
      } else {
#pragma unroll
        for (int k = 0; k < N / 16; ++k) {
          const uint64_t ko = (uint64_t)(((k / 4) * kTileBytes + (k % 4) * 32) >> 4);
          umma_f16(tmem + kColX, dBk + ko, dDSmn + (uint64_t)(k * 128), kId64km, k > 0 ? 1u : 0u);
        }
      }
      umma_commit(bar1);
    }
    // the next chunk's decays (its dt read a chunk ago), its successor's dt in flight
    if (warp == kWarpDecay && n + 1 < nwalk) {
      chunk_decays(n + 1);
      if (n + 2 < nwalk) load_dt(n + 2);
    }
    mbar_wait(bar1, ph, P.status);
    tmem_fence_after_sync();

    // ---- 3: the masked, decayed images and the chunk's row / column sums
    float part_rs = 0.f;  // sum over this thread's rows s of w delta (B dS)_s . x_s
    {
      float gv[16], zv[16], cv[16], xb[16];
      __syncwarp();
      tmem_ld16x2_16(tquarter + kColG + (uint32_t)(32 * kq), gv);
      tmem_ld16x2_16(tquarter + kColZ + (uint32_t)(32 * kq), zv);
      tmem_ld16x2_16(tquarter + kColCS + (uint32_t)(32 * kq), cv);
      tmem_ld16x2_16(tquarter + kColX + (uint32_t)(32 * kq), xb);
      const float ct = vc[64 + row];
      float glv[16], zlv[16], rowf = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int s2 = col0 + j;
        const float lts = s2 <= row ? fast_exp(ct - vc[64 + s2]) : 0.f;
        const float lg = lts * gv[j];
        const float dd = lg * zv[j];  // (L o G o Z)[row][s2]
        glv[j] = lg * vc[s2];
        zlv[j] = lts * zv[j] * vc[s2];
        rowf = fmaf(dd, vc[s2], rowf);
        d2[row * 65 + s2] = dd;
      }
      put8(SM::kGl, row, col0 / 8, glv);
      put8(SM::kGl, row, col0 / 8 + 1, glv + 8);
      put8(SM::kZl, row, col0 / 8, zlv);
      put8(SM::kZl, row, col0 / 8 + 1, zlv + 8);
      // dy_t . (C S_in)_t and (B dS)_s . x_s over this thread's 16 columns
      float yv[16], xv[16];
      get8(SM::kDY + s * SM::kBuf, row, col0 / 8, yv);
      get8(SM::kDY + s * SM::kBuf, row, col0 / 8 + 1, yv + 8);
      get8(SM::kX + s * SM::kBuf, row, col0 / 8, xv);
      get8(SM::kX + s * SM::kBuf, row, col0 / 8 + 1, xv + 8);
      float rcs = 0.f, rq = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        rcs = fmaf(yv[j], cv[j], rcs);
        rq = fmaf(xb[j], xv[j], rq);
      }
      // X <- w delta (B dS), the first term of dx (its second accumulates on top)
      const float wd = vc[320 + row];
#pragma unroll
      for (int j = 0; j < 16; ++j) xb[j] *= wd;
      __syncwarp();
      tmem_st16x2_16(tquarter + kColX + (uint32_t)(32 * kq), xb);
      tmem_wait_st();
      part_rs = wd * rq;
      // row partials: part index kq * 2 + lane half
      const int pi = 2 * kq + (lane >> 4);
      rowp[(0 * 64 + row) * 4 + pi] = rowf;
      rowp[(1 * 64 + row) * 4 + pi] = rcs;
      rowp[(2 * 64 + row) * 4 + pi] = rq;
    }
    // block sums of <dS, S_in>, dy . x and the w delta (B dS) . x terms
    {
      float v3[3] = {part_dss, part_dyx, part_rs};
#pragma unroll
      for (int i = 0; i < 3; ++i)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v3[i] += __shfl_xor_sync(0xffffffffu, v3[i], o);
      if (lane == 0) {
        red[warp] = v3[0];
        red[8 + warp] = v3[1];
        red[16 + warp] = v3[2];
      }
    }
    fence_proxy_async_smem();
    tmem_fence_before_sync();
    __syncthreads();

    // ---- 4: dx += (L o G o delta)^T dy; dB = (L o Z o delta)^T C + x'' dS^T;
    // dC = dy' S_in^T + (L o Z o delta) B
    // (dB on issuer 0, dC on issuer 1, dx on issuer 2)
    if (issuer) {
      tmem_fence_after_sync();
      const uint64_t dDYmn = mnmaj(stb[s] + SM::kDY), dCmn = mnmaj(stb[s] + SM::kCo), dBmn = mnmaj(stb[s] + SM::kBo);
      const uint64_t dSk = kmaj(stb[s] + SM::kSo);
      if (iss == 0) {
#pragma unroll
        for (int k = 0; k < 4; ++k)  // K = t
          umma_f16(tmem + kColB, dZlmn + (uint64_t)(k * 128), dCmn + (uint64_t)(k * 128), kIdBmm, k > 0 ? 1u : 0u);
#pragma unroll
        for (int k = 0; k < 4; ++k)  // K = p
          umma_f16(tmem + kColB, dXw + (uint64_t)(2 * k), dDSk + (uint64_t)(2 * k), kIdBkk, 1u);
      } else if (iss == 1) {
#pragma unroll
        for (int k = 0; k < 4; ++k)  // K = p
          umma_f16(tmem + kColC, dDYek + (uint64_t)(2 * k), dSk + (uint64_t)(2 * k), kIdBkk, k > 0 ? 1u : 0u);
#pragma unroll
        for (int k = 0; k < 4; ++k)  // K = s
          umma_f16(tmem + kColC, dZlk + (uint64_t)(2 * k), dBmn + (uint64_t)(k * 128), kIdCkm, 1u);
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k)  // K = t
          umma_f16(tmem + kColX, dGlmn + (uint64_t)(k * 128), dDYmn + (uint64_t)(k * 128), kId64mm, 1u);
      }
      umma_commit(bar2);
    }
    // the gradient of the log-decays, delta and A (warps 4 and 5: step t = tid - 128)
    if (tid >= kTidDcum && tid < kTidDcum + 64) {
      const int t = tid - kTidDcum;
      float colD2 = 0.f;
      for (int r = t; r < 64; ++r) colD2 += d2[r * 65 + t];  // rows r >= t (L is 0 above the diagonal)
      const float* rp0 = rowp + (0 * 64 + t) * 4;
      const float* rp1 = rowp + (1 * 64 + t) * 4;
      const float* rp2 = rowp + (2 * 64 + t) * 4;
      const float rowF = (rp0[0] + rp0[1]) + (rp0[2] + rp0[3]);
      const float rCS = (rp1[0] + rp1[1]) + (rp1[2] + rp1[3]);
      const float qv = (rp2[0] + rp2[1]) + (rp2[2] + rp2[3]);
      const float dl = vc[t], ec = vc[128 + t], wt = vc[192 + t];
      float dcum = rowF - dl * colD2 + ec * rCS - wt * dl * qv;
      if (t == 63) {
        // <dS, S_out> = e^(cum_end) <dS, S_in> + sum_s w_s delta_s (B dS)_s . x_s
        float dss = 0.f, rs = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
          dss += red[w];
          rs += red[16 + w];
        }
        dcum += vc[384] * dss + rs;
      }
      // suffix sums over t (two warps: within-warp inclusive suffix scan, then
      // the upper warp's total added to the lower one)
      float suf = dcum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float u = __shfl_down_sync(0xffffffffu, suf, o);
        if (lane + o < 32) suf += u;
      }
      if (t == 32) red[24] = suf;  // total of steps 32..63
      named_bar_sync(3, 64);
      if (t < 32) suf += red[24];
      const float ddl = colD2 + wt * qv + A * suf;
      const float graw = ddl * vc[256 + t];
      if (t0 + t < P.L) {
        if (P.m == 1)
          P.ddt_raw[((size_t)b * P.L + t0 + t) * Hr + hr] = __float2bfloat16_rn(graw);
        else  // the head's sub-heads are added by the reduce kernel
          P.ws_ddt[((size_t)b * P.L + t0 + t) * P.H + h] = graw;
      }
      // chunk sums of dA terms and of ddt_raw, fixed order
      float va = dl * suf, vb = t0 + t < P.L ? graw : 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        va += __shfl_xor_sync(0xffffffffu, va, o);
        vb += __shfl_xor_sync(0xffffffffu, vb, o);
      }
      if (lane == 0) {
        red[32 + 2 * (warp - kTidDcum / 32)] = va;
        red[33 + 2 * (warp - kTidDcum / 32)] = vb;
      }
      named_bar_sync(3, 64);
      if (t == 0) {
        accA += red[32] + red[34];
        accB += red[33] + red[35];
        float dyx = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) dyx += red[8 + w];
        accD += dyx;
      }
    }
    mbar_wait(bar2, ph, P.status);
    tmem_fence_after_sync();

    // ---- 5: dx = D dy + X; the per-head dB and dC rows
    {
      float xv[16];
      __syncwarp();
      tmem_ld16x2_16(tquarter + kColX + (uint32_t)(32 * kq), xv);
      float yv[16];
      get8(SM::kDY + s * SM::kBuf, row, col0 / 8, yv);
      get8(SM::kDY + s * SM::kBuf, row, col0 / 8 + 1, yv + 8);
      if (t0 + row < P.L && col0 < P.w) {
        uint4* dst = reinterpret_cast<uint4*>(P.dx + (((size_t)b * P.L + t0 + row) * P.H + h) * P.w + col0);
        uint32_t o[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) o[k] = pack_bf16(fmaf(Dh, yv[2 * k], xv[2 * k]), fmaf(Dh, yv[2 * k + 1], xv[2 * k + 1]));
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
      }
#pragma unroll
      for (int half = 0; half < NT; ++half) {
        float bv[16], cv[16];
        __syncwarp();
        tmem_ld16x2_16(tquarter + kColB + (uint32_t)(64 * half + 32 * kq), bv);
        tmem_ld16x2_16(tquarter + kColC + (uint32_t)(64 * half + 32 * kq), cv);
        if (t0 + row < P.L) {
          const size_t o = (((size_t)b * P.L + t0 + row) * P.H + h) * N + 64 * half + col0;
          float4* db = reinterpret_cast<float4*>(P.ws_dB + o);
          float4* dc = reinterpret_cast<float4*>(P.ws_dC + o);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            db[k] = make_float4(bv[4 * k], bv[4 * k + 1], bv[4 * k + 2], bv[4 * k + 3]);
            dc[k] = make_float4(cv[4 * k], cv[4 * k + 1], cv[4 * k + 2], cv[4 * k + 3]);
          }
        }
      }
    }
    tmem_fence_before_sync();
    __syncthreads();  // every product of this stage done and read; images free
    if (kCut && c == wp.c_lo) piece_end(wp, b, h, hr, st_c0);
  }
  if (!kCut && ok) piece_end(wp, b, h, hr, st_c0);  // the sequence's end (dh0)
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// dBm / dCm[b,t,g,n] = sum over the group's sub-heads (ascending) of the
// per-sub-head terms; dA_log[h] = A_h sum_b sum_j sum_k dA, dDp[h] = sum_b
// sum_j sum_k, ddt_bias[h] = sum_b sum_j sum_k (ascending b, then the head's
// sub-heads j, then the sequence's pieces k: first, last); with
// m > 1 sub-heads per head also ddt_raw[b,t,h] = sum_j (ascending).  H counts
// sub-heads.
__global__ void s6_ssd_bwd_reduce_kernel(const float* __restrict__ ws_dB, const float* __restrict__ ws_dC,
                                         const float* __restrict__ ws_sc, const float* __restrict__ A_log,
                                         int B, int L, int H, int G, int N, int m,
                                         __nv_bfloat16* __restrict__ dBm, __nv_bfloat16* __restrict__ dCm,
                                         float* __restrict__ dA_log, float* __restrict__ dDp,
                                         float* __restrict__ ddt_bias) {
  const int hpg = H / G;
  const size_t total = (size_t)B * L * G * N;
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (size_t)gridDim.x * blockDim.x) {
    const int n = (int)(e % N);
    const size_t btg = e / N;
    const int gg = (int)(btg % G);
    const size_t bt = btg / G;
    const size_t src = (bt * H + (size_t)gg * hpg) * N + n;
    float sb = 0.f, scv = 0.f;
    for (int k = 0; k < hpg; ++k) {
      sb += ws_dB[src + (size_t)k * N];
      scv += ws_dC[src + (size_t)k * N];
    }
    dBm[e] = __float2bfloat16_rn(sb);
    dCm[e] = __float2bfloat16_rn(scv);
  }
  if (blockIdx.x == 0) {
    for (int hh = threadIdx.x; hh < H / m; hh += blockDim.x) {
      float a = 0.f, d = 0.f, tb = 0.f;
      for (int bb = 0; bb < B; ++bb)
        for (int j = 0; j < m; ++j) {
          const float* w6 = ws_sc + ((size_t)bb * H + (size_t)hh * m + j) * 6;
          a += w6[0];
          a += w6[3];
          d += w6[1];
          d += w6[4];
          tb += w6[2];
          tb += w6[5];
        }
      dA_log[hh] = -expf(A_log[hh]) * a;
      dDp[hh] = d;
      ddt_bias[hh] = tb;
    }
  }
}

// m > 1 sub-heads per head: ddt_raw[b,t,h] = sum over the head's sub-heads
// (ascending) of their terms ws_ddt[b][t][h m + j]
__global__ void s6_ssd_bwd_ddt_kernel(const float* __restrict__ ws_ddt, size_t n_out, int m,
                                      __nv_bfloat16* __restrict__ ddt_raw) {
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < n_out; e += (size_t)gridDim.x * blockDim.x) {
    const float* w = ws_ddt + e * m;
    float v = w[0];
    for (int j = 1; j < m; ++j) v += w[j];
    ddt_raw[e] = __float2bfloat16_rn(v);
  }
}

// One CTA per sequence when they fit the SMs at once; with more sequences
// than SMs, one range per SM (no tail wave), launched cooperatively so that
// every CTA is resident while they hand state gradients over.  Where this
// GPU cannot hold them all, the one-per-sequence grid (the same results).
template <int N>
cudaError_t launch_bwd_n(const SsdBwdParams& P, cudaStream_t stream) {
  const size_t smem = BwdSmem<N>::kBytes + 1024;
  const int seqs = P.B * P.H;
  const int sms = device_sm_count();
  cudaError_t e;
  if (sms > 0 && seqs > sms) {
    auto kern = s6_ssd_bwd_kernel<N, true>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm >= 1) {
      e = cudaMemsetAsync(P.seq_flag, 0, sizeof(int) * (size_t)seqs, stream);
      if (e != cudaSuccess) return e;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)sms);
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = smem;
      cfg.stream = stream;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeCooperative;
      attr[0].val.cooperative = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      e = cudaLaunchKernelEx(&cfg, kern, P);
      if (e != cudaErrorCooperativeLaunchTooLarge) return e;
    }
    (void)cudaGetLastError();
    note_plan_fallback();
  }
  auto kern = s6_ssd_bwd_kernel<N, false>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)seqs, kThreads, smem, stream>>>(P);
  return cudaGetLastError();
}

}  // namespace

size_t ssd_bwd_workspace_bytes(int B, int L, int H, int m, int G, int N) {
  (void)G;
  const size_t Hs = (size_t)H * m;  // sub-heads
  const size_t terms = (size_t)B * L * Hs * N * sizeof(float);
  const size_t sc = ((size_t)B * Hs * 6 * sizeof(float) + 255) / 256 * 256;
  const size_t ddt = m > 1 ? ((size_t)B * L * Hs * sizeof(float) + 255) / 256 * 256 : 0;
  const size_t flags = ((size_t)B * Hs * sizeof(int) + 255) / 256 * 256;
  const size_t carry = (size_t)B * Hs * N * kP * sizeof(float);
  return 2 * ((terms + 255) / 256 * 256) + sc + ddt + flags + carry;
}

cudaError_t launch_ssd_bwd(const SsdBwdArgs& a, cudaStream_t stream) {
  const SsdArgs& f = a.f;
  SsdBwdParams P;
  memset(&P, 0, sizeof(P));
  const uint64_t e = 2;
  if (!ssd_encode_x_map(&P.map_x, f.x, f) || !ssd_encode_x_map(&P.map_dy, a.dy, f)) return cudaErrorInvalidValue;
  {
    const uint64_t dims[3] = {(uint64_t)f.G * f.N, (uint64_t)f.L, (uint64_t)f.B};
    const uint64_t strides[2] = {(uint64_t)f.G * f.N * e, (uint64_t)f.L * f.G * f.N * e};
    const uint32_t box[3] = {64, kQ, 1};
    if (!encode_tile_map(&P.map_B, f.Bm, true, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tile_map(&P.map_C, f.Cm, true, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  {
    const uint64_t nch = (uint64_t)(f.L + kQ - 1) / kQ;
    // the saves [B][H][nch][N][w m]: rows of w m, a sub-head's 64 columns at
    // (h % m) * 64 (w = 32: the box's columns 32..63 are zeros)
    const uint64_t dims[2] = {(uint64_t)f.w * f.m, (uint64_t)f.B * f.H * nch * f.N};
    const uint64_t strides[1] = {(uint64_t)f.w * f.m * e};
    const uint32_t box[2] = {64, 64};
    if (!encode_tile_map(&P.map_S, f.chunk_states, true, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  P.dt_raw = static_cast<const __nv_bfloat16*>(f.dt_raw);
  P.dt_bias = f.dt_bias;
  P.A_log = f.A_log;
  P.Dp = f.Dp;
  P.dh_last = a.dh_last;
  P.dx = static_cast<__nv_bfloat16*>(a.dx);
  P.ddt_raw = static_cast<__nv_bfloat16*>(a.ddt_raw);
  P.dh0 = a.dh0;
  const size_t Hs = (size_t)f.H * f.m;
  const size_t terms = ((size_t)f.B * f.L * Hs * f.N * sizeof(float) + 255) / 256 * 256;
  const size_t scb = ((size_t)f.B * Hs * 6 * sizeof(float) + 255) / 256 * 256;
  const size_t ddtb = f.m > 1 ? ((size_t)f.B * f.L * Hs * sizeof(float) + 255) / 256 * 256 : 0;
  const size_t flagb = ((size_t)f.B * Hs * sizeof(int) + 255) / 256 * 256;
  char* wsb = reinterpret_cast<char*>(a.ws);
  P.ws_dB = a.ws;
  P.ws_dC = reinterpret_cast<float*>(wsb + terms);
  P.ws_sc = reinterpret_cast<float*>(wsb + 2 * terms);
  P.ws_ddt = f.m > 1 ? reinterpret_cast<float*>(wsb + 2 * terms + scb) : nullptr;
  P.seq_flag = reinterpret_cast<int*>(wsb + 2 * terms + scb + ddtb);
  P.carry = reinterpret_cast<float*>(wsb + 2 * terms + scb + ddtb + flagb);
  P.status = f.status;
  P.dt_min = f.dt_min;
  P.dt_max = f.dt_max;
  P.B = f.B;
  P.L = f.L;
  P.H = (int)Hs;
  P.m = f.m;
  P.w = f.w;
  P.Hr = f.H;
  P.G = f.G;
  P.N = f.N;
  cudaError_t err = f.N == 128 ? launch_bwd_n<128>(P, stream) : launch_bwd_n<64>(P, stream);
  if (err != cudaSuccess) return err;
  const size_t total = (size_t)f.B * f.L * f.G * f.N;
  const int threads = 256;
  const int blocks = (int)std::min<size_t>(std::max<size_t>((total + threads - 1) / threads, 1), 152 * 8);
  s6_ssd_bwd_reduce_kernel<<<blocks, threads, 0, stream>>>(
      P.ws_dB, P.ws_dC, P.ws_sc, f.A_log, f.B, f.L, (int)Hs, f.G, f.N, f.m, static_cast<__nv_bfloat16*>(a.dBm),
      static_cast<__nv_bfloat16*>(a.dCm), a.dA_log, a.dDp, a.ddt_bias);
  err = cudaGetLastError();
  if (err != cudaSuccess || f.m == 1) return err;
  const size_t n_ddt = (size_t)f.B * f.L * f.H;
  const int dblocks = (int)std::min<size_t>(std::max<size_t>((n_ddt + threads - 1) / threads, 1), 152 * 8);
  s6_ssd_bwd_ddt_kernel<<<dblocks, threads, 0, stream>>>(P.ws_ddt, n_ddt, f.m, static_cast<__nv_bfloat16*>(a.ddt_raw));
  return cudaGetLastError();
}

}  // namespace s6
