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
// A CTA owns one (batch, head) sequence and walks its chunks in order,
// carrying S (N x 64, f32) in the accumulator registers of its four warps;
// the chunk's x, Bm and Cm tiles arrive by TMA (128-byte swizzled boxes of
// 64 steps x 64 columns) into a two-deep ring.  The four products run on
// the tensor cores with mma.sync (bf16 operands, f32 accumulation): C B^T
// and C S_in share their A operand; the masked, scaled C B^T goes from the
// accumulators straight into the A operand of the next product; the causal
// structure skips the blocks above the diagonal.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>

#include "s6_internal.cuh"
#include "s6_math.cuh"
#include "s6_tma.cuh"

namespace s6 {

namespace {

constexpr int kQ = 64;           // steps per chunk
constexpr int kP = 64;           // head dimension
constexpr int kSsdThreads = 128;  // 4 warps: warp w owns rows 16w..16w+15 of a chunk, 32w..32w+31 of S
constexpr int kTileBytes = 64 * 128;  // one 64 x 64 bf16 box (128-byte rows)

struct SsdParams {
  CUtensorMap map_x, map_B, map_C;  // 64-byte aligned members first
  const __nv_bfloat16* dt_raw;      // [B][L][H]
  const float* dt_bias;             // [H]
  const float* A_log;               // [H]
  const float* Dp;                  // [H]
  const float* h0;                  // [B][H][N][P] or null
  __nv_bfloat16* y;                 // [B][L][H][P]
  float* h_last;                    // [B][H][N][P] or null
  unsigned int* status;
  float dt_min, dt_max;
  int B, L, H, G, N;
};

// byte offset of the 16-byte chunk `c8` (elements 8 c8 .. 8 c8 + 7) of row r
// in a 128-byte swizzled box of 128-byte rows (the TMA's 128B swizzle: the
// chunk index is XORed with the row's position in its 8-row group)
__device__ __forceinline__ uint32_t swz(int r, int c8) { return (uint32_t)(r * 128 + ((c8 ^ (r & 7)) << 4)); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// d += a (16 x 16, row) * b (16 x 8, col), bf16 operands, f32 accumulators
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ float2 unpack_bf16(uint32_t v) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
}
__device__ __forceinline__ float fast_exp(float x) { return ex2_approx(x * kLog2e); }

// ---- tcgen05 (5th-generation tensor core) helpers for the state update
// Shared-memory matrix descriptor of a 128-byte-swizzled operand: start
// address, leading-dimension byte offset (between 64-element blocks of the
// M/N dimension for an MN-major operand), stride byte offset (between 8-row
// groups of K), descriptor version 1, swizzle mode 128B.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor, kind::f16: f32 accumulator, bf16 A and B, both
// MN-major, N = 64, M = 128.
constexpr uint32_t kUmmaIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | (1u << 16) | ((64u >> 3) << 17) |
                                ((128u >> 4) << 24);
// D[tmem] (+)= A (smem) x B (smem), issued by one thread
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// arrive on `bar` once every tcgen05 operation this thread issued has completed
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
// make this thread's generic-proxy shared-memory writes visible to the tensor core
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

template <int N>
struct SsdSmem {
  static constexpr int NT = N / 64;                    // 64-column boxes of Bm / Cm
  static constexpr int kX = 0;                         // x box [64 s][64 p]
  static constexpr int kBo = kTileBytes;               // Bm boxes [NT][64 s][64 n]
  static constexpr int kCo = kBo + NT * kTileBytes;    // Cm boxes
  static constexpr int kBuf = kCo + NT * kTileBytes;   // one stage
  static constexpr int kStage = 2 * kBuf;              // x' / y staging box [64][64]
  static constexpr int kS = kStage + kTileBytes;       // S_in (bf16) [N n][64 p]
  static constexpr int kVec = kS + N * 128;            // two sets of cum, delta, w*delta [3][64] f32 + decay
  static constexpr int kBar = kVec + 2 * 4 * 64 * 4;   // three mbarriers and the TMEM address
  static constexpr int kBytes = kBar + 64;
  static constexpr uint32_t kTx = (1 + 2 * NT) * kTileBytes;
  static_assert(kBuf % 1024 == 0 && kStage % 1024 == 0 && kS % 1024 == 0, "swizzled boxes on 1024-byte boundaries");
};

template <int N>
__global__ void __launch_bounds__(kSsdThreads) s6_ssd_fwd_kernel(const __grid_constant__ SsdParams P) {
  using SM = SsdSmem<N>;
  constexpr int NT = SM::NT;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // the 128B swizzle repeats every 1024 bytes: align the base
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* smem = smem_raw + (base - raw);
  // per chunk set (two sets, by chunk parity): (cum, delta) pairs of steps
  // [0, 64) interleaved [0, 128), w*delta [128, 192), e^(cum_end) [192]
  float* vec = reinterpret_cast<float*>(smem + SM::kVec);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SM::kBar);
  uint64_t* mma_bar = full + 2;  // the state update's completion (tcgen05 path)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(full + 3);
  // N = 128: the state lives in tensor memory (128 lanes = rows n, 64 columns
  // = p, f32) and its update S = e^(cum_end) S + B^T x' runs as tcgen05.mma;
  // N = 64: in the accumulators of the four warps (mma.sync)
  constexpr bool kUmma = N == 128;

  const int b = blockIdx.x / P.H, h = blockIdx.x % P.H;
  const int g = h / (P.H / P.G);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, cq = lane & 3;  // fragment row group, column pair
  const int nch = (P.L + kQ - 1) / kQ;
  const float A = -expf(P.A_log[h]);
  const float bias = P.dt_bias[h];
  const float Dh = P.Dp[h];

  if (tid == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    mbar_init(mma_bar, 1);
    fence_mbar_init();
  }
  if (kUmma && warp == 0) tmem_alloc(tmem_slot, 64);
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  const uint32_t tmem = kUmma ? *tmem_slot : 0u;
  const uint32_t trow = tmem + ((uint32_t)(32 * warp) << 16);  // this thread's lane (row n = tid)
  auto issue = [&](int c) {  // chunk c's boxes into stage c & 1 (one thread)
    const int s = c & 1;
    unsigned char* st = smem + s * SM::kBuf;
    mbar_arrive_expect_tx(&full[s], SM::kTx);
    tma_load_3d(st + SM::kX, &P.map_x, &full[s], h * kP, c * kQ, b);
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      tma_load_3d(st + SM::kBo + j * kTileBytes, &P.map_B, &full[s], g * N + 64 * j, c * kQ, b);
      tma_load_3d(st + SM::kCo + j * kTileBytes, &P.map_C, &full[s], g * N + 64 * j, c * kQ, b);
    }
  };
  if (tid == 0) {
    tma_prefetch_desc(&P.map_x);
    if (nch > 0) issue(0);
    if (nch > 1) issue(1);
  }

  // the state (mma.sync path): warp w holds rows n = 32w + 16 mt + {gq, gq + 8}, columns p = 8 j + 2 cq + {0, 1}
  constexpr int kMT = N / 64;  // 16-row tiles of S per warp (N / 4 rows per warp)
  float S[kMT][8][4];  // (unused on the tcgen05 path)
  // tcgen05 path: thread tid owns row n = tid of S (one TMEM lane, 64 columns)
  auto row_to_smem_bf16 = [&](const float (&v)[64]) {  // S_in for the next readout, [n][p] swizzled
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8)
      *reinterpret_cast<uint4*>(smem + SM::kS + swz(tid, c8)) =
          make_uint4(pack_bf16(v[8 * c8], v[8 * c8 + 1]), pack_bf16(v[8 * c8 + 2], v[8 * c8 + 3]),
                     pack_bf16(v[8 * c8 + 4], v[8 * c8 + 5]), pack_bf16(v[8 * c8 + 6], v[8 * c8 + 7]));
  };
  auto tmem_row_ld = [&](float (&v)[64]) {
    float a[32], c[32];
    tmem_ld32(trow, a);
    tmem_ld32(trow + 32u, c);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = a[i], v[32 + i] = c[i];
  };
  auto tmem_row_st = [&](const float (&v)[64]) {
    float a[32], c[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) a[i] = v[i], c[i] = v[32 + i];
    tmem_st32(trow, a);
    tmem_st32(trow + 32u, c);
  };
  if constexpr (kUmma) {
    float v[64];
    const float* h0 = P.h0 ? P.h0 + (((size_t)b * P.H + h) * N + tid) * kP : nullptr;
#pragma unroll
    for (int i = 0; i < 64; ++i) v[i] = h0 ? h0[i] : 0.f;
    row_to_smem_bf16(v);
    tmem_row_st(v);
    tmem_wait_st();
  } else {
    const float* h0 = P.h0 ? P.h0 + ((size_t)b * P.H + h) * N * kP : nullptr;
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int n = warp * (N / 4) + 16 * mt + gq + 8 * (e >> 1), p = 8 * j + 2 * cq + (e & 1);
          S[mt][j][e] = h0 ? h0[(size_t)n * kP + p] : 0.f;
        }
  }
  auto store_S_bf16 = [&]() {  // S_in for the next chunk's readout, [n][p] swizzled
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int hlf = 0; hlf < 2; ++hlf) {
          const int n = warp * (N / 4) + 16 * mt + gq + 8 * hlf;
          *reinterpret_cast<uint32_t*>(smem + SM::kS + swz(n, j) + 4 * cq) =
              pack_bf16(S[mt][j][2 * hlf], S[mt][j][2 * hlf + 1]);
        }
  };
  if constexpr (!kUmma) store_S_bf16();

  // Warp 0 reads each chunk's dt one chunk ahead (two steps per lane) and,
  // during the state update of the chunk before, turns them into delta, the
  // running sum of delta*A, the weights e^(cum_end - cum_s) delta_s and the
  // chunk's total decay (set c & 1 of `vec`).
  float raw_next[2] = {0.f, 0.f};
  auto load_dt = [&](int c) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int t = c * kQ + 2 * lane + i;
      raw_next[i] = (c < nch && t < P.L) ? __bfloat162float(P.dt_raw[((size_t)b * P.L + t) * P.H + h]) : 0.f;
    }
  };
  auto chunk_decays = [&](int c) {
    float* v = vec + (c & 1) * 256;
    float d2[2], a2[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int t = c * kQ + 2 * lane + i;
      const float d = t < P.L ? clamp_dt(softplus_fast(raw_next[i] + bias), P.dt_min, P.dt_max) : 0.f;
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
    // (cum, delta) of steps 2 lane and 2 lane + 1 side by side: one 16-byte read per pair
    *reinterpret_cast<float4*>(v + 4 * lane) = make_float4(c0, d2[0], c1, d2[1]);
    v[128 + 2 * lane] = fast_exp(end - c0) * d2[0];
    v[128 + 2 * lane + 1] = fast_exp(end - c1) * d2[1];
    if (lane == 0) v[192] = fast_exp(end);
  };
  if (warp == 0) {
    load_dt(0);
    chunk_decays(0);
    load_dt(1);
  }
  __syncthreads();

  for (int c = 0; c < nch; ++c) {
    const int s = c & 1;
    const int t0 = c * kQ;
    const bool ok = mbar_wait(&full[s], (c >> 1) & 1, P.status);
    if (__syncthreads_or(!ok)) break;  // the copy never came: stop, uniformly
    unsigned char* st = smem + s * SM::kBuf;
    const uint32_t xs = base + s * SM::kBuf + SM::kX;
    const uint32_t bs = base + s * SM::kBuf + SM::kBo;
    const uint32_t cs = base + s * SM::kBuf + SM::kCo;
    const uint32_t ss = base + SM::kS;
    const float* cum = vec + s * 256;  // cum of step t at cum[2 t], delta at cum[2 t + 1]
    const float* wd = cum + 128;
    if constexpr (kUmma) {  // S_in in TMEM takes the chunk's decay before the update accumulates onto it
      tmem_fence_after_sync();
      float v[64];
      tmem_row_ld(v);
      const float dec0 = cum[192];
#pragma unroll
      for (int i = 0; i < 64; ++i) v[i] *= dec0;
      tmem_row_st(v);
      tmem_wait_st();
      tmem_fence_before_sync();
    }

    // ---- y rows 16w .. 16w+15: (C B^T o L)(delta x) + e^cum (C S_in) + D x
    const int r0 = 16 * warp;
    float G[8][4], CS[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) G[j][e] = CS[j][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < N / 16; ++kk) {
      const int k0 = 16 * kk;
      const int sub = k0 / 64, kc = (k0 % 64) / 8;
      uint32_t a[4];
      ldsm_x4(cs + sub * kTileBytes + swz(r0 + (lane & 7) + 8 * ((lane >> 3) & 1), kc + (lane >> 4)), a);
      // C B^T: only the s blocks at or below this warp's rows
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        if (jj > warp) break;
        uint32_t bb[4];
        ldsm_x4(bs + sub * kTileBytes + swz(16 * jj + (lane & 7) + 8 * (lane >> 4), kc + ((lane >> 3) & 1)), bb);
        mma16816(G[2 * jj], a, bb[0], bb[1]);
        mma16816(G[2 * jj + 1], a, bb[2], bb[3]);
      }
      // C S_in
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        uint32_t bb[4];
        ldsm_x4_t(ss + swz(k0 + (lane & 7) + 8 * ((lane >> 3) & 1), 2 * jj + (lane >> 4)), bb);
        mma16816(CS[2 * jj], a, bb[0], bb[1]);
        mma16816(CS[2 * jj + 1], a, bb[2], bb[3]);
      }
    }
    // mask and scale: M[t][s] = G[t][s] e^(cum_t - cum_s) delta_s for s <= t
    const int ta = r0 + gq, tb = ta + 8;
    const float cta = cum[2 * ta], ctb = cum[2 * tb];
    uint32_t M[4][4];  // A operand of (M)(x): k block kk2 = s in [16 kk2, 16 kk2 + 16)
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int s0 = 8 * j + 2 * cq;
      const float4 cd = *reinterpret_cast<const float4*>(cum + 2 * s0);  // steps s0, s0 + 1
      float m[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int t = (e < 2) ? ta : tb;
        const int sx = s0 + (e & 1);
        const float ct = (e < 2) ? cta : ctb;
        const float cs_ = (e & 1) ? cd.z : cd.x, ds_ = (e & 1) ? cd.w : cd.y;
        m[e] = (sx <= t) ? G[j][e] * fast_exp(ct - cs_) * ds_ : 0.f;
      }
      M[j >> 1][(j & 1) * 2] = pack_bf16(m[0], m[1]);
      M[j >> 1][(j & 1) * 2 + 1] = pack_bf16(m[2], m[3]);
    }
    float Y[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) Y[j][e] = 0.f;
#pragma unroll
    for (int kk2 = 0; kk2 < 4; ++kk2) {
      if (kk2 > warp) break;
      const uint32_t a[4] = {M[kk2][0], M[kk2][1], M[kk2][2], M[kk2][3]};
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        uint32_t bb[4];
        ldsm_x4_t(xs + swz(16 * kk2 + (lane & 7) + 8 * ((lane >> 3) & 1), 2 * jj + (lane >> 4)), bb);
        mma16816(Y[2 * jj], a, bb[0], bb[1]);
        mma16816(Y[2 * jj + 1], a, bb[2], bb[3]);
      }
    }
    const float eta = fast_exp(cta), etb = fast_exp(ctb);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float2 xa = unpack_bf16(*reinterpret_cast<const uint32_t*>(st + SM::kX + swz(ta, j) + 4 * cq));
      const float2 xb = unpack_bf16(*reinterpret_cast<const uint32_t*>(st + SM::kX + swz(tb, j) + 4 * cq));
      const float y0 = Y[j][0] + eta * CS[j][0] + Dh * xa.x;
      const float y1 = Y[j][1] + eta * CS[j][1] + Dh * xa.y;
      const float y2 = Y[j][2] + etb * CS[j][2] + Dh * xb.x;
      const float y3 = Y[j][3] + etb * CS[j][3] + Dh * xb.y;
      *reinterpret_cast<uint32_t*>(smem + SM::kStage + swz(ta, j) + 4 * cq) = pack_bf16(y0, y1);
      *reinterpret_cast<uint32_t*>(smem + SM::kStage + swz(tb, j) + 4 * cq) = pack_bf16(y2, y3);
    }
    __syncthreads();  // y rows staged; every read of x done
    // the chunk's y rows to global memory (16 bytes per thread and pass), and
    // x' = w o delta x in place of x
    {
      __nv_bfloat16* yb = P.y + ((size_t)b * P.L) * P.H * kP + (size_t)h * kP;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int q = tid + kSsdThreads * i;  // 512 chunks of 16 bytes
        const int row = q >> 3, c8 = q & 7;
        if (t0 + row < P.L) {
          const uint4 v = *reinterpret_cast<const uint4*>(smem + SM::kStage + swz(row, c8));
          *reinterpret_cast<uint4*>(yb + (size_t)(t0 + row) * P.H * kP + 8 * c8) = v;
        }
        const float f = wd[row];
        const uint4 xv = *reinterpret_cast<const uint4*>(st + SM::kX + swz(row, c8));
        const uint32_t in[4] = {xv.x, xv.y, xv.z, xv.w};
        uint32_t out[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 e = unpack_bf16(in[k]);
          out[k] = pack_bf16(f * e.x, f * e.y);
        }
        *reinterpret_cast<uint4*>(st + SM::kX + swz(row, c8)) = make_uint4(out[0], out[1], out[2], out[3]);
      }
    }
    if constexpr (kUmma) fence_proxy_async_smem();  // x' is read by the tensor core
    __syncthreads();
    // ---- S = e^(cum_end) S + B^T x'
    if constexpr (kUmma) {
      // one thread issues the 128 x 64 x 64 product as four K = 16 steps:
      // A = B^T from the Bm boxes (MN-major: n contiguous, the two 64-column
      // boxes 8 KB apart), B = x' (MN-major), D = S in TMEM (already scaled)
      if (tid == 0) {
        tmem_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t da = umma_desc_sw128(bs + kk * 2048u, kTileBytes, 1024u);
          const uint64_t db = umma_desc_sw128(xs + kk * 2048u, kTileBytes, 1024u);
          umma_f16(tmem, da, db, kUmmaIdesc, 1u);
        }
        umma_commit(mma_bar);
      }
    } else {  // warp w: rows n = 16 w .. 16 w + 15 of S (N = 64)
      const float dec = cum[192];
#pragma unroll
      for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) S[mt][j][e] *= dec;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {  // s blocks
        uint32_t bx[4][4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
          ldsm_x4_t(xs + swz(16 * kk + (lane & 7) + 8 * ((lane >> 3) & 1), 2 * jj + (lane >> 4)), bx[jj]);
#pragma unroll
        for (int mt = 0; mt < kMT; ++mt) {
          const int m0 = warp * (N / 4) + 16 * mt;  // rows n
          const int sub = m0 / 64, mc = (m0 % 64) / 8;
          uint32_t a[4];
          ldsm_x4_t(bs + sub * kTileBytes + swz(16 * kk + (lane & 7) + 8 * (lane >> 4), mc + ((lane >> 3) & 1)), a);
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            mma16816(S[mt][2 * jj], a, bx[jj][0], bx[jj][1]);
            mma16816(S[mt][2 * jj + 1], a, bx[jj][2], bx[jj][3]);
          }
        }
      }
    }
    if (warp == 0 && c + 1 < nch) {  // the next chunk's decays; its successor's dt in flight
      chunk_decays(c + 1);
      load_dt(c + 2);
    }
    if constexpr (kUmma) {
      // the updated state: S_in of the next chunk's readout (bf16), or h_last
      mbar_wait(mma_bar, (uint32_t)(c & 1), P.status);
      tmem_fence_after_sync();
      float v[64];
      tmem_row_ld(v);
      if (c + 1 < nch) {
        row_to_smem_bf16(v);
      } else if (P.h_last) {
        float* hl = P.h_last + (((size_t)b * P.H + h) * N + tid) * kP;
#pragma unroll
        for (int i = 0; i < 64; i += 2) *reinterpret_cast<float2*>(hl + i) = make_float2(v[i], v[i + 1]);
      }
      tmem_fence_before_sync();
    }
    __syncthreads();  // every warp is done with S_in, the stage and x'
    if constexpr (!kUmma) store_S_bf16();
    if (tid == 0 && c + 2 < nch) issue(c + 2);
  }
  if constexpr (kUmma) {
    __syncthreads();
    tmem_fence_after_sync();
    if (warp == 0) tmem_dealloc(tmem, 64);
  } else if (P.h_last) {
    float* hl = P.h_last + ((size_t)b * P.H + h) * N * kP;
#pragma unroll
    for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int hlf = 0; hlf < 2; ++hlf) {
          const int n = warp * (N / 4) + 16 * mt + gq + 8 * hlf, p = 8 * j + 2 * cq;
          *reinterpret_cast<float2*>(hl + (size_t)n * kP + p) = make_float2(S[mt][j][2 * hlf], S[mt][j][2 * hlf + 1]);
        }
  }
}

template <int N>
cudaError_t launch_n(const SsdParams& P, cudaStream_t stream) {
  auto kern = s6_ssd_fwd_kernel<N>;
  const size_t smem = SsdSmem<N>::kBytes + 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)(P.B * P.H), kSsdThreads, smem, stream>>>(P);
  return cudaGetLastError();
}

}  // namespace

bool ssd_supported(int act, int P, int N) { return act == SSM_BF16 && P == kP && (N == 64 || N == 128); }

cudaError_t launch_ssd_fwd(const SsdArgs& a, cudaStream_t stream) {
  SsdParams P;
  memset(&P, 0, sizeof(P));
  const uint64_t e = 2;
  {
    const uint64_t dims[3] = {(uint64_t)a.H * kP, (uint64_t)a.L, (uint64_t)a.B};
    const uint64_t strides[2] = {(uint64_t)a.H * kP * e, (uint64_t)a.L * a.H * kP * e};
    const uint32_t box[3] = {64, kQ, 1};
    if (!encode_tile_map(&P.map_x, a.x, true, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
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
  P.status = a.status;
  P.dt_min = a.dt_min;
  P.dt_max = a.dt_max;
  P.B = a.B;
  P.L = a.L;
  P.H = a.H;
  P.G = a.G;
  P.N = a.N;
  return a.N == 128 ? launch_n<128>(P, stream) : launch_n<64>(P, stream);
}

}  // namespace s6
