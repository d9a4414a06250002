// Host side of the C ABI declared in include/ssm_scan.h: argument checks,
// workspace sizing and kernel dispatch.  No allocation, no synchronisation.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "s6_internal.cuh"
#include "s6_tma.cuh"

namespace s6 {

// The library's device status word: bounded device-side waits that give up
// set bits here (kStatusWaitTimeout); ssm_check_device_status() reads and
// clears it.  One copy per device; its address is looked up per device.
__device__ unsigned int g_s6_status = 0;

void* current_context() {
  using GetCtx = int (*)(void**);  // cuCtxGetCurrent(CUcontext*), CUresult 0 = success
  static GetCtx fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return (GetCtx) nullptr;
    return reinterpret_cast<GetCtx>(f);
  }();
  void* ctx = nullptr;
  if (!fn || fn(&ctx) != 0) return nullptr;
  return ctx;
}

cudaError_t symbol_address(SymbolCache& cache, const void* symbol, void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= SymbolCache::kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(cache.mu);
  void* ctx = current_context();
  if (!cache.addr[dev] || !ctx || cache.ctx[dev] != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, symbol);
    if (e != cudaSuccess) return e;
    cache.addr[dev] = p;
    cache.ctx[dev] = current_context();  // the lookup made the device's context current
  }
  *out = cache.addr[dev];
  return cudaSuccess;
}

int device_sm_count() {
  static std::mutex mu;
  static int sms[SymbolCache::kMaxDevices] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= SymbolCache::kMaxDevices) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (sms[dev] <= 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    sms[dev] = n;
  }
  return sms[dev];
}

static std::atomic<long long> g_plan_fallbacks{0};
void note_plan_fallback() { g_plan_fallbacks.fetch_add(1, std::memory_order_relaxed); }
long long plan_fallbacks() { return g_plan_fallbacks.load(std::memory_order_relaxed); }

unsigned int* device_status_word() {
  static SymbolCache cache;
  void* a = nullptr;
  if (symbol_address(cache, &g_s6_status, &a) != cudaSuccess) return nullptr;
  return static_cast<unsigned int*>(a);
}

}  // namespace s6

namespace {

thread_local char g_last_error[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* where) {
  return fail(SSM_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

size_t act_size(int act) { return act == SSM_BF16 ? 2 : 4; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

constexpr int64_t kMaxElems = (int64_t)1 << 31;  // every per-tensor index fits in 31 bits

int check_shape(int64_t B, int64_t L, int64_t D, int64_t N, int act) {
  if (act != SSM_F32 && act != SSM_BF16) return fail(SSM_ERR_INVALID_ARG, "act must be SSM_F32 or SSM_BF16, got %d", act);
  if (B < 0 || L < 0 || D < 0) return fail(SSM_ERR_INVALID_ARG, "negative shape (B=%lld L=%lld D=%lld)", (long long)B, (long long)L, (long long)D);
  if (N < 1) return fail(SSM_ERR_INVALID_ARG, "dstate must be >= 1, got %lld", (long long)N);
  if (N > SSM_MAX_DSTATE) return fail(SSM_ERR_UNSUPPORTED, "dstate %lld > %d is not supported", (long long)N, SSM_MAX_DSTATE);
  if (B > 65535) return fail(SSM_ERR_UNSUPPORTED, "batch %lld > 65535 is not supported", (long long)B);
  if (B * L * D >= kMaxElems || B * L * N >= kMaxElems || B * D * N * (L / SSM_CHUNK_LEN + 1) >= kMaxElems)
    return fail(SSM_ERR_UNSUPPORTED, "problem too large for 31-bit indexing");
  return SSM_OK;
}

// A required pointer to `count` elements must be non-NULL (unless the tensor
// is empty) and aligned to its element size.
int need(const void* p, int64_t count, size_t align, const char* name) {
  if (!p) {
    if (count == 0) return SSM_OK;
    return fail(SSM_ERR_INVALID_ARG, "%s must not be NULL", name);
  }
  if (!aligned(p, align)) return fail(SSM_ERR_INVALID_ARG, "%s is not %zu-byte aligned", name, align);
  return SSM_OK;
}
int opt(const void* p, size_t align, const char* name) {
  return p ? need(p, 1, align, name) : SSM_OK;
}

#define S6_TRY(x)                    \
  do {                               \
    const int _rc = (x);             \
    if (_rc != SSM_OK) return _rc;   \
  } while (0)

int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

int check_ws(const void* ws, size_t ws_bytes, int64_t total) {
  if (total <= 0) return SSM_OK;
  if (!ws) return fail(SSM_ERR_WORKSPACE, "ws is NULL but %lld bytes are required", (long long)total);
  if ((int64_t)ws_bytes < total)
    return fail(SSM_ERR_WORKSPACE, "ws_bytes=%zu < required %lld", ws_bytes, (long long)total);
  if (!aligned(ws, 256)) return fail(SSM_ERR_INVALID_ARG, "ws is not 256-byte aligned");
  return SSM_OK;
}

// The forward's segment plan and the backward's work plan are functions of
// the shape only (they target a 152-SM GB300), so workspace sizes and results
// never depend on the device.
constexpr int kPlanSms = 152;

struct FwdWorkspace {
  s6::FwdPlan plan;  // stream plan (plan.handover) or not
  int nseg, seg_len;
  int64_t agg_off, start_off, flag_off, carry_off, total;
};

FwdWorkspace fwd_ws_layout(int64_t B, int64_t L, int64_t D, int64_t N, int act) {
  FwdWorkspace w;
  w.plan = s6::fwd_stream_plan((int)B, (int)L, (int)D, (int)N, act, kPlanSms);
  w.nseg = w.plan.handover ? 1 : s6::fwd_segments((int)B, (int)L, (int)D, (int)N, kPlanSms);
  w.seg_len = (int)L;
  w.agg_off = w.start_off = w.flag_off = w.carry_off = w.total = 0;
  if (w.plan.handover) {
    // one flag and one hand-over state (128/TPC channels x N = 512 floats) per sequence
    const int64_t nseq = B * (int64_t)w.plan.ndt;
    w.flag_off = 0;
    w.carry_off = align_up(nseq * (int64_t)sizeof(int), 256);
    w.total = align_up(w.carry_off + nseq * 512 * (int64_t)sizeof(float), 256);
  } else if (w.nseg > 1) {
    w.seg_len = (int)(((L + w.nseg - 1) / w.nseg + SSM_CHUNK_LEN - 1) / SSM_CHUNK_LEN * SSM_CHUNK_LEN);
    w.nseg = (int)((L + w.seg_len - 1) / w.seg_len);
    const int64_t cells = B * w.nseg * D * N;
    w.agg_off = 0;
    w.start_off = align_up(cells * 2 * (int64_t)sizeof(float), 256);
    w.total = align_up(w.start_off + cells * (int64_t)sizeof(float), 256);
  }
  return w;
}

struct BwdWorkspace {
  s6::BwdPlan plan;
  int nseg, nslot;
  int64_t hdr_off, dbc_off, dbc_bytes, param_off, param_bytes, agg_off, carry_off, flag_off, total;
};

BwdWorkspace bwd_ws_layout(int64_t B, int64_t L, int64_t D, int64_t N) {
  BwdWorkspace w;
  w.plan = s6::bwd_plan((int)B, (int)L, (int)D, (int)N, kPlanSms);
  w.nseg = w.plan.maxp;
  // tile rows of the dBm/dCm partials: 128-channel tiles (TMA kernel) or
  // 64-channel tiles (generic kernel); room for the larger count.  The kernel
  // that fills them writes their count into the header at offset 0.
  const int64_t ndt = (D + s6::kDTile - 1) / s6::kDTile;
  w.hdr_off = 0;
  w.dbc_off = 256;
  w.dbc_bytes = ndt * B * L * 2 * N * (int64_t)sizeof(float);
  w.param_off = align_up(w.dbc_off + w.dbc_bytes, 256);
  w.param_bytes = B * w.nseg * D * (N + 2) * (int64_t)sizeof(float);
  w.agg_off = align_up(w.param_off + w.param_bytes, 256);
  w.nslot = w.nseg > 1 ? s6::agg_slots(w.plan) : 0;
  const int64_t cells = w.nseg > 1 ? B * w.nseg * D * N : 0;
  const int64_t agg_cells = B * (int64_t)w.nslot * D * N;
  w.carry_off = align_up(w.agg_off + agg_cells * 2 * (int64_t)sizeof(float), 256);
  // one hand-over flag per (batch, channel tile) sequence
  const int64_t nseq = w.nseg > 1 ? B * (int64_t)w.plan.ndt : 0;
  w.flag_off = align_up(w.carry_off + cells * (int64_t)sizeof(float), 256);
  w.total = align_up(w.flag_off + nseq * (int64_t)sizeof(int), 256);
  return w;
}

// dt_limit of an options struct (NULL: 0, +inf); 0 <= dt_min <= dt_max
int read_opts(const ssm_scan_options* o, float* lo, float* hi) {
  *lo = 0.f;
  *hi = INFINITY;
  if (!o) return SSM_OK;
  if (!(o->dt_min >= 0.f) || !(o->dt_min <= o->dt_max))
    return fail(SSM_ERR_INVALID_ARG, "dt limit needs 0 <= dt_min <= dt_max, got [%g, %g]", (double)o->dt_min,
                (double)o->dt_max);
  *lo = o->dt_min;
  *hi = o->dt_max;
  return SSM_OK;
}

int fwd_common(int64_t B, int64_t L, int64_t D, int64_t N, int act, const void* u,
               const void* delta_raw, const void* z, const void* Bm, const void* Cm,
               const float* A_log, const float* Dp, const float* delta_bias, const float* h0,
               void* out, float* h_last, float* chunk_states, bool save, void* ws,
               size_t ws_bytes, void* stream, const ssm_scan_options* opts, bool step = false) {
  float dt_lo, dt_hi;
  S6_TRY(read_opts(opts, &dt_lo, &dt_hi));
  S6_TRY(check_shape(B, L, D, N, act));
  const size_t e = act_size(act);
  const int64_t bld = B * L * D, bln = B * L * N, dn = D * N;
  S6_TRY(need(u, bld, e, "u"));
  S6_TRY(need(delta_raw, bld, e, "delta_raw"));
  S6_TRY(opt(z, e, "z"));
  S6_TRY(need(Bm, bln, e, "Bm"));
  S6_TRY(need(Cm, bln, e, "Cm"));
  S6_TRY(need(A_log, dn, 4, "A_log"));
  S6_TRY(need(Dp, D, 4, "Dp"));
  S6_TRY(need(delta_bias, D, 4, "delta_bias"));
  S6_TRY(opt(h0, 4, "h0"));
  S6_TRY(need(out, bld, e, "out"));
  S6_TRY(opt(h_last, 4, "h_last"));
  if (save) S6_TRY(need(chunk_states, B * ssm_num_chunks(L) * dn, 4, "chunk_states"));
  g_last_error[0] = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (B == 0 || D == 0) return SSM_OK;
  if (L == 0) {
    // No steps: the final state is the initial state.
    if (h_last) {
      cudaError_t ce = h0 ? cudaMemcpyAsync(h_last, h0, sizeof(float) * B * D * N, cudaMemcpyDeviceToDevice, st)
                          : cudaMemsetAsync(h_last, 0, sizeof(float) * B * D * N, st);
      if (ce != cudaSuccess) return cuda_fail(ce, "ssm_scan_fwd(L=0)");
    }
    return SSM_OK;
  }
  s6::FwdParams p;
  p.u = u; p.delta_raw = delta_raw; p.z = z; p.Bm = Bm; p.Cm = Cm;
  p.A_log = A_log; p.Dp = Dp; p.delta_bias = delta_bias; p.h0 = h0;
  p.out = out; p.h_last = h_last; p.chunk_states = save ? chunk_states : nullptr;
  p.B = (int)B; p.L = (int)L; p.D = (int)D; p.N = (int)N;
  p.nchunks = (int)ssm_num_chunks(L);
  p.dt_min = dt_lo;
  p.dt_max = dt_hi;
  p.status = s6::device_status_word();
  if (!p.status) return fail(SSM_ERR_CUDA, "cannot locate the device status word");
  const FwdWorkspace w = fwd_ws_layout(B, L, D, N, act);
  S6_TRY(check_ws(ws, ws_bytes, w.total));
  p.nseg = 1;
  p.seg_len = (int)L;
  p.seg_agg = p.seg_start = nullptr;
  p.plan = w.plan;
  p.seq_flag = nullptr;
  p.seq_carry = nullptr;
  const bool tma = s6::fwd_tma_supported(p, act);
  if (tma && w.plan.handover && !step) {
    p.seq_flag = reinterpret_cast<int*>(static_cast<char*>(ws) + w.flag_off);
    p.seq_carry = reinterpret_cast<float*>(static_cast<char*>(ws) + w.carry_off);
  }
  if (tma && w.nseg > 1) {
    p.nseg = w.nseg;
    p.seg_len = w.seg_len;
    p.seg_agg = reinterpret_cast<float*>(static_cast<char*>(ws) + w.agg_off);
    p.seg_start = reinterpret_cast<float*>(static_cast<char*>(ws) + w.start_off);
  }
  cudaError_t ce;
  if (step && L == 1 && s6::step_supported(p, act))
    ce = s6::launch_step(p, act, st);
  else
    ce = tma ? s6::launch_fwd_tma(p, act, st) : s6::launch_fwd(p, act, st);
  if (ce != cudaSuccess) return cuda_fail(ce, "ssm_scan_fwd launch");
  return SSM_OK;
}

}  // namespace

namespace s6 {

// Records a message for ssm_last_error() and returns `code` (for entry points
// defined in other translation units).
int report_error(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return code;
}

}  // namespace s6

// One thread waits on an mbarrier phase that nothing completes: the bounded
// wait gives up after kWaitCycles and sets the timeout bit (self-test of the
// give-up path used by every pipeline wait).
__global__ void s6_selftest_wait_kernel(unsigned int* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    s6::mbar_init(&bar, 1);
    s6::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) s6::mbar_wait(&bar, 0, status);
}

extern "C" {

const char* ssm_status_string(int status) {
  switch (status) {
    case SSM_OK: return "SSM_OK";
    case SSM_ERR_INVALID_ARG: return "SSM_ERR_INVALID_ARG";
    case SSM_ERR_UNSUPPORTED: return "SSM_ERR_UNSUPPORTED";
    case SSM_ERR_WORKSPACE: return "SSM_ERR_WORKSPACE";
    case SSM_ERR_CUDA: return "SSM_ERR_CUDA";
    case SSM_ERR_TIMEOUT: return "SSM_ERR_TIMEOUT";
    case SSM_ERR_INTERNAL: return "SSM_ERR_INTERNAL";
    default: return "SSM_ERR_UNKNOWN";
  }
}

const char* ssm_last_error(void) { return g_last_error; }

int ssm_version(void) { return 100; }

int ssm_check_device_status(void* stream) {
  unsigned int* w = s6::device_status_word();
  if (!w) return fail(SSM_ERR_CUDA, "cannot locate the device status word");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned int v = 0;
  cudaError_t ce = cudaMemcpyAsync(&v, w, sizeof(v), cudaMemcpyDeviceToHost, st);
  if (ce == cudaSuccess) ce = cudaStreamSynchronize(st);
  if (ce == cudaSuccess && v != 0) ce = cudaMemsetAsync(w, 0, sizeof(v), st);
  if (ce == cudaSuccess) ce = cudaStreamSynchronize(st);
  if (ce != cudaSuccess) return cuda_fail(ce, "ssm_check_device_status");
  if (v & s6::kStatusWaitTimeoutBit) return fail(SSM_ERR_TIMEOUT, "a device-side wait gave up (status 0x%x)", v);
  if (v & s6::kStatusLayoutBit)
    return fail(SSM_ERR_INTERNAL, "a kernel found its shared memory misaligned for swizzled tiles (status 0x%x)", v);
  return SSM_OK;
}

int ssm_selftest_wait_timeout(void* stream) {
  unsigned int* w = s6::device_status_word();
  if (!w) return fail(SSM_ERR_CUDA, "cannot locate the device status word");
  s6_selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(w);
  const cudaError_t ce = cudaGetLastError();
  return ce == cudaSuccess ? SSM_OK : cuda_fail(ce, "ssm_selftest_wait_timeout");
}

int64_t ssm_num_chunks(int64_t seqlen) {
  return seqlen <= 0 ? 0 : (seqlen + SSM_CHUNK_LEN - 1) / SSM_CHUNK_LEN;
}

int64_t ssm_fwd_workspace_bytes(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, int act) {
  if (check_shape(batch, seqlen, dim, dstate, act) != SSM_OK) return -1;
  return fwd_ws_layout(batch, seqlen, dim, dstate, act).total;
}

int64_t ssm_bwd_workspace_bytes(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, int act) {
  if (check_shape(batch, seqlen, dim, dstate, act) != SSM_OK) return -1;
  return bwd_ws_layout(batch, seqlen, dim, dstate).total;
}

int64_t ssm_plan_fallbacks(void) { return (int64_t)s6::plan_fallbacks(); }

int ssm_plan_segments(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, int act,
                      int* fwd_segments, int* bwd_segments) {
  const int rc = check_shape(batch, seqlen, dim, dstate, act);
  if (rc != SSM_OK) return rc;
  if (fwd_segments) *fwd_segments = fwd_ws_layout(batch, seqlen, dim, dstate, act).nseg;
  if (bwd_segments) {
    const BwdWorkspace w = bwd_ws_layout(batch, seqlen, dim, dstate);
    *bwd_segments = w.plan.handover ? 1 : w.nseg;
  }
  return SSM_OK;
}

int ssm_scan_fwd(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, int act,
                 const void* u, const void* delta_raw, const void* z, const void* Bm,
                 const void* Cm, const float* A_log, const float* Dp, const float* delta_bias,
                 const float* h0, void* out, float* h_last, float* chunk_states, void* ws,
                 size_t ws_bytes, void* stream) {
  return fwd_common(batch, seqlen, dim, dstate, act, u, delta_raw, z, Bm, Cm, A_log, Dp,
                    delta_bias, h0, out, h_last, chunk_states, true, ws, ws_bytes, stream, nullptr);
}

int ssm_scan_fwd_ex(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, int act,
                    const void* u, const void* delta_raw, const void* z, const void* Bm,
                    const void* Cm, const float* A_log, const float* Dp, const float* delta_bias,
                    const float* h0, void* out, float* h_last, float* chunk_states, void* ws,
                    size_t ws_bytes, void* stream, const ssm_scan_options* opts) {
  return fwd_common(batch, seqlen, dim, dstate, act, u, delta_raw, z, Bm, Cm, A_log, Dp,
                    delta_bias, h0, out, h_last, chunk_states, chunk_states != nullptr, ws, ws_bytes,
                    stream, opts);
}

int ssm_scan_fwd_nosave(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, int act,
                        const void* u, const void* delta_raw, const void* z, const void* Bm,
                        const void* Cm, const float* A_log, const float* Dp,
                        const float* delta_bias, const float* h0, void* out, float* h_last,
                        void* ws, size_t ws_bytes, void* stream) {
  return fwd_common(batch, seqlen, dim, dstate, act, u, delta_raw, z, Bm, Cm, A_log, Dp,
                    delta_bias, h0, out, h_last, nullptr, false, ws, ws_bytes, stream, nullptr);
}

int ssm_scan_bwd_partials(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, int act,
                          const void* u, const void* delta_raw, const void* z, const void* Bm,
                          const void* Cm, const float* A_log, const float* Dp,
                          const float* delta_bias, const float* chunk_states, const void* dout,
                          const float* dh_last, void* du, void* d_delta_raw, void* dz,
                          float* dh0, void* ws, size_t ws_bytes, void* stream) {
  return ssm_scan_bwd_partials_ex(batch, seqlen, dim, dstate, act, u, delta_raw, z, Bm, Cm, A_log, Dp,
                                  delta_bias, chunk_states, dout, dh_last, du, d_delta_raw, dz, dh0, ws,
                                  ws_bytes, stream, nullptr);
}

int ssm_scan_bwd_partials_ex(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, int act,
                             const void* u, const void* delta_raw, const void* z, const void* Bm,
                             const void* Cm, const float* A_log, const float* Dp,
                             const float* delta_bias, const float* chunk_states, const void* dout,
                             const float* dh_last, void* du, void* d_delta_raw, void* dz,
                             float* dh0, void* ws, size_t ws_bytes, void* stream,
                             const ssm_scan_options* opts) {
  const int64_t B = batch, L = seqlen, D = dim, N = dstate;
  float dt_lo, dt_hi;
  S6_TRY(read_opts(opts, &dt_lo, &dt_hi));
  S6_TRY(check_shape(B, L, D, N, act));
  const size_t e = act_size(act);
  const int64_t bld = B * L * D, bln = B * L * N, dn = D * N;
  S6_TRY(need(u, bld, e, "u"));
  S6_TRY(need(delta_raw, bld, e, "delta_raw"));
  S6_TRY(opt(z, e, "z"));
  S6_TRY(need(Bm, bln, e, "Bm"));
  S6_TRY(need(Cm, bln, e, "Cm"));
  S6_TRY(need(A_log, dn, 4, "A_log"));
  S6_TRY(need(Dp, D, 4, "Dp"));
  S6_TRY(need(delta_bias, D, 4, "delta_bias"));
  S6_TRY(need(chunk_states, B * ssm_num_chunks(L) * dn, 4, "chunk_states"));
  S6_TRY(need(dout, bld, e, "dout"));
  S6_TRY(opt(dh_last, 4, "dh_last"));
  S6_TRY(need(du, bld, e, "du"));
  S6_TRY(need(d_delta_raw, bld, e, "d_delta_raw"));
  if (z) S6_TRY(need(dz, bld, e, "dz (required when z is given)"));
  S6_TRY(opt(dh0, 4, "dh0"));
  const BwdWorkspace w = bwd_ws_layout(B, L, D, N);
  S6_TRY(check_ws(ws, ws_bytes, w.total));
  g_last_error[0] = 0;
  if (B == 0 || D == 0) return SSM_OK;
  s6::BwdParams p;
  p.u = u; p.delta_raw = delta_raw; p.z = z; p.Bm = Bm; p.Cm = Cm;
  p.A_log = A_log; p.Dp = Dp; p.delta_bias = delta_bias; p.chunk_states = chunk_states;
  p.dout = dout; p.dh_last = dh_last; p.du = du; p.d_delta_raw = d_delta_raw; p.dz = dz;
  p.dh0 = dh0;
  p.ws_dbc = reinterpret_cast<float*>(static_cast<char*>(ws) + w.dbc_off);
  p.ws_ndt = reinterpret_cast<int*>(static_cast<char*>(ws) + w.hdr_off);
  p.ws_param = reinterpret_cast<float*>(static_cast<char*>(ws) + w.param_off);
  p.B = (int)B; p.L = (int)L; p.D = (int)D; p.N = (int)N;
  p.nchunks = (int)ssm_num_chunks(L);
  p.dt_min = dt_lo;
  p.dt_max = dt_hi;
  p.status = s6::device_status_word();
  if (!p.status) return fail(SSM_ERR_CUDA, "cannot locate the device status word");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  p.plan = w.plan;
  p.nseg = w.nseg;
  p.nslot = w.nslot;
  p.seg_agg = reinterpret_cast<float*>(static_cast<char*>(ws) + w.agg_off);
  p.seg_carry = reinterpret_cast<float*>(static_cast<char*>(ws) + w.carry_off);
  p.seq_flag = w.nseg > 1 ? reinterpret_cast<int*>(static_cast<char*>(ws) + w.flag_off) : nullptr;
  cudaError_t ce;
  if (L > 0 && s6::bwd_tma_supported(p, act)) {
    ce = s6::launch_bwd_tma(p, act, st);
  } else {
    // the generic kernel does not split time: it fills segment row 0 of the
    // parameter partials; the other rows of the plan's layout are zeroed
    if (w.nseg > 1) {
      ce = cudaMemsetAsync(p.ws_param, 0, (size_t)w.param_bytes, st);
      if (ce != cudaSuccess) return cuda_fail(ce, "ssm_scan_bwd_partials");
    }
    ce = s6::launch_bwd(p, act, st);
  }
  if (ce != cudaSuccess) return cuda_fail(ce, "ssm_scan_bwd_partials launch");
  return SSM_OK;
}

int ssm_scan_bwd_finalize(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, int act,
                          void* dBm, void* dCm, float* dA_log, float* dDp, float* d_delta_bias,
                          const void* ws, size_t ws_bytes, void* stream) {
  const int64_t B = batch, L = seqlen, D = dim, N = dstate;
  S6_TRY(check_shape(B, L, D, N, act));
  const size_t e = act_size(act);
  S6_TRY(need(dBm, B * L * N, e, "dBm"));
  S6_TRY(need(dCm, B * L * N, e, "dCm"));
  S6_TRY(need(dA_log, D * N, 4, "dA_log"));
  S6_TRY(need(dDp, D, 4, "dDp"));
  S6_TRY(need(d_delta_bias, D, 4, "d_delta_bias"));
  const BwdWorkspace w = bwd_ws_layout(B, L, D, N);
  S6_TRY(check_ws(ws, ws_bytes, w.total));
  g_last_error[0] = 0;
  if (D == 0) return SSM_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const float* ws_dbc = reinterpret_cast<const float*>(static_cast<const char*>(ws) + w.dbc_off);
  const float* ws_param = reinterpret_cast<const float*>(static_cast<const char*>(ws) + w.param_off);
  cudaError_t ce;
  if (B > 0) {
    const int* ndt = reinterpret_cast<const int*>(static_cast<const char*>(ws) + w.hdr_off);
    ce = s6::launch_reduce_dbc(ws_dbc, ndt, (int)B, (int)L, (int)N, dBm, dCm, act, st);
    if (ce != cudaSuccess) return cuda_fail(ce, "ssm_scan_bwd_finalize dBm/dCm reduction");
  }
  ce = s6::launch_reduce_params(ws_param, (int)(B * w.nseg), (int)D, (int)N, dA_log, dDp, d_delta_bias, st);
  if (ce != cudaSuccess) return cuda_fail(ce, "ssm_scan_bwd_finalize parameter reduction");
  return SSM_OK;
}

int ssm_scan_bwd(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, int act,
                 const void* u, const void* delta_raw, const void* z, const void* Bm,
                 const void* Cm, const float* A_log, const float* Dp, const float* delta_bias,
                 const float* h0, const float* chunk_states, const void* dout,
                 const float* dh_last, void* du, void* d_delta_raw, void* dz, void* dBm,
                 void* dCm, float* dA_log, float* dDp, float* d_delta_bias, float* dh0,
                 void* ws, size_t ws_bytes, void* stream) {
  return ssm_scan_bwd_ex(batch, seqlen, dim, dstate, act, u, delta_raw, z, Bm, Cm, A_log, Dp, delta_bias, h0,
                         chunk_states, dout, dh_last, du, d_delta_raw, dz, dBm, dCm, dA_log, dDp, d_delta_bias,
                         dh0, ws, ws_bytes, stream, nullptr);
}

int ssm_scan_bwd_ex(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, int act,
                    const void* u, const void* delta_raw, const void* z, const void* Bm,
                    const void* Cm, const float* A_log, const float* Dp, const float* delta_bias,
                    const float* h0, const float* chunk_states, const void* dout,
                    const float* dh_last, void* du, void* d_delta_raw, void* dz, void* dBm,
                    void* dCm, float* dA_log, float* dDp, float* d_delta_bias, float* dh0,
                    void* ws, size_t ws_bytes, void* stream, const ssm_scan_options* opts) {
  // h0 is not read: the chunk states already start from it.  It is checked so
  // that a caller passing a bad pointer hears about it.
  S6_TRY(opt(h0, 4, "h0"));
  float dt_lo, dt_hi;
  S6_TRY(read_opts(opts, &dt_lo, &dt_hi));
  const size_t e = (act == SSM_BF16) ? 2 : 4;
  // validate the finalize outputs before enqueueing the first half
  S6_TRY(check_shape(batch, seqlen, dim, dstate, act));
  S6_TRY(need(dBm, batch * seqlen * dstate, e, "dBm"));
  S6_TRY(need(dCm, batch * seqlen * dstate, e, "dCm"));
  S6_TRY(need(dA_log, dim * dstate, 4, "dA_log"));
  S6_TRY(need(dDp, dim, 4, "dDp"));
  S6_TRY(need(d_delta_bias, dim, 4, "d_delta_bias"));
  S6_TRY(ssm_scan_bwd_partials_ex(batch, seqlen, dim, dstate, act, u, delta_raw, z, Bm, Cm, A_log,
                                  Dp, delta_bias, chunk_states, dout, dh_last, du, d_delta_raw, dz,
                                  dh0, ws, ws_bytes, stream, opts));
  return ssm_scan_bwd_finalize(batch, seqlen, dim, dstate, act, dBm, dCm, dA_log, dDp,
                               d_delta_bias, ws, ws_bytes, stream);
}

int ssm_step(int64_t batch, int64_t dim, int64_t dstate, int act, const void* u,
             const void* delta_raw, const void* z, const void* Bm, const void* Cm,
             const float* A_log, const float* Dp, const float* delta_bias, float* h, void* out,
             void* stream) {
  return ssm_step_ex(batch, dim, dstate, act, u, delta_raw, z, Bm, Cm, A_log, Dp, delta_bias, h, out, stream,
                     nullptr);
}

int ssm_step_ex(int64_t batch, int64_t dim, int64_t dstate, int act, const void* u,
                const void* delta_raw, const void* z, const void* Bm, const void* Cm,
                const float* A_log, const float* Dp, const float* delta_bias, float* h, void* out,
                void* stream, const ssm_scan_options* opts) {
  S6_TRY(need(h, batch * dim * (dstate > 0 ? dstate : 0), 4, "h"));
  return fwd_common(batch, 1, dim, dstate, act, u, delta_raw, z, Bm, Cm, A_log, Dp, delta_bias,
                    h, out, h, nullptr, false, nullptr, 0, stream, opts, /*step=*/true);
}

// ---------------------------------------------------------------- conv1d

int check_conv(int64_t B, int64_t L, int64_t D, int64_t K, int act) {
  if (act != SSM_F32 && act != SSM_BF16) return fail(SSM_ERR_INVALID_ARG, "act must be SSM_F32 or SSM_BF16, got %d", act);
  if (B < 0 || L < 0 || D < 0) return fail(SSM_ERR_INVALID_ARG, "negative shape");
  if (K < 1) return fail(SSM_ERR_INVALID_ARG, "width must be >= 1, got %lld", (long long)K);
  if (K > SSM_MAX_CONV_WIDTH) return fail(SSM_ERR_UNSUPPORTED, "width %lld > %d is not supported", (long long)K, SSM_MAX_CONV_WIDTH);
  if (B * L * D >= kMaxElems || B * D * K >= kMaxElems) return fail(SSM_ERR_UNSUPPORTED, "problem too large for 31-bit indexing");
  return SSM_OK;
}

int ssm_conv1d_fwd(int64_t batch, int64_t seqlen, int64_t dim, int64_t width, int act, const void* x,
                   const float* w, const float* bias, const void* state0, void* out, void* state_last,
                   void* stream) {
  const int64_t B = batch, L = seqlen, D = dim, K = width;
  S6_TRY(check_conv(B, L, D, K, act));
  const size_t e = act_size(act);
  S6_TRY(need(x, B * L * D, e, "x"));
  S6_TRY(need(w, D * K, 4, "w"));
  S6_TRY(need(bias, D, 4, "bias"));
  S6_TRY(opt(state0, e, "state0"));
  S6_TRY(need(out, B * L * D, e, "out"));
  S6_TRY(opt(state_last, e, "state_last"));
  g_last_error[0] = 0;
  if (B == 0 || D == 0) return SSM_OK;
  s6::ConvParams p = {};
  p.x = x; p.w = w; p.bias = bias; p.state0 = state0; p.out = out; p.state_last = state_last;
  p.B = (int)B; p.L = (int)L; p.D = (int)D; p.K = (int)K;
  p.status = s6::device_status_word();
  if (!p.status) return fail(SSM_ERR_CUDA, "cannot locate the device status word");
  const cudaError_t ce = s6::launch_conv1d(p, act, false, static_cast<cudaStream_t>(stream));
  return ce == cudaSuccess ? SSM_OK : cuda_fail(ce, "ssm_conv1d_fwd launch");
}

int64_t ssm_conv1d_bwd_workspace_bytes(int64_t batch, int64_t seqlen, int64_t dim, int64_t width, int act) {
  if (check_conv(batch, seqlen, dim, width, act) != SSM_OK) return -1;
  return (int64_t)s6::conv1d_bwd_workspace_bytes((int)batch, (int)seqlen, (int)dim, (int)width);
}

int ssm_conv1d_bwd(int64_t batch, int64_t seqlen, int64_t dim, int64_t width, int act, const void* x,
                   const float* w, const float* bias, const void* state0, const void* dout, void* dx,
                   float* dw, float* dbias, float* dstate0, void* ws, size_t ws_bytes, void* stream) {
  const int64_t B = batch, L = seqlen, D = dim, K = width;
  S6_TRY(check_conv(B, L, D, K, act));
  const size_t e = act_size(act);
  S6_TRY(need(x, B * L * D, e, "x"));
  S6_TRY(need(w, D * K, 4, "w"));
  S6_TRY(need(bias, D, 4, "bias"));
  S6_TRY(opt(state0, e, "state0"));
  S6_TRY(need(dout, B * L * D, e, "dout"));
  S6_TRY(need(dx, B * L * D, e, "dx"));
  S6_TRY(need(dw, D * K, 4, "dw"));
  S6_TRY(need(dbias, D, 4, "dbias"));
  S6_TRY(opt(dstate0, 4, "dstate0"));
  const int64_t total = (int64_t)s6::conv1d_bwd_workspace_bytes((int)B, (int)L, (int)D, (int)K);
  S6_TRY(check_ws(ws, ws_bytes, total));
  g_last_error[0] = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (D == 0) return SSM_OK;
  if (B == 0 || L == 0) {
    // no steps: zero weight and bias gradients (and the state's)
    cudaError_t ce = cudaMemsetAsync(dw, 0, sizeof(float) * D * K, st);
    if (ce == cudaSuccess) ce = cudaMemsetAsync(dbias, 0, sizeof(float) * D, st);
    if (ce == cudaSuccess && dstate0 && B > 0 && K > 1) ce = cudaMemsetAsync(dstate0, 0, sizeof(float) * B * D * (K - 1), st);
    return ce == cudaSuccess ? SSM_OK : cuda_fail(ce, "ssm_conv1d_bwd");
  }
  s6::ConvParams p = {};
  p.x = x; p.w = w; p.bias = bias; p.state0 = state0; p.dout = dout; p.dx = dx; p.dw = dw; p.dbias = dbias;
  p.dstate0 = dstate0; p.ws = static_cast<float*>(ws);
  p.B = (int)B; p.L = (int)L; p.D = (int)D; p.K = (int)K;
  p.status = s6::device_status_word();
  if (!p.status) return fail(SSM_ERR_CUDA, "cannot locate the device status word");
  const cudaError_t ce = s6::launch_conv1d(p, act, true, st);
  return ce == cudaSuccess ? SSM_OK : cuda_fail(ce, "ssm_conv1d_bwd launch");
}

int ssm_conv1d_path(int64_t batch, int64_t seqlen, int64_t dim, int64_t width, int act, const void* x,
                    const void* dout, const void* y) {
  const int st = check_conv(batch, seqlen, dim, width, act);
  if (st != SSM_OK) return -st;
  s6::ConvParams p = {};
  p.x = x;
  p.dout = dout;
  if (dout)
    p.dx = const_cast<void*>(y);
  else
    p.out = const_cast<void*>(y);
  p.B = (int)batch; p.L = (int)seqlen; p.D = (int)dim; p.K = (int)width;
  return s6::conv1d_path(p, act, dout != nullptr);
}

// shape checks shared by the SSD entry points
int check_ssd(int64_t B, int64_t L, int64_t H, int64_t P, int64_t G, int64_t N, int act, const char* what) {
  if (act != SSM_F32 && act != SSM_BF16) return fail(SSM_ERR_INVALID_ARG, "act must be SSM_F32 or SSM_BF16, got %d", act);
  if (B < 0 || L < 0 || H < 1 || P < 1 || G < 1 || N < 1)
    return fail(SSM_ERR_INVALID_ARG, "bad SSD shape (B=%lld L=%lld H=%lld P=%lld G=%lld N=%lld)", (long long)B,
                (long long)L, (long long)H, (long long)P, (long long)G, (long long)N);
  if (H % G != 0) return fail(SSM_ERR_INVALID_ARG, "nheads %lld is not a multiple of ngroups %lld", (long long)H, (long long)G);
  if (!s6::ssd_supported(act, (int)P, (int)N))
    return fail(SSM_ERR_UNSUPPORTED, "SSD %s supports bf16 activations, headdim 32 or a multiple of 64 (up to 256) and dstate 64 or 128", what);
  const int64_t nch = (L + SSM_SSD_CHUNK_LEN - 1) / SSM_SSD_CHUNK_LEN;
  if (B * L * H * P >= kMaxElems || B * L * H * N >= kMaxElems || B * H * nch * N >= kMaxElems || L >= kMaxElems)
    return fail(SSM_ERR_UNSUPPORTED, "problem too large for 31-bit indexing");
  return SSM_OK;
}

int ssd_fwd_common(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim, int64_t ngroups,
                   int64_t dstate, int act, const void* x, const void* dt_raw, const float* dt_bias,
                   const float* A_log, const void* Bm, const void* Cm, const float* Dp, const float* h0,
                   void* y, float* h_last, void* chunk_states, const ssm_scan_options* opts, void* stream) {
  const int64_t B = batch, L = seqlen, H = nheads, P = headdim, G = ngroups, N = dstate;
  float dt_lo, dt_hi;
  S6_TRY(read_opts(opts, &dt_lo, &dt_hi));
  S6_TRY(check_ssd(B, L, H, P, G, N, act, "forward"));
  S6_TRY(need(x, B * L * H * P, 16, "x"));
  S6_TRY(need(dt_raw, B * L * H, 2, "dt_raw"));
  S6_TRY(need(dt_bias, H, 4, "dt_bias"));
  S6_TRY(need(A_log, H, 4, "A_log"));
  S6_TRY(need(Bm, B * L * G * N, 16, "Bm"));
  S6_TRY(need(Cm, B * L * G * N, 16, "Cm"));
  S6_TRY(need(Dp, H, 4, "Dp"));
  S6_TRY(opt(h0, 4, "h0"));
  S6_TRY(need(y, B * L * H * P, 16, "y"));
  S6_TRY(opt(h_last, 8, "h_last"));
  S6_TRY(opt(chunk_states, 16, "chunk_states"));
  g_last_error[0] = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (B == 0) return SSM_OK;
  if (L == 0) {
    if (h_last) {
      const size_t bytes = sizeof(float) * (size_t)(B * H * N * P);
      const cudaError_t ce = h0 ? cudaMemcpyAsync(h_last, h0, bytes, cudaMemcpyDeviceToDevice, st)
                                : cudaMemsetAsync(h_last, 0, bytes, st);
      if (ce != cudaSuccess) return cuda_fail(ce, "ssm_ssd_fwd(L=0)");
    }
    return SSM_OK;
  }
  s6::SsdArgs a = {};
  a.x = x; a.dt_raw = dt_raw; a.Bm = Bm; a.Cm = Cm; a.dt_bias = dt_bias; a.A_log = A_log; a.Dp = Dp;
  a.h0 = h0; a.y = y; a.h_last = h_last; a.chunk_states = chunk_states;
  a.status = s6::device_status_word();
  if (!a.status) return fail(SSM_ERR_CUDA, "cannot locate the device status word");
  a.dt_min = dt_lo; a.dt_max = dt_hi;
  a.B = (int)B; a.L = (int)L; a.H = (int)H; a.G = (int)G; a.N = (int)N; a.m = (int)std::max<int64_t>(P / 64, 1);
  a.w = (int)std::min<int64_t>(P, 64);
  const cudaError_t ce = s6::launch_ssd_fwd(a, st);
  return ce == cudaSuccess ? SSM_OK : cuda_fail(ce, "ssm_ssd_fwd launch");
}

int ssm_ssd_fwd(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim, int64_t ngroups,
                int64_t dstate, int act, const void* x, const void* dt_raw, const float* dt_bias,
                const float* A_log, const void* Bm, const void* Cm, const float* Dp, const float* h0,
                void* y, float* h_last, const ssm_scan_options* opts, void* stream) {
  return ssd_fwd_common(batch, seqlen, nheads, headdim, ngroups, dstate, act, x, dt_raw, dt_bias, A_log, Bm, Cm,
                        Dp, h0, y, h_last, nullptr, opts, stream);
}

int ssm_ssd_fwd_save(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim, int64_t ngroups,
                     int64_t dstate, int act, const void* x, const void* dt_raw, const float* dt_bias,
                     const float* A_log, const void* Bm, const void* Cm, const float* Dp, const float* h0,
                     void* y, float* h_last, void* chunk_states, const ssm_scan_options* opts, void* stream) {
  const int64_t nch = seqlen > 0 ? (seqlen + SSM_SSD_CHUNK_LEN - 1) / SSM_SSD_CHUNK_LEN : 0;
  S6_TRY(need(chunk_states, batch * nheads * nch * dstate * headdim, 16, "chunk_states"));
  return ssd_fwd_common(batch, seqlen, nheads, headdim, ngroups, dstate, act, x, dt_raw, dt_bias, A_log, Bm, Cm,
                        Dp, h0, y, h_last, chunk_states, opts, stream);
}

int64_t ssm_ssd_bwd_workspace_bytes(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim,
                                    int64_t ngroups, int64_t dstate, int act) {
  if (check_ssd(batch, seqlen, nheads, headdim, ngroups, dstate, act, "backward") != SSM_OK) return -1;
  return (int64_t)s6::ssd_bwd_workspace_bytes((int)batch, (int)seqlen, (int)nheads, (int)std::max<int64_t>(headdim / 64, 1),
                                              (int)ngroups, (int)dstate);
}

int ssm_ssd_bwd(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim, int64_t ngroups,
                int64_t dstate, int act, const void* x, const void* dt_raw, const float* dt_bias,
                const float* A_log, const void* Bm, const void* Cm, const float* Dp,
                const void* chunk_states, const void* dy, const float* dh_last, void* dx, void* ddt_raw,
                float* ddt_bias, float* dA_log, void* dBm, void* dCm, float* dDp, float* dh0, void* ws,
                size_t ws_bytes, const ssm_scan_options* opts, void* stream) {
  const int64_t B = batch, L = seqlen, H = nheads, P = headdim, G = ngroups, N = dstate;
  float dt_lo, dt_hi;
  S6_TRY(read_opts(opts, &dt_lo, &dt_hi));
  S6_TRY(check_ssd(B, L, H, P, G, N, act, "backward"));
  const int64_t nch = L > 0 ? (L + SSM_SSD_CHUNK_LEN - 1) / SSM_SSD_CHUNK_LEN : 0;
  S6_TRY(need(x, B * L * H * P, 16, "x"));
  S6_TRY(need(dt_raw, B * L * H, 2, "dt_raw"));
  S6_TRY(need(dt_bias, H, 4, "dt_bias"));
  S6_TRY(need(A_log, H, 4, "A_log"));
  S6_TRY(need(Bm, B * L * G * N, 16, "Bm"));
  S6_TRY(need(Cm, B * L * G * N, 16, "Cm"));
  S6_TRY(need(Dp, H, 4, "Dp"));
  S6_TRY(need(chunk_states, B * H * nch * N * P, 16, "chunk_states"));
  S6_TRY(need(dy, B * L * H * P, 16, "dy"));
  S6_TRY(opt(dh_last, 16, "dh_last"));
  S6_TRY(need(dx, B * L * H * P, 16, "dx"));
  S6_TRY(need(ddt_raw, B * L * H, 2, "ddt_raw"));
  S6_TRY(need(ddt_bias, H, 4, "ddt_bias"));
  S6_TRY(need(dA_log, H, 4, "dA_log"));
  S6_TRY(need(dBm, B * L * G * N, 2, "dBm"));
  S6_TRY(need(dCm, B * L * G * N, 2, "dCm"));
  S6_TRY(need(dDp, H, 4, "dDp"));
  S6_TRY(opt(dh0, 16, "dh0"));
  S6_TRY(check_ws(ws, ws_bytes, (int64_t)s6::ssd_bwd_workspace_bytes((int)B, (int)L, (int)H, (int)std::max<int64_t>(P / 64, 1), (int)G, (int)N)));
  g_last_error[0] = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t ce;
  if (B == 0 || L == 0) {
    // no steps: no gradient but the one passing straight through to h0
    ce = cudaMemsetAsync(ddt_bias, 0, sizeof(float) * H, st);
    if (ce == cudaSuccess) ce = cudaMemsetAsync(dA_log, 0, sizeof(float) * H, st);
    if (ce == cudaSuccess) ce = cudaMemsetAsync(dDp, 0, sizeof(float) * H, st);
    if (ce == cudaSuccess && dh0 && B > 0) {
      const size_t bytes = sizeof(float) * (size_t)(B * H * N * P);
      ce = dh_last ? cudaMemcpyAsync(dh0, dh_last, bytes, cudaMemcpyDeviceToDevice, st) : cudaMemsetAsync(dh0, 0, bytes, st);
    }
    return ce == cudaSuccess ? SSM_OK : cuda_fail(ce, "ssm_ssd_bwd(empty)");
  }
  s6::SsdBwdArgs a = {};
  a.f.x = x; a.f.dt_raw = dt_raw; a.f.Bm = Bm; a.f.Cm = Cm; a.f.dt_bias = dt_bias; a.f.A_log = A_log; a.f.Dp = Dp;
  a.f.chunk_states = const_cast<void*>(chunk_states);
  a.f.status = s6::device_status_word();
  if (!a.f.status) return fail(SSM_ERR_CUDA, "cannot locate the device status word");
  a.f.dt_min = dt_lo; a.f.dt_max = dt_hi;
  a.f.B = (int)B; a.f.L = (int)L; a.f.H = (int)H; a.f.G = (int)G; a.f.N = (int)N; a.f.m = (int)std::max<int64_t>(P / 64, 1);
  a.f.w = (int)std::min<int64_t>(P, 64);
  a.dy = dy; a.dh_last = dh_last; a.dx = dx; a.ddt_raw = ddt_raw; a.dBm = dBm; a.dCm = dCm;
  a.dA_log = dA_log; a.ddt_bias = ddt_bias; a.dDp = dDp; a.dh0 = dh0;
  a.ws = static_cast<float*>(ws);
  ce = s6::launch_ssd_bwd(a, st);
  return ce == cudaSuccess ? SSM_OK : cuda_fail(ce, "ssm_ssd_bwd launch");
}

int ssm_conv1d_step(int64_t batch, int64_t dim, int64_t width, int act, const void* x, const float* w,
                    const float* bias, void* state, void* out, void* stream) {
  const int64_t B = batch, D = dim, K = width;
  S6_TRY(check_conv(B, 1, D, K, act));
  const size_t e = act_size(act);
  S6_TRY(need(x, B * D, e, "x"));
  S6_TRY(need(w, D * K, 4, "w"));
  S6_TRY(need(bias, D, 4, "bias"));
  S6_TRY(need(state, K > 1 ? B * D * (K - 1) : 0, e, "state"));
  S6_TRY(need(out, B * D, e, "out"));
  g_last_error[0] = 0;
  if (B == 0 || D == 0) return SSM_OK;
  s6::ConvParams p = {};
  p.x = x; p.w = w; p.bias = bias; p.state_last = state; p.out = out;
  p.B = (int)B; p.L = 1; p.D = (int)D; p.K = (int)K;
  const cudaError_t ce = s6::launch_conv1d_step(p, act, static_cast<cudaStream_t>(stream));
  return ce == cudaSuccess ? SSM_OK : cuda_fail(ce, "ssm_conv1d_step launch");
}

}  // extern "C"
