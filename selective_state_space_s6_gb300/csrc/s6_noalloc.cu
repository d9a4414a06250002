// ssm_scan_bwd_noalloc: the backward scan for callers that cannot allocate
// device memory.
//
// ssm_scan_bwd needs a scratch buffer (`ws`) for its per-tile and per-batch
// partial sums, which its caller normally allocates.  Some callers cannot do
// that: code running inside a host framework that owns the device allocator
// and forbids raw cudaMalloc, plugin interfaces that hand over only input and
// output pointers, and latency-critical loops that must not allocate (or
// synchronise, as cudaMalloc/cudaFree may) at all.  For them this entry point
// takes its scratch from a fixed array that is part of the library image: it
// is reserved on every GPU that loads the library and stays there until the
// process exits.  Nothing is allocated or freed per call.
//
// Limits and rules (also in include/ssm_scan.h):
//   - the scratch holds kNoAllocScratchBytes (16 MiB); a shape whose
//     ssm_bwd_workspace_bytes() exceeds that is rejected with
//     SSM_ERR_UNSUPPORTED before anything is enqueued;
//   - the first call on a device looks the array's device address up
//     (cudaGetSymbolAddress) with that device current, and so does the first
//     call after the device's context was reset (cudaDeviceReset reloads the
//     library's device image); make those calls before any stream capture;
//   - every call on a device shares the one array, which keeps the last
//     call's contents: calls whose GPU work overlaps (different streams
//     without ordering between them) race on it.  Nothing in the array has
//     to start at zero: the backward writes every partial it later reads.
#include <mutex>

#include "s6_internal.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

s6::SymbolCache g_scratch_cache;

// Device address of g_noalloc_scratch on the current device.  In host code
// the symbol names a host-side stand-in, not device memory, so kernels must
// only ever be given this looked-up address.  It is looked up once per device
// (and again if the device's context was reset since, as the array may then
// have moved).
cudaError_t scratch_address(void** out) { return s6::symbol_address(g_scratch_cache, &g_noalloc_scratch, out); }

}  // namespace

extern "C" {

size_t ssm_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

int ssm_scan_bwd_noalloc(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, int act,
                         const void* u, const void* delta_raw, const void* z, const void* Bm,
                         const void* Cm, const float* A_log, const float* Dp,
                         const float* delta_bias, const float* h0, const float* chunk_states,
                         const void* dout, const float* dh_last, void* du, void* d_delta_raw,
                         void* dz, void* dBm, void* dCm, float* dA_log, float* dDp,
                         float* d_delta_bias, float* dh0, void* stream) {
  const int64_t need = ssm_bwd_workspace_bytes(batch, seqlen, dim, dstate, act);
  if (need < 0) {
    // invalid shape: let the regular entry point report which argument
    return ssm_scan_bwd(batch, seqlen, dim, dstate, act, u, delta_raw, z, Bm, Cm, A_log, Dp,
                        delta_bias, h0, chunk_states, dout, dh_last, du, d_delta_raw, dz, dBm,
                        dCm, dA_log, dDp, d_delta_bias, dh0, nullptr, 0, stream);
  }
  if ((size_t)need > kNoAllocScratchBytes)
    return s6::report_error(SSM_ERR_UNSUPPORTED,
                            "ssm_scan_bwd_noalloc: this shape needs %lld bytes of scratch, more than "
                            "the fixed %zu bytes; use ssm_scan_bwd with a caller buffer",
                            (long long)need, kNoAllocScratchBytes);
  void* ws = nullptr;
  const cudaError_t e = scratch_address(&ws);
  if (e != cudaSuccess)
    return s6::report_error(SSM_ERR_CUDA, "ssm_scan_bwd_noalloc: cudaGetSymbolAddress: %s",
                            cudaGetErrorString(e));
  return ssm_scan_bwd(batch, seqlen, dim, dstate, act, u, delta_raw, z, Bm, Cm, A_log, Dp,
                      delta_bias, h0, chunk_states, dout, dh_last, du, d_delta_raw, dz, dBm, dCm,
                      dA_log, dDp, d_delta_bias, dh0, ws, kNoAllocScratchBytes, stream);
}

}  // extern "C"
