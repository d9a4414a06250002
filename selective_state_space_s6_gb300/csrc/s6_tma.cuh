// TMA (cp.async.bulk.tensor), mbarrier and packed-f32 helpers for sm_103a,
// written as inline PTX.  Every wait is bounded: a wait that runs out sets a
// bit in the library's device status word and returns false, and the caller
// leaves its loop (see ssm_check_device_status()).
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace s6 {

// Bits of the library's device status word (see ssm_check_device_status);
// kernels receive the word's address as a parameter.
constexpr unsigned int kStatusWaitTimeout = 1u;
// a kernel found its shared-memory layout unusable (a swizzled TMA tile not
// on a 1024-byte boundary) and did no work
constexpr unsigned int kStatusLayout = 2u;
// about 2 s at 2 GHz; a healthy pipeline waits microseconds
constexpr long long kWaitCycles = 4000000000LL;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete; after ~2 s give up,
// set kStatusWaitTimeout in *status and return false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitCycles) {
      atomicOr(status, kStatusWaitTimeout);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2D tiled TMA load of the box at (x = inner coordinate, y = row) into smem,
// completing `bytes` transaction bytes on `bar`.  x must be a multiple of
// 16 bytes / element size (it always is: x is a multiple of the 64-channel tile).
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---- packed f32x2 arithmetic (one instruction for two lanes' worth of FP32 work)

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// 2^x on the special-function unit (the hardware instruction, ~2 ulp).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Shared-memory image of a [kRows][kCh] activation tile delivered by TMA
// boxes of at most 128 bytes per row (kNBox boxes of kChBox channels side by
// side) with the swizzle of the box row width (128, 64 or 32 bytes): in each
// byte offset the 16-byte unit index (bits 4..) is XORed with the 128-byte
// line index (bits 7..), masked to the row width.  The lanes of a channel
// read different rows at once; the XOR spreads those rows over the banks.
// Tiles start on a 1024-byte boundary.
template <typename Act, int kCh, int kRows>
struct SwzTile {
  static constexpr int kE = (int)sizeof(Act);
  static constexpr int kRowB = kCh * kE < 128 ? kCh * kE : 128;  // bytes per box row
  static constexpr int kChBox = kRowB / kE;                       // channels per box
  static constexpr int kNBox = kCh / kChBox;
  static constexpr int kBoxBytes = kRows * kRowB;
  static constexpr int kMask = kRowB / 16 - 1;  // 7 (128 B), 3 (64 B), 1 (32 B)
  static_assert(kRowB >= 32 && kCh % kChBox == 0 && kBoxBytes % 1024 == 0, "unsupported swizzled tile");
  __host__ __device__ static constexpr int swz(int o) { return o ^ (((o >> 7) & kMask) << 4); }
  // byte offset of (row, channel)
  __host__ __device__ static constexpr int off(int row, int ch) {
    return swz((ch / kChBox) * kBoxBytes + row * kRowB + (ch % kChBox) * kE);
  }
  // off(row, ch) - row * kRowB, which depends on row % 8 only
  __host__ __device__ static constexpr int col(int row, int ch) { return off(row & 7, ch) - (row & 7) * kRowB; }
};

// tensor-map swizzle mode matching SwzTile's box row width
inline CUtensorMapSwizzle swizzle_for_row_bytes(int row_bytes) {
  return row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
         : row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                           : CU_TENSOR_MAP_SWIZZLE_32B;
}

}  // namespace s6
