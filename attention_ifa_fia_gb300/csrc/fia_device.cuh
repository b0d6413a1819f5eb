// fia_device.cuh -- device-side helpers shared by the attention kernels.
//
// Inline PTX wrappers for mbarriers, bulk/tensor TMA copies, named barriers
// and tcgen05, the fp32 antiquant step, storage-format conversions, and the
// device status word that bounded waits write when they give up.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "fia_internal.h"

namespace fia {

// ----------------------------------------------------------------------------
// Device status word.  Kernels OR bits into it instead of trapping; the host
// reads and clears it through fia_device_status().  Every kernel receives its
// address as a parameter.
// ----------------------------------------------------------------------------
__device__ __forceinline__ void raise_status(unsigned int* status, unsigned int bits) {
  if (status) atomicOr(status, bits);
}

// Bounded waits give up after this many SM clock cycles (about one second).
constexpr long long kWaitLimitCycles = 2000000000LL;

// ----------------------------------------------------------------------------
// Shared-memory addresses and mbarriers
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete.  Returns false (and
// raises kStatusWaitTimeout) if it has not completed within kWaitLimitCycles.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitLimitCycles) {
      raise_status(status, kStatusWaitTimeout);
      return false;
    }
  }
  return true;
}

// ----------------------------------------------------------------------------
// TMA: tiled tensor loads and plain bulk copies, completing on an mbarrier
// ----------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* m, int32_t c0, int32_t c1,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* m, int32_t c0, int32_t c1, int32_t c2,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// 1-D bulk copy global -> shared; both addresses 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ----------------------------------------------------------------------------
// Named barriers (id 0 is __syncthreads)
// ----------------------------------------------------------------------------
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ----------------------------------------------------------------------------
// Shared loads
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// Byte offset inside a TMA box written with the 128-byte (mask 7) or 64-byte
// (mask 3) swizzle: the 16-byte chunk index is XORed with address bits 7 and up.
__device__ __forceinline__ uint32_t swz(uint32_t off, uint32_t mask) { return off ^ (((off >> 7) & mask) << 4); }

// ----------------------------------------------------------------------------
// Storage-format conversions (exact widenings)
// ----------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }
__device__ __forceinline__ float f16lo(uint32_t x) { return __half2float(__ushort_as_half((unsigned short)(x & 0xffff))); }
__device__ __forceinline__ float f16hi(uint32_t x) { return __half2float(__ushort_as_half((unsigned short)(x >> 16))); }

// int8 code (byte i of x, two's complement) -> exact fp32, via the 2^23 magic.
__device__ __forceinline__ float i8_to_f32(uint32_t x, int i) {
  const uint32_t u = ((x >> (8 * i)) ^ 0x80u) & 0xffu;           // code + 128 in [0, 255]
  return __fsub_rn(__uint_as_float(0x4B000000u | u), 8388736.0f);  // (2^23 + u) - (2^23 + 128)
}

// Per-channel antiquant of one code: fl(fl(x - offset) * scale), two separate
// round-to-nearest fp32 operations, never contracted into an FMA.  The same
// function serves the attention kernels and the fia_debug_dequant probe.
__device__ __forceinline__ float dequant_i8(float x, float offset, float scale) {
  return __fmul_rn(__fsub_rn(x, offset), scale);
}

// Round-to-nearest-even stores of fp32 into the output storage types.
template <int DT>
__device__ __forceinline__ void store_out(void* base, int64_t idx, float v);
template <>
__device__ __forceinline__ void store_out<kF32>(void* base, int64_t idx, float v) {
  static_cast<float*>(base)[idx] = v;
}
template <>
__device__ __forceinline__ void store_out<kF16>(void* base, int64_t idx, float v) {
  static_cast<__half*>(base)[idx] = __float2half_rn(v);
}
template <>
__device__ __forceinline__ void store_out<kBF16>(void* base, int64_t idx, float v) {
  static_cast<__nv_bfloat16*>(base)[idx] = __float2bfloat16_rn(v);
}

template <int DT>
__device__ __forceinline__ float load_elem(const void* base, int64_t idx);
template <>
__device__ __forceinline__ float load_elem<kF32>(const void* base, int64_t idx) {
  return static_cast<const float*>(base)[idx];
}
template <>
__device__ __forceinline__ float load_elem<kF16>(const void* base, int64_t idx) {
  return __half2float(static_cast<const __half*>(base)[idx]);
}
template <>
__device__ __forceinline__ float load_elem<kBF16>(const void* base, int64_t idx) {
  return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[idx]);
}

}  // namespace fia
