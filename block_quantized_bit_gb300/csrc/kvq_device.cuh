// kvq_device.cuh -- device helpers shared by the libkvq kernels (sm_103a).
//
// Inline-PTX wrappers for mbarriers and 1-D bulk copies (TMA engine, no tensor map), the fp8/int8
// code conversions of the store, and the dequantization of the decode.  Conversions call CUDA's own
// intrinsics (cuda_fp8.h / cuda_bf16.h); nothing here re-implements a library routine.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "../../include/kvq.h"
#include "kvq_internal.h"

namespace kvq {

constexpr int kBlock = 32;              // elements per scale block
constexpr float kFp8Max = 448.0f;       // largest finite E4M3 value
constexpr float kQ8Max = 127.0f;        // int8 code range
constexpr float kScaleMax = 65504.0f;   // largest finite fp16
constexpr int kPage = kPageTokens;      // tokens per page supported by the decode kernels
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // bounded waits give up after 2 s

// Values a kernel writes to the workspace status word: it gave up a bounded wait; or a block-table
// entry pointed past the pool (that page was skipped).
constexpr uint32_t kStatusTimeout = 0x7100u;
constexpr uint32_t kStatusBadPage = 0x7200u;

// ------------------------------------------------------------------------------------------ PTX
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the async proxy (bulk copies complete on it).
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` to complete; gives up after kWaitLimitNs.  Returns false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// 1-D bulk copy global -> shared, completing `bytes` of transaction count on `bar`.
// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t code) {
  if (status) atomicExch(status, code);
}

// ------------------------------------------------------------------------------ store conversions
// fp16 block scale from the block's fp32 amax: fp16_RNE(min(amax / Q, 65504)), IEEE division.
template <int KIND>
__device__ __forceinline__ __half block_scale(float amax) {
  const float q = (KIND == KVQ_FP8_E4M3) ? kFp8Max : kQ8Max;
  float s = __fdiv_rn(amax, q);
  s = fminf(s, kScaleMax);
  return __float2half_rn(s);
}

// Two fp8 codes (low byte = a) of already-scaled values: clamp to +-448 and round once to nearest-even.
__device__ __forceinline__ uint16_t encode_fp8x2(float a, float b) {
  return static_cast<uint16_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

// One q8_0 code: round half away from zero, clamp to +-127.
__device__ __forceinline__ uint8_t encode_q8(float y) {
  float r = roundf(y);  // C semantics: halfway cases away from zero
  r = fminf(fmaxf(r, -kQ8Max), kQ8Max);
  return static_cast<uint8_t>(static_cast<int8_t>(static_cast<int>(r)));
}

// --------------------------------------------------------------------------- decode dequantization
// Value of one code pair as exact fp32 (fp8: via the hardware E4M3 -> f16 conversion, exact).
__device__ __forceinline__ float2 fp8x2_to_float2(uint16_t two) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two), __NV_E4M3);
  __half2 hh = *reinterpret_cast<__half2*>(&h);
  return __half22float2(hh);
}

// bf16 RNE of an exact fp32 product, returned widened back to fp32.
__device__ __forceinline__ float round_bf16(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

// Dequantize 16 codes (one 16-byte chunk) of one scale block into fp32 values that are exactly the
// bf16 numbers RNE(code * scale).  The code * scale product is exact in fp32 (<= 18 significant bits).
template <int KIND>
__device__ __forceinline__ void dequant16(const uint4 c, float scale, float out[16]) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (KIND == KVQ_FP8_E4M3) {
      float2 lo = fp8x2_to_float2(static_cast<uint16_t>(w[i] & 0xFFFFu));
      float2 hi = fp8x2_to_float2(static_cast<uint16_t>(w[i] >> 16));
      out[4 * i + 0] = round_bf16(lo.x * scale);
      out[4 * i + 1] = round_bf16(lo.y * scale);
      out[4 * i + 2] = round_bf16(hi.x * scale);
      out[4 * i + 3] = round_bf16(hi.y * scale);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int8_t q = static_cast<int8_t>((w[i] >> (8 * j)) & 0xFFu);
        out[4 * i + j] = round_bf16(static_cast<float>(q) * scale);
      }
    }
  }
}

__device__ __forceinline__ float half_bits_to_float(uint16_t h) {
  return __half2float(__ushort_as_half(h));
}

}  // namespace kvq
