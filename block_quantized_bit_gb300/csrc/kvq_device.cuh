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
#include <string.h>

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
constexpr uint32_t kStatusBadExtend = 0x7300u;  // q_start inconsistent with seq_lens or total_q

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

// Non-blocking probe: has phase `parity` of `bar` completed?
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
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

// q8_0 codes: round half away from zero, clamp to +-127, in two steps.
// (1) q8_trunc_code: truncating y + copysign(0.5 - 2^-25, y) toward zero rounds half away from zero exactly
//     (the fp32 sum is correctly rounded).  At a tie k + 0.5 the sum k + 1 - 2^-25 rounds up to k + 1 (for
//     k = 0 it is the midpoint below 1, which goes to the even 1.0).  Just below a tie the sum stays below
//     k + 1, because its distance to k + 1 exceeds half an ulp there; and 0.5 - 2^-25 itself, whose sum
//     with 0.5 would round up to 1, gives 1 - 2^-24 with this offset, truncated to 0.  The sum is clamped
//     at -127.5 so that the negative side saturates at -127; infinities saturate in the conversion.
// (2) pack_q8x4: four such integers to int8 with saturation at +127 (cvt.pack.sat), element 0 in the
//     lowest byte.
// The kernels' quantize and encode probes compare this with the oracle's exact round-half-away on every
// bf16 value against every fp16 scale and on a dense fp32 sweep with every tie.
__device__ __forceinline__ int32_t q8_trunc_code(float y) {
  const float half_below = copysignf(__uint_as_float(0x3EFFFFFFu), y);  // 0.5 - 2^-25, signed as y
  return __float2int_rz(fmaxf(y + half_below, -127.5f));
}

__device__ __forceinline__ uint32_t pack_q8x4(int32_t e0, int32_t e1, int32_t e2, int32_t e3) {
  uint32_t hi, r;
  asm("cvt.pack.sat.s8.s32.b32 %0, %1, %2, 0;" : "=r"(hi) : "r"(e3), "r"(e2));
  asm("cvt.pack.sat.s8.s32.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(e1), "r"(e0), "r"(hi));
  return r;
}

// One q8_0 code (the probe's single-element form).
__device__ __forceinline__ uint8_t encode_q8(float y) {
  return static_cast<uint8_t>(pack_q8x4(q8_trunc_code(y), 0, 0, 0) & 0xFFu);
}

// --------------------------------------------------------------------------- decode dequantization
// Dequantize to bf16: kd = RNE_bf16(value(code) * s), where s is the block's fp16 scale.
//   1. the codes become exact f16 values: fp8 through the hardware E4M3 -> f16x2 conversion; q8_0
//      through the 1024-offset f16 pattern 0x6400 | (q + 128), whose offset is removed in step 2;
//   2. one mixed-precision FMA per element, f16 x f16 + f32 -> f32, forms code * s exactly (an
//      11-bit by 11-bit product fits fp32's 24 bits; for q8_0 the addend -1152 * s removes the offset
//      exactly, because (q + 1152) * s and 1152 * s are exact and the result q * s is representable);
//   3. one bf16x2 conversion rounds the pair to nearest-even.
// The result is packed bf16x2 (element 2p in the low half), exactly the bf16 numbers of the oracle.
__device__ __forceinline__ float fma_f32_bf16(uint16_t a, uint16_t b, float c) {
  float d;
  asm("fma.rn.f32.bf16 %0, %1, %2, %3;" : "=f"(d) : "h"(a), "h"(b), "f"(c));
  return d;
}

// bf16x2 of (lo, hi), round to nearest-even; lo lands in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Packed fp32 FMA on two lanes of a 64-bit register pair (d = a * b + c elementwise).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  uint64_t A, B, C, D;
  memcpy(&A, &a, 8);
  memcpy(&B, &b, 8);
  memcpy(&C, &c, 8);
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(D) : "l"(A), "l"(B), "l"(C));
  float2 d;
  memcpy(&d, &D, 8);
  return d;
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t v) {
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}

__device__ __forceinline__ uint16_t lo16(uint32_t v) { return static_cast<uint16_t>(v & 0xFFFFu); }
__device__ __forceinline__ uint16_t hi16(uint32_t v) { return static_cast<uint16_t>(v >> 16); }

// Kinds with one fp16 scale per 32 elements (a scale array beside the codes); the unscaled kinds
// ("Add fp8 KV-cache quantization (--kv-dtype)", section "How it works": the plain fp8 cast, scale 1.0)
// have codes only.
template <int KIND>
struct KindTraits {
  static constexpr bool kScaled = (KIND == KVQ_FP8_E4M3 || KIND == KVQ_Q8_0);
};

// fp16 bits of 1.0: the scale of every element of an unscaled pool.
constexpr uint16_t kHalfOne = 0x3C00u;

// Addend that completes step 2 for a block with fp16 scale bits s_bits.
template <int KIND>
__device__ __forceinline__ float dequant_addend(uint16_t s_bits) {
  if (KIND != KVQ_Q8_0) return -0.0f;
  return -1152.0f * __half2float(__ushort_as_half(s_bits));
}

// Exact f16 values of the four codes of a 32-bit word: lo = codes 0-1, hi = codes 2-3.  The 16-bit
// halves are taken with mov.b32 {l, h} inside the asm, so the conversions read register halves
// instead of shifted and masked copies.
// E5M2 codes are the upper byte of the binary16 of the same value (1 sign, 5 exponent bits with
// bias 15, the leading 2 fraction bits), so each code only moves into the high byte of a half.
template <int KIND>
__device__ __forceinline__ void codes_to_f16x2(uint32_t word, uint32_t& lo, uint32_t& hi) {
  if (KIND == KVQ_FP8_E4M3 || KIND == KVQ_FP8_E4M3_UNSCALED) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(word));
  } else if (KIND == KVQ_FP8_E5M2_UNSCALED) {
    lo = __byte_perm(word, 0u, 0x1404u);  // codes 0, 1 -> bytes 1, 3
    hi = __byte_perm(word, 0u, 0x3424u);  // codes 2, 3 -> bytes 1, 3
  } else {
    const uint32_t u = word ^ 0x80808080u;  // q + 128 in each byte
    lo = __byte_perm(u, 0x64646464u, 0x5140u);
    hi = __byte_perm(u, 0x64646464u, 0x5342u);
  }
}

// bf16x2 of RN(f16 pair * s + z) per half, each product formed exactly by the mixed-precision FMA.
__device__ __forceinline__ uint32_t scale_pack_bf16x2(uint32_t f16x2, uint16_t s_bits, float z) {
  uint32_t r;
  asm("{\n\t.reg .b16 l, h;\n\t.reg .f32 a, b;\n\tmov.b32 {l, h}, %1;\n\t"
      "fma.rn.f32.f16 a, l, %2, %3;\n\tfma.rn.f32.f16 b, h, %2, %3;\n\t"
      "cvt.rn.bf16x2.f32 %0, b, a;\n\t}"
      : "=r"(r)
      : "r"(f16x2), "h"(s_bits), "f"(z));
  return r;
}

// Dequantize 16 codes (one 16-byte chunk, one scale) into 8 bf16x2 words.  The unscaled kinds ignore
// s_bits: their values are the codes' own, exact in bf16 (the FMA by 1.0 and the bf16 rounding change
// nothing).
template <int KIND>
__device__ __forceinline__ void dequant16(const uint4 c, uint16_t s_bits, uint32_t kd[8]) {
  if (!KindTraits<KIND>::kScaled) s_bits = kHalfOne;
  const float z = dequant_addend<KIND>(s_bits);
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t lo, hi;
    codes_to_f16x2<KIND>(w[i], lo, hi);
    kd[2 * i] = scale_pack_bf16x2(lo, s_bits, z);
    kd[2 * i + 1] = scale_pack_bf16x2(hi, s_bits, z);
  }
}

__device__ __forceinline__ float half_bits_to_float(uint16_t h) {
  return __half2float(__ushort_as_half(h));
}

}  // namespace kvq
