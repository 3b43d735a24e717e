// kvq_tc.cuh -- tcgen05 / TMA helpers shared by the tensor-core kernels over the paged 8-bit pool:
// TMA boxes of the code pool, tcgen05.mma issue and commit, shared-memory matrix descriptors, tensor
// memory loads and stores, and the host-side tensor-map encoder.
#pragma once
#include <cuda.h>  // CUtensorMap and its enums (the encoder is fetched from the driver at run time)
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "kvq_device.cuh"

namespace kvq {

// TMA tile load of one box of the code pool: the 128-byte slice `slice` of the rows `row`..`row+15`
// (row = kv head * 16 + token) of K (kv = 0) or V (kv = 1) in physical page `page`, completing on `bar`.
__device__ __forceinline__ void tma_load_codes(uint32_t dst, const CUtensorMap* map, int slice, int row, int kv,
                                               int page, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, "
      "%6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(slice), "r"(row), "r"(kv), "r"(page), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// The MMA and commit helpers are warp-collective: all 32 lanes of the converged MMA warp call them with the
// same operands and the lane chosen by elect.sync issues, so the descriptors stay in uniform registers (an
// elected issue beat a lane-0 branch).  The full mask elects the same lane every time, so a commit tracks
// every MMA issued before it.
__device__ __forceinline__ void mma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                                uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // descriptor version for tcgen05; no swizzle, base offset 0
  return d;
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// Eight MMAs of one accumulator chain from a single elect.sync: k-step k reads A at a + k * a_step and B at
// b + k * b_step (descriptor units); the first accumulates when acc_first is nonzero, the rest always.  Below
// N = 128 an MMA costs mostly its issue (elect.sync and predicate set-up), so grouping them took a probe of
// 64 dependent MMAs at N = 16 from 42 to 11 clocks each with A in tensor memory and from 58 to 40 with both
// operands in shared memory.
__device__ __forceinline__ void mma8_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint32_t a_step, uint64_t b,
                                                 uint64_t b_step, uint32_t idesc, uint32_t acc_first) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b32 a1, a2, a3, a4, a5, a6, a7;\n\t"
      ".reg .b64 b1, b2, b3, b4, b5, b6, b7;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "add.u32 a1, %1, %5;\n\tadd.u32 a2, a1, %5;\n\tadd.u32 a3, a2, %5;\n\tadd.u32 a4, a3, %5;\n\t"
      "add.u32 a5, a4, %5;\n\tadd.u32 a6, a5, %5;\n\tadd.u32 a7, a6, %5;\n\t"
      "add.u64 b1, %2, %6;\n\tadd.u64 b2, b1, %6;\n\tadd.u64 b3, b2, %6;\n\tadd.u64 b4, b3, %6;\n\t"
      "add.u64 b5, b4, %6;\n\tadd.u64 b6, b5, %6;\n\tadd.u64 b7, b6, %6;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %3, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %3, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a4], b4, %3, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a5], b5, %3, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a6], b6, %3, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a7], b7, %3, 1;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc_first), "r"(a_step), "l"(b_step)
      : "memory");
}

__device__ __forceinline__ void mma8_bf16(uint32_t d_tmem, uint64_t a, uint64_t a_step, uint64_t b, uint64_t b_step,
                                          uint32_t idesc, uint32_t acc_first) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b64 a1, a2, a3, a4, a5, a6, a7, b1, b2, b3, b4, b5, b6, b7;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "add.u64 a1, %1, %5;\n\tadd.u64 a2, a1, %5;\n\tadd.u64 a3, a2, %5;\n\tadd.u64 a4, a3, %5;\n\t"
      "add.u64 a5, a4, %5;\n\tadd.u64 a6, a5, %5;\n\tadd.u64 a7, a6, %5;\n\t"
      "add.u64 b1, %2, %6;\n\tadd.u64 b2, b1, %6;\n\tadd.u64 b3, b2, %6;\n\tadd.u64 b4, b3, %6;\n\t"
      "add.u64 b5, b4, %6;\n\tadd.u64 b6, b5, %6;\n\tadd.u64 b7, b6, %6;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a2, b2, %3, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a3, b3, %3, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a4, b4, %3, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a5, b5, %3, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a6, b6, %3, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a7, b7, %3, 1;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc_first), "l"(a_step), "l"(b_step)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// The first 8 columns only (32x32b.x8): what a group of at most 8 heads needs, in half the registers.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const float (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
               "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
               "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
               "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
               : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// N = 8 or 16 columns of one lane quarter.
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[N]) {
  static_assert(N == 8 || N == 16, "8 or 16 columns");
  if constexpr (N == 8) tmem_ld8(taddr, v);
  else tmem_ld16(taddr, v);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]);

template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const float (&v)[N]) {
  static_assert(N == 8 || N == 16, "8 or 16 columns");
  if constexpr (N == 8) tmem_st8(taddr, v);
  else tmem_st16(taddr, v);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
      "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
      "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once through the runtime (no link against libcuda).
inline EncodeTiledFn tensor_map_encoder() {
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// 5-D view of the code pool [page][kv][head][token][D] as (128-byte slice offset, slice, head*16 + token,
// kv, page); a box is one slice of the 16 rows of one head, of K or of V: 2 KB, 128-byte swizzled.
inline bool encode_code_map(CUtensorMap* map, const uint8_t* codes, int64_t num_pages, int32_t num_kv_heads, int D) {
  const EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t H = static_cast<cuuint64_t>(num_kv_heads);
  const cuuint64_t pages = static_cast<cuuint64_t>(std::max<int64_t>(num_pages, 1));  // no copy reads past it
  const cuuint64_t dims[5] = {128, static_cast<cuuint64_t>(D / 128), H * kPage, 2, pages};
  const cuuint64_t Dc = static_cast<cuuint64_t>(D);
  const cuuint64_t strides[4] = {128, Dc, H * kPage * Dc, 2 * H * kPage * Dc};
  const cuuint32_t box[5] = {128, 1, kPage, 1, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<uint8_t*>(codes), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace kvq
