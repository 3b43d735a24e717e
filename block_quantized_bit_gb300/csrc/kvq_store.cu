// kvq_store.cu -- quantize-and-scatter store of bf16 K/V rows into the 8-bit paged pool.
//
// "feat(kvcache): 8-bit KV cache (q8_0 / fp8_e4m3) behind --kv-cache-dtype", section "What" (the
// store kernel: per-block max-abs -> codes + scales, one fp16 scale per 32 elements along head_dim)
// and its review comment "A bug on sm_89" (int8 rounds half away from zero then clamps; fp8 clamps
// then rounds once to nearest-even -- never through a truncated fp16).
//
// Mapping: one lane owns one 32-element block (four 16-byte loads, 64 contiguous bytes).  The input
// is walked as a flat stream of blocks, K first then V; a warp covers 2 KiB of contiguous input per
// sweep.  The grid is persistent (four CTAs per SM) and every lane loads its next block while it
// quantizes the current one.  The lane computes amax, the fp16 scale, the 32 codes (two 16-byte
// stores) and the scale without any cross-lane traffic.
//
// Division.  The codes must be those of the IEEE fp32 quotient x / s.  Per block the lane takes
// r = RN(1/s) (IEEE reciprocal) once; per element it forms q0 = x*r, the exact remainder
// e = q0*s - x by FMA, and y = q0 - e*r (one Newton-Raphson step with an FMA remainder, Markstein,
// "Computation of elementary functions on the IBM RISC System/6000 processor", IBM J. Res. Dev.
// 34(1), 1990).  y is not the correctly rounded quotient for every (x, s), but its fp8 and q8_0 codes
// equal the codes of the IEEE quotient for every bf16 x and every fp16 s; the GPU test sweeps all of
// them through kvq_quantize_probe against the oracle's IEEE division.  The operand order keeps the
// sign of zero (x = -0 gives y = -0, code 0x80).
#include <algorithm>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

namespace {

constexpr int kStoreThreads = 256;
constexpr int kStoreCtasPerSm = 4;  // resident CTAs per SM (64 registers per thread)

// Unsigned division by a run-time constant d >= 1 via a multiply-high (Granlund & Montgomery,
// "Division by invariant integers using multiplication", PLDI 1994): q = (umulhi(n, m) + n) >> s,
// valid for n < 2^31.
struct FastDiv {
  uint32_t m, s, d;
};

FastDiv make_fastdiv(uint32_t d) {
  uint32_t s = 0;
  while ((1ull << s) < d) ++s;  // s = ceil(log2 d)
  const uint64_t m = ((1ull << 32) * ((1ull << s) - d)) / d + 1;
  return FastDiv{static_cast<uint32_t>(m), s, d};
}

__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv& f) {
  return (__umulhi(n, f.m) + n) >> f.s;
}

// Code step shared by the store kernel and kvq_quantize_probe.
__device__ __forceinline__ float quotient(float x, float s, float r) {
  const float q0 = x * r;
  const float e = fmaf(q0, s, -x);
  return fmaf(e, -r, q0);
}

template <int KIND>
__device__ __forceinline__ uint32_t encode4(float a, float b, float c, float d) {
  if (KIND == KVQ_FP8_E4M3) {
    return static_cast<uint32_t>(encode_fp8x2(a, b)) | (static_cast<uint32_t>(encode_fp8x2(c, d)) << 16);
  } else {
    return pack_q8x4(q8_trunc_code(a), q8_trunc_code(b), q8_trunc_code(c), q8_trunc_code(d));
  }
}

struct StoreArgs {
  uint8_t* codes;
  __half* scales;
  const uint4* k;
  const uint4* v;
  const int64_t* slot_mapping;
  int32_t blocks_per_kv;  // T * Hkv * nb
  int32_t total;          // blocks_per_kv * n_kv  (< 2^31)
  FastDiv row_blocks;     // Hkv * nb
  FastDiv nb;             // blocks per row of one head
  int32_t Hkv, D, n_kv;
  int32_t page_shift;     // log2(page_size) if a power of two, else -1
  int32_t P;
  int64_t num_slots;
};

// Load one 32-element block (64 contiguous bytes: four 16-byte pieces) of the flat K-then-V stream.
__device__ __forceinline__ void load_block(const StoreArgs& a, int32_t blk, uint4 (&x)[4]) {
  const int kv = blk >= a.blocks_per_kv;
  const int32_t local = blk - (kv ? a.blocks_per_kv : 0);
  const uint4* src = (kv ? a.v : a.k) + static_cast<int64_t>(local) * 4;
#pragma unroll
  for (int i = 0; i < 4; ++i) x[i] = __ldcs(src + i);
}

// amax, fp16 scale, codes and scatter of one block whose bf16 values are in x.
template <int KIND>
__device__ __forceinline__ void store_block(const StoreArgs& a, int32_t blk, const uint4 (&x)[4]) {
  const int kv = blk >= a.blocks_per_kv;
  const uint32_t local = static_cast<uint32_t>(blk - (kv ? a.blocks_per_kv : 0));
  const uint32_t t = fdiv(local, a.row_blocks);
  const uint32_t in_row = local - t * a.row_blocks.d;
  const uint32_t h = fdiv(in_row, a.nb);
  const uint32_t j = in_row - h * a.nb.d;
  const int64_t slot = __ldg(a.slot_mapping + t);
  if (slot < 0 || slot >= a.num_slots) return;  // -1 skips; out-of-range slots are never written
  int64_t page, off;
  if (a.page_shift >= 0) {
    page = slot >> a.page_shift;
    off = slot & (a.P - 1);
  } else {
    page = slot / a.P;
    off = slot - page * a.P;
  }
  const int64_t dst_row = ((page * a.n_kv + kv) * a.Hkv + h) * a.P + off;
  const uint32_t w[16] = {x[0].x, x[0].y, x[0].z, x[0].w, x[1].x, x[1].y, x[1].z, x[1].w,
                          x[2].x, x[2].y, x[2].z, x[2].w, x[3].x, x[3].y, x[3].z, x[3].w};
  // bf16 pair (lo, hi) of word e: lo = w << 16, hi = w & 0xFFFF0000 as fp32 bit patterns
  float amax = 0.0f;
#pragma unroll
  for (int e = 0; e < 16; ++e)
    amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[e] << 16)), fabsf(__uint_as_float(w[e] & 0xFFFF0000u))));
  const __half s16 = block_scale<KIND>(amax);
  const float sf = __half2float(s16);
  uint32_t o[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
  if (sf != 0.0f) {
    const float r = __frcp_rn(sf);
#pragma unroll
    for (int q = 0; q < 8; ++q)  // four elements (two words) per code word
      o[q] = encode4<KIND>(quotient(__uint_as_float(w[2 * q] << 16), sf, r),
                           quotient(__uint_as_float(w[2 * q] & 0xFFFF0000u), sf, r),
                           quotient(__uint_as_float(w[2 * q + 1] << 16), sf, r),
                           quotient(__uint_as_float(w[2 * q + 1] & 0xFFFF0000u), sf, r));
  }
  uint4* dst = reinterpret_cast<uint4*>(a.codes + dst_row * a.D + (static_cast<int64_t>(j) << 5));
  __stcs(dst, make_uint4(o[0], o[1], o[2], o[3]));
  __stcs(dst + 1, make_uint4(o[4], o[5], o[6], o[7]));
  a.scales[dst_row * (a.D >> 5) + j] = (sf != 0.0f) ? s16 : __ushort_as_half(0);
}

// Persistent grid-stride store: a few CTAs per SM stay resident and every thread loads its next block
// while it quantizes the current one, so the input stream never waits for a wave of CTAs to finish.
template <int KIND>
__global__ void __launch_bounds__(kStoreThreads, kStoreCtasPerSm) store_kernel(StoreArgs a) {
  const int32_t stride = gridDim.x * kStoreThreads;
  int32_t blk = blockIdx.x * kStoreThreads + threadIdx.x;
  if (blk >= a.total) return;
  uint4 x[4];
  load_block(a, blk, x);
  for (; blk < a.total; blk += stride) {
    uint4 nx[4] = {x[0], x[1], x[2], x[3]};
    if (blk + stride < a.total) load_block(a, blk + stride, nx);
    store_block<KIND>(a, blk, x);
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = nx[i];
  }
}

template <int KIND>
__global__ void encode_probe_kernel(const float* __restrict__ y, uint8_t* __restrict__ codes, int64_t n) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t e = i; e < n; e += stride) {
    if (KIND == KVQ_FP8_E4M3)
      codes[e] = static_cast<uint8_t>(encode_fp8x2(y[e], 0.0f) & 0xFFu);
    else
      codes[e] = encode_q8(y[e]);
  }
}

// codes[i * nx + j] = code of x[j] against the nonzero fp16 scale s[i], by the store's own routine.
template <int KIND>
__global__ void quantize_probe_kernel(const uint16_t* __restrict__ x, int64_t nx, const uint16_t* __restrict__ s,
                                      int64_t ns, uint8_t* __restrict__ codes) {
  const int64_t n = nx * ns;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < n; e += stride) {
    const int64_t i = e / nx, j = e - i * nx;
    const float sf = half_bits_to_float(s[i]);
    const float xf = __uint_as_float(static_cast<uint32_t>(x[j]) << 16);
    const float y = quotient(xf, sf, __frcp_rn(sf));
    codes[e] = static_cast<uint8_t>(encode4<KIND>(y, 0.0f, 0.0f, 0.0f) & 0xFFu);
  }
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 152;
  return n;
}

}  // namespace

kvq_status launch_store(void* pool, void* scales, const void* k, const void* v, const int64_t* slot_mapping,
                        int64_t num_tokens, const kvq_layout& L, kvq_kind kind, cudaStream_t stream) {
  const int n_kv = L.mla ? 1 : 2;
  const int32_t nb = L.head_dim / 32;
  const int64_t row_blocks = static_cast<int64_t>(L.num_kv_heads) * nb;
  const int64_t max_rows = std::max<int64_t>(1, ((int64_t(1) << 30) / (row_blocks * n_kv)));
  const int64_t row_elems = static_cast<int64_t>(L.num_kv_heads) * L.head_dim;
  const int sms = sm_count();
  int page_shift = -1;
  for (int s = 0; s < 31; ++s)
    if ((1 << s) == L.page_size) page_shift = s;
  for (int64_t t0 = 0; t0 < num_tokens; t0 += max_rows) {
    const int64_t T = std::min(max_rows, num_tokens - t0);
    StoreArgs a;
    a.codes = static_cast<uint8_t*>(pool);
    a.scales = static_cast<__half*>(scales);
    a.k = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(k) + t0 * row_elems);
    a.v = v ? reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(v) + t0 * row_elems) : nullptr;
    a.slot_mapping = slot_mapping + t0;
    a.blocks_per_kv = static_cast<int32_t>(T * row_blocks);
    a.total = a.blocks_per_kv * n_kv;
    a.row_blocks = make_fastdiv(static_cast<uint32_t>(row_blocks));
    a.nb = make_fastdiv(static_cast<uint32_t>(nb));
    a.Hkv = L.num_kv_heads;
    a.D = L.head_dim;
    a.n_kv = n_kv;
    a.page_shift = page_shift;
    a.P = L.page_size;
    a.num_slots = L.num_pages * L.page_size;
    int64_t grid = (static_cast<int64_t>(a.total) + kStoreThreads - 1) / kStoreThreads;
    grid = std::max<int64_t>(1, std::min<int64_t>(grid, static_cast<int64_t>(sms) * kStoreCtasPerSm));
    if (kind == KVQ_FP8_E4M3)
      store_kernel<KVQ_FP8_E4M3><<<static_cast<unsigned>(grid), kStoreThreads, 0, stream>>>(a);
    else
      store_kernel<KVQ_Q8_0><<<static_cast<unsigned>(grid), kStoreThreads, 0, stream>>>(a);
    if (cudaGetLastError() != cudaSuccess) return KVQ_ECUDA;
  }
  return KVQ_OK;
}

kvq_status launch_encode_probe(kvq_kind kind, const float* y, uint8_t* codes, int64_t n, cudaStream_t stream) {
  if (n == 0) return KVQ_OK;
  const int threads = 256;
  const int64_t grid = std::min<int64_t>((n + threads - 1) / threads, static_cast<int64_t>(sm_count()) * 16);
  if (kind == KVQ_FP8_E4M3)
    encode_probe_kernel<KVQ_FP8_E4M3><<<static_cast<unsigned>(grid), threads, 0, stream>>>(y, codes, n);
  else
    encode_probe_kernel<KVQ_Q8_0><<<static_cast<unsigned>(grid), threads, 0, stream>>>(y, codes, n);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ECUDA;
}

kvq_status launch_quantize_probe(kvq_kind kind, const uint16_t* x, int64_t nx, const uint16_t* s, int64_t ns,
                                 uint8_t* codes, cudaStream_t stream) {
  const int64_t n = nx * ns;
  if (n == 0) return KVQ_OK;
  const int threads = 256;
  const int64_t grid = std::min<int64_t>((n + threads - 1) / threads, static_cast<int64_t>(sm_count()) * 16);
  if (kind == KVQ_FP8_E4M3)
    quantize_probe_kernel<KVQ_FP8_E4M3><<<static_cast<unsigned>(grid), threads, 0, stream>>>(x, nx, s, ns, codes);
  else
    quantize_probe_kernel<KVQ_Q8_0><<<static_cast<unsigned>(grid), threads, 0, stream>>>(x, nx, s, ns, codes);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ECUDA;
}

}  // namespace kvq

// ------------------------------------------------------------------------ the store fused with act_quant
// "feat(kvcache): 8-bit DSV4 window/compressed KV", section "Why the precision cost is small": the model
// rounds each MLA latent row onto the E4M3 grid with one scale per 64 elements immediately before every
// store (the rope tail stays bf16).  Fused here: one thread takes one 64-element unit of a row, rounds it
// in registers when it belongs to the latent (fp32 scale amax / 448, code = E4M3 of x / s by IEEE
// division, value = code * s in fp32, rounded to bf16; an all-zero unit stays as it is), and stores the
// unit's two 32-element blocks exactly as the plain store does.  One pass over the bf16 rows instead of a
// rounding pass that reads and writes them and then the store.
namespace kvq {
namespace {

struct ActQuantStoreArgs {
  uint8_t* codes;
  __half* scales;
  const uint4* kv;             // bf16 rows [T][D]
  const int64_t* slot_mapping;
  int64_t num_tokens;
  int32_t D, latent, P;        // latent = D - rope_dim: the rounded part (a multiple of 64)
  int64_t num_slots;
};

template <int KIND>
__global__ void __launch_bounds__(256) act_quant_store_kernel(ActQuantStoreArgs a) {
  const int32_t units = a.D / 64;
  const int64_t n = a.num_tokens * units;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u < n; u += stride) {
    const int64_t t = u / units;
    const int32_t c = static_cast<int32_t>(u - t * units);
    const int64_t slot = __ldg(a.slot_mapping + t);
    if (slot < 0 || slot >= a.num_slots) continue;  // -1 skips; out-of-range slots are never written
    float f[64];
    const uint4* src = a.kv + (t * a.D + c * 64) / 8;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint4 x = __ldcs(src + i);
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        f[8 * i + 2 * e] = __uint_as_float(w[e] << 16);
        f[8 * i + 2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
      }
    }
    if (c * 64 < a.latent) {
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 64; ++i) amax = fmaxf(amax, fabsf(f[i]));
      if (amax != 0.0f) {
        const float s = __fdiv_rn(amax, kFp8Max);
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
          const uint16_t pair = encode_fp8x2(__fdiv_rn(f[i], s), __fdiv_rn(f[i + 1], s));
          const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(pair), __NV_E4M3);
          f[i] = __bfloat162float(__float2bfloat16_rn(__fmul_rn(__half2float(__ushort_as_half(h.x)), s)));
          f[i + 1] = __bfloat162float(__float2bfloat16_rn(__fmul_rn(__half2float(__ushort_as_half(h.y)), s)));
        }
      }
    }
    const int64_t page = slot / a.P, off = slot - (slot / a.P) * a.P;
    const int64_t dst_row = page * a.P + off;  // one latent row per token: n_kv = 1, one kv head
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const float* g = f + 32 * half;
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(g[i]));
      const __half s16 = block_scale<KIND>(amax);
      const float sf = __half2float(s16);
      uint32_t o[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
      if (sf != 0.0f) {
        const float r = __frcp_rn(sf);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          o[q] = encode4<KIND>(quotient(g[4 * q], sf, r), quotient(g[4 * q + 1], sf, r), quotient(g[4 * q + 2], sf, r),
                               quotient(g[4 * q + 3], sf, r));
      }
      const int32_t j = 2 * c + half;  // 32-element block of the row
      uint4* dst = reinterpret_cast<uint4*>(a.codes + dst_row * a.D + static_cast<int64_t>(j) * 32);
      __stcs(dst, make_uint4(o[0], o[1], o[2], o[3]));
      __stcs(dst + 1, make_uint4(o[4], o[5], o[6], o[7]));
      a.scales[dst_row * (a.D / 32) + j] = (sf != 0.0f) ? s16 : __ushort_as_half(0);
    }
  }
}

}  // namespace
}  // namespace kvq

extern "C" kvq_status kvq_store_act_quant(void* pool, void* scales, const void* kv, const int64_t* slot_mapping,
                                          int64_t num_tokens, int32_t rope_dim, const kvq_layout* layout,
                                          kvq_kind kind, void* stream) {
  using namespace kvq;
  if (!layout) return KVQ_EINVAL;
  if (kind != KVQ_FP8_E4M3 && kind != KVQ_Q8_0) return KVQ_EKIND;
  if (!layout->mla || layout->num_kv_heads != 1 || layout->num_pages < 0 || layout->page_size <= 0)
    return KVQ_EINVAL;
  if (layout->head_dim <= 0 || layout->head_dim % 64 != 0 || rope_dim < 0 || rope_dim % 64 != 0 ||
      rope_dim > layout->head_dim)
    return KVQ_EUNSUPPORTED;
  if (num_tokens < 0) return KVQ_EINVAL;
  if (num_tokens == 0) return KVQ_OK;
  if (!pool || !scales || !kv || !slot_mapping) return KVQ_EINVAL;
  if ((reinterpret_cast<uintptr_t>(pool) | reinterpret_cast<uintptr_t>(scales) | reinterpret_cast<uintptr_t>(kv)) % 16 ||
      reinterpret_cast<uintptr_t>(slot_mapping) % 8)
    return KVQ_EALIGN;
  const kvq_status st = kvq_device_check();
  if (st != KVQ_OK) return st;
  ActQuantStoreArgs a;
  a.codes = static_cast<uint8_t*>(pool);
  a.scales = static_cast<__half*>(scales);
  a.kv = static_cast<const uint4*>(kv);
  a.slot_mapping = slot_mapping;
  a.num_tokens = num_tokens;
  a.D = layout->head_dim;
  a.latent = layout->head_dim - rope_dim;
  a.P = layout->page_size;
  a.num_slots = static_cast<int64_t>(layout->num_pages) * layout->page_size;
  const int64_t units = num_tokens * (layout->head_dim / 64);
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>((units + 255) / 256, static_cast<int64_t>(sm_count()) * 8));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (kind == KVQ_FP8_E4M3)
    act_quant_store_kernel<KVQ_FP8_E4M3><<<static_cast<unsigned>(grid), 256, 0, s>>>(a);
  else
    act_quant_store_kernel<KVQ_Q8_0><<<static_cast<unsigned>(grid), 256, 0, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ECUDA;
}

// ------------------------------------------------------------------------ store into an unscaled fp8 pool
// "Add fp8 KV-cache quantization (--kv-dtype)", section "How it works": the store casts the incoming bf16
// K/V straight to the pool's fp8 type (scale 1.0; e4m3, or e5m2 wired the same way).  One thread casts 16
// consecutive elements of a row (two 16-byte loads, one 16-byte store); the conversion rounds once to
// nearest-even and saturates at the largest finite value.
namespace kvq {
namespace {

struct UnscaledStoreArgs {
  uint8_t* codes;
  const uint4* k;
  const uint4* v;
  const int64_t* slot_mapping;
  int64_t num_tokens;
  int32_t Hkv, D, n_kv, P;
  int64_t num_slots;
};

template <int FMT>  // __NV_E4M3 or __NV_E5M2
__global__ void __launch_bounds__(256) unscaled_store_kernel(UnscaledStoreArgs a) {
  const int32_t chunks = a.D / 16;                            // 16-element pieces of a head row
  const int64_t per_kv = a.num_tokens * a.Hkv * chunks;
  const int64_t n = per_kv * a.n_kv;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u < n; u += stride) {
    const int kv = u >= per_kv;
    const int64_t local = u - (kv ? per_kv : 0);              // (token, head, chunk) of K or of V
    const int64_t t = local / (static_cast<int64_t>(a.Hkv) * chunks);
    const int32_t rem = static_cast<int32_t>(local - t * a.Hkv * chunks);
    const int32_t h = rem / chunks, c = rem - h * chunks;
    const int64_t slot = __ldg(a.slot_mapping + t);
    if (slot < 0 || slot >= a.num_slots) continue;            // -1 skips; out-of-range slots are never written
    const uint4* src = (kv ? a.v : a.k) + local * 2;          // 16 bf16 = two 16-byte pieces
    const uint4 x0 = __ldcs(src), x1 = __ldcs(src + 1);
    const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 lo = make_float2(__uint_as_float(w[2 * q] << 16), __uint_as_float(w[2 * q] & 0xFFFF0000u));
      const float2 hi = make_float2(__uint_as_float(w[2 * q + 1] << 16), __uint_as_float(w[2 * q + 1] & 0xFFFF0000u));
      const uint32_t a2 = __nv_cvt_float2_to_fp8x2(lo, __NV_SATFINITE, static_cast<__nv_fp8_interpretation_t>(FMT));
      const uint32_t b2 = __nv_cvt_float2_to_fp8x2(hi, __NV_SATFINITE, static_cast<__nv_fp8_interpretation_t>(FMT));
      o[q] = (a2 & 0xFFFFu) | (b2 << 16);
    }
    const int64_t page = slot / a.P, off = slot - (slot / a.P) * a.P;
    const int64_t dst_row = ((page * a.n_kv + kv) * a.Hkv + h) * a.P + off;
    __stcs(reinterpret_cast<uint4*>(a.codes + dst_row * a.D + static_cast<int64_t>(c) * 16),
           make_uint4(o[0], o[1], o[2], o[3]));
  }
}

}  // namespace
}  // namespace kvq

extern "C" kvq_status kvq_store_unscaled(void* pool, const void* k, const void* v, const int64_t* slot_mapping,
                                         int64_t num_tokens, const kvq_layout* layout, kvq_kind kind, void* stream) {
  using namespace kvq;
  if (!layout) return KVQ_EINVAL;
  if (kind != KVQ_FP8_E4M3_UNSCALED && kind != KVQ_FP8_E5M2_UNSCALED) return KVQ_EKIND;
  if (layout->num_pages < 0 || layout->page_size <= 0 || layout->num_kv_heads <= 0) return KVQ_EINVAL;
  if (layout->head_dim <= 0 || layout->head_dim % 32 != 0) return KVQ_EHEADDIM;
  if (num_tokens < 0) return KVQ_EINVAL;
  if (num_tokens == 0) return KVQ_OK;
  if (!pool || !k || !slot_mapping || (layout->mla ? v != nullptr : v == nullptr)) return KVQ_EINVAL;
  if ((reinterpret_cast<uintptr_t>(pool) | reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) % 16 ||
      reinterpret_cast<uintptr_t>(slot_mapping) % 8)
    return KVQ_EALIGN;
  const kvq_status st = kvq_device_check();
  if (st != KVQ_OK) return st;
  UnscaledStoreArgs a;
  a.codes = static_cast<uint8_t*>(pool);
  a.k = static_cast<const uint4*>(k);
  a.v = static_cast<const uint4*>(v);
  a.slot_mapping = slot_mapping;
  a.num_tokens = num_tokens;
  a.Hkv = layout->num_kv_heads;
  a.D = layout->head_dim;
  a.n_kv = layout->mla ? 1 : 2;
  a.P = layout->page_size;
  a.num_slots = static_cast<int64_t>(layout->num_pages) * layout->page_size;
  const int64_t n = num_tokens * a.Hkv * (a.D / 16) * a.n_kv;
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>((n + 255) / 256, static_cast<int64_t>(sm_count()) * 8));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (kind == KVQ_FP8_E4M3_UNSCALED)
    unscaled_store_kernel<__NV_E4M3><<<static_cast<unsigned>(grid), 256, 0, s>>>(a);
  else
    unscaled_store_kernel<__NV_E5M2><<<static_cast<unsigned>(grid), 256, 0, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ECUDA;
}
