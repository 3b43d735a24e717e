// kvq_store.cu -- quantize-and-scatter store of bf16 K/V rows into the 8-bit paged pool.
//
// "feat(kvcache): 8-bit KV cache (q8_0 / fp8_e4m3) behind --kv-cache-dtype", section "What" (the
// store kernel: per-block max-abs -> codes + scales, one fp16 scale per 32 elements along head_dim)
// and its review comment "A bug on sm_89" (int8 rounds half away from zero then clamps; fp8 clamps
// then rounds once to nearest-even -- never through a truncated fp16).
//
// Mapping: four lanes own one 32-element block (8 bf16 = one 16-byte load each).  The input is
// walked as a flat stream of blocks, K first then V, so every warp load is 512 contiguous bytes.
// amax is a 2-step xor shuffle inside the 4-lane group; each lane writes its 8 code bytes, the
// group's first lane the fp16 scale.  UNROLL independent blocks per lane are loaded before any is
// processed, to keep enough bytes in flight for HBM.
#include <algorithm>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

namespace {

constexpr int kStoreThreads = 256;
constexpr int kStoreUnroll = 4;

template <int KIND, int UNROLL>
__global__ void __launch_bounds__(kStoreThreads)
    store_kernel(uint8_t* __restrict__ codes, __half* __restrict__ scales, const uint4* __restrict__ k,
                 const uint4* __restrict__ v, const int64_t* __restrict__ slot_mapping, int32_t T,
                 int32_t Hkv, int32_t D, int32_t P, int32_t n_kv, int64_t num_slots) {
  const int32_t nb = D >> 5;
  const int32_t row_blocks = Hkv * nb;            // blocks in one token row (all heads)
  const int32_t blocks_per_kv = T * row_blocks;   // host guarantees n_kv * this < 2^31
  const int32_t total = blocks_per_kv * n_kv;
  const int lane = threadIdx.x & 31;
  const int sub = lane & 3;
  const int32_t warp_global = (blockIdx.x * kStoreThreads + threadIdx.x) >> 5;
  const int32_t nwarps = (gridDim.x * kStoreThreads) >> 5;
  const int32_t step = nwarps * 8;  // groups per sweep of all warps

  for (int32_t wbase = warp_global * 8; wbase < total; wbase += step * UNROLL) {
    uint4 x[UNROLL];
    int32_t blk[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      blk[u] = wbase + u * step + (lane >> 2);
      x[u] = make_uint4(0u, 0u, 0u, 0u);
      if (blk[u] < total) {
        const int kv = blk[u] >= blocks_per_kv;
        const int32_t local = blk[u] - (kv ? blocks_per_kv : 0);
        x[u] = __ldcs((kv ? v : k) + (static_cast<int64_t>(local) * 4 + sub));
      }
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      float f[8];
      const __nv_bfloat162* xp = reinterpret_cast<const __nv_bfloat162*>(&x[u]);
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 t = __bfloat1622float2(xp[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
        amax = fmaxf(amax, fmaxf(fabsf(t.x), fabsf(t.y)));
      }
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      if (blk[u] >= total) continue;
      const int kv = blk[u] >= blocks_per_kv;
      const int32_t local = blk[u] - (kv ? blocks_per_kv : 0);
      const int32_t t = local / row_blocks;
      const int32_t in_row = local - t * row_blocks;
      const int32_t h = in_row / nb;
      const int32_t j = in_row - h * nb;
      const int64_t slot = __ldg(slot_mapping + t);
      if (slot < 0 || slot >= num_slots) continue;  // -1 skips; out-of-range slots are never written
      const int64_t page = slot / P;
      const int32_t off = static_cast<int32_t>(slot - page * P);
      const int64_t dst_row = ((page * n_kv + kv) * Hkv + h) * P + off;

      const __half s16 = block_scale<KIND>(amax);
      const float sf = __half2float(s16);
      uint2 out = make_uint2(0u, 0u);
      if (sf != 0.0f) {
        float y[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) y[i] = __fdiv_rn(f[i], sf);
        if (KIND == KVQ_FP8_E4M3) {
          out.x = static_cast<uint32_t>(encode_fp8x2(y[0], y[1])) |
                  (static_cast<uint32_t>(encode_fp8x2(y[2], y[3])) << 16);
          out.y = static_cast<uint32_t>(encode_fp8x2(y[4], y[5])) |
                  (static_cast<uint32_t>(encode_fp8x2(y[6], y[7])) << 16);
        } else {
          out.x = static_cast<uint32_t>(encode_q8(y[0])) | (static_cast<uint32_t>(encode_q8(y[1])) << 8) |
                  (static_cast<uint32_t>(encode_q8(y[2])) << 16) | (static_cast<uint32_t>(encode_q8(y[3])) << 24);
          out.y = static_cast<uint32_t>(encode_q8(y[4])) | (static_cast<uint32_t>(encode_q8(y[5])) << 8) |
                  (static_cast<uint32_t>(encode_q8(y[6])) << 16) | (static_cast<uint32_t>(encode_q8(y[7])) << 24);
        }
      }
      uint2* dst = reinterpret_cast<uint2*>(codes + dst_row * D + (j << 5) + (sub << 3));
      __stcs(dst, out);
      if (sub == 0) scales[dst_row * nb + j] = (sf != 0.0f) ? s16 : __ushort_as_half(0);
    }
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
  const int64_t row_blocks = static_cast<int64_t>(L.num_kv_heads) * (L.head_dim / 32);
  const int64_t max_rows = std::max<int64_t>(1, ((int64_t(1) << 30) / (row_blocks * n_kv)));
  const int64_t row_elems = static_cast<int64_t>(L.num_kv_heads) * L.head_dim;
  const int sms = sm_count();
  const int64_t num_slots = L.num_pages * L.page_size;
  for (int64_t t0 = 0; t0 < num_tokens; t0 += max_rows) {
    const int32_t T = static_cast<int32_t>(std::min(max_rows, num_tokens - t0));
    const int64_t total_blocks = static_cast<int64_t>(T) * row_blocks * n_kv;
    const int64_t groups_per_cta = kStoreThreads / 4;
    int64_t grid = (total_blocks + groups_per_cta * kStoreUnroll - 1) / (groups_per_cta * kStoreUnroll);
    grid = std::min<int64_t>(grid, static_cast<int64_t>(sms) * 8);
    grid = std::max<int64_t>(grid, 1);
    const uint4* kp = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(k) + t0 * row_elems);
    const uint4* vp =
        v ? reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(v) + t0 * row_elems) : nullptr;
    const int64_t* sm = slot_mapping + t0;
    if (kind == KVQ_FP8_E4M3)
      store_kernel<KVQ_FP8_E4M3, kStoreUnroll><<<static_cast<unsigned>(grid), kStoreThreads, 0, stream>>>(
          static_cast<uint8_t*>(pool), static_cast<__half*>(scales), kp, vp, sm, T, L.num_kv_heads, L.head_dim,
          L.page_size, n_kv, num_slots);
    else
      store_kernel<KVQ_Q8_0, kStoreUnroll><<<static_cast<unsigned>(grid), kStoreThreads, 0, stream>>>(
          static_cast<uint8_t*>(pool), static_cast<__half*>(scales), kp, vp, sm, T, L.num_kv_heads, L.head_dim,
          L.page_size, n_kv, num_slots);
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

}  // namespace kvq
