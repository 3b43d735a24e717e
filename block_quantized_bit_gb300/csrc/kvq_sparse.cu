// kvq_sparse.cu -- sparse (top-K) decode: gather the columns a sequence's index list selects into a
// compact pool; the dense split-K decode then runs over that pool.
//
// "Experimental FP8 KV Cache" (its SPARSE_MLA_DECODE profile line: one query reads K = 256 selected
// tokens of a 163840-token latent pool) and "feat(kvcache): 8-bit DSV4 window/compressed KV", section
// "Testing" (masked -1 columns).  A column is valid when its position p satisfies 0 <= p < seq_len and
// block_table[b][p / 16] is not -1; each valid column is one term of the softmax, a position listed twice
// counting twice.  Attention does not depend on the order of its columns, so the valid columns of
// sequence b are packed, in list order, into the compact pages b * cpages .. of a pool with the same
// layout; the compact sequence has as many tokens as valid columns and an identity block table.  The
// gather moves codes and scales byte for byte: the decode then sees exactly the stored values.
#include <cuda_runtime.h>

#include <algorithm>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kGatherThreads = 256;

// Grid (sequence, share): every CTA of a sequence numbers the valid columns in list order (a block-wide
// scan over per-thread runs of the list, recomputed by each CTA, which is cheaper than a second launch)
// and then copies its share of the columns: every (column, kv, head) row's D code bytes as 16-byte
// pieces and D/32 scales as 4-byte words (D is a multiple of 64, checked on the host, so a row's
// scales are whole, 4-byte aligned words).  The shares spread the copies' load latency over many SMs.
__global__ void __launch_bounds__(kGatherThreads) sparse_gather_kernel(SparseGatherArgs a) {
  extern __shared__ int32_t s_src[];  // [topk] source slot of the column at each packed position
  __shared__ int32_t s_warp[kGatherThreads / 32];
  __shared__ int32_t s_count;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t b = blockIdx.x;
  const int32_t L = __ldg(a.seq_lens + b);
  const int32_t* idx = a.indices + static_cast<int64_t>(b) * a.topk;
  const int32_t per = (a.topk + kGatherThreads - 1) / kGatherThreads;
  const int32_t i0 = min(tid * per, a.topk), i1 = min(i0 + per, a.topk);
  auto slot_of = [&](int32_t i) -> int32_t {
    const int32_t p = __ldg(idx + i);
    if (p < 0 || p >= L || p / kPage >= a.max_pages) return -1;  // (seq_len past the table: never read)
    const int32_t page = __ldg(a.block_table + static_cast<int64_t>(b) * a.max_pages + p / kPage);
    if (page < 0) return -1;
    if (page >= a.num_pages) {  // never dereferenced; reported in the status word
      set_status(a.status, kStatusBadPage);
      return -1;
    }
    return page * kPage + p % kPage;
  };
  int32_t mine = 0;
  for (int32_t i = i0; i < i1; ++i) mine += slot_of(i) >= 0;
  int32_t incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  int32_t base = 0, total = 0;
#pragma unroll
  for (int w = 0; w < kGatherThreads / 32; ++w) {
    base += (w < warp) ? s_warp[w] : 0;
    total += s_warp[w];
  }
  int32_t pos = base + incl - mine;
  for (int32_t i = i0; i < i1; ++i) {
    const int32_t s = slot_of(i);
    if (s >= 0) s_src[pos++] = s;
  }
  if (tid == 0) s_count = total;
  if (blockIdx.y == 0) {
    if (tid == 0) a.dst_lens[b] = total;
    for (int32_t j = tid; j < a.cpages; j += kGatherThreads)
      a.dst_table[static_cast<int64_t>(b) * a.cpages + j] = b * a.cpages + j;
  }
  __syncthreads();
  // this CTA's share of the packed columns
  const int32_t share = (s_count + gridDim.y - 1) / gridDim.y;
  const int32_t c0 = min(static_cast<int32_t>(blockIdx.y) * share, s_count);
  const int32_t count = min(c0 + share, s_count) - c0;
  const int32_t rows = a.n_kv * a.Hkv;          // rows per column
  const int32_t pieces = a.D / 16;              // 16-byte pieces per code row
  const int64_t total_pieces = static_cast<int64_t>(count) * rows * pieces;
  for (int64_t u = tid; u < total_pieces; u += kGatherThreads) {
    const int32_t c = c0 + static_cast<int32_t>(u / (rows * pieces));
    const int32_t r = static_cast<int32_t>((u / pieces) % rows);  // kv * Hkv + h
    const int32_t k = static_cast<int32_t>(u % pieces);
    const int32_t src = s_src[c];
    const int32_t dpos = b * a.cpages * kPage + c;  // packed slot in the compact pool
    const int64_t srow = (static_cast<int64_t>(src / kPage) * rows + r) * kPage + src % kPage;
    const int64_t drow = (static_cast<int64_t>(dpos / kPage) * rows + r) * kPage + dpos % kPage;
    reinterpret_cast<uint4*>(a.dst_codes + drow * a.D)[k] =
        __ldg(reinterpret_cast<const uint4*>(a.codes + srow * a.D) + k);
  }
  if (a.dst_scales == nullptr) return;           // an unscaled pool: codes only
  const int32_t words = a.D / 64;               // 4-byte words of scales per row (D/32 fp16 values)
  const int64_t total_words = static_cast<int64_t>(count) * rows * words;
  for (int64_t u = tid; u < total_words; u += kGatherThreads) {
    const int32_t c = c0 + static_cast<int32_t>(u / (rows * words));
    const int32_t r = static_cast<int32_t>((u / words) % rows);
    const int32_t k = static_cast<int32_t>(u % words);
    const int32_t src = s_src[c];
    const int32_t dpos = b * a.cpages * kPage + c;
    const int64_t srow = (static_cast<int64_t>(src / kPage) * rows + r) * kPage + src % kPage;
    const int64_t drow = (static_cast<int64_t>(dpos / kPage) * rows + r) * kPage + dpos % kPage;
    reinterpret_cast<uint32_t*>(a.dst_scales + drow * (a.D / 32))[k] =
        __ldg(reinterpret_cast<const uint32_t*>(a.scales + srow * (a.D / 32)) + k);
  }
}

}  // namespace

kvq_status launch_sparse_gather(const SparseGatherArgs& g, cudaStream_t stream) {
  if (g.batch == 0) return KVQ_OK;
  const size_t smem = static_cast<size_t>(g.topk > 0 ? g.topk : 1) * sizeof(int32_t);
  // about eight columns per CTA, at most 64 CTAs per sequence
  const unsigned shares = static_cast<unsigned>(std::min<int32_t>(64, std::max<int32_t>(1, (g.topk + 7) / 8)));
  sparse_gather_kernel<<<dim3(static_cast<unsigned>(g.batch), shares), kGatherThreads, smem, stream>>>(g);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ECUDA;
}

}  // namespace kvq
