// kvq_plan.cuh -- work-item planning shared by the decode kernels and the merge kernel.
//
// A decode work item is (sequence b, query group, split): a query group is a kv head together with a
// tile of the query heads that read it, and a split is a run of C consecutive pages of the sequence.
// C = pages_per_split when the caller fixes it; otherwise C = max(4, ceil(sum_b pages_b * groups /
// target)) rounded up to `split_align` pages; the host sets the target per kernel (about two waves of
// the CUDA-core kernel's resident CTAs, two items per SM for the GQA tensor-core kernel, one for MLA).
// The GQA tensor-core kernel first tries the target of one item per SM and keeps it when the batch's
// items fit in that many (the rounding of C can push them over; then two per SM).
// Every CTA derives the same plan from seq_lens on the device, so no planning launch and no host
// read-back are needed.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr float kLog2e = 1.4426950408889634f;


struct KParams {
  int32_t split_align;    // automatic split sizes are rounded up to a multiple of this
  const __nv_bfloat16* q;
  const uint8_t* codes;
  const __half* scales;
  const int32_t* block_table;
  const int32_t* bt_row;  // block-table row of each sequence, or null: row b (the extend's per-token prefixes)
  const int32_t* seq_lens;
  float* part_acc;
  float* part_ml;
  int32_t* plan_tab;      // [batch][2] first item, splits per query group; CTA 0 of the decode writes it
  int32_t* split_cnt;     // [batch][groups] splits finished (zeroed per call), or null: no fused merge
  void* out;              // [batch][num_q_heads][v_dim], bf16 or fp32 (out_f32)
  int32_t out_f32;
  uint32_t* status;
  int64_t num_pages;      // pages in the pool: larger block-table entries are treated as masked
  int64_t max_items;      // work items the workspace holds
  int32_t max_pages;
  int32_t batch;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t group;          // Hq / Hkv
  int32_t head_tiles;     // group / heads_per_item
  int32_t pages_per_split;
  int32_t target_items;   // automatic split sizes aim at about this many items
  int32_t one_wave_items; // nonzero: first try about this many items, kept when the items fit in it
  int32_t min_one_split;  // nonzero: a sequence without pages still gets one (empty) split per group, so
                          // that the kernel which merges in-kernel writes its zero output
  float score_scale;      // sm_scale * log2(e)
};

// Block-table entry of page pg of sequence b.
__device__ __forceinline__ int32_t bt_entry(const KParams& p, int32_t b, int32_t pg) {
  const int64_t row = p.bt_row ? __ldg(p.bt_row + b) : b;
  return __ldg(p.block_table + row * p.max_pages + pg);
}

__device__ __forceinline__ int32_t seq_pages(const KParams& p, int32_t b) {
  const int32_t L = max(__ldg(p.seq_lens + b), 0);
  return min((L + kPage - 1) / kPage, p.max_pages);
}

// Block-wide plan: pages per split C, and for `want_b` (or the sequence that owns item `want_item`)
// its first item index and split count.  Every thread of the CTA must call it (blockDim a multiple of 32).
struct Plan {
  int32_t C;
  int32_t b;        // sequence
  int32_t base;     // first item of sequence b
  int32_t nsplit;   // splits per query group of sequence b
  int32_t n_items;  // items over the whole batch
};

__device__ Plan make_plan(const KParams& p, int32_t want_item, int32_t want_b) {
  __shared__ long long s_red[32];
  __shared__ unsigned long long s_scan[32];
  __shared__ Plan s_plan;
  const int tid = threadIdx.x, nthr = blockDim.x, nwarp = nthr >> 5;
  const int lane = tid & 31, warp = tid >> 5;
  const int32_t groups = p.num_kv_heads * p.head_tiles;
  const int32_t per = (p.batch + nthr - 1) / nthr;
  const int32_t b0 = tid * per, b1 = min(b0 + per, p.batch);
  // 1) total page-units
  long long units = 0;
  for (int32_t b = b0; b < b1; ++b) units += seq_pages(p, b);
  for (int o = 16; o > 0; o >>= 1) units += __shfl_xor_sync(0xffffffffu, units, o);
  if (lane == 0) s_red[warp] = units;
  __syncthreads();
  long long tot = 0;
  for (int w = 0; w < nwarp; ++w) tot += s_red[w];
  tot *= groups;
  auto split_size = [&](int32_t target) {
    long long c = (tot + target - 1) / target;
    int32_t cc = static_cast<int32_t>(c > kMinPagesPerSplit ? c : static_cast<long long>(kMinPagesPerSplit));
    return (cc + p.split_align - 1) / p.split_align * p.split_align;
  };
  // C2: the fixed or the target split size; C1: the one-wave size (C2 when there is none)
  const int32_t C2 = p.pages_per_split > 0 ? p.pages_per_split : split_size(p.target_items);
  const int32_t C1 = (p.pages_per_split <= 0 && p.one_wave_items > 0) ? split_size(p.one_wave_items) : C2;
  auto splits_of = [&](int32_t b, int32_t c) { return max((seq_pages(p, b) + c - 1) / c, p.min_one_split ? 1 : 0); };
  // 2) items per sequence under both sizes (low half C1, high half C2), exclusive scan over the batch
  unsigned long long mine = 0;
  for (int32_t b = b0; b < b1; ++b)
    mine += static_cast<unsigned long long>(groups * splits_of(b, C1)) |
            (static_cast<unsigned long long>(groups * splits_of(b, C2)) << 32);
  unsigned long long incl = mine;
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_scan[warp] = incl;
  __syncthreads();
  unsigned long long warp_off = 0, totals = 0;
  for (int w = 0; w < nwarp; ++w) {
    if (w < warp) warp_off += s_scan[w];
    totals += s_scan[w];
  }
  // one wave when every item has a resident CTA
  const bool one = C1 != C2 && static_cast<uint32_t>(totals) <= static_cast<uint32_t>(p.one_wave_items);
  const int32_t C = one ? C1 : C2;
  auto pick = [&](unsigned long long v) { return static_cast<int32_t>(one ? (v & 0xFFFFFFFFull) : (v >> 32)); };
  const int32_t total_items = pick(totals);
  int32_t run = pick(warp_off + incl - mine);  // first item of b0
  for (int32_t b = b0; b < b1; ++b) {
    const int32_t ns = splits_of(b, C);
    const int32_t n = groups * ns;
    if (blockIdx.x == 0 && p.plan_tab) {  // for the merge, which then needs no plan of its own
      p.plan_tab[2 * b] = run;
      p.plan_tab[2 * b + 1] = ns;
    }
    const bool hit = (want_b >= 0) ? (b == want_b) : (want_item >= run && want_item < run + n);
    if (hit) {
      s_plan.C = C;
      s_plan.b = b;
      s_plan.base = run;
      s_plan.nsplit = ns;
    }
    run += n;
  }
  if (tid == 0 && want_b < 0 && want_item >= total_items) {
    s_plan.C = C;
    s_plan.b = -1;
    s_plan.base = 0;
    s_plan.nsplit = 0;
  }
  __syncthreads();
  Plan r = s_plan;
  r.n_items = total_items;
  r.C = C;
  __syncthreads();
  return r;
}

inline KParams make_kparams(const DecodeArgs& a) {
  KParams p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.codes = a.codes;
  p.scales = reinterpret_cast<const __half*>(a.scales);
  p.block_table = a.block_table;
  p.bt_row = a.bt_row;
  p.seq_lens = a.seq_lens;
  p.part_acc = a.part_acc;
  p.part_ml = a.part_ml;
  p.plan_tab = a.plan_tab;
  p.split_cnt = a.split_cnt;
  p.out = a.out;
  p.out_f32 = a.out_dtype == KVQ_OUT_F32;
  p.status = a.status;
  p.num_pages = a.num_pages;
  p.max_items = a.max_items;
  p.max_pages = a.max_pages;
  p.batch = a.batch;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.group = a.num_q_heads / a.num_kv_heads;
  p.head_tiles = p.group / a.heads_per_item;
  p.pages_per_split = a.pages_per_split;
  p.score_scale = a.sm_scale * kLog2e;
  p.split_align = a.split_align;
  p.target_items = a.target_items > 0 ? a.target_items : kTargetItems;
  p.one_wave_items = a.one_wave_items;
  p.min_one_split = a.min_one_split;
  return p;
}

}  // namespace
}  // namespace kvq
