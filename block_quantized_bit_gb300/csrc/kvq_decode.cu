// kvq_decode.cu -- split-K decode attention over the 8-bit paged pool, CUDA-core path, and the merge.
//
// "feat(kvcache): 8-bit KV cache (q8_0 / fp8_e4m3) behind --kv-cache-dtype", section "What": the scale
// varies along head_dim, the reduction dim, so K and V are dequantized to bf16 before the dot.
// "feat(kvcache): 8-bit DSV4 window/compressed KV", section "Testing": the split-k decode kernel and
// masked (-1) columns; section "What this adds": an MLA latent row serves as both K and V.
//
// Work decomposition (computed identically by every CTA and by the merge kernel from seq_lens, so no
// planning launch and no host read-back is needed):
//   query group qg = (kv head g, head tile ht): `heads_per_item` query heads that share kv head g;
//   pages of sequence b are cut into splits of C pages; one work item = (b, qg, split);
//   C = pages_per_split, or max(4, ceil(sum_b pages_b * groups / 1216)) when automatic.
// One CTA runs one item.  Each of its warps walks every WARPS-th page of the split with its own
// STAGES-deep pipeline of 1-D bulk copies (codes and scales of the page's K and V chunks into shared
// memory, completion on an mbarrier).  Lanes read 16-byte code chunks, dequantize to bf16-exact fp32,
// and run the fp32 online softmax in the exp2 domain; the CTA combines its warps and writes one
// (m, l, acc) partial per query head.  The merge kernel combines the partials of a (b, qg).
#include <math.h>

#include <algorithm>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kPlanThreads = 128;

struct KParams {
  const __nv_bfloat16* q;
  const uint8_t* codes;
  const __half* scales;
  const int32_t* block_table;
  const int32_t* seq_lens;
  float* part_acc;
  float* part_ml;
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
  float score_scale;      // sm_scale * log2(e)
};

__device__ __forceinline__ int32_t seq_pages(const KParams& p, int32_t b) {
  const int32_t L = max(__ldg(p.seq_lens + b), 0);
  return min((L + kPage - 1) / kPage, p.max_pages);
}

// Block-wide plan: pages per split C, and for `want_b` (or the sequence that owns item `want_item`)
// its first item index and split count.  Must be called by all kPlanThreads threads of the CTA.
struct Plan {
  int32_t C;
  int32_t b;        // sequence
  int32_t base;     // first item of sequence b
  int32_t nsplit;   // splits per query group of sequence b
  int32_t n_items;  // items over the whole batch
};

__device__ Plan make_plan(const KParams& p, int32_t want_item, int32_t want_b) {
  __shared__ long long s_red[kPlanThreads / 32];
  __shared__ int32_t s_scan[kPlanThreads / 32];
  __shared__ Plan s_plan;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int32_t groups = p.num_kv_heads * p.head_tiles;
  const int32_t per = (p.batch + kPlanThreads - 1) / kPlanThreads;
  const int32_t b0 = tid * per, b1 = min(b0 + per, p.batch);
  // 1) total page-units
  long long units = 0;
  for (int32_t b = b0; b < b1; ++b) units += seq_pages(p, b);
  for (int o = 16; o > 0; o >>= 1) units += __shfl_xor_sync(0xffffffffu, units, o);
  if (lane == 0) s_red[warp] = units;
  __syncthreads();
  long long tot = 0;
  for (int w = 0; w < kPlanThreads / 32; ++w) tot += s_red[w];
  tot *= groups;
  int32_t C = p.pages_per_split;
  if (C <= 0) {
    long long c = (tot + kTargetItems - 1) / kTargetItems;
    C = static_cast<int32_t>(c > kMinPagesPerSplit ? c : static_cast<long long>(kMinPagesPerSplit));
  }
  // 2) items per sequence, exclusive scan over the batch
  int32_t mine = 0;
  for (int32_t b = b0; b < b1; ++b) mine += groups * ((seq_pages(p, b) + C - 1) / C);
  int32_t incl = mine;
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_scan[warp] = incl;
  __syncthreads();
  int32_t warp_off = 0, total_items = 0;
  for (int w = 0; w < kPlanThreads / 32; ++w) {
    if (w < warp) warp_off += s_scan[w];
    total_items += s_scan[w];
  }
  int32_t run = warp_off + incl - mine;  // first item of b0
  for (int32_t b = b0; b < b1; ++b) {
    const int32_t ns = (seq_pages(p, b) + C - 1) / C;
    const int32_t n = groups * ns;
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

// ---------------------------------------------------------------------------- CUDA-core kernel
template <int D>
struct RowGeom {
  static constexpr int NCH = D / 16;                  // 16-byte code chunks per row
  static constexpr int LPT = NCH < 32 ? NCH : 32;     // lanes per token
  static constexpr int CPL = (NCH + 31) / 32;         // chunks per lane
  static constexpr int TPI = 32 / LPT;                // tokens per warp iteration
  static constexpr int ITERS = kPage / TPI;
  static constexpr int NB = D / 32;
  static_assert(32 % LPT == 0, "lanes per token must divide the warp");
};

template <int D, int DV, int GT, int KIND, bool MLA, int WARPS, int STAGES>
struct CCConfig {
  using G = RowGeom<D>;
  static constexpr int NKV = MLA ? 1 : 2;
  static constexpr int CODE_BYTES = kPage * D;           // one page of one head
  static constexpr int SCALE_BYTES = kPage * G::NB * 2;
  static constexpr int STAGE_BYTES = NKV * (CODE_BYTES + SCALE_BYTES);
  static constexpr int PIPE_BYTES = WARPS * STAGES * STAGE_BYTES;
  static constexpr int COMBINE_BYTES = WARPS * GT * (DV + 2) * 4;
  static constexpr int DATA_BYTES = PIPE_BYTES > COMBINE_BYTES ? PIPE_BYTES : COMBINE_BYTES;
  static constexpr int SMEM_BYTES = DATA_BYTES + WARPS * STAGES * 8 + WARPS * STAGES * 4;
  static constexpr int CPL_V = (DV / 16 + 31) / 32;       // value chunks per lane
  static_assert(CODE_BYTES % 16 == 0 && SCALE_BYTES % 16 == 0, "bulk copy sizes");
};

template <int D, int DV, int GT, int KIND, bool MLA, int WARPS, int STAGES>
__global__ void __launch_bounds__(WARPS * 32) decode_cc_kernel(KParams p) {
  using Cfg = CCConfig<D, DV, GT, KIND, MLA, WARPS, STAGES>;
  using Geo = RowGeom<D>;
  constexpr int NCH = Geo::NCH, LPT = Geo::LPT, CPL = Geo::CPL, TPI = Geo::TPI, ITERS = Geo::ITERS;
  constexpr int NB = Geo::NB;
  static_assert(WARPS * 32 == kPlanThreads, "plan helper assumes 128 threads");

  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::DATA_BYTES);
  int32_t* s_phys = reinterpret_cast<int32_t*>(smem + Cfg::DATA_BYTES + WARPS * STAGES * 8);

  const Plan plan = make_plan(p, static_cast<int32_t>(blockIdx.x), -1);
  if (plan.b < 0) return;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t b = plan.b;
  const int32_t groups = p.num_kv_heads * p.head_tiles;
  const int32_t local = static_cast<int32_t>(blockIdx.x) - plan.base;
  const int32_t qg = local / plan.nsplit;
  const int32_t split = local - qg * plan.nsplit;
  const int32_t g = qg / p.head_tiles;
  const int32_t ht = qg - g * p.head_tiles;
  const int32_t L = __ldg(p.seq_lens + b);
  const int32_t npages = seq_pages(p, b);
  const int32_t pg0 = split * plan.C;
  const int32_t pg1 = min(pg0 + plan.C, npages);
  const int32_t head0 = g * p.group + ht * GT;  // first query head of this item
  (void)groups;

  if (tid < WARPS * STAGES) mbar_init(&bars[tid], 1);
  fence_mbar_init();
  __syncthreads();

  // Query rows of this item's heads, for the chunk(s) this lane owns.
  const int tg = lane / LPT;  // token group within the warp
  const int c0 = lane % LPT;  // first chunk of this lane
  float qreg[GT][CPL][16];
#pragma unroll
  for (int h = 0; h < GT; ++h) {
    const __nv_bfloat16* qrow = p.q + (static_cast<int64_t>(b) * p.num_q_heads + head0 + h) * D;
#pragma unroll
    for (int k = 0; k < CPL; ++k) {
      const int c = c0 + 32 * k;
#pragma unroll
      for (int i = 0; i < 16; ++i) qreg[h][k][i] = 0.0f;
      if (c < NCH) {
        const uint4* src = reinterpret_cast<const uint4*>(qrow + c * 16);
        const uint4 a = __ldg(src), bq = __ldg(src + 1);
        const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
        const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&bq);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 x = __bfloat1622float2(pa[i]);
          const float2 y = __bfloat1622float2(pb[i]);
          qreg[h][k][2 * i] = x.x;
          qreg[h][k][2 * i + 1] = x.y;
          qreg[h][k][8 + 2 * i] = y.x;
          qreg[h][k][8 + 2 * i + 1] = y.y;
        }
      }
    }
  }

  float m[GT], l[GT], acc[GT][Cfg::CPL_V][16];
#pragma unroll
  for (int h = 0; h < GT; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.0f;
#pragma unroll
    for (int k = 0; k < Cfg::CPL_V; ++k)
#pragma unroll
      for (int i = 0; i < 16; ++i) acc[h][k][i] = 0.0f;
  }

  // Pages of this warp: pg0 + warp + i * WARPS.
  const int32_t np = pg1 - pg0;
  const int32_t nw = (np > warp) ? (np - warp + WARPS - 1) / WARPS : 0;
  uint8_t* wbuf = smem + warp * STAGES * Cfg::STAGE_BYTES;
  uint64_t* wbar = bars + warp * STAGES;
  int32_t* wphys = s_phys + warp * STAGES;
  const int64_t head_chunk = static_cast<int64_t>(Cfg::CODE_BYTES);
  const int64_t head_scale = static_cast<int64_t>(kPage * NB);  // fp16 elements

  auto issue = [&](int32_t i) {
    const int s = i % STAGES;
    if (lane == 0) {
      const int32_t pg = pg0 + warp + i * WARPS;
      int32_t phys = __ldg(p.block_table + static_cast<int64_t>(b) * p.max_pages + pg);
      if (phys >= p.num_pages) {  // out-of-range page: never dereferenced, reported in the status word
        set_status(p.status, kStatusBadPage);
        phys = -1;
      }
      wphys[s] = phys;
      uint8_t* dst = wbuf + s * Cfg::STAGE_BYTES;
      if (phys >= 0) {
        mbar_arrive_expect_tx(&wbar[s], Cfg::STAGE_BYTES);
#pragma unroll
        for (int kv = 0; kv < Cfg::NKV; ++kv) {
          const int64_t row = (static_cast<int64_t>(phys) * Cfg::NKV + kv) * p.num_kv_heads + g;
          bulk_g2s(dst + kv * Cfg::CODE_BYTES, p.codes + row * head_chunk, Cfg::CODE_BYTES, &wbar[s]);
          bulk_g2s(dst + Cfg::NKV * Cfg::CODE_BYTES + kv * Cfg::SCALE_BYTES, p.scales + row * head_scale,
                   Cfg::SCALE_BYTES, &wbar[s]);
        }
      } else {
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&wbar[s])) : "memory");
      }
    }
  };

  const int32_t prologue = min(nw, STAGES);
  for (int32_t i = 0; i < prologue; ++i) issue(i);
  __syncwarp();

  bool ok = true;
  int32_t consumed = 0;
  for (int32_t i = 0; i < nw; ++i) {
    const int s = i % STAGES;
    const uint32_t parity = (i / STAGES) & 1;
    if (!mbar_wait_bounded(&wbar[s], parity)) {
      ok = false;
      break;
    }
    consumed = i + 1;
    const int32_t phys = wphys[s];
    if (phys >= 0) {
      const int32_t pg = pg0 + warp + i * WARPS;
      const uint8_t* kc = wbuf + s * Cfg::STAGE_BYTES;
      const uint8_t* vc = MLA ? kc : kc + Cfg::CODE_BYTES;
      const __half* ks = reinterpret_cast<const __half*>(kc + Cfg::NKV * Cfg::CODE_BYTES);
      const __half* vs = MLA ? ks : ks + kPage * NB;

      // ---- scores for the 16 tokens of the page
      float sc[ITERS][GT];
#pragma unroll
      for (int it = 0; it < ITERS; ++it) {
        const int t = it * TPI + tg;
        float part[GT];
#pragma unroll
        for (int h = 0; h < GT; ++h) part[h] = 0.0f;
#pragma unroll
        for (int k = 0; k < CPL; ++k) {
          const int c = c0 + 32 * k;
          if (c < NCH) {
            const uint4 code = *reinterpret_cast<const uint4*>(kc + t * D + c * 16);
            const float sf = __half2float(ks[t * NB + (c >> 1)]);
            float kd[16];
            dequant16<KIND>(code, sf, kd);
#pragma unroll
            for (int h = 0; h < GT; ++h)
#pragma unroll
              for (int e = 0; e < 16; ++e) part[h] = fmaf(qreg[h][k][e], kd[e], part[h]);
          }
        }
#pragma unroll
        for (int h = 0; h < GT; ++h) {
#pragma unroll
          for (int o = 1; o < LPT; o <<= 1) part[h] += __shfl_xor_sync(0xffffffffu, part[h], o);
          const bool valid = pg * kPage + t < L;
          sc[it][h] = valid ? part[h] * p.score_scale : -INFINITY;
        }
      }
      // ---- online softmax update (page max is warp-uniform)
#pragma unroll
      for (int h = 0; h < GT; ++h) {
        float mx = -INFINITY;
#pragma unroll
        for (int it = 0; it < ITERS; ++it) mx = fmaxf(mx, sc[it][h]);
#pragma unroll
        for (int o = LPT; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float mnew = fmaxf(m[h], mx);
        const float alpha = (mnew == -INFINITY) ? 1.0f : exp2f(m[h] - mnew);
        m[h] = mnew;
        l[h] *= alpha;
#pragma unroll
        for (int k = 0; k < Cfg::CPL_V; ++k)
#pragma unroll
          for (int e = 0; e < 16; ++e) acc[h][k][e] *= alpha;
#pragma unroll
        for (int it = 0; it < ITERS; ++it) {
          const float pr = (sc[it][h] == -INFINITY) ? 0.0f : exp2f(sc[it][h] - mnew);
          sc[it][h] = pr;
          l[h] += pr;
        }
      }
      // ---- P.V
#pragma unroll
      for (int it = 0; it < ITERS; ++it) {
        const int t = it * TPI + tg;
        if (pg * kPage + t >= L) continue;  // never touch rows past the sequence end
#pragma unroll
        for (int k = 0; k < Cfg::CPL_V; ++k) {
          const int c = c0 + 32 * k;
          if (c * 16 < DV) {
            const uint4 code = *reinterpret_cast<const uint4*>(vc + t * D + c * 16);
            const float sf = __half2float(vs[t * NB + (c >> 1)]);
            float vd[16];
            dequant16<KIND>(code, sf, vd);
#pragma unroll
            for (int h = 0; h < GT; ++h)
#pragma unroll
              for (int e = 0; e < 16; ++e) acc[h][k][e] = fmaf(sc[it][h], vd[e], acc[h][k][e]);
          }
        }
      }
    }
    // release the stage and refill it
    fence_proxy_async_smem();
    __syncwarp();
    if (i + STAGES < nw) issue(i + STAGES);
    __syncwarp();
  }

  if (!ok) {
    set_status(p.status, kStatusTimeout);
    // drain this warp's copies still in flight (bounded) before the CTA may exit
    for (int32_t i = consumed; i < min(nw, consumed + STAGES); ++i)
      (void)mbar_wait_bounded(&wbar[i % STAGES], (i / STAGES) & 1);
  }

  // ---- reduce over token groups inside the warp
#pragma unroll
  for (int h = 0; h < GT; ++h) {
#pragma unroll
    for (int o = LPT; o < 32; o <<= 1) l[h] += __shfl_xor_sync(0xffffffffu, l[h], o);
#pragma unroll
    for (int k = 0; k < Cfg::CPL_V; ++k)
#pragma unroll
      for (int e = 0; e < 16; ++e)
#pragma unroll
        for (int o = LPT; o < 32; o <<= 1) acc[h][k][e] += __shfl_xor_sync(0xffffffffu, acc[h][k][e], o);
  }

  // ---- combine warps through shared memory (pipeline buffers are free now)
  __syncthreads();
  float* cm = reinterpret_cast<float*>(smem);            // [WARPS][GT] m
  float* cl = cm + WARPS * GT;                             // [WARPS][GT] l
  float* ca = cl + WARPS * GT;                             // [WARPS][GT][DV]
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < GT; ++h) {
      cm[warp * GT + h] = m[h];
      cl[warp * GT + h] = l[h];
    }
  }
  if (tg == 0) {
#pragma unroll
    for (int h = 0; h < GT; ++h)
#pragma unroll
      for (int k = 0; k < Cfg::CPL_V; ++k) {
        const int c = c0 + 32 * k;
        if (c * 16 < DV) {
          float4* dst = reinterpret_cast<float4*>(ca + (warp * GT + h) * DV + c * 16);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[e] = make_float4(acc[h][k][4 * e], acc[h][k][4 * e + 1], acc[h][k][4 * e + 2], acc[h][k][4 * e + 3]);
        }
      }
  }
  __syncthreads();
  const int64_t item = blockIdx.x;
  for (int idx = tid; idx < GT * DV; idx += WARPS * 32) {
    const int h = idx / DV, d = idx - h * DV;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) M = fmaxf(M, cm[w * GT + h]);
    float a = 0.0f, lsum = 0.0f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < WARPS; ++w) {
        const float mw = cm[w * GT + h];
        if (mw == -INFINITY) continue;
        const float wgt = exp2f(mw - M);
        a = fmaf(ca[(w * GT + h) * DV + d], wgt, a);
        lsum = fmaf(cl[w * GT + h], wgt, lsum);
      }
    }
    p.part_acc[(item * GT + h) * DV + d] = a;
    if (d == 0) {
      p.part_ml[(item * GT + h) * 2 + 0] = M;
      p.part_ml[(item * GT + h) * 2 + 1] = lsum;
    }
  }
}

// ------------------------------------------------------------------------------------- merge
// One CTA per (b, query group): combine the group's split partials per head and write the output.
template <typename OutT>
__global__ void __launch_bounds__(kPlanThreads) merge_kernel(KParams p, OutT* __restrict__ out, int32_t heads_per_item,
                                                             int32_t DV) {
  const int32_t groups = p.num_kv_heads * p.head_tiles;
  const int32_t b = blockIdx.x / groups;
  const int32_t qg = blockIdx.x - b * groups;
  const Plan plan = make_plan(p, -1, b);
  const int32_t g = qg / p.head_tiles, ht = qg - g * p.head_tiles;
  const int32_t head0 = g * p.group + ht * heads_per_item;
  int32_t ns = plan.nsplit;
  const int64_t first = static_cast<int64_t>(plan.base) + static_cast<int64_t>(qg) * ns;
  if (first + ns > p.max_items) {  // cannot happen when the workspace bound holds; never read past it
    if (threadIdx.x == 0) set_status(p.status, kStatusBadPage);
    ns = 0;
  }
  for (int idx = threadIdx.x; idx < heads_per_item * DV; idx += blockDim.x) {
    const int h = idx / DV, d = idx - h * DV;
    float M = -INFINITY;
    for (int32_t s = 0; s < ns; ++s) M = fmaxf(M, p.part_ml[((first + s) * heads_per_item + h) * 2]);
    float a = 0.0f, lsum = 0.0f;
    if (M != -INFINITY) {
      for (int32_t s = 0; s < ns; ++s) {
        const int64_t it = (first + s) * heads_per_item + h;
        const float ms = p.part_ml[it * 2];
        if (ms == -INFINITY) continue;
        const float w = exp2f(ms - M);
        lsum = fmaf(p.part_ml[it * 2 + 1], w, lsum);
        a = fmaf(p.part_acc[it * DV + d], w, a);
      }
    }
    const float o = (lsum > 0.0f) ? a / lsum : 0.0f;
    const int64_t dst = (static_cast<int64_t>(b) * p.num_q_heads + head0 + h) * DV + d;
    if constexpr (sizeof(OutT) == 2)
      out[dst] = __float2bfloat16_rn(o);
    else
      out[dst] = o;
  }
}

// --------------------------------------------------------------------------------- dequant probe
template <int KIND>
__global__ void dequant_probe_kernel(const uint8_t* __restrict__ codes, const uint16_t* __restrict__ scales,
                                     uint16_t* __restrict__ out, int64_t nchunks) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t c = i; c < nchunks; c += stride) {
    const uint4 code = reinterpret_cast<const uint4*>(codes)[c];
    float v[16];
    dequant16<KIND>(code, half_bits_to_float(scales[c]), v);
#pragma unroll
    for (int e = 0; e < 16; ++e) out[c * 16 + e] = __bfloat16_as_ushort(__float2bfloat16_rn(v[e]));
  }
}

KParams make_kparams(const DecodeArgs& a) {
  KParams p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.codes = a.codes;
  p.scales = reinterpret_cast<const __half*>(a.scales);
  p.block_table = a.block_table;
  p.seq_lens = a.seq_lens;
  p.part_acc = a.part_acc;
  p.part_ml = a.part_ml;
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
  return p;
}

template <int D, int DV, int GT, int KIND, bool MLA, int WARPS, int STAGES>
kvq_status launch_cc(const DecodeArgs& a, cudaStream_t stream) {
  using Cfg = CCConfig<D, DV, GT, KIND, MLA, WARPS, STAGES>;
  auto kern = decode_cc_kernel<D, DV, GT, KIND, MLA, WARPS, STAGES>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) != cudaSuccess)
    return KVQ_ECUDA;
  const KParams p = make_kparams(a);
  kern<<<static_cast<unsigned>(a.max_items), WARPS * 32, Cfg::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ECUDA;
}

template <int D, int DV, int GT, bool MLA, int STAGES>
kvq_status launch_cc_kind(const DecodeArgs& a, cudaStream_t stream) {
  if (a.kind == KVQ_FP8_E4M3) return launch_cc<D, DV, GT, KVQ_FP8_E4M3, MLA, 4, STAGES>(a, stream);
  return launch_cc<D, DV, GT, KVQ_Q8_0, MLA, 4, STAGES>(a, stream);
}

}  // namespace

int32_t cc_heads_per_item(int32_t group, int32_t head_dim, int32_t mla) {
  const int32_t cap = mla ? 2 : 4;
  int32_t gt = 1;
  while (gt * 2 <= cap && group % (gt * 2) == 0) gt *= 2;
  (void)head_dim;
  return gt;
}

bool decode_cc_supported(int32_t head_dim, int32_t v_dim, int32_t mla) {
  if (mla) return head_dim == 576 && v_dim == 512;
  return v_dim == head_dim && (head_dim == 64 || head_dim == 128 || head_dim == 256);
}

kvq_status launch_decode_cc(const DecodeArgs& a, cudaStream_t stream) {
  const int gt = a.heads_per_item;
  if (a.mla) {
    if (gt == 1) return launch_cc_kind<576, 512, 1, true, 2>(a, stream);
    return launch_cc_kind<576, 512, 2, true, 2>(a, stream);
  }
#define KVQ_CC_CASE(DD, STG)                                                        \
  if (a.head_dim == DD) {                                                           \
    if (gt == 1) return launch_cc_kind<DD, DD, 1, false, STG>(a, stream);           \
    if (gt == 2) return launch_cc_kind<DD, DD, 2, false, STG>(a, stream);           \
    return launch_cc_kind<DD, DD, 4, false, STG>(a, stream);                        \
  }
  KVQ_CC_CASE(64, 4)
  KVQ_CC_CASE(128, 4)
  KVQ_CC_CASE(256, 3)
#undef KVQ_CC_CASE
  return KVQ_EUNSUPPORTED;
}

kvq_status launch_merge(const DecodeArgs& a, int32_t query_groups, cudaStream_t stream) {
  const KParams p = make_kparams(a);
  const unsigned grid = static_cast<unsigned>(static_cast<int64_t>(a.batch) * query_groups);
  if (grid == 0) return KVQ_OK;
  if (a.out_dtype == KVQ_OUT_BF16)
    merge_kernel<__nv_bfloat16><<<grid, kPlanThreads, 0, stream>>>(p, static_cast<__nv_bfloat16*>(a.out),
                                                                    a.heads_per_item, a.v_dim);
  else
    merge_kernel<float><<<grid, kPlanThreads, 0, stream>>>(p, static_cast<float*>(a.out), a.heads_per_item, a.v_dim);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ECUDA;
}

kvq_status launch_dequant_probe(kvq_kind kind, const uint8_t* codes, const uint16_t* scales, uint16_t* out,
                                int64_t n, cudaStream_t stream) {
  const int64_t nchunks = n / 16;
  if (nchunks == 0) return KVQ_OK;
  const int threads = 256;
  const int64_t grid = std::min<int64_t>((nchunks + threads - 1) / threads, 152 * 16);
  if (kind == KVQ_FP8_E4M3)
    dequant_probe_kernel<KVQ_FP8_E4M3><<<static_cast<unsigned>(grid), threads, 0, stream>>>(codes, scales, out,
                                                                                           nchunks);
  else
    dequant_probe_kernel<KVQ_Q8_0><<<static_cast<unsigned>(grid), threads, 0, stream>>>(codes, scales, out, nchunks);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ECUDA;
}

}  // namespace kvq
