// kvq_decode.cu -- split-K decode attention over the 8-bit paged pool, CUDA-core path, and the merge.
//
// "feat(kvcache): 8-bit KV cache (q8_0 / fp8_e4m3) behind --kv-cache-dtype", section "What": the scale
// varies along head_dim, the reduction dim, so K and V are dequantized to bf16 before the dot.
// "feat(kvcache): 8-bit DSV4 window/compressed KV", section "Testing": the split-k decode kernel and
// masked (-1) columns; section "What this adds": an MLA latent row serves as both K and V.
//
// Work decomposition (computed identically by every CTA from seq_lens, so no planning launch and no
// host read-back is needed; CTA 0 also leaves each sequence's first item and split count for the merge):
//   query group qg = (kv head g, head tile ht): `heads_per_item` query heads that share kv head g;
//   pages of sequence b are cut into splits of C pages; one work item = (b, qg, split);
//   C = pages_per_split, or max(4, ceil(sum_b pages_b * groups / target)) when automatic, target a little
//   under two waves of the resident CTAs (the host's plan).
// One CTA runs one item.  Each of its warps walks every WARPS-th page of the split with its own
// STAGES-deep pipeline of 1-D bulk copies (codes and scales of the page's K and V chunks into shared
// memory, completion on an mbarrier).  Lanes read 16-byte code chunks, dequantize to bf16-exact fp32,
// and run the fp32 online softmax in the exp2 domain; the CTA combines its warps and writes one
// (m, l, acc) partial per query head.  The CTA that finishes the last split of a (b, qg) merges the
// group's partials itself (a split counter in the workspace), so this path needs no merge launch; a
// group with one split writes its output directly.  The merge kernel below combines the partials of
// the tensor-core kernels.
#include <math.h>

#include <algorithm>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_plan.cuh"

namespace kvq {

namespace {

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

template <int N>
struct Log2 {
  static constexpr int value = 1 + Log2<N / 2>::value;
};
template <>
struct Log2<1> {
  static constexpr int value = 0;
};

template <int D, int DV, int GT, int KIND, bool MLA, int WARPS, int STAGES>
struct CCConfig {
  using G = RowGeom<D>;
  static constexpr int NKV = MLA ? 1 : 2;
  static constexpr int CODE_BYTES = kPage * D;           // one page of one head
  static constexpr int SCALE_BYTES = KindTraits<KIND>::kScaled ? kPage * G::NB * 2 : 0;  // none when unscaled
  static constexpr int STAGE_BYTES = NKV * (CODE_BYTES + SCALE_BYTES);
  static constexpr int PIPE_BYTES = WARPS * STAGES * STAGE_BYTES;
  static constexpr int COMBINE_BYTES = WARPS * GT * (DV + 2) * 4;
  static constexpr int DATA_BYTES = PIPE_BYTES > COMBINE_BYTES ? PIPE_BYTES : COMBINE_BYTES;
  static constexpr int SMEM_BYTES = DATA_BYTES + WARPS * STAGES * 8 + WARPS * STAGES * 4;
  static constexpr int CPL_V = (DV / 16 + 31) / 32;       // value chunks per lane
  static constexpr int LOG_GT = Log2<GT>::value;
  static_assert(CODE_BYTES % 16 == 0 && SCALE_BYTES % 16 == 0, "bulk copy sizes");
  static_assert(GT <= G::LPT, "a token's lanes must cover every head of the tile");
};

// Lane (within a token group) that ends up holding head h after the transposed reduction.
template <int LPT, int GT>
__device__ __forceinline__ int head_lane(int h) {
  constexpr int LG = Log2<GT>::value;
  int c = 0;
#pragma unroll
  for (int k = 0; k < LG; ++k)
    if ((h >> (LG - 1 - k)) & 1) c |= LPT >> (k + 1);
  return c;
}

// Sum v[h] over the LPT lanes of a token while distributing heads: after the call, v[0] of a lane
// holds the full dot for head H(lane) (the first log2(GT) xor steps exchange half of the remaining
// heads each, the rest add the single value).  Every lane of the warp must call it.
template <int LPT, int GT>
__device__ __forceinline__ float reduce_heads(float (&v)[GT], int lane) {
  constexpr int LG = Log2<GT>::value;
#pragma unroll
  for (int k = 0; k < LG; ++k) {
    const int o = LPT >> (k + 1);
    const bool upper = (lane & o) != 0;
    constexpr int dummy = 0;
    (void)dummy;
    const int n = GT >> k;
#pragma unroll
    for (int i = 0; i < GT / 2; ++i) {
      if (i < n / 2) {
        const float send = upper ? v[i] : v[i + n / 2];
        const float keep = upper ? v[i + n / 2] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
    }
  }
  float r = v[0];
#pragma unroll
  for (int o = LPT >> (LG + 1); o >= 1; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
  return r;
}

// One element of the decode output, bf16 (round to nearest-even) or fp32.
__device__ __forceinline__ void store_out(const KParams& p, int64_t idx, float v) {
  if (p.out_f32)
    static_cast<float*>(p.out)[idx] = v;
  else
    static_cast<__nv_bfloat16*>(p.out)[idx] = __float2bfloat16_rn(v);
}

template <int D, int DV, int GT, int KIND, bool MLA, int WARPS, int STAGES, int MINB>
__global__ void __launch_bounds__(WARPS * 32, MINB) decode_cc_kernel(KParams p) {
  using Cfg = CCConfig<D, DV, GT, KIND, MLA, WARPS, STAGES>;
  using Geo = RowGeom<D>;
  constexpr int NCH = Geo::NCH, LPT = Geo::LPT, CPL = Geo::CPL, TPI = Geo::TPI, ITERS = Geo::ITERS;
  constexpr int NB = Geo::NB, CPL_V = Cfg::CPL_V, LG = Cfg::LOG_GT;

  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::DATA_BYTES);
  int32_t* s_phys = reinterpret_cast<int32_t*>(smem + Cfg::DATA_BYTES + WARPS * STAGES * 8);

  const Plan plan = make_plan(p, static_cast<int32_t>(blockIdx.x), -1);
  if (plan.b < 0) return;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t b = plan.b;
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

  if (tid < WARPS * STAGES) mbar_init(&bars[tid], 1);
  fence_mbar_init();
  __syncthreads();

  const int tg = lane / LPT;  // token group within the warp
  const int c0 = lane % LPT;  // first 16-element chunk of this lane
  // head whose score this lane ends up owning after reduce_heads
  int my_head = 0;
#pragma unroll
  for (int k = 0; k < LG; ++k)
    if (c0 & (LPT >> (k + 1))) my_head |= GT >> (k + 1);

  // q rows of this item's heads for the lane's chunk(s), as packed bf16 pairs
  uint32_t qb[GT][CPL][8];
#pragma unroll
  for (int h = 0; h < GT; ++h) {
    const __nv_bfloat16* qrow = p.q + (static_cast<int64_t>(b) * p.num_q_heads + head0 + h) * D;
#pragma unroll
    for (int k = 0; k < CPL; ++k) {
      const int c = c0 + 32 * k;
      uint4 a = make_uint4(0u, 0u, 0u, 0u), bq = a;
      if (c < NCH) {
        const uint4* src = reinterpret_cast<const uint4*>(qrow + c * 16);
        a = __ldg(src);
        bq = __ldg(src + 1);
      }
      qb[h][k][0] = a.x; qb[h][k][1] = a.y; qb[h][k][2] = a.z; qb[h][k][3] = a.w;
      qb[h][k][4] = bq.x; qb[h][k][5] = bq.y; qb[h][k][6] = bq.z; qb[h][k][7] = bq.w;
    }
  }

  float m = -INFINITY, l = 0.0f;  // online-softmax state of head my_head
  float2 acc[GT][CPL_V][8];
#pragma unroll
  for (int h = 0; h < GT; ++h)
#pragma unroll
    for (int k = 0; k < CPL_V; ++k)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[h][k][e] = make_float2(0.0f, 0.0f);

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
      int32_t phys = bt_entry(p, b, pg);
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
          if (KindTraits<KIND>::kScaled)
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
      const uint16_t* ks = reinterpret_cast<const uint16_t*>(kc + Cfg::NKV * Cfg::CODE_BYTES);
      const uint16_t* vs = MLA ? ks : ks + kPage * NB;

      // ---- scores of this lane's head for its tokens of the page
      float sc[ITERS];
#pragma unroll
      for (int it = 0; it < ITERS; ++it) {
        const int t = it * TPI + tg;
        float part[GT][2];
#pragma unroll
        for (int h = 0; h < GT; ++h) part[h][0] = part[h][1] = 0.0f;
#pragma unroll
        for (int k = 0; k < CPL; ++k) {
          const int c = c0 + 32 * k;
          if (c < NCH) {
            const uint4 code = *reinterpret_cast<const uint4*>(kc + t * D + c * 16);
            uint32_t kd[8];
            dequant16<KIND>(code, KindTraits<KIND>::kScaled ? ks[t * NB + (c >> 1)] : kHalfOne, kd);
#pragma unroll
            for (int e = 0; e < 8; ++e)
#pragma unroll
              for (int h = 0; h < GT; ++h) {
                part[h][0] = fma_f32_bf16(lo16(qb[h][k][e]), lo16(kd[e]), part[h][0]);
                part[h][1] = fma_f32_bf16(hi16(qb[h][k][e]), hi16(kd[e]), part[h][1]);
              }
          }
        }
        float v[GT];
#pragma unroll
        for (int h = 0; h < GT; ++h) v[h] = part[h][0] + part[h][1];
        const float dot = reduce_heads<LPT, GT>(v, lane);
        sc[it] = (pg * kPage + t < L) ? dot * p.score_scale : -INFINITY;
      }
      // ---- online softmax for this lane's head; the page max is uniform over the head's lanes
      float mx = -INFINITY;
#pragma unroll
      for (int it = 0; it < ITERS; ++it) mx = fmaxf(mx, sc[it]);
#pragma unroll
      for (int o = LPT; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float mnew = fmaxf(m, mx);
      const float alpha = (mnew == -INFINITY) ? 1.0f : exp2f(m - mnew);
      m = mnew;
      l *= alpha;
#pragma unroll
      for (int it = 0; it < ITERS; ++it) {
        sc[it] = (sc[it] == -INFINITY) ? 0.0f : exp2f(sc[it] - mnew);
        l += sc[it];
      }
      if (__any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll
        for (int h = 0; h < GT; ++h) {
          const float ah = __shfl_sync(0xffffffffu, alpha, tg * LPT + head_lane<LPT, GT>(h));
#pragma unroll
          for (int k = 0; k < CPL_V; ++k)
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              acc[h][k][e].x *= ah;
              acc[h][k][e].y *= ah;
            }
        }
      }
      // ---- P.V
#pragma unroll
      for (int it = 0; it < ITERS; ++it) {
        const int t = it * TPI + tg;
        float ph[GT];
#pragma unroll
        for (int h = 0; h < GT; ++h) ph[h] = __shfl_sync(0xffffffffu, sc[it], tg * LPT + head_lane<LPT, GT>(h));
        if (pg * kPage + t >= L) continue;  // never touch rows past the sequence end
#pragma unroll
        for (int k = 0; k < CPL_V; ++k) {
          const int c = c0 + 32 * k;
          if (c * 16 < DV) {
            const uint4 code = *reinterpret_cast<const uint4*>(vc + t * D + c * 16);
            uint32_t vd[8];
            dequant16<KIND>(code, KindTraits<KIND>::kScaled ? vs[t * NB + (c >> 1)] : kHalfOne, vd);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float2 v2 = unpack_bf16x2(vd[e]);
#pragma unroll
              for (int h = 0; h < GT; ++h) acc[h][k][e] = ffma2(v2, make_float2(ph[h], ph[h]), acc[h][k][e]);
            }
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
  for (int o = LPT; o < 32; o <<= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
#pragma unroll
  for (int h = 0; h < GT; ++h)
#pragma unroll
    for (int k = 0; k < CPL_V; ++k)
#pragma unroll
      for (int e = 0; e < 8; ++e)
#pragma unroll
        for (int o = LPT; o < 32; o <<= 1) {
          acc[h][k][e].x += __shfl_xor_sync(0xffffffffu, acc[h][k][e].x, o);
          acc[h][k][e].y += __shfl_xor_sync(0xffffffffu, acc[h][k][e].y, o);
        }

  // ---- combine warps through shared memory (pipeline buffers are free now)
  __syncthreads();
  float* cm = reinterpret_cast<float*>(smem);            // [WARPS][GT] m
  float* cl = cm + WARPS * GT;                             // [WARPS][GT] l
  float* ca = cl + WARPS * GT;                             // [WARPS][GT][DV]
  if (tg == 0 && lane < LPT) {
#pragma unroll
    for (int h = 0; h < GT; ++h)
      if (c0 == head_lane<LPT, GT>(h)) {
        cm[warp * GT + h] = m;
        cl[warp * GT + h] = l;
      }
  }
  if (tg == 0) {
#pragma unroll
    for (int h = 0; h < GT; ++h)
#pragma unroll
      for (int k = 0; k < CPL_V; ++k) {
        const int c = c0 + 32 * k;
        if (c * 16 < DV) {
          float4* dst = reinterpret_cast<float4*>(ca + (warp * GT + h) * DV + c * 16);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[e] = make_float4(acc[h][k][2 * e].x, acc[h][k][2 * e].y, acc[h][k][2 * e + 1].x,
                                 acc[h][k][2 * e + 1].y);
        }
      }
  }
  __syncthreads();
  const int64_t item = blockIdx.x;
  const bool only_split = (plan.nsplit == 1) && (p.split_cnt != nullptr);
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
    if (only_split) {  // the group's only split: its normalised output, no partial
      store_out(p, (static_cast<int64_t>(b) * p.num_q_heads + head0 + h) * DV + d, lsum > 0.0f ? a / lsum : 0.0f);
      continue;
    }
    p.part_acc[(item * GT + h) * DV + d] = a;
    if (d == 0) {
      p.part_ml[(item * GT + h) * 2 + 0] = M;
      p.part_ml[(item * GT + h) * 2 + 1] = lsum;
    }
  }
  if (only_split || p.split_cnt == nullptr) return;

  // ---- fused merge: the CTA that finishes the last split of its (b, query group) merges the group.
  // Every CTA publishes its partial (fence) before it counts itself in; the last one fences again
  // before reading the others' partials, which it reads from L2 (ld.cg: its L1 may hold stale lines).
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  const int32_t groups = p.num_kv_heads * p.head_tiles;
  if (tid == 0) s_last = atomicAdd(p.split_cnt + static_cast<int64_t>(b) * groups + qg, 1) == plan.nsplit - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int64_t first = static_cast<int64_t>(plan.base) + static_cast<int64_t>(qg) * plan.nsplit;
  const int32_t ns = plan.nsplit;
  // (1) M_h = max_s m_s,h.  The (split, head) pairs are contiguous and the stride is a multiple of GT,
  // so every thread sees one head only: tid % GT.
  float* sM = reinterpret_cast<float*>(smem);  // [WARPS][GT]
  float* sL = sM + WARPS * GT;                  // [WARPS][GT]
  float* sA = sL + WARPS * GT;                  // [WARPS][GT][DV]
  {
    float mt = -INFINITY;
    for (int32_t i = tid; i < ns * GT; i += WARPS * 32) mt = fmaxf(mt, __ldcg(p.part_ml + (first * GT + i) * 2));
#pragma unroll
    for (int o = 16; o >= GT; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
    if (lane < GT) sM[warp * GT + lane] = mt;
  }
  __syncthreads();
  float Mh[GT];
#pragma unroll
  for (int h = 0; h < GT; ++h) {
    Mh[h] = -INFINITY;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) Mh[h] = fmaxf(Mh[h], sM[w * GT + h]);
  }
  // (2) warp w sums the splits s = w, w + WARPS, ...; lane = dim (mod 32)
  constexpr int DPL = DV / 32;  // dims per lane
  float am[GT][DPL], lw[GT];
#pragma unroll
  for (int h = 0; h < GT; ++h) {
    lw[h] = 0.0f;
#pragma unroll
    for (int j = 0; j < DPL; ++j) am[h][j] = 0.0f;
  }
#pragma unroll 2
  for (int32_t sp = warp; sp < ns; sp += WARPS) {
#pragma unroll
    for (int h = 0; h < GT; ++h) {
      const int64_t it = (first + sp) * GT + h;
      const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.part_ml + it * 2));
      const float wgt = (ml.x == -INFINITY) ? 0.0f : exp2f(ml.x - Mh[h]);
      lw[h] = fmaf(ml.y, wgt, lw[h]);
#pragma unroll
      for (int j = 0; j < DPL; ++j) am[h][j] = fmaf(__ldcg(p.part_acc + it * DV + lane + 32 * j), wgt, am[h][j]);
    }
  }
#pragma unroll
  for (int h = 0; h < GT; ++h) {
    if (lane == 0) sL[warp * GT + h] = lw[h];
#pragma unroll
    for (int j = 0; j < DPL; ++j) sA[(warp * GT + h) * DV + lane + 32 * j] = am[h][j];
  }
  __syncthreads();
  // (3) sum over the warps, normalise
  for (int idx = tid; idx < GT * DV; idx += WARPS * 32) {
    const int h = idx / DV, d = idx - h * DV;
    float at = 0.0f, lt = 0.0f;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) {
      at += sA[(w * GT + h) * DV + d];
      lt += sL[w * GT + h];
    }
    store_out(p, (static_cast<int64_t>(b) * p.num_q_heads + head0 + h) * DV + d, lt > 0.0f ? at / lt : 0.0f);
  }
}

// ------------------------------------------------------------------------------------- merge
constexpr int kMergeThreads = 256;
constexpr int kMergeWarps = kMergeThreads / 32;
constexpr int kMergeSubs = 4;  // splits a warp reads at once: 8 lanes x float4 = the 32 dims of a slice

// One CTA per (sequence, query group, head of the item, 32-dim slice of v): the log-sum-exp merge of
// the sequence's split partials, out = sum_s 2^(m_s - M) acc_s / sum_s 2^(m_s - M) l_s, M = max_s m_s.
// A warp reads four splits at a time (lanes 8j..8j+7 take split j, four dims each), so the CTA has 32
// splits' loads in flight per round; the sums are reduced across the lane groups and the warps.  The
// decode kernel's CTA 0 left each sequence's first item and split count in plan_tab, so no plan is
// recomputed here.
template <typename OutT>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(KParams p, OutT* __restrict__ out, int32_t heads_per_item,
                                                              int32_t DV, int32_t units_per_seq) {
  __shared__ float s_m[kMergeWarps];
  __shared__ __align__(16) float s_a[kMergeWarps][32];
  __shared__ float s_l[kMergeWarps];
  // Launched as a programmatic dependent of the decode kernel: its CTAs may start while the decode's last
  // CTAs still run; this waits until that grid has completed and its partials are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sub = lane >> 3, q = lane & 7;  // split of the four, float4 of the slice
  const int32_t b = blockIdx.x / units_per_seq;
  const int32_t u = blockIdx.x - b * units_per_seq;
  const int32_t slices = DV / 32;
  const int32_t slice = u % slices;
  const int32_t h = (u / slices) % heads_per_item;
  const int32_t qg = u / (slices * heads_per_item);
  const int32_t g = qg / p.head_tiles, ht = qg - g * p.head_tiles;
  const int32_t head = g * p.group + ht * heads_per_item + h;
  int32_t ns = p.plan_tab[2 * b + 1];
  const int64_t first = static_cast<int64_t>(p.plan_tab[2 * b]) + static_cast<int64_t>(qg) * ns;
  if (ns < 0 || first < 0 || first + ns > p.max_items) {  // cannot happen when the workspace bound holds
    if (tid == 0) set_status(p.status, kStatusBadPage);
    ns = 0;
  }
  float M = -INFINITY;
  for (int32_t s = tid; s < ns; s += kMergeThreads) M = fmaxf(M, p.part_ml[((first + s) * heads_per_item + h) * 2]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if (lane == 0) s_m[warp] = M;
  __syncthreads();
#pragma unroll
  for (int w = 0; w < kMergeWarps; ++w) M = fmaxf(M, s_m[w]);
  float4 a = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  float l = 0.0f;
  if (M != -INFINITY) {
    const float* acc = p.part_acc + slice * 32 + q * 4;
#pragma unroll 2
    for (int32_t s = warp * kMergeSubs + sub; s < ns; s += kMergeWarps * kMergeSubs) {
      const int64_t it = (first + s) * heads_per_item + h;
      const float2 ml = *reinterpret_cast<const float2*>(p.part_ml + it * 2);
      const float w = (ml.x == -INFINITY) ? 0.0f : exp2f(ml.x - M);
      const float4 v = *reinterpret_cast<const float4*>(acc + it * DV);
      a.x = fmaf(v.x, w, a.x);
      a.y = fmaf(v.y, w, a.y);
      a.z = fmaf(v.z, w, a.z);
      a.w = fmaf(v.w, w, a.w);
      l = fmaf(ml.y, w, l);
    }
  }
#pragma unroll
  for (int o = 8; o < 32; o <<= 1) {  // over the four lane groups (the same q)
    a.x += __shfl_xor_sync(0xffffffffu, a.x, o);
    a.y += __shfl_xor_sync(0xffffffffu, a.y, o);
    a.z += __shfl_xor_sync(0xffffffffu, a.z, o);
    a.w += __shfl_xor_sync(0xffffffffu, a.w, o);
    l += __shfl_xor_sync(0xffffffffu, l, o);
  }
  if (lane < 8) *reinterpret_cast<float4*>(&s_a[warp][q * 4]) = a;
  if (lane == 0) s_l[warp] = l;
  __syncthreads();
  if (warp == 0) {
    float at = 0.0f, lt = 0.0f;
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) {
      at += s_a[w][lane];
      lt += s_l[w];
    }
    const float o = (lt > 0.0f) ? at / lt : 0.0f;
    const int64_t dst = (static_cast<int64_t>(b) * p.num_q_heads + head) * DV + slice * 32 + lane;
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
    uint32_t kd[8];
    dequant16<KIND>(code, KindTraits<KIND>::kScaled ? scales[c] : kHalfOne, kd);
    uint4* dst = reinterpret_cast<uint4*>(out + c * 16);
    dst[0] = make_uint4(kd[0], kd[1], kd[2], kd[3]);
    dst[1] = make_uint4(kd[4], kd[5], kd[6], kd[7]);
  }
}


template <int D, int DV, int GT, int KIND, bool MLA, int STAGES, int MINB>
kvq_status launch_cc(const DecodeArgs& a, cudaStream_t stream) {
  constexpr int WARPS = 4;
  using Cfg = CCConfig<D, DV, GT, KIND, MLA, WARPS, STAGES>;
  auto kern = decode_cc_kernel<D, DV, GT, KIND, MLA, WARPS, STAGES, MINB>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) != cudaSuccess)
    return KVQ_ECUDA;
  const KParams p = make_kparams(a);
  kern<<<static_cast<unsigned>(a.max_items), WARPS * 32, Cfg::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ECUDA;
}

template <int D, int DV, int GT, bool MLA, int STAGES, int MINB>
kvq_status launch_cc_kind(const DecodeArgs& a, cudaStream_t stream) {
  switch (a.kind) {
    case KVQ_FP8_E4M3: return launch_cc<D, DV, GT, KVQ_FP8_E4M3, MLA, STAGES, MINB>(a, stream);
    case KVQ_Q8_0: return launch_cc<D, DV, GT, KVQ_Q8_0, MLA, STAGES, MINB>(a, stream);
    case KVQ_FP8_E4M3_UNSCALED: return launch_cc<D, DV, GT, KVQ_FP8_E4M3_UNSCALED, MLA, STAGES, MINB>(a, stream);
    case KVQ_FP8_E5M2_UNSCALED: return launch_cc<D, DV, GT, KVQ_FP8_E5M2_UNSCALED, MLA, STAGES, MINB>(a, stream);
  }
  return KVQ_EKIND;
}

}  // namespace

int32_t cc_heads_per_item(int32_t group, int32_t head_dim, int32_t mla) {
  const int32_t cap = mla ? 2 : 4;
  int32_t gt = 1;
  while (gt * 2 <= cap && group % (gt * 2) == 0) gt *= 2;
  (void)head_dim;
  return gt;
}

// CTAs per SM that launch_decode_cc's configuration keeps resident (its MINB).
int32_t cc_ctas_per_sm(int32_t head_dim, int32_t mla, int32_t gt) {
  if (mla) return 1;
  if (head_dim == 64) return 4;
  if (head_dim == 128) return gt == 2 ? 5 : 4;
  return 3;
}

bool decode_cc_supported(int32_t head_dim, int32_t v_dim, int32_t mla) {
  if (mla) return head_dim == 576 && v_dim == 512;
  return v_dim == head_dim && (head_dim == 64 || head_dim == 128 || head_dim == 256);
}

kvq_status launch_decode_cc(const DecodeArgs& a, cudaStream_t stream) {
  const int gt = a.heads_per_item;
  if (a.mla) {
    if (gt == 1) return launch_cc_kind<576, 512, 1, true, 2, 1>(a, stream);
    return launch_cc_kind<576, 512, 2, true, 2, 1>(a, stream);
  }
// (stages, CTAs per SM) per head_dim and heads per item: two heads at D = 128 fit 93 registers, so five
// CTAs of two stages each stay resident (qwen3_1p7b 58 -> 55 us); four heads need the registers of four.
#define KVQ_CC_CASE(DD, STG, MB, STG2, MB2)                                         \
  if (a.head_dim == DD) {                                                           \
    if (gt == 1) return launch_cc_kind<DD, DD, 1, false, STG, MB>(a, stream);       \
    if (gt == 2) return launch_cc_kind<DD, DD, 2, false, STG2, MB2>(a, stream);     \
    return launch_cc_kind<DD, DD, 4, false, STG, MB>(a, stream);                    \
  }
  KVQ_CC_CASE(64, 4, 4, 4, 4)
  KVQ_CC_CASE(128, 3, 4, 2, 5)
  KVQ_CC_CASE(256, 2, 3, 2, 3)
#undef KVQ_CC_CASE
  return KVQ_EUNSUPPORTED;
}

kvq_status launch_merge(const DecodeArgs& a, int32_t query_groups, cudaStream_t stream) {
  const KParams p = make_kparams(a);
  const int32_t units = query_groups * a.heads_per_item * (a.v_dim / 32);
  const int64_t grid = static_cast<int64_t>(a.batch) * units;
  if (grid == 0) return KVQ_OK;
  // programmatic stream serialization: the merge grid launches as the decode grid winds down instead of after it
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (a.out_dtype == KVQ_OUT_BF16)
    e = cudaLaunchKernelEx(&cfg, merge_kernel<__nv_bfloat16>, p, static_cast<__nv_bfloat16*>(a.out), a.heads_per_item,
                           a.v_dim, units);
  else
    e = cudaLaunchKernelEx(&cfg, merge_kernel<float>, p, static_cast<float*>(a.out), a.heads_per_item, a.v_dim,
                           units);
  return (e == cudaSuccess && cudaGetLastError() == cudaSuccess) ? KVQ_OK : KVQ_ECUDA;
}

// ------------------------------------------------------------------------------------ wait probe
// One thread initialises an mbarrier expecting one arrival that never comes, and waits on it with
// mbar_wait_bounded, the wait every decode kernel uses; it gives up after kWaitLimitNs and reports the
// timeout exactly as a decode kernel would.
__global__ void wait_probe_kernel(uint32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_mbar_init();
  if (!mbar_wait_bounded(&bar, 0)) set_status(status, kStatusTimeout);
}

kvq_status launch_wait_probe(uint32_t* status, cudaStream_t stream) {
  wait_probe_kernel<<<1, 32, 0, stream>>>(status);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ECUDA;
}

kvq_status launch_dequant_probe(kvq_kind kind, const uint8_t* codes, const uint16_t* scales, uint16_t* out,
                                int64_t n, cudaStream_t stream) {
  const int64_t nchunks = n / 16;
  if (nchunks == 0) return KVQ_OK;
  const int threads = 256;
  const int64_t grid = std::min<int64_t>((nchunks + threads - 1) / threads, 152 * 16);
  const unsigned g = static_cast<unsigned>(grid);
  switch (kind) {
    case KVQ_FP8_E4M3: dequant_probe_kernel<KVQ_FP8_E4M3><<<g, threads, 0, stream>>>(codes, scales, out, nchunks); break;
    case KVQ_Q8_0: dequant_probe_kernel<KVQ_Q8_0><<<g, threads, 0, stream>>>(codes, scales, out, nchunks); break;
    case KVQ_FP8_E4M3_UNSCALED:
      dequant_probe_kernel<KVQ_FP8_E4M3_UNSCALED><<<g, threads, 0, stream>>>(codes, scales, out, nchunks);
      break;
    case KVQ_FP8_E5M2_UNSCALED:
      dequant_probe_kernel<KVQ_FP8_E5M2_UNSCALED><<<g, threads, 0, stream>>>(codes, scales, out, nchunks);
      break;
  }
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ECUDA;
}

}  // namespace kvq
