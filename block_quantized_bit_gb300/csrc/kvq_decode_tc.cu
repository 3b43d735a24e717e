// kvq_decode_tc.cu -- split-K decode on the 5th-generation tensor cores (tcgen05) for wide GQA groups.
//
// "feat(kvcache): 8-bit KV cache (q8_0 / fp8_e4m3) behind --kv-cache-dtype", section "What": K and V
// are dequantized to bf16 before the dot (the scale varies along the reduction dim).  Here the
// dequantized bf16 tiles are the operands of tcgen05.mma, with fp32 accumulators in tensor memory.
// "feat(kvcache): 8-bit DSV4 window/compressed KV", section "Testing": split-k decode, masked -1 pages.
//
// With G = 8..16 query heads per kv head, QK^T and PV are small dense contractions.  They run
// swapped so that the 128 tokens of a tile are the MMA's M dimension:
//   S^T[128 tok][16] = Kd[128 tok][D] . Q[16][D]^T     (A = K tile, K-major; B = Q, K-major)
//   O^T[d][16]     += Vd^T[d][128 tok] . P[16][128]^T  (A = the V tile read MN-major; B = P, MN-major)
// (heads beyond G are zero rows of Q and P).  Both tiles use the canonical no-swizzle core-matrix
// layout  off(t, d) = (t%8)*16 + (t/8)*RS + (d%8)*2 + (d/8)*128  with RS = D*16, which is K-major for
// the K operand (descriptor LBO = 128, SBO = RS) and MN-major for V^T (LBO = RS, SBO = 128).
//
// One persistent CTA per SM, 13 warps:
//   warps 0-3   softmax: TMEM lane = token; fp32 online softmax in the exp2 domain with lazy
//               rescaling (the running max moves only when a tile's max exceeds it by 2^8); writes P
//               (bf16) and, when the max moves, rescales O in TMEM; finally writes the item partial.
//   warps 4-11  dequant: each thread owns half a token row; codes are loaded from the pool one tile
//               ahead, dequantized exactly as on the CUDA-core path, and stored as bf16 tiles.
//   warp 12     TMEM allocation and the single thread that issues tcgen05.mma / tcgen05.commit.
// The roles hand tiles over with mbarriers; every wait is bounded (2 s) and reports a timeout in the
// workspace status word instead of hanging.
#include <math.h>

#include <algorithm>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_plan.cuh"

namespace kvq {
namespace {

constexpr int kTile = 128;        // tokens per tile (8 pages)
constexpr int kPagesPerTile = kTile / kPage;
constexpr int kN = 16;            // MMA N: query heads, padded
constexpr int kSmWarps = 4;
constexpr int kDwWarps = 8;
constexpr int kMmaWarp = kSmWarps + kDwWarps;
constexpr int kThreads = (kMmaWarp + 1) * 32;
constexpr int kMaxPlanBatch = 2048;  // sequences whose item bases fit the shared table
constexpr float kLazyRescale = 8.0f;  // log2 headroom before the running max must move
constexpr int kTmemCols = 64;

template <int D>
struct TcCfg {
  static constexpr int RS = D * 16;                 // bytes between 8-token groups of a tile
  static constexpr int TILE_BYTES = kTile * D * 2;  // one bf16 tile
  static constexpr int Q_BYTES = kN * D * 2;
  static constexpr int P_BYTES = kN * kTile * 2;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = TILE_BYTES;
  static constexpr int Q_OFF = 2 * TILE_BYTES;
  static constexpr int P_OFF = Q_OFF + Q_BYTES;
  static constexpr int RED_OFF = P_OFF + P_BYTES;                  // softmax cross-warp scratch
  static constexpr int TAB_OFF = RED_OFF + kSmWarps * kN * 4;      // item bases of the batch
  static constexpr int BAR_OFF = TAB_OFF + kMaxPlanBatch * 4;
  static constexpr int SMEM_BYTES = BAR_OFF + 8 * 8 + 16;
  static constexpr int HALF = D / 2;                // dims per dequant thread
  static constexpr int NCH_T = HALF / 16;           // 16-code chunks per dequant thread
  static constexpr int NB = D / 32;
  static constexpr int O_CHUNKS = D / 128;          // M=128 slices of O^T
  static_assert(D % 128 == 0, "tensor-core decode needs head_dim a multiple of 128");
  static_assert(16 + O_CHUNKS * kN <= kTmemCols, "TMEM columns");
};

__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // descriptor version for tcgen05; no swizzle, base offset 0
  return d;
}

// kind::f16 instruction descriptor: fp32 accumulate, bf16 A and B, M = 128, N = 16.
__device__ __forceinline__ uint32_t mma_idesc(bool a_mn_major, bool b_mn_major) {
  uint32_t d = 0;
  d |= 1u << 4;   // D: f32
  d |= 1u << 7;   // A: bf16
  d |= 1u << 10;  // B: bf16
  d |= static_cast<uint32_t>(a_mn_major) << 15;
  d |= static_cast<uint32_t>(b_mn_major) << 16;
  d |= static_cast<uint32_t>(kN >> 3) << 17;
  d |= static_cast<uint32_t>(kTile >> 4) << 24;
  return d;
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
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

// Item -> (sequence, group, split) through the shared table of per-sequence first items.
struct ItemPos {
  int32_t b, qg, split, nsplit;
};

__device__ __forceinline__ ItemPos locate(const int32_t* tab, const KParams& p, int32_t groups, int32_t C,
                                          int32_t item) {
  int lo = 0, hi = p.batch;  // first b with tab[b] > item
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (tab[mid] <= item) lo = mid + 1;
    else hi = mid;
  }
  ItemPos r;
  r.b = lo - 1;
  r.nsplit = (seq_pages(p, r.b) + C - 1) / C;
  const int32_t local = item - tab[r.b];
  r.qg = local / r.nsplit;
  r.split = local - r.qg * r.nsplit;
  return r;
}

// The flattened sequence of (item, tile) pairs a persistent CTA works through.
struct TileIter {
  int32_t item, i, ntiles, b, g, pg0, pg1, L;
  bool live;
};

__device__ __forceinline__ void tile_load_item(TileIter& t, const int32_t* tab, const KParams& p, int32_t groups,
                                               int32_t C) {
  const ItemPos ip = locate(tab, p, groups, C, t.item);
  t.b = ip.b;
  t.g = ip.qg;
  t.L = __ldg(p.seq_lens + ip.b);
  t.pg0 = ip.split * C;
  t.pg1 = min(t.pg0 + C, seq_pages(p, ip.b));
  t.ntiles = (t.pg1 - t.pg0 + kPagesPerTile - 1) / kPagesPerTile;
  t.i = 0;
}

__device__ __forceinline__ void tile_first(TileIter& t, const int32_t* tab, const KParams& p, int32_t groups,
                                           int32_t C, int32_t n_items) {
  t.item = blockIdx.x;
  t.live = t.item < n_items;
  if (t.live) tile_load_item(t, tab, p, groups, C);
}

__device__ __forceinline__ void tile_next(TileIter& t, const int32_t* tab, const KParams& p, int32_t groups,
                                          int32_t C, int32_t n_items) {
  if (++t.i < t.ntiles) return;
  t.item += gridDim.x;
  t.live = t.item < n_items;
  if (t.live) tile_load_item(t, tab, p, groups, C);
}

template <int D, int KIND>
__global__ void __launch_bounds__(kThreads, 1) decode_tc_kernel(KParams p) {
  using Cfg = TcCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* sK = smem + Cfg::K_OFF;
  uint8_t* sV = smem + Cfg::V_OFF;
  uint8_t* sQ = smem + Cfg::Q_OFF;
  uint8_t* sP = smem + Cfg::P_OFF;
  float* sRed = reinterpret_cast<float*>(smem + Cfg::RED_OFF);
  int32_t* sTab = reinterpret_cast<int32_t*>(smem + Cfg::TAB_OFF);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::BAR_OFF);
  uint64_t* bar_k_full = bars + 0;
  uint64_t* bar_v_full = bars + 1;
  uint64_t* bar_qk_done = bars + 2;
  uint64_t* bar_p_full = bars + 3;
  uint64_t* bar_pv_done = bars + 4;
  uint32_t* sTmem = reinterpret_cast<uint32_t*>(smem + Cfg::BAR_OFF + 8 * 8);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t groups = p.num_kv_heads;  // one item covers all G heads of a kv head
  const int32_t G = p.group;

  // ---- plan: split size, total items, first item of every sequence
  const Plan plan = make_plan(p, 0, -1);
  const int32_t C = plan.C;
  const int32_t n_items = plan.n_items;
  {
    // exclusive scan of items per sequence into sTab (batch <= kMaxPlanBatch, checked by the host)
    if (tid == 0) {
      int32_t run = 0;
      for (int32_t b = 0; b < p.batch; ++b) {
        sTab[b] = run;
        run += groups * ((seq_pages(p, b) + C - 1) / C);
      }
    }
  }
  if (tid == 0) {
    for (int i = 0; i < 5; ++i) mbar_init(&bars[i], (i == 0 || i == 1) ? kDwWarps : (i == 3 ? kSmWarps : 1));
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(sTmem)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  // zero P (heads beyond G stay zero) and Q padding rows once
  for (int i = tid; i < Cfg::P_BYTES / 16; i += kThreads) reinterpret_cast<uint4*>(sP)[i] = make_uint4(0, 0, 0, 0);
  for (int i = tid; i < Cfg::Q_BYTES / 16; i += kThreads) reinterpret_cast<uint4*>(sQ)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sTmem;
  const uint32_t tS = tmem;           // S^T: columns [0, 16)
  const uint32_t tO = tmem + 16;      // O^T slices: columns [16 + 16 c, 32 + 16 c)

  bool ok = true;
  uint32_t gtile = 0;  // tiles processed by this CTA so far (mbarrier phases)

  if (warp >= kSmWarps && warp < kMmaWarp) {
    // ===================================================================== dequant warps
    // Each thread owns half of one token row of the tile.  The codes of the next tile are requested
    // right after the current tile's K (resp. V) row has been written, one tile ahead of their use.
    const int dw = tid - kSmWarps * 32;  // 0..255
    const int tt = dw & (kTile - 1);     // token slot in the tile
    const int half = dw >> 7;            // which half of the row
    const int pi = tt / kPage, off = tt % kPage;
    TileIter cur;
    tile_first(cur, sTab, p, groups, C, n_items);
    uint4 kc[Cfg::NCH_T], vc[Cfg::NCH_T];
    uint16_t ksc[Cfg::NB / 2], vsc[Cfg::NB / 2];
    bool cvalid = false;
    int64_t rowK = 0, rowV = 0;
    auto rows_of = [&](const TileIter& t, bool& valid, int64_t& rk, int64_t& rv) {
      const int32_t pg = t.pg0 + t.i * kPagesPerTile + pi;
      int32_t phys = -1;
      if (pg < t.pg1) {
        phys = __ldg(p.block_table + static_cast<int64_t>(t.b) * p.max_pages + pg);
        if (phys >= p.num_pages) {
          set_status(p.status, kStatusBadPage);
          phys = -1;
        }
      }
      valid = phys >= 0 && (pg * kPage + off < t.L);
      rk = ((static_cast<int64_t>(phys) * 2 + 0) * p.num_kv_heads + t.g) * kPage + off;
      rv = ((static_cast<int64_t>(phys) * 2 + 1) * p.num_kv_heads + t.g) * kPage + off;
    };
    auto load_row = [&](bool valid, int64_t row, uint4 (&c)[Cfg::NCH_T], uint16_t (&sc)[Cfg::NB / 2]) {
      if (!valid) return;
      const uint4* src = reinterpret_cast<const uint4*>(p.codes + row * D + half * Cfg::HALF);
#pragma unroll
      for (int k = 0; k < Cfg::NCH_T; ++k) c[k] = __ldcs(src + k);
      const uint16_t* ss = reinterpret_cast<const uint16_t*>(p.scales) + row * Cfg::NB + half * (Cfg::NB / 2);
#pragma unroll
      for (int j = 0; j < Cfg::NB / 2; ++j) sc[j] = __ldg(ss + j);
    };
    auto store_row = [&](uint8_t* tile, bool valid, const uint4 (&c)[Cfg::NCH_T], const uint16_t (&sc)[Cfg::NB / 2]) {
      const uint32_t rowoff = (tt % 8) * 16 + (tt / 8) * Cfg::RS;
#pragma unroll
      for (int k = 0; k < Cfg::NCH_T; ++k) {
        uint32_t w[8];
        if (valid) {
          dequant16<KIND>(c[k], sc[k >> 1], w);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) w[e] = 0u;
        }
        const int d8 = (half * Cfg::HALF) / 8 + 2 * k;
        *reinterpret_cast<uint4*>(tile + rowoff + d8 * 128) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(tile + rowoff + (d8 + 1) * 128) = make_uint4(w[4], w[5], w[6], w[7]);
      }
    };
    if (cur.live) {
      rows_of(cur, cvalid, rowK, rowV);
      load_row(cvalid, rowK, kc, ksc);
      load_row(cvalid, rowV, vc, vsc);
    }
    while (cur.live && ok) {
      TileIter nxt = cur;
      tile_next(nxt, sTab, p, groups, C, n_items);
      bool nvalid = false;
      int64_t nK = 0, nV = 0;
      if (nxt.live) rows_of(nxt, nvalid, nK, nV);
      // the K tile (and, at an item's first tile, q) may be rewritten once the previous QK is done
      if (gtile > 0 && !mbar_wait_bounded(bar_qk_done, (gtile - 1) & 1)) { ok = false; break; }
      if (cur.i == 0) {
        const int32_t head0 = cur.g * G;
        for (int idx = dw; idx < G * (D / 8); idx += kDwWarps * 32) {
          const int h = idx / (D / 8), c8 = idx % (D / 8);
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(
              p.q + (static_cast<int64_t>(cur.b) * p.num_q_heads + head0 + h) * D + c8 * 8));
          *reinterpret_cast<uint4*>(sQ + (h % 8) * 16 + (h / 8) * Cfg::RS + c8 * 128) = v;
        }
      }
      store_row(sK, cvalid, kc, ksc);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar_k_full)) : "memory");
      if (nxt.live) load_row(nvalid, nK, kc, ksc);
      // the V tile may be rewritten once the previous PV is done
      if (gtile > 0 && !mbar_wait_bounded(bar_pv_done, (gtile - 1) & 1)) { ok = false; break; }
      store_row(sV, cvalid, vc, vsc);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar_v_full)) : "memory");
      if (nxt.live) load_row(nvalid, nV, vc, vsc);
      cur = nxt;
      cvalid = nvalid;
      ++gtile;
    }
  } else if (warp == kMmaWarp) {
    // ===================================================================== MMA issuer
    const uint32_t idesc_qk = mma_idesc(false, false);
    const uint32_t idesc_pv = mma_idesc(true, true);
    const uint32_t aK = smem_u32(sK), aV = smem_u32(sV), aQ = smem_u32(sQ), aP = smem_u32(sP);
    for (int32_t item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
      const ItemPos ip = locate(sTab, p, groups, C, item);
      const int32_t pg0 = ip.split * C;
      const int32_t pg1 = min(pg0 + C, seq_pages(p, ip.b));
      const int32_t ntiles = (pg1 - pg0 + kPagesPerTile - 1) / kPagesPerTile;
      for (int32_t i = 0; i < ntiles && ok; ++i, ++gtile) {
        if (!mbar_wait_bounded(bar_k_full, gtile & 1)) { ok = false; break; }
        tc_fence_after();
        if (lane == 0) {
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)
            mma_bf16(tS, smem_desc(aK + ks * 256, 128, Cfg::RS), smem_desc(aQ + ks * 256, 128, Cfg::RS), idesc_qk,
                     ks > 0);
          mma_commit(bar_qk_done);
        }
        __syncwarp();
        if (!mbar_wait_bounded(bar_v_full, gtile & 1)) { ok = false; break; }
        if (!mbar_wait_bounded(bar_p_full, gtile & 1)) { ok = false; break; }
        tc_fence_after();
        if (lane == 0) {
#pragma unroll
          for (int oc = 0; oc < Cfg::O_CHUNKS; ++oc)
#pragma unroll
            for (int ks = 0; ks < kTile / 16; ++ks)
              mma_bf16(tO + oc * kN, smem_desc(aV + oc * 16 * 128 + ks * 2 * Cfg::RS, Cfg::RS, 128),
                       smem_desc(aP + ks * 2 * 128, 128, 2048), idesc_pv, (i > 0 || ks > 0) ? 1u : 0u);
          mma_commit(bar_pv_done);
        }
        __syncwarp();
      }
    }
    // before TMEM is freed, every MMA this thread issued must have completed
    if (gtile > 0) (void)mbar_wait_bounded(bar_pv_done, (gtile - 1) & 1);
  } else {
    // ===================================================================== softmax warps
    const int tt = tid;  // token slot / O^T row / TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    for (int32_t item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
      const ItemPos ip = locate(sTab, p, groups, C, item);
      const int32_t L = __ldg(p.seq_lens + ip.b);
      const int32_t pg0 = ip.split * C;
      const int32_t pg1 = min(pg0 + C, seq_pages(p, ip.b));
      const int32_t ntiles = (pg1 - pg0 + kPagesPerTile - 1) / kPagesPerTile;
      float m_used[kN], l_t[kN];
#pragma unroll
      for (int h = 0; h < kN; ++h) {
        m_used[h] = -INFINITY;
        l_t[h] = 0.0f;
      }
      bool o_live = false;  // O holds contributions that a rescale must scale
      for (int32_t i = 0; i < ntiles && ok; ++i, ++gtile) {
        const int32_t pg = pg0 + i * kPagesPerTile + tt / kPage;
        bool valid = false;
        if (pg < pg1) {
          const int32_t phys = __ldg(p.block_table + static_cast<int64_t>(ip.b) * p.max_pages + pg);
          valid = phys >= 0 && phys < p.num_pages && (pg * kPage + tt % kPage < L);
        }
        if (!mbar_wait_bounded(bar_qk_done, gtile & 1)) { ok = false; break; }
        tc_fence_after();
        float s[16];
        tmem_ld16(tS + lane_base, s);
        float tmax[kN];
#pragma unroll
        for (int h = 0; h < kN; ++h) {
          s[h] = (valid && h < G) ? s[h] * p.score_scale : -INFINITY;
          float mx = s[h];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          tmax[h] = mx;
        }
        if (lane == 0) {
#pragma unroll
          for (int h = 0; h < kN; ++h) sRed[warp * kN + h] = tmax[h];
        }
        named_sync(1, kSmWarps * 32);
        float alpha[kN];
        bool rescale = false;
#pragma unroll
        for (int h = 0; h < kN; ++h) {
          float mx = sRed[h];
#pragma unroll
          for (int w = 1; w < kSmWarps; ++w) mx = fmaxf(mx, sRed[w * kN + h]);
          alpha[h] = 1.0f;
          if (mx > -INFINITY && (m_used[h] == -INFINITY || mx > m_used[h] + kLazyRescale)) {
            if (m_used[h] != -INFINITY) {
              alpha[h] = exp2f(m_used[h] - mx);
              rescale = true;
            }
            m_used[h] = mx;
          }
        }
        named_sync(1, kSmWarps * 32);  // sRed is rewritten next tile
        // P row of this token (bf16), and the matching fp32 row sums
        uint32_t pw[8];
#pragma unroll
        for (int h2 = 0; h2 < kN / 2; ++h2) {
          float pr[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int h = 2 * h2 + e;
            pr[e] = (s[h] == -INFINITY || m_used[h] == -INFINITY) ? 0.0f : exp2f(s[h] - m_used[h]);
          }
          pw[h2] = pack_bf16x2(pr[0], pr[1]);
          const float2 pb = unpack_bf16x2(pw[h2]);
          l_t[2 * h2] = fmaf(l_t[2 * h2], alpha[2 * h2], pb.x);
          l_t[2 * h2 + 1] = fmaf(l_t[2 * h2 + 1], alpha[2 * h2 + 1], pb.y);
        }
        // P and O may be touched only after the previous PV finished
        if (gtile > 0 && !mbar_wait_bounded(bar_pv_done, (gtile - 1) & 1)) { ok = false; break; }
        tc_fence_after();
        if (rescale && o_live) {
#pragma unroll
          for (int oc = 0; oc < Cfg::O_CHUNKS; ++oc) {
            float o[16];
            tmem_ld16(tO + oc * kN + lane_base, o);
#pragma unroll
            for (int h = 0; h < kN; ++h) o[h] *= alpha[h];
            tmem_st16(tO + oc * kN + lane_base, o);
          }
        }
        *reinterpret_cast<uint4*>(sP + (tt % 8) * 16 + (tt / 8) * 128) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
        if (G > 8)
          *reinterpret_cast<uint4*>(sP + 2048 + (tt % 8) * 16 + (tt / 8) * 128) =
              make_uint4(pw[4], pw[5], pw[6], pw[7]);
        o_live = true;
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar_p_full)) : "memory");
      }
      if (!ok) break;
      // ---- item epilogue: O^T rows -> partial accumulators; (m, l) per head
      if (!mbar_wait_bounded(bar_pv_done, (gtile - 1) & 1)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int oc = 0; oc < Cfg::O_CHUNKS; ++oc) {
        float o[16];
        tmem_ld16(tO + oc * kN + lane_base, o);
        const int d = oc * 128 + tt;
        for (int h = 0; h < G; ++h) p.part_acc[(static_cast<int64_t>(item) * G + h) * D + d] = o[h];
      }
#pragma unroll
      for (int h = 0; h < kN; ++h) {
        float v = l_t[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        l_t[h] = v;
      }
      if (lane == 0) {
#pragma unroll
        for (int h = 0; h < kN; ++h) sRed[warp * kN + h] = l_t[h];
      }
      named_sync(1, kSmWarps * 32);
      if (tt == 0) {  // m_used is identical in every softmax thread
#pragma unroll
        for (int h = 0; h < kN; ++h) {
          if (h < G) {
            float lsum = 0.0f;
#pragma unroll
            for (int w = 0; w < kSmWarps; ++w) lsum += sRed[w * kN + h];
            p.part_ml[(static_cast<int64_t>(item) * G + h) * 2 + 0] = m_used[h];
            p.part_ml[(static_cast<int64_t>(item) * G + h) * 2 + 1] = lsum;
          }
        }
      }
      tc_fence_before();
      named_sync(1, kSmWarps * 32);
    }
  }
  if (!ok) set_status(p.status, kStatusTimeout);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
}

template <int D>
kvq_status launch_tc_d(const DecodeArgs& a, cudaStream_t stream) {
  using Cfg = TcCfg<D>;
  auto kern = (a.kind == KVQ_FP8_E4M3) ? decode_tc_kernel<D, KVQ_FP8_E4M3> : decode_tc_kernel<D, KVQ_Q8_0>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) != cudaSuccess)
    return KVQ_ECUDA;
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const KParams p = make_kparams(a);
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(a.max_items, sms));
  kern<<<static_cast<unsigned>(grid), kThreads, Cfg::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ECUDA;
}

}  // namespace

bool decode_tc_supported(int32_t head_dim, int32_t v_dim, int32_t mla, int32_t group, int32_t batch) {
  if (mla || v_dim != head_dim) return false;
  if (head_dim != 128 && head_dim != 256) return false;
  return group >= 8 && group <= kN && batch <= kMaxPlanBatch;
}

kvq_status launch_decode_tc(const DecodeArgs& a, cudaStream_t stream) {
  if (a.head_dim == 128) return launch_tc_d<128>(a, stream);
  if (a.head_dim == 256) return launch_tc_d<256>(a, stream);
  return KVQ_EUNSUPPORTED;
}

}  // namespace kvq
