// kvq_decode_tc.cu -- split-K decode on the 5th-generation tensor cores (tcgen05) for wide GQA groups.
//
// "feat(kvcache): 8-bit KV cache (q8_0 / fp8_e4m3) behind --kv-cache-dtype", section "What": K and V
// are dequantized to bf16 before the dot (the scale varies along the reduction dim).  Here the
// dequantized bf16 tiles are the operands of tcgen05.mma, with fp32 accumulators in tensor memory.
// "feat(kvcache): 8-bit DSV4 window/compressed KV", section "Testing": split-k decode, masked -1 pages.
//
// With G = 8 or 16 query heads per kv head, QK^T and PV are small dense contractions.  They run
// swapped so that the 128 tokens of a tile are the MMA's M dimension:
//   S^T[128 tok][16] = Kd[128 tok][D] . Q[16][D]^T     (A = K tile in tensor memory; B = Q, K-major smem)
//   O^T[d][16]     += Vd^T[d][128 tok] . P[16][128]^T  (A = the V tile read MN-major; B = P, MN-major)
// (heads beyond G are zero rows of Q and P).  The V tile uses the canonical no-swizzle core-matrix
// layout  off(t, d) = (t%8)*16 + (t/8)*RS + (d%8)*2 + (d/8)*128  with RS = D*16, read MN-major with
// descriptor LBO = RS (token groups) and SBO = 128 (8-dim groups); Q uses the same form, K-major.
// The K tile lives in tensor memory (lane = token, two bf16 per column), double-buffered.
//
// One persistent CTA per SM, 14 warps (at most 4 per SM sub-partition):
//   warp 13     producer: one lane per page of a tile reads the block table and issues TMA copies of
//               the page's codes (a 5-D tensor map over the pool, one 4 KB box = 16 tokens x 128 code
//               bytes of K and of V, stored with the 128-byte swizzle) and 1-D bulk copies of its K and V
//               scales into a multi-stage staging ring; the tile's valid-token counts go with it.
//   warps 4-11  dequant: each thread owns half of a token row.  It reads its codes from the swizzled
//               staging rows (bank-conflict free: the 16-byte chunk index is XORed with token % 8),
//               dequantizes them exactly as on the CUDA-core path, K into tensor memory, V into shared.
//   warp 12     allocates TMEM; one thread issues every tcgen05.mma / tcgen05.commit, taking QK of the
//               next tile and PV of the oldest tile in whichever order their inputs become ready.
//   warps 0-3   softmax: TMEM lane = token; fp32 online softmax in the exp2 domain with lazy
//               rescaling: the running max of a head moves only when some token exceeds it by 2^8,
//               detected by one vote per tile; only then are the exact tile maxima reduced across
//               warps and O rescaled in TMEM.  Writes P (bf16, double-buffered); finally the partial.
// The roles hand tiles over with mbarriers; every wait is bounded (2 s) and reports a timeout in the
// workspace status word instead of hanging.
#include <cuda.h>  // CUtensorMap and its enums (the encoder is fetched from the driver at run time)
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
constexpr int kMmaWarp = kSmWarps + kDwWarps;          // warp 12
constexpr int kProdWarp = kMmaWarp + 1;                // warp 13
constexpr int kThreads = (kProdWarp + 1) * 32;         // 14 warps: at most 4 per sub-partition
constexpr int kDwThreads = kDwWarps * 32;
constexpr int kMaxPlanBatch = 2048;   // sequences whose item bases fit the shared table
constexpr float kLazyRescale = 8.0f;  // log2 headroom before the running max must move
constexpr int kTmemCols = 512;
constexpr int kBox = 2 * kPage * 128;  // one TMA box: 16 tokens x 128 code bytes, of K and of V

template <int D>
struct TcCfg {
  static constexpr int RS = D * 16;                 // bytes between 8-token groups of a tile
  static constexpr int TILE_BYTES = kTile * D * 2;  // one bf16 tile
  static constexpr int Q_BYTES = kN * D * 2;
  static constexpr int P_BYTES = kN * kTile * 2;   // one P buffer (two are kept)
  static constexpr int PARTS = kDwThreads / kTile;  // dequant threads per token row
  static constexpr int HALF = D / PARTS;            // dims per dequant thread
  static constexpr int NCH_T = HALF / 16;           // 16-code chunks per dequant thread
  static constexpr int NBT = HALF / 32;             // scale blocks per dequant thread
  static constexpr int NB = D / 32;
  static constexpr int NSL = D / 128;               // 128-byte column slices of a code row
  static constexpr int O_CHUNKS = D / 128;          // M=128 slices of O^T
  static constexpr int KCOLS = D / 2;               // TMEM columns of one K tile
  static constexpr int STAGES = (D == 128) ? 4 : 2; // staging ring depth (tiles)
  // one stage: codes [page][slice][kv][token][128 B] as TMA wrote them (128-byte swizzle), then the
  // scales [page][kv][token][NB] (fp16)
  static constexpr int SC_KV = kPage * NB * 2;      // scale bytes of one page, K or V
  static constexpr int ST_SC = kPagesPerTile * NSL * kBox;
  static constexpr int STAGE_BYTES = ST_SC + kPagesPerTile * 2 * SC_KV;
  static constexpr int ST_OFF = 0;                  // 1024-byte aligned: swizzle atoms
  static constexpr int V_OFF = ST_OFF + STAGES * STAGE_BYTES;
  static constexpr int Q_OFF = V_OFF + TILE_BYTES;
  static constexpr int P_OFF = Q_OFF + Q_BYTES;
  static constexpr int RED_OFF = P_OFF + 2 * P_BYTES;
  static constexpr int FLAG_OFF = RED_OFF + kSmWarps * kN * 4;  // per-warp "max moved" votes
  static constexpr int VAL_OFF = FLAG_OFF + 16;                  // token validity of each K buffer's tile
  static constexpr int META_OFF = VAL_OFF + 2 * kTile;           // valid tokens per page of each stage
  static constexpr int TAB_OFF = META_OFF + STAGES * kPagesPerTile * 4;
  static constexpr int NBARS = 9 + 2 * STAGES;
  static constexpr int BAR_OFF = TAB_OFF + kMaxPlanBatch * 4;
  static constexpr int SMEM_BYTES = BAR_OFF + NBARS * 8 + 16 + 1024;  // + slack to align the base
  static_assert(D % 128 == 0, "tensor-core decode needs head_dim a multiple of 128");
  static_assert(STAGE_BYTES % 1024 == 0, "stages keep the boxes 1024-byte aligned");
  static_assert(NCH_T % 2 == 0, "32 codes per tcgen05.st");
  static_assert(64 + 2 * KCOLS <= kTmemCols && 32 + O_CHUNKS * kN <= 64, "TMEM columns");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

// TMA tile load of one box of the code pool: the 128-byte slice `slice` of the rows `row`..`row+15`
// (row = kv head * 16 + token) of K and V in physical page `page`, completing on `bar`.
__device__ __forceinline__ void tma_load_codes(uint32_t dst, const CUtensorMap* map, int slice, int row, int page,
                                               uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, "
      "%6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(slice), "r"(row), "r"(0), "r"(page), "r"(smem_u32(bar))
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

__device__ __forceinline__ void mma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                                uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
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
  if (!t.live) return;
  if (++t.i < t.ntiles) return;
  t.item += gridDim.x;
  t.live = t.item < n_items;
  if (t.live) tile_load_item(t, tab, p, groups, C);
}

template <int D, int KIND, int GN>
__global__ void __launch_bounds__(kThreads, 1) decode_tc_kernel(const KParams p, const __grid_constant__ CUtensorMap tmap) {
  using Cfg = TcCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);  // swizzle atoms are 1024 B
  uint8_t* sV = smem + Cfg::V_OFF;
  uint8_t* sQ = smem + Cfg::Q_OFF;
  uint8_t* sP = smem + Cfg::P_OFF;  // [2] buffers
  uint8_t* sSt = smem + Cfg::ST_OFF;
  float* sRed = reinterpret_cast<float*>(smem + Cfg::RED_OFF);
  int32_t* sFlag = reinterpret_cast<int32_t*>(smem + Cfg::FLAG_OFF);
  int32_t* sTab = reinterpret_cast<int32_t*>(smem + Cfg::TAB_OFF);
  int32_t* sMeta = reinterpret_cast<int32_t*>(smem + Cfg::META_OFF);
  uint8_t* sValid = smem + Cfg::VAL_OFF;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::BAR_OFF);
  // Every barrier completes once per use of its buffer, so a waiter names an unambiguous phase.
  uint64_t* bar_k_full = bars + 0;   // [2] K tile in TMEM buffer b written (dequant warps)
  uint64_t* bar_qk_done = bars + 2;  // [2] QK into S buffer b (reading K buffer b) completed (commit)
  uint64_t* bar_p_full = bars + 4;   // [2] P buffer b written, S buffer b read, O rescaled (softmax warps)
  uint64_t* bar_pv_done = bars + 6;  // [2] PV that read P buffer b completed (commit)
  uint64_t* bar_v_full = bars + 8;   // V tile written (dequant warps), once per tile
  uint64_t* bar_full = bars + 9;               // [STAGES] stage s landed (producer arrival + bytes)
  uint64_t* bar_empty = bars + 9 + Cfg::STAGES;  // [STAGES] stage s read by every dequant warp
  uint32_t* sTmem = reinterpret_cast<uint32_t*>(smem + Cfg::BAR_OFF + Cfg::NBARS * 8);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t groups = p.num_kv_heads;  // one item covers all GN heads of a kv head

  // ---- plan: split size, total items, first item of every sequence
  const Plan plan = make_plan(p, 0, -1);
  const int32_t C = plan.C;
  const int32_t n_items = plan.n_items;
  if (tid == 0) {
    int32_t run = 0;
    for (int32_t b = 0; b < p.batch; ++b) {
      sTab[b] = run;
      run += groups * ((seq_pages(p, b) + C - 1) / C);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar_k_full[b], kDwWarps);
      mbar_init(&bar_qk_done[b], 1);
      mbar_init(&bar_p_full[b], kSmWarps);
      mbar_init(&bar_pv_done[b], 1);
    }
    mbar_init(bar_v_full, kDwWarps);
    for (int s = 0; s < Cfg::STAGES; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], kDwWarps);
    }
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(sTmem)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  for (int i = tid; i < 2 * Cfg::P_BYTES / 16; i += kThreads) reinterpret_cast<uint4*>(sP)[i] = make_uint4(0, 0, 0, 0);
  for (int i = tid; i < Cfg::Q_BYTES / 16; i += kThreads) reinterpret_cast<uint4*>(sQ)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sTmem;
  const uint32_t tS = tmem;       // S^T buffers: columns [16 b, 16 b + 16)
  const uint32_t tO = tmem + 32;  // O^T slices: columns [32 + 16 c, 48 + 16 c)
  const uint32_t tK = tmem + 64;  // K tiles: buffer b at columns [64 + b * KCOLS, 64 + (b + 1) * KCOLS)
  const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;

  bool ok = true;
  uint32_t gtile = 0;  // tiles processed by this CTA so far

  if (warp == kProdWarp) {
    // ===================================================================== producer
    // Lane pi (< 8) owns page pi of the tile: block-table entry, valid tokens, and its copies.
    const uint32_t st_base = smem_u32(sSt);
    TileIter t;
    tile_first(t, sTab, p, groups, C, n_items);
    uint32_t n = 0;  // tiles issued
    while (ok && t.live) {
      const int st = n % Cfg::STAGES;
      const uint32_t use = n / Cfg::STAGES;
      if (use > 0 && !mbar_wait_bounded(&bar_empty[st], (use - 1) & 1)) { ok = false; break; }
      int32_t phys = -1, nvalid = 0;
      if (lane < kPagesPerTile) {
        const int32_t pg = t.pg0 + t.i * kPagesPerTile + lane;
        if (pg < t.pg1) {
          phys = __ldg(p.block_table + static_cast<int64_t>(t.b) * p.max_pages + pg);
          if (phys >= p.num_pages) {
            set_status(p.status, kStatusBadPage);
            phys = -1;
          }
          if (phys >= 0) nvalid = min(kPage, t.L - pg * kPage);  // >= 1: pg < the sequence's page count
        }
      }
      const uint32_t bytes =
          __reduce_add_sync(0xffffffffu, phys >= 0 ? static_cast<uint32_t>(Cfg::NSL * kBox + 2 * Cfg::SC_KV) : 0u);
      int32_t nv[kPagesPerTile];
#pragma unroll
      for (int i = 0; i < kPagesPerTile; ++i) nv[i] = __shfl_sync(0xffffffffu, nvalid, i);
      if (lane == 0) {
#pragma unroll
        for (int i = 0; i < kPagesPerTile; ++i) sMeta[st * kPagesPerTile + i] = nv[i];
        mbar_arrive_expect_tx(&bar_full[st], bytes);  // releases sMeta with the stage
      }
      __syncwarp();
      if (phys >= 0) {
        const uint32_t dst = st_base + st * Cfg::STAGE_BYTES;
#pragma unroll
        for (int sl = 0; sl < Cfg::NSL; ++sl)
          tma_load_codes(dst + (lane * Cfg::NSL + sl) * kBox, &tmap, sl, t.g * kPage, phys, &bar_full[st]);
        const uint8_t* sk = reinterpret_cast<const uint8_t*>(p.scales) +
                            ((static_cast<int64_t>(phys) * 2 * p.num_kv_heads + t.g) * kPage) * Cfg::NB * 2;
        const uint8_t* sv = sk + static_cast<int64_t>(p.num_kv_heads) * Cfg::SC_KV;
        uint8_t* sdst = sSt + st * Cfg::STAGE_BYTES + Cfg::ST_SC + lane * 2 * Cfg::SC_KV;
        bulk_g2s(sdst, sk, Cfg::SC_KV, &bar_full[st]);
        bulk_g2s(sdst + Cfg::SC_KV, sv, Cfg::SC_KV, &bar_full[st]);
      }
      tile_next(t, sTab, p, groups, C, n_items);
      ++n;
    }
    // no copy may still be in flight when the CTA exits
    for (uint32_t j = 1; j <= n && j <= static_cast<uint32_t>(Cfg::STAGES); ++j) {
      const uint32_t m = n - j;
      (void)mbar_wait_bounded(&bar_full[m % Cfg::STAGES], (m / Cfg::STAGES) & 1);
    }
  } else if (warp >= kSmWarps && warp < kMmaWarp) {
    // ===================================================================== dequant warps
    const int dw = tid - kSmWarps * 32;   // 0 .. kDwThreads-1
    const int tt = dw & (kTile - 1);      // token slot = TMEM lane (warp & 3 selects the lane quarter)
    const int part = dw / kTile;          // which part of the row
    const int pi = tt / kPage, off = tt % kPage;
    const int swz = off & 7;              // 128-byte swizzle phase of this token's staging rows
    const uint32_t voff = (tt % 8) * 16 + (tt / 8) * Cfg::RS;
    // staging address of 16-code chunk k of this thread's part of the K (kv = 0) or V (kv = 1) row
    auto chunk_addr = [&](const uint8_t* sb, int kv, int k) -> const uint4* {
      const int c = part * Cfg::NCH_T + k;  // chunk index along the row
      const int sl = c / 8, cw = c % 8;
      return reinterpret_cast<const uint4*>(sb + (pi * Cfg::NSL + sl) * kBox + (kv * kPage + off) * 128 +
                                            ((cw ^ swz) * 16));
    };
    TileIter tc;
    tile_first(tc, sTab, p, groups, C, n_items);
    while (ok && tc.live) {
      const int st = gtile % Cfg::STAGES;  // staging stage
      const int kb = gtile & 1;            // K buffer = S / P buffer = validity slot of this tile
      if (!mbar_wait_bounded(&bar_full[st], (gtile / Cfg::STAGES) & 1)) { ok = false; break; }
      const uint8_t* sb = sSt + st * Cfg::STAGE_BYTES;
      const bool v_ok = off < sMeta[st * kPagesPerTile + pi];
      const uint16_t* scl = reinterpret_cast<const uint16_t*>(sb + Cfg::ST_SC + pi * 2 * Cfg::SC_KV) +
                            off * Cfg::NB + part * Cfg::NBT;  // K scales; V scales SC_KV bytes on
      // ---- K tile into TMEM buffer kb, once the QK that last read that buffer is complete
      if (gtile >= 2 && !mbar_wait_bounded(&bar_qk_done[kb], ((gtile >> 1) - 1) & 1)) { ok = false; break; }
      if (tc.i == 0) {
        // this item's q rows; the previous tile's QK must have read the old ones
        if (gtile >= 1 && !mbar_wait_bounded(&bar_qk_done[(gtile - 1) & 1], ((gtile - 1) >> 1) & 1)) {
          ok = false;
          break;
        }
        const int32_t head0 = tc.g * p.group;
        for (int idx = dw; idx < GN * (D / 8); idx += kDwThreads) {
          const int h = idx / (D / 8), c8 = idx % (D / 8);
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(
              p.q + (static_cast<int64_t>(tc.b) * p.num_q_heads + head0 + h) * D + c8 * 8));
          *reinterpret_cast<uint4*>(sQ + (h % 8) * 16 + (h / 8) * Cfg::RS + c8 * 128) = v;
        }
        fence_proxy_async_smem();
      }
      // the validity slot kb was last read by the softmax of tile gtile - 2
      if (gtile >= 2 && !mbar_wait_bounded(&bar_p_full[kb], ((gtile >> 1) - 1) & 1)) { ok = false; break; }
      if (part == 0) sValid[kb * kTile + tt] = v_ok ? 1 : 0;  // published to the softmax warps with k_full
      {
#pragma unroll
        for (int k2 = 0; k2 < Cfg::NCH_T / 2; ++k2) {  // 32 codes -> 16 TMEM columns per tcgen05.st
          uint32_t w[16];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int k = 2 * k2 + h;
            if (v_ok) {
              uint32_t ww[8];
              dequant16<KIND>(*chunk_addr(sb, 0, k), scl[k >> 1], ww);
#pragma unroll
              for (int e = 0; e < 8; ++e) w[8 * h + e] = ww[e];
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e) w[8 * h + e] = 0u;
            }
          }
          tmem_st16u(tK + kb * Cfg::KCOLS + lane_base + part * (Cfg::HALF / 2) + k2 * 16, w);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&bar_k_full[kb])) : "memory");
      }
      // ---- V tile into shared memory, once the previous PV is complete
      if (gtile >= 1 && !mbar_wait_bounded(&bar_pv_done[(gtile - 1) & 1], ((gtile - 1) >> 1) & 1)) { ok = false; break; }
      {
        const uint16_t* vs = scl + Cfg::SC_KV / 2;
#pragma unroll
        for (int k = 0; k < Cfg::NCH_T; ++k) {
          uint32_t w[8];
          if (v_ok) {
            dequant16<KIND>(*chunk_addr(sb, 1, k), vs[k >> 1], w);
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) w[e] = 0u;
          }
          const int d8 = (part * Cfg::HALF) / 8 + 2 * k;
          *reinterpret_cast<uint4*>(sV + voff + d8 * 128) = make_uint4(w[0], w[1], w[2], w[3]);
          *reinterpret_cast<uint4*>(sV + voff + (d8 + 1) * 128) = make_uint4(w[4], w[5], w[6], w[7]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar_v_full)) : "memory");
          asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&bar_empty[st])) : "memory");
        }
      }
      tile_next(tc, sTab, p, groups, C, n_items);
      ++gtile;
    }
  } else if (warp == kMmaWarp) {
    // ===================================================================== MMA issue (lane 0)
    // QK(nq) needs K tile nq in TMEM and S buffer nq&1 read by the softmax of tile nq-2; PV(np) needs
    // V tile np and P tile np.  Whichever is ready is issued first; lane 0 polls, the warp follows.
    const uint32_t idesc_qk = mma_idesc(false, false);
    const uint32_t idesc_pv = mma_idesc(true, true);
    const uint32_t aV = smem_u32(sV), aQ = smem_u32(sQ), aP = smem_u32(sP);
    TileIter tq, tp;  // next tile to QK; next tile to PV
    tile_first(tq, sTab, p, groups, C, n_items);
    tp = tq;
    uint32_t nq = 0, np = 0;  // tiles QK'd / PV'd
    uint64_t idle_since = 0;
    while (tp.live) {
      bool progressed = false;
      if (tq.live && nq < np + 2) {
        const int b = nq & 1;
        int ready = 0;
        if (lane == 0)
          ready = mbar_test_wait(&bar_k_full[b], (nq >> 1) & 1) &&
                  (nq < 2 || mbar_test_wait(&bar_p_full[b], ((nq >> 1) - 1) & 1));
        if (__shfl_sync(0xffffffffu, ready, 0)) {
          tc_fence_after();
          if (lane == 0) {
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
              mma_bf16_tmem_a(tS + b * kN, tK + b * Cfg::KCOLS + ks * 8, smem_desc(aQ + ks * 256, 128, Cfg::RS),
                              idesc_qk, ks > 0);
            mma_commit(&bar_qk_done[b]);
          }
          __syncwarp();
          ++nq;
          tile_next(tq, sTab, p, groups, C, n_items);
          progressed = true;
        }
      }
      if (np < nq) {
        const int b = np & 1;
        int ready = 0;
        if (lane == 0)
          ready = mbar_test_wait(bar_v_full, np & 1) && mbar_test_wait(&bar_p_full[b], (np >> 1) & 1);
        if (__shfl_sync(0xffffffffu, ready, 0)) {
          tc_fence_after();
          if (lane == 0) {
#pragma unroll
            for (int oc = 0; oc < Cfg::O_CHUNKS; ++oc)
#pragma unroll
              for (int ks = 0; ks < kTile / 16; ++ks)
                mma_bf16(tO + oc * kN, smem_desc(aV + oc * 16 * 128 + ks * 2 * Cfg::RS, Cfg::RS, 128),
                         smem_desc(aP + b * Cfg::P_BYTES + ks * 2 * 128, 128, 2048), idesc_pv,
                         (tp.i > 0 || ks > 0) ? 1u : 0u);
            mma_commit(&bar_pv_done[b]);
          }
          __syncwarp();
          ++np;
          tile_next(tp, sTab, p, groups, C, n_items);
          progressed = true;
        }
      }
      if (progressed) {
        idle_since = 0;
      } else {
        const uint64_t now = global_timer_ns();
        if (idle_since == 0) idle_since = now;
        else if (now - idle_since > kWaitLimitNs) { ok = false; break; }
      }
    }
    // before TMEM is freed, every MMA issued must have completed (in order: the last commit implies all)
    if (np > 0) (void)mbar_wait_bounded(&bar_pv_done[(np - 1) & 1], ((np - 1) >> 1) & 1);
    if (nq > np) (void)mbar_wait_bounded(&bar_qk_done[(nq - 1) & 1], ((nq - 1) >> 1) & 1);
  } else {
    // ===================================================================== softmax warps
    const int tt = tid;  // token slot / O^T row / TMEM lane
    for (int32_t item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
      const ItemPos ip = locate(sTab, p, groups, C, item);
      const int32_t pg0 = ip.split * C;
      const int32_t pg1 = min(pg0 + C, seq_pages(p, ip.b));
      const int32_t ntiles = (pg1 - pg0 + kPagesPerTile - 1) / kPagesPerTile;
      float m_used[GN], l_t[GN];
#pragma unroll
      for (int h = 0; h < GN; ++h) {
        m_used[h] = -INFINITY;
        l_t[h] = 0.0f;
      }
      bool o_live = false;  // O holds contributions that a rescale must scale
      for (int32_t i = 0; i < ntiles && ok; ++i, ++gtile) {
        const int b = gtile & 1;
        if (!mbar_wait_bounded(&bar_qk_done[b], (gtile >> 1) & 1)) { ok = false; break; }
        // token validity was published before k_full[b] completed (already complete: QK followed it)
        if (!mbar_wait_bounded(&bar_k_full[b], (gtile >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
        const bool valid = sValid[b * kTile + tt] != 0;
        float s[16];
        tmem_ld16(tS + b * kN + lane_base, s);
        bool moved = false;
#pragma unroll
        for (int h = 0; h < GN; ++h) {
          s[h] = valid ? s[h] * p.score_scale : -INFINITY;
          moved |= (s[h] > -INFINITY) && (m_used[h] == -INFINITY || s[h] > m_used[h] + kLazyRescale);
        }
        // does any token of the tile move any head's running max?  (one vote per warp, one barrier)
        const int wv = __any_sync(0xffffffffu, moved);
        if (lane == 0) sFlag[warp] = wv;
        named_sync(1, kSmWarps * 32);
        const bool any_moved = (sFlag[0] | sFlag[1] | sFlag[2] | sFlag[3]) != 0;
        float alpha[GN];
        bool rescale = false;
#pragma unroll
        for (int h = 0; h < GN; ++h) alpha[h] = 1.0f;
        if (any_moved) {  // uniform branch: exact tile maxima, then the new running max per head
          named_sync(1, kSmWarps * 32);  // sFlag has been read by every warp
#pragma unroll
          for (int h = 0; h < GN; ++h) {
            float mx = s[h];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            if (lane == 0) sRed[warp * kN + h] = mx;
          }
          named_sync(1, kSmWarps * 32);
#pragma unroll
          for (int h = 0; h < GN; ++h) {
            float mx = sRed[h];
#pragma unroll
            for (int w = 1; w < kSmWarps; ++w) mx = fmaxf(mx, sRed[w * kN + h]);
            if (mx > -INFINITY && (m_used[h] == -INFINITY || mx > m_used[h] + kLazyRescale)) {
              if (m_used[h] != -INFINITY) {
                alpha[h] = exp2f(m_used[h] - mx);
                rescale = true;
              }
              m_used[h] = mx;
            }
          }
        }
        named_sync(1, kSmWarps * 32);  // sFlag / sRed are rewritten next tile
        // P row of this token (bf16), and the row sums of exactly those bf16 values
        uint32_t pw[GN / 2];
#pragma unroll
        for (int h2 = 0; h2 < GN / 2; ++h2) {
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
        // P buffer b is free once the PV two tiles back has read it
        if (gtile >= 2 && !mbar_wait_bounded(&bar_pv_done[b], ((gtile >> 1) - 1) & 1)) { ok = false; break; }
        if (rescale && o_live) {  // O must hold every earlier PV before it is scaled
          if (!mbar_wait_bounded(&bar_pv_done[(gtile - 1) & 1], ((gtile - 1) >> 1) & 1)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int oc = 0; oc < Cfg::O_CHUNKS; ++oc) {
            float o[16];
            tmem_ld16(tO + oc * kN + lane_base, o);
#pragma unroll
            for (int h = 0; h < GN; ++h) o[h] *= alpha[h];
            tmem_st16(tO + oc * kN + lane_base, o);
          }
        }
        uint8_t* pb = sP + b * Cfg::P_BYTES;
        *reinterpret_cast<uint4*>(pb + (tt % 8) * 16 + (tt / 8) * 128) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
        if constexpr (GN > 8)
          *reinterpret_cast<uint4*>(pb + 2048 + (tt % 8) * 16 + (tt / 8) * 128) =
              make_uint4(pw[4], pw[5], pw[6], pw[7]);
        o_live = true;
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&bar_p_full[b])) : "memory");
      }
      if (!ok) break;
      // ---- item epilogue: O^T rows -> partial accumulators; (m, l) per head
      if (!mbar_wait_bounded(&bar_pv_done[(gtile - 1) & 1], ((gtile - 1) >> 1) & 1)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int oc = 0; oc < Cfg::O_CHUNKS; ++oc) {
        float o[16];
        tmem_ld16(tO + oc * kN + lane_base, o);
        const int d = oc * 128 + tt;
#pragma unroll
        for (int h = 0; h < GN; ++h) p.part_acc[(static_cast<int64_t>(item) * GN + h) * D + d] = o[h];
      }
#pragma unroll
      for (int h = 0; h < GN; ++h) {
        float v = l_t[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) sRed[warp * kN + h] = v;
      }
      named_sync(1, kSmWarps * 32);
      if (tt == 0) {  // m_used is identical in every softmax thread
#pragma unroll
        for (int h = 0; h < GN; ++h) {
          float lsum = 0.0f;
#pragma unroll
          for (int w = 0; w < kSmWarps; ++w) lsum += sRed[w * kN + h];
          p.part_ml[(static_cast<int64_t>(item) * GN + h) * 2 + 0] = m_used[h];
          p.part_ml[(static_cast<int64_t>(item) * GN + h) * 2 + 1] = lsum;
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

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once through the runtime (no link against libcuda).
EncodeTiledFn tensor_map_encoder() {
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
// kv, page); a box is one slice of the 16 rows of one head, for K and V: 4 KB, 128-byte swizzled.
template <int D>
bool encode_code_map(CUtensorMap* map, const DecodeArgs& a) {
  const EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t H = static_cast<cuuint64_t>(a.num_kv_heads);
  const cuuint64_t pages = static_cast<cuuint64_t>(std::max<int64_t>(a.num_pages, 1));  // no copy reads past it
  const cuuint64_t dims[5] = {128, D / 128, H * kPage, 2, pages};
  const cuuint64_t strides[4] = {128, D, H * kPage * D, 2 * H * kPage * D};
  const cuuint32_t box[5] = {128, 1, kPage, 2, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<uint8_t*>(a.codes), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
kvq_status launch_tc_d(const DecodeArgs& a, cudaStream_t stream) {
  using Cfg = TcCfg<D>;
  const bool g16 = (a.num_q_heads / a.num_kv_heads) == 16;
  auto kern = (a.kind == KVQ_FP8_E4M3) ? (g16 ? decode_tc_kernel<D, KVQ_FP8_E4M3, 16> : decode_tc_kernel<D, KVQ_FP8_E4M3, 8>)
                                       : (g16 ? decode_tc_kernel<D, KVQ_Q8_0, 16> : decode_tc_kernel<D, KVQ_Q8_0, 8>);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) != cudaSuccess)
    return KVQ_ECUDA;
  CUtensorMap map;
  if (!encode_code_map<D>(&map, a)) return KVQ_ECUDA;
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const KParams p = make_kparams(a);
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(a.max_items, sms));
  kern<<<static_cast<unsigned>(grid), kThreads, Cfg::SMEM_BYTES, stream>>>(p, map);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ECUDA;
}

}  // namespace

bool decode_tc_supported(int32_t head_dim, int32_t v_dim, int32_t mla, int32_t group, int32_t batch) {
  if (mla || v_dim != head_dim) return false;
  if (head_dim != 128 && head_dim != 256) return false;
  return (group == 8 || group == 16) && batch <= kMaxPlanBatch;
}

kvq_status launch_decode_tc(const DecodeArgs& a, cudaStream_t stream) {
  if (a.head_dim == 128) return launch_tc_d<128>(a, stream);
  if (a.head_dim == 256) return launch_tc_d<256>(a, stream);
  return KVQ_EUNSUPPORTED;
}

}  // namespace kvq
