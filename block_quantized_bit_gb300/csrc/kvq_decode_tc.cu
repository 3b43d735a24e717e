// kvq_decode_tc.cu -- split-K decode on the 5th-generation tensor cores (tcgen05) for wide GQA groups.
//
// "feat(kvcache): 8-bit KV cache (q8_0 / fp8_e4m3) behind --kv-cache-dtype", section "What": K and V
// are dequantized to bf16 before the dot (the scale varies along the reduction dim).  Here the
// dequantized bf16 tiles are the operands of tcgen05.mma, with fp32 accumulators in tensor memory.
// "feat(kvcache): 8-bit DSV4 window/compressed KV", section "Testing": split-k decode, masked -1 pages.
//
// With G <= 16 query heads per kv head (padded to the MMA N = 16), QK^T and PV are small dense
// contractions.  They run swapped so that the 128 tokens of a tile are the MMA's M dimension:
//   S^T[128 tok][16] = Kd[128 tok][D] . Q[16][D]^T     (A = K tile in tensor memory; B = Q, K-major smem)
//   O^T[d][16]     += Vd^T[d][128 tok] . P[16][128]^T  (A = the V tile read MN-major; B = P, MN-major)
// (heads beyond G are zero rows of Q and P).  The V tile uses the canonical no-swizzle core-matrix
// layout  off(t, d) = (t%8)*16 + (t/8)*RS + (d%8)*2 + (d/8)*128  with RS = D*16, read MN-major with
// descriptor LBO = RS (token groups) and SBO = 128 (8-dim groups); Q uses the same form, K-major.
// The K tile lives in tensor memory (lane = token, two bf16 per column), double-buffered.
//
// One persistent CTA per SM, 23 warps (80 registers each):
//   warps 21-22 producers, one for K and one for V: one lane per page of a tile reads the block table
//               and issues TMA copies of the page's codes (a 5-D tensor map over the pool, one 2 KB box
//               = 16 tokens x 128 code bytes, stored with the 128-byte swizzle) and a 1-D bulk copy of
//               its scales into that producer's multi-stage staging ring; the tile's valid-token counts
//               go with it.
//   warps 4-19  dequant: each thread owns a quarter of a token row.  It reads its codes from the
//               swizzled staging rows (bank-conflict free: the 16-byte chunk index is XORed with
//               token % 8), dequantizes them exactly as on the CUDA-core path, K into tensor memory, V
//               into shared.  Its loops are deliberately not fully unrolled: with five roles sharing
//               each SM sub-partition, instruction-cache misses cost more than the loop overhead.
//               Sixteen dequant warps (instead of eight) and the elected-lane MMA issue below together
//               took the long-context decode from 526 to 502 us; either alone gained nothing, because
//               the other then paced the tile.
//   warp 20     allocates TMEM and issues every tcgen05.mma / tcgen05.commit (one lane elected by the
//               converged warp), taking QK of the next tile and PV of the oldest tile in whichever
//               order their inputs become ready.
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
#include "kvq_tc.cuh"

namespace kvq {
namespace {

constexpr int kTile = 128;        // tokens per tile (8 pages)
constexpr int kPagesPerTile = kTile / kPage;
constexpr int kN = 16;            // MMA N: query heads, padded
constexpr int kSmWarps = 4;
constexpr int kDwWarps = 16;
constexpr int kMmaWarp = kSmWarps + kDwWarps;          // warp 20
constexpr int kProdWarp = kMmaWarp + 1;                // warps 21 (K ring) and 22 (V ring)
constexpr int kThreads = (kProdWarp + 2) * 32;         // 23 warps
constexpr int kDwThreads = kDwWarps * 32;
constexpr int kMaxPlanBatch = 2048;   // sequences whose item bases fit the shared table
constexpr float kLazyRescale = 8.0f;  // log2 headroom before the running max must move
// running max of a head before its first valid score: finite, so that s * scale - m stays finite and the
// tile's vote fires; padded heads (G .. GN - 1) hold +inf, so that their probabilities are 2^-inf = 0
constexpr float kNoMax = -1.0e30f;
constexpr int kTmemCols = 512;
constexpr int kBox = kPage * 128;  // one TMA box: 16 tokens x 128 code bytes of K or of V

// 2^x by the hardware approximation, subnormal results flushed to 0 (far below the bf16 rounding of P);
// 2^-inf = 0.
__device__ __forceinline__ float tc_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

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
  static constexpr int STAGES = (D == 128) ? 4 : 2; // depth of each staging ring (tiles)
  // one ring slot (K ring and V ring alike): codes [page][slice][token][128 B] as TMA wrote them
  // (128-byte swizzle), then the scales [page][token][NB] (fp16)
  static constexpr int SC_KV = kPage * NB * 2;      // scale bytes of one page
  static constexpr int SL_SC = kPagesPerTile * NSL * kBox;
  static constexpr int SLOT_BYTES = SL_SC + kPagesPerTile * SC_KV;
  static constexpr int KR_OFF = 0;                  // 1024-byte aligned: swizzle atoms
  static constexpr int VR_OFF = KR_OFF + STAGES * SLOT_BYTES;
  static constexpr int V_OFF = VR_OFF + STAGES * SLOT_BYTES;
  static constexpr int Q_OFF = V_OFF + TILE_BYTES;
  static constexpr int P_OFF = Q_OFF + Q_BYTES;
  static constexpr int RED_OFF = P_OFF + 2 * P_BYTES;
  static constexpr int FLAG_OFF = RED_OFF + kSmWarps * kN * 4;  // per-warp "max moved" votes [2 tile parities]
  static constexpr int VAL_OFF = FLAG_OFF + 2 * 16;              // token validity of each K buffer's tile
  static constexpr int META_OFF = VAL_OFF + 2 * kTile;           // valid tokens per page: [ring][slot][page]
  static constexpr int TAB_OFF = META_OFF + 2 * STAGES * kPagesPerTile * 4;
  static constexpr int NBARS = 11 + 4 * STAGES;
  static constexpr int BAR_OFF = TAB_OFF + kMaxPlanBatch * 4;
  static constexpr int SMEM_BYTES = BAR_OFF + NBARS * 8 + 16 + 1024;  // + slack to align the base
  static_assert(D % 128 == 0, "tensor-core decode needs head_dim a multiple of 128");
  static_assert(SLOT_BYTES % 1024 == 0, "slots keep the boxes 1024-byte aligned");
  static_assert(NCH_T % 2 == 0, "32 codes per tcgen05.st");
  static_assert(96 + 2 * KCOLS <= kTmemCols && O_CHUNKS * kN <= 32, "TMEM columns");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

// This thread's NBT (<= 4) block scales of a staged row, in one load: 16 bits each, lowest first.  A
// 2-byte load per scale would hit each bank four times (the token rows are 16 bytes apart).
template <int NBT>
__device__ __forceinline__ uint64_t load_scales(const uint8_t* p) {
  static_assert(NBT == 1 || NBT == 2 || NBT == 4, "scale blocks per dequant thread");
  if (NBT == 1) return *reinterpret_cast<const uint16_t*>(p);
  if (NBT == 4) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    return static_cast<uint64_t>(v.x) | (static_cast<uint64_t>(v.y) << 32);
  }
  return *reinterpret_cast<const uint32_t*>(p);
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

// Which of the two O accumulators an item uses: items alternate within a CTA.
__device__ __forceinline__ int item_obuf(int32_t item) { return ((item - static_cast<int32_t>(blockIdx.x)) / gridDim.x) & 1; }

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
  uint8_t* sKr = smem + Cfg::KR_OFF;  // K ring
  uint8_t* sVr = smem + Cfg::VR_OFF;  // V ring
  float* sRed = reinterpret_cast<float*>(smem + Cfg::RED_OFF);
  int32_t* sFlag = reinterpret_cast<int32_t*>(smem + Cfg::FLAG_OFF);
  int32_t* sTab = reinterpret_cast<int32_t*>(smem + Cfg::TAB_OFF);
  int32_t* sMeta = reinterpret_cast<int32_t*>(smem + Cfg::META_OFF);  // [ring][slot][page]
  uint8_t* sValid = smem + Cfg::VAL_OFF;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::BAR_OFF);
  // Every barrier completes once per use of its buffer, so a waiter names an unambiguous phase.
  uint64_t* bar_k_full = bars + 0;   // [2] K tile in TMEM buffer b written (dequant warps)
  uint64_t* bar_qk_done = bars + 2;  // [2] QK into S buffer b (reading K buffer b) completed (commit)
  uint64_t* bar_p_full = bars + 4;   // [2] P buffer b written, S buffer b read, O rescaled (softmax warps)
  uint64_t* bar_pv_done = bars + 6;  // [2] PV that read P buffer b completed (commit)
  uint64_t* bar_v_full = bars + 8;   // V tile written (dequant warps), once per tile
  uint64_t* bar_pv_lo = bars + 9;    // [2] the PV MMAs of O^T slice 0 (d < 128) reading P buffer b completed
  uint64_t* bar_full = bars + 11;                     // [ring][STAGES] slot landed (producer arrival + bytes)
  uint64_t* bar_empty = bars + 11 + 2 * Cfg::STAGES;  // [ring][STAGES] slot read by every dequant warp
  uint32_t* sTmem = reinterpret_cast<uint32_t*>(smem + Cfg::BAR_OFF + Cfg::NBARS * 8);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t groups = p.num_kv_heads;  // one item covers all G heads of a kv head
  const int32_t G = p.group;              // query heads per kv head, 1 <= G <= GN (the rest is padding)

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
      mbar_init(&bar_pv_lo[b], 1);
    }
    mbar_init(bar_v_full, kDwWarps);
    for (int s = 0; s < 2 * Cfg::STAGES; ++s) {
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
  const uint32_t tO = tmem + 32;  // O^T of item parity o, slice c: columns [32 + 32 o + 16 c, +16)
  const uint32_t tK = tmem + 96;  // K tiles: buffer b at columns [96 + b * KCOLS, 96 + (b + 1) * KCOLS)
  const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;

  // the merge kernel that follows may launch now; it waits for this grid to complete before it reads
  asm volatile("griddepcontrol.launch_dependents;");
  bool ok = true;
  uint32_t gtile = 0;  // tiles processed by this CTA so far

  if (warp >= kProdWarp) {
    // ===================================================================== producers
    // Warp 21 fills the K ring, warp 22 the V ring, each running ahead on its own ring.  Lane pi (< 8)
    // owns page pi of a tile: block-table entry (requested one tile ahead), valid tokens, its copies.
    const int kv = warp - kProdWarp;
    uint8_t* ring_base = kv ? sVr : sKr;
    TileIter t;
    tile_first(t, sTab, p, groups, C, n_items);
    auto page_entry = [&](const TileIter& ti) -> int32_t {
      if (!ti.live || lane >= kPagesPerTile) return -1;
      const int32_t pg = ti.pg0 + ti.i * kPagesPerTile + lane;
      return pg < ti.pg1 ? bt_entry(p, ti.b, pg) : -1;
    };
    uint32_t n = 0;              // tiles issued
    int32_t bt = page_entry(t);  // block-table entry of tile n
    while (ok && t.live) {
      int32_t phys = bt, nvalid = 0;
      if (phys >= p.num_pages) {
        set_status(p.status, kStatusBadPage);
        phys = -1;
      }
      if (phys >= 0) nvalid = min(kPage, t.L - (t.pg0 + t.i * kPagesPerTile + lane) * kPage);  // >= 1
      TileIter nx = t;
      tile_next(nx, sTab, p, groups, C, n_items);
      bt = page_entry(nx);
      const int sl = n % Cfg::STAGES;
      const int ring = kv * Cfg::STAGES + sl;
      const uint32_t use = n / Cfg::STAGES;
      if (use > 0 && !mbar_wait_bounded(&bar_empty[ring], (use - 1) & 1)) { ok = false; break; }
      constexpr uint32_t kPageBytes = Cfg::NSL * kBox + (KindTraits<KIND>::kScaled ? Cfg::SC_KV : 0);
      const uint32_t bytes = __reduce_add_sync(0xffffffffu, phys >= 0 ? kPageBytes : 0u);
      int32_t nv[kPagesPerTile];
#pragma unroll
      for (int i = 0; i < kPagesPerTile; ++i) nv[i] = __shfl_sync(0xffffffffu, nvalid, i);
      if (lane == 0) {
#pragma unroll
        for (int i = 0; i < kPagesPerTile; ++i) sMeta[ring * kPagesPerTile + i] = nv[i];
        mbar_arrive_expect_tx(&bar_full[ring], bytes);  // releases the page counts with the slot
      }
      __syncwarp();
      if (phys >= 0) {
        uint8_t* slot = ring_base + sl * Cfg::SLOT_BYTES;
#pragma unroll
        for (int c = 0; c < Cfg::NSL; ++c)
          tma_load_codes(smem_u32(slot + (lane * Cfg::NSL + c) * kBox), &tmap, c, t.g * kPage, kv, phys,
                         &bar_full[ring]);
        if (KindTraits<KIND>::kScaled) {  // an unscaled pool has codes only
          const uint8_t* src = reinterpret_cast<const uint8_t*>(p.scales) +
                               ((static_cast<int64_t>(phys) * 2 + kv) * p.num_kv_heads + t.g) * Cfg::SC_KV;
          bulk_g2s(slot + Cfg::SL_SC + lane * Cfg::SC_KV, src, Cfg::SC_KV, &bar_full[ring]);
        }
      }
      t = nx;
      ++n;
    }
    // no copy may still be in flight when the CTA exits
    for (uint32_t j = 1; j <= n && j <= static_cast<uint32_t>(Cfg::STAGES); ++j) {
      const uint32_t m = n - j;
      (void)mbar_wait_bounded(&bar_full[kv * Cfg::STAGES + m % Cfg::STAGES], (m / Cfg::STAGES) & 1);
    }
  } else if (warp >= kSmWarps && warp < kMmaWarp) {
    // ===================================================================== dequant warps
    const int dw = tid - kSmWarps * 32;   // 0 .. kDwThreads-1
    const int tt = dw & (kTile - 1);      // token slot = TMEM lane (warp & 3 selects the lane quarter)
    const int part = dw / kTile;          // which part of the row
    const int pi = tt / kPage, off = tt % kPage;
    const int swz = off & 7;              // 128-byte swizzle phase of this token's staging rows
    const uint32_t voff = (tt % 8) * 16 + (tt / 8) * Cfg::RS;
    // address, in a ring slot, of 16-code chunk k of this thread's part of its token's row
    auto chunk_addr = [&](const uint8_t* slot, int k) -> const uint4* {
      const int c = part * Cfg::NCH_T + k;  // chunk index along the row
      const int sl = c / 8, cw = c % 8;
      return reinterpret_cast<const uint4*>(slot + (pi * Cfg::NSL + sl) * kBox + off * 128 + ((cw ^ swz) * 16));
    };
    const int sc_off = Cfg::SL_SC + pi * Cfg::SC_KV + (off * Cfg::NB + part * Cfg::NBT) * 2;
    // q rows of an item (G x D bf16), at most QPT 16-byte pieces per thread, loaded one tile ahead of use;
    // the padding rows G..GN-1 of the shared q tile stay zero
    constexpr int QPT = (GN * (D / 8) + kDwThreads - 1) / kDwThreads;
    const int QPIECES = G * (D / 8);
    uint4 qreg[QPT];
    auto load_q = [&](const TileIter& t) {
      const int32_t head0 = t.g * p.group;
#pragma unroll
      for (int j = 0; j < QPT; ++j) {
        const int idx = dw + j * kDwThreads;
        if (idx < QPIECES) {
          const int h = idx / (D / 8), c8 = idx % (D / 8);
          qreg[j] = __ldg(reinterpret_cast<const uint4*>(
              p.q + (static_cast<int64_t>(t.b) * p.num_q_heads + head0 + h) * D + c8 * 8));
        }
      }
    };
    // K of tile n+1 is dequantized before V of tile n: the PV that frees the V tile for tile n+1 then
    // has two dequant steps of slack instead of none.
    TileIter tk;  // next tile whose K is dequantized
    tile_first(tk, sTab, p, groups, C, n_items);
    if (tk.live) load_q(tk);
    uint32_t nk = 0, nv = 0;  // tiles whose K / V have been written
    while (ok && (tk.live || nv < nk)) {
      if (tk.live) {
        // ================================================================ K of tile nk -> TMEM buffer kb
        const int kb = nk & 1;  // K buffer = S / P buffer = validity slot of this tile
        const int ring = nk % Cfg::STAGES;
        if (!mbar_wait_bounded(&bar_full[ring], (nk / Cfg::STAGES) & 1)) { ok = false; break; }
        const uint8_t* slot = sKr + ring * Cfg::SLOT_BYTES;
        const bool v_ok = off < sMeta[ring * kPagesPerTile + pi];
        const uint64_t scw = KindTraits<KIND>::kScaled ? load_scales<Cfg::NBT>(slot + sc_off) : 0u;
        // the buffer was last read by the QK of tile nk - 2
        if (nk >= 2 && !mbar_wait_bounded(&bar_qk_done[kb], ((nk >> 1) - 1) & 1)) { ok = false; break; }
        if (tk.i == 0) {
          // this item's q rows; the previous tile's QK must have read the old ones
          if (nk >= 1 && !mbar_wait_bounded(&bar_qk_done[(nk - 1) & 1], ((nk - 1) >> 1) & 1)) {
            ok = false;
            break;
          }
#pragma unroll
          for (int j = 0; j < QPT; ++j) {
            const int idx = dw + j * kDwThreads;
            if (idx < QPIECES) {
              const int h = idx / (D / 8), c8 = idx % (D / 8);
              *reinterpret_cast<uint4*>(sQ + (h % 8) * 16 + (h / 8) * Cfg::RS + c8 * 128) = qreg[j];
            }
          }
          fence_proxy_async_smem();
        }
        if (tk.i == tk.ntiles - 1) {  // the next item's q rows travel while this tile is dequantized
          TileIter nx = tk;
          tile_next(nx, sTab, p, groups, C, n_items);
          if (nx.live) load_q(nx);
        }
        // the validity slot kb was last read by the softmax of tile nk - 2
        if (nk >= 2 && !mbar_wait_bounded(&bar_p_full[kb], ((nk >> 1) - 1) & 1)) { ok = false; break; }
        if (part == 0) sValid[kb * kTile + tt] = v_ok ? 1 : 0;  // published to the softmax warps with k_full
#pragma unroll 1
        for (int k2 = 0; k2 < Cfg::NCH_T / 2; ++k2) {  // 32 codes (one scale) -> 16 TMEM columns per tcgen05.st
          uint32_t w[16];
          const uint16_t s_k = static_cast<uint16_t>(scw >> (16 * k2));
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int k = 2 * k2 + h;
            if (v_ok) {
              uint32_t ww[8];
              dequant16<KIND>(*chunk_addr(slot, k), s_k, ww);
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
        if (lane == 0) {
          asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&bar_k_full[kb])) : "memory");
          asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&bar_empty[ring])) : "memory");
        }
        tile_next(tk, sTab, p, groups, C, n_items);
        ++nk;
        if (nk == 1 && tk.live) continue;  // K runs one tile ahead of V
      }
      // ================================================================== V of tile nv -> shared memory
      {
        const int ring = Cfg::STAGES + nv % Cfg::STAGES;
        if (!mbar_wait_bounded(&bar_full[ring], (nv / Cfg::STAGES) & 1)) { ok = false; break; }
        const uint8_t* slot = sVr + (nv % Cfg::STAGES) * Cfg::SLOT_BYTES;
        const bool v_ok = off < sMeta[ring * kPagesPerTile + pi];
        const uint64_t scw = KindTraits<KIND>::kScaled ? load_scales<Cfg::NBT>(slot + sc_off) : 0u;
        // the previous PV must have read this thread's rows of the V tile (with two O^T slices, a part
        // that writes dims of slice 0 only waits for the first half of the PV)
        if (nv >= 1) {
          const bool lo = Cfg::O_CHUNKS == 2 && part * Cfg::HALF < 128;
          uint64_t* vbar = lo ? &bar_pv_lo[(nv - 1) & 1] : &bar_pv_done[(nv - 1) & 1];
          if (!mbar_wait_bounded(vbar, ((nv - 1) >> 1) & 1)) { ok = false; break; }
        }
#pragma unroll 2
        for (int k = 0; k < Cfg::NCH_T; ++k) {
          uint32_t w[8];
          if (v_ok) {
            dequant16<KIND>(*chunk_addr(slot, k), static_cast<uint16_t>(scw >> (16 * (k >> 1))), w);
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
          asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&bar_empty[ring])) : "memory");
        }
        ++nv;
      }
    }
  } else if (warp == kMmaWarp) {
    // ===================================================================== MMA issue (elected lane)
    // QK(nq) needs K tile nq in TMEM and S buffer nq&1 read by the softmax of tile nq-2; PV(np) needs
    // V tile np and P tile np.  Whichever is ready is issued first; lane 0 polls,
    // the converged warp issues (one elected lane).
    const uint32_t idesc_qk = mma_idesc(false, false);
    const uint32_t idesc_pv = mma_idesc(true, true);
    // descriptors of the first K-step; later steps add their byte offset >> 4 to the address field
    const uint64_t dQ = smem_desc(smem_u32(sQ), 128, Cfg::RS);
    const uint64_t dV = smem_desc(smem_u32(sV), Cfg::RS, 128);
    const uint64_t dP0 = smem_desc(smem_u32(sP), 128, 2048);
    TileIter tq, tp;  // next tile to QK; next tile to PV
    tile_first(tq, sTab, p, groups, C, n_items);
    tp = tq;
    uint32_t nq = 0, np = 0;  // tiles QK'd / PV'd
    uint64_t idle_since = 0;
    while (tp.live) {
      bool progressed = false;
      // PV first: the dequant warps wait for it before they rewrite the V tile
      if (np < nq) {
        const int b = np & 1;
        int ready = 0;
        if (lane == 0)
          ready = mbar_test_wait(bar_v_full, np & 1) && mbar_test_wait(&bar_p_full[b], (np >> 1) & 1);
        if (__shfl_sync(0xffffffffu, ready, 0)) {
          tc_fence_after();
          {
            const uint32_t o = tO + item_obuf(tp.item) * 32;
            const uint64_t dP = dP0 + static_cast<uint64_t>((b * Cfg::P_BYTES) >> 4);
#pragma unroll
            for (int oc = 0; oc < Cfg::O_CHUNKS; ++oc) {
              static_assert(kTile / 16 == 8, "one group of eight k-steps per O chunk");
              mma8_bf16(o + oc * kN, dV + static_cast<uint64_t>((oc * 16 * 128) >> 4),
                        static_cast<uint64_t>((2 * Cfg::RS) >> 4), dP, static_cast<uint64_t>((2 * 128) >> 4),
                        idesc_pv, tp.i > 0 ? 1u : 0u);
              if (oc == 0 && Cfg::O_CHUNKS == 2) mma_commit(&bar_pv_lo[b]);
            }
            mma_commit(&bar_pv_done[b]);
          }
          __syncwarp();
          ++np;
          tile_next(tp, sTab, p, groups, C, n_items);
          progressed = true;
        }
      }
      if (tq.live && nq < np + 2) {
        const int b = nq & 1;
        int ready = 0;
        if (lane == 0)
          ready = mbar_test_wait(&bar_k_full[b], (nq >> 1) & 1) &&
                  (nq < 2 || mbar_test_wait(&bar_p_full[b], ((nq >> 1) - 1) & 1));
        if (__shfl_sync(0xffffffffu, ready, 0)) {
          tc_fence_after();
          {
            const uint32_t ka = tK + b * Cfg::KCOLS;
#pragma unroll
            for (int g8 = 0; g8 < D / 128; ++g8)  // k-steps 8 g8 .. 8 g8 + 7
              mma8_bf16_tmem_a(tS + b * kN, ka + g8 * 64, 8u, dQ + static_cast<uint64_t>((g8 * 8 * 256) >> 4),
                               static_cast<uint64_t>(256 >> 4), idesc_qk, g8 > 0 ? 1u : 0u);
            mma_commit(&bar_qk_done[b]);
          }
          __syncwarp();
          ++nq;
          tile_next(tq, sTab, p, groups, C, n_items);
          progressed = true;
        }
      }
      if (progressed) {
        idle_since = 0;
      } else {
        // back off while nothing is ready: the poll shares its SM sub-partition with four dequant warps
        // (long_gqa batch 8 x 262144: 493 -> 489 us)
        __nanosleep(128);
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
    // O^T of an item is read out of TMEM (its "flush") only after the next item's first P has been
    // handed to the MMA thread: the two items use different O accumulators, so the readout overlaps
    // the next item's first PV instead of stalling the pipeline.
    const int tt = tid;  // token slot / O^T row / TMEM lane
    int32_t pend_item = -1;  // item whose O^T is still in TMEM
    uint32_t pend_tile = 0;  // its last tile (CTA tile count), whose PV completes it
    auto flush_o = [&]() -> bool {
      if (!mbar_wait_bounded(&bar_pv_done[pend_tile & 1], (pend_tile >> 1) & 1)) return false;
      tc_fence_after();
      const uint32_t ob = tO + item_obuf(pend_item) * 32;
#pragma unroll
      for (int oc = 0; oc < Cfg::O_CHUNKS; ++oc) {
        float o[GN];  // the padding heads' columns are not read
        tmem_ld_cols<GN>(ob + oc * kN + lane_base, o);
        const int d = oc * 128 + tt;
#pragma unroll
        for (int h = 0; h < GN; ++h)
          if (h < G) p.part_acc[(static_cast<int64_t>(pend_item) * G + h) * D + d] = o[h];
      }
      tc_fence_before();  // the reads are ordered before this warp's later arrivals
      pend_item = -1;
      return true;
    };
    for (int32_t item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
      const ItemPos ip = locate(sTab, p, groups, C, item);
      const int32_t pg0 = ip.split * C;
      const int32_t pg1 = min(pg0 + C, seq_pages(p, ip.b));
      const int32_t ntiles = (pg1 - pg0 + kPagesPerTile - 1) / kPagesPerTile;
      const uint32_t ob = tO + item_obuf(item) * 32;
      float m_used[GN], l_t[GN];
#pragma unroll
      for (int h = 0; h < GN; ++h) {
        m_used[h] = h < G ? kNoMax : INFINITY;
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
        float s[GN];
        tmem_ld_cols<GN>(tS + b * kN + lane_base, s);
        // d = s * scale - m per head (-inf for an invalid token or a padded head); a max moves when d > 2^8
        // headroom, which a head without a max yet always reports
        bool moved = false;
#pragma unroll
        for (int h = 0; h < GN; ++h) moved |= valid && fmaf(s[h], p.score_scale, -m_used[h]) > kLazyRescale;
        // does any token of the tile move any head's running max?  (one vote per warp, one barrier)
        const int wv = __any_sync(0xffffffffu, moved);
        // the votes alternate by tile parity: a warp writes the next tile's only after every warp has passed
        // this tile's barrier below, and nobody reads this tile's after the next tile's barrier
        int32_t* flags = sFlag + b * kSmWarps;
        if (lane == 0) flags[warp] = wv;
        named_sync(1, kSmWarps * 32);
        const bool any_moved = (flags[0] | flags[1] | flags[2] | flags[3]) != 0;
        float alpha[GN];
        bool rescale = false;
#pragma unroll
        for (int h = 0; h < GN; ++h) alpha[h] = 1.0f;
        if (any_moved) {  // uniform branch: exact tile maxima, then the new running max per head
          named_sync(1, kSmWarps * 32);  // every warp has read the votes
#pragma unroll
          for (int h = 0; h < GN; ++h) {
            float mx = (valid && h < G) ? s[h] * p.score_scale : -INFINITY;
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
            if (mx > -INFINITY && mx > m_used[h] + kLazyRescale) {  // (never for a padded head: m = +inf)
              if (m_used[h] != kNoMax) {
                alpha[h] = exp2f(m_used[h] - mx);
                rescale = true;
              }
              m_used[h] = mx;
            }
          }
        }
        // P row of this token (bf16), and the row sums of exactly those bf16 values
        uint32_t pw[GN / 2];
#pragma unroll
        for (int h2 = 0; h2 < GN / 2; ++h2) {
          float pr[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int h = 2 * h2 + e;
            pr[e] = tc_ex2(valid ? fmaf(s[h], p.score_scale, -m_used[h]) : -INFINITY);
          }
          pw[h2] = pack_bf16x2(pr[0], pr[1]);
          const float2 pb = unpack_bf16x2(pw[h2]);
          l_t[2 * h2] = fmaf(l_t[2 * h2], alpha[2 * h2], pb.x);
          l_t[2 * h2 + 1] = fmaf(l_t[2 * h2 + 1], alpha[2 * h2 + 1], pb.y);
        }
        // P buffer b is free once the PV two tiles back has read it
        if (gtile >= 2 && !mbar_wait_bounded(&bar_pv_done[b], ((gtile >> 1) - 1) & 1)) { ok = false; break; }
        if (rescale && o_live) {  // O must hold every earlier PV of this item before it is scaled
          if (!mbar_wait_bounded(&bar_pv_done[(gtile - 1) & 1], ((gtile - 1) >> 1) & 1)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int oc = 0; oc < Cfg::O_CHUNKS; ++oc) {
            float o[GN];
            tmem_ld_cols<GN>(ob + oc * kN + lane_base, o);
#pragma unroll
            for (int h = 0; h < GN; ++h) o[h] *= alpha[h];
            tmem_st_cols<GN>(ob + oc * kN + lane_base, o);
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
        // the previous item's O^T, now that this item's first PV can run into the other accumulator
        if (pend_item >= 0 && !flush_o()) { ok = false; break; }
      }
      if (!ok) break;
      // ---- item end: (m, l) per head now; O^T at the next item's first tile (or after the last item)
      named_sync(1, kSmWarps * 32);  // the last tile's maxima in sRed have been read by every warp
#pragma unroll
      for (int h = 0; h < GN; ++h) {
        float v = l_t[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) sRed[warp * kN + h] = v;
      }
      named_sync(1, kSmWarps * 32);
      if (tt < G) {  // m_used is identical in every softmax thread; thread h writes head h
        float lsum = 0.0f, mh = -INFINITY;
#pragma unroll
        for (int w = 0; w < kSmWarps; ++w) lsum += sRed[w * kN + tt];
#pragma unroll
        for (int h = 0; h < GN; ++h)
          if (h == tt) mh = m_used[h];
        p.part_ml[(static_cast<int64_t>(item) * G + tt) * 2 + 0] = mh == kNoMax ? -INFINITY : mh;
        p.part_ml[(static_cast<int64_t>(item) * G + tt) * 2 + 1] = lsum;
      }
      named_sync(1, kSmWarps * 32);
      pend_item = item;
      pend_tile = gtile - 1;
    }
    if (ok && pend_item >= 0 && !flush_o()) ok = false;
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
  const bool g16 = (a.num_q_heads / a.num_kv_heads) > 8;
  decltype(&decode_tc_kernel<D, KVQ_FP8_E4M3, 8>) kern = nullptr;
  switch (a.kind) {
#define KVQ_TC_KIND(K) \
  case K: kern = g16 ? decode_tc_kernel<D, K, 16> : decode_tc_kernel<D, K, 8>; break;
    KVQ_TC_KIND(KVQ_FP8_E4M3)
    KVQ_TC_KIND(KVQ_Q8_0)
    KVQ_TC_KIND(KVQ_FP8_E4M3_UNSCALED)
    KVQ_TC_KIND(KVQ_FP8_E5M2_UNSCALED)
#undef KVQ_TC_KIND
  }
  if (kern == nullptr) return KVQ_EKIND;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) != cudaSuccess)
    return KVQ_ECUDA;
  CUtensorMap map;
  if (!encode_code_map(&map, a.codes, a.num_pages, a.num_kv_heads, D)) return KVQ_ECUDA;
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
  return group >= 1 && group <= kN && batch <= kMaxPlanBatch;
}

kvq_status launch_decode_tc(const DecodeArgs& a, cudaStream_t stream) {
  if (a.head_dim == 128) return launch_tc_d<128>(a, stream);
  if (a.head_dim == 256) return launch_tc_d<256>(a, stream);
  return KVQ_EUNSUPPORTED;
}

}  // namespace kvq
