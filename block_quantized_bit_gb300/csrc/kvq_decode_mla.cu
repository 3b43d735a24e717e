// kvq_decode_mla.cu -- split-K MLA decode on the 5th-generation tensor cores (tcgen05).
//
// "feat(kvcache): 8-bit DSV4 window/compressed KV", section "What this adds": one latent row per
// token (512 latent dims + 64 rope dims = 576) is both K and, through its first 512 dims, V; 128 query
// heads read it.  "feat(kvcache): 8-bit KV cache (q8_0 / fp8_e4m3) behind --kv-cache-dtype", section
// "What": the row is dequantized to bf16 (RNE of code * fp16 block scale) before the dot.
//
// A work item is (sequence, group of up to 64 query heads, split of pages); the head groups of a split
// read the same codes (after the first time from L2).  A group of fewer than 64 heads is padded with
// zero query rows whose probabilities are forced to zero.  A tile is 128 tokens (8 pages), the M of every MMA:
//   S^T[128 tok][64 h]  = Kd[128 tok][576] . Q[64 h][576]^T   A = K slab in TMEM, B = Q (K-major smem)
//   O^T[128 d][64 h]   += Vd^T[128 d][128 tok] . P[64 h][128 tok]^T, four 128-dim blocks of V
//                        A = V^T block (MN-major smem), B = P (MN-major smem)
// Q, V^T blocks and P use the canonical no-swizzle core-matrix layout (8 rows x 16 bytes per core
// matrix), so one V^T block written token-major serves as the MN-major A operand.
//
// One persistent CTA per SM, 26 warps (72 registers each):
//   warp 25     producer: per tile, TMA copies of five 128-byte-wide code slabs (d = 0, 128, 256, 384 and
//               448; the last one's upper half is the rope part) into a 3-slot ring, one 2 KB box per
//               page (128-byte swizzle), and the tile's scales with the first slab.
//   warps 8-15  K dequant: thread = (token, half of the slab's dims); each slab to bf16 in a TMEM slot
//               (two slots).
//   warps 16-23 V dequant: thread = (token, half of the block's dims); reads its codes of each 128-dim
//               block straight from global memory (the K pass just brought them into L2), one block
//               ahead in registers, and writes the bf16 V^T block into one of two shared buffers.
//   warp 24     MMA issue (one elected lane): QK slab by slab into S (double-buffered in TMEM), PV
//               block by block into O; whichever is ready first.
//   warps 0-7   softmax: thread = (token, 32 of the 64 heads); fp32 online softmax in the exp2 domain
//               with lazy rescaling (a head's running max moves only when a score exceeds it by 2^8),
//               one pass over the scores that forms P with the current maxima (again only if one
//               moved); P to shared memory as bf16; O rescaled in TMEM when a max moves; the partial.
// TMEM: S[2] 128 columns, O^T 4 x 64, K slots 2 x 64 = 512.  Every wait is bounded (2 s) and reports a
// timeout in the workspace status word instead of hanging.
#include <cuda.h>  // CUtensorMap and its enums (the encoder is fetched from the driver at run time)
#include <math.h>

#include <algorithm>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_plan.cuh"
#include "kvq_tc.cuh"

namespace kvq {
namespace {
namespace mla {

constexpr int kD = 576, kDV = 512, kNB = kD / 32;   // row width, V width, scale blocks per row
constexpr int kTile = 128;                         // tokens per tile = MMA M
constexpr int kPagesPerTile = kTile / kPage;       // 8
constexpr int kHG = 64;                            // query heads per item = MMA N
constexpr int kSlabs = 5;                          // K slabs per tile
constexpr int kVBlocks = kDV / 128;                // 4 V^T blocks per tile
constexpr int kRing = 3;                           // code ring slots
constexpr int kBox = kPage * 128;                  // 2 KB TMA box: 16 rows x 128 code bytes of one page
constexpr int kSlab = kPagesPerTile * kBox;        // 16 KB
constexpr int kScPage = kPage * kNB * 2;           // 576 B of scales per page
constexpr int kScTile = kPagesPerTile * kScPage;   // 4608 B
constexpr int kQS = (kD / 8) * 128;                // 9216: bytes between 8-head groups of Q
constexpr int kVRS = 128 * 16;                     // 2048: bytes between 8-token groups of a V^T block
constexpr int kPS = (kTile / 8) * 128;             // 2048: bytes between 8-head groups of P
constexpr int kMaxBatch = 1024;                    // sequences whose item bases fit the shared table
constexpr float kLazyRescale = 8.0f;
// running max of a head before its first valid score: finite, so that s * scale - m stays finite and the
// first tile's vote fires; padded heads keep +inf, so that their probabilities come out as 2^-inf = 0
constexpr float kNoMax = -1.0e30f;
constexpr int kTmemCols = 512;

constexpr int kSmWarps = 8;   // 0-7: warp w covers TMEM lane quarter w % 4 and heads 32 (w / 4) ..
constexpr int kKWarp0 = 8;    // 8-15: quarter w % 4, dims 64 ((w - 8) / 4) .. of each slab
constexpr int kVWarp0 = 16;   // 16-23: quarter w % 4, dims 64 ((w - 16) / 4) .. of each V block
constexpr int kMmaWarp = 24;
constexpr int kProdWarp = 25;
constexpr int kThreads = 26 * 32;  // 72 registers per thread
constexpr int kHS = kHG / 2;       // query heads per softmax thread

constexpr int RING_OFF = 0;                               // 1024-byte aligned (swizzle atoms)
constexpr int VT_OFF = RING_OFF + kRing * kSlab;          // 2 x 32 KB
constexpr int Q_OFF = VT_OFF + 2 * kTile * 128 * 2;       // 72 KB
constexpr int P_OFF = Q_OFF + kHG * kD * 2;               // 16 KB
constexpr int SC_OFF = P_OFF + kTile * kHG * 2;           // 2 x 4608
constexpr int RED_OFF = SC_OFF + 2 * kScTile;             // softmax cross-warp scratch [8][32]
constexpr int M_OFF = RED_OFF + kSmWarps * kHS * 4;       // running max per head [64]
constexpr int A_OFF = M_OFF + kHG * 4;                    // rescale factor per head [64]
constexpr int FLAG_OFF = A_OFF + kHG * 4;                 // one vote per softmax warp
constexpr int VAL_OFF = FLAG_OFF + kSmWarps * 4;          // [2][128] token validity by tile parity
constexpr int META_OFF = VAL_OFF + 2 * kTile;             // [kRing][8] valid tokens per page
constexpr int TAB_OFF = META_OFF + kRing * kPagesPerTile * 4;
constexpr int NBARS = 18 + 2 * kRing;
constexpr int BAR_OFF = TAB_OFF + kMaxBatch * 4;
constexpr int SMEM_BYTES = BAR_OFF + NBARS * 8 + 16 + 1024;  // + slack to align the base
static_assert(kSlab % 1024 == 0 && VT_OFF % 1024 == 0, "swizzle atoms");
static_assert(SMEM_BYTES <= 226 * 1024, "shared memory (with the plan's static part)");

}  // namespace mla

// 2^x by the hardware approximation, subnormal results flushed to 0 (far below the bf16 rounding of P);
// 2^-inf = 0.
__device__ __forceinline__ float mla_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint64_t mla_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // descriptor version for tcgen05; no swizzle, base offset 0
  return d;
}

// kind::f16 instruction descriptor: fp32 accumulate, bf16 A and B, M = 128, N = 64.
__device__ __forceinline__ uint32_t mla_idesc(bool a_mn_major, bool b_mn_major) {
  uint32_t d = 0;
  d |= 1u << 4;
  d |= 1u << 7;
  d |= 1u << 10;
  d |= static_cast<uint32_t>(a_mn_major) << 15;
  d |= static_cast<uint32_t>(b_mn_major) << 16;
  d |= static_cast<uint32_t>(mla::kHG >> 3) << 17;
  d |= static_cast<uint32_t>(mla::kTile >> 4) << 24;
  return d;
}

// Warp-collective MMA and commit: all 32 lanes of the converged MMA warp call them with the same operands
// and the lane chosen by elect.sync issues (the descriptors stay in uniform registers, which a probe measured
// at 15 to 40 clocks per MMA against 56 from a lane-0 branch).  The full mask elects the same lane every
// time, so a commit tracks every MMA issued before it.
__device__ __forceinline__ void mla_mma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mla_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                           uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mla_commit(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void mla_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void mla_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void mla_ld16(uint32_t taddr, float (&v)[16]) {
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

__device__ __forceinline__ void mla_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void mla_named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void mla_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// TMA load of one box: code bytes [x, x+128) of the 16 token rows of physical page `page`.
__device__ __forceinline__ void mla_tma(uint32_t dst, const CUtensorMap* map, int x, int page, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(page * kPage), "r"(smem_u32(bar))
      : "memory");
}

// Item -> (sequence, head group, split) through the shared table of per-sequence first items.
struct MlaPos {
  int32_t b, hg, split;
};

__device__ __forceinline__ MlaPos mla_locate(const int32_t* tab, const KParams& p, int32_t C, int32_t item) {
  int lo = 0, hi = p.batch;  // first b with tab[b] > item
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (tab[mid] <= item) lo = mid + 1;
    else hi = mid;
  }
  MlaPos r;
  r.b = lo - 1;
  const int32_t nsplit = (seq_pages(p, r.b) + C - 1) / C;
  const int32_t local = item - tab[r.b];
  r.hg = local / nsplit;
  r.split = local - r.hg * nsplit;
  return r;
}

struct MlaIter {
  int32_t item, i, ntiles, b, hg, pg0, pg1, L;
  bool live;
};

__device__ __forceinline__ void mla_load_item(MlaIter& t, const int32_t* tab, const KParams& p, int32_t C) {
  const MlaPos ip = mla_locate(tab, p, C, t.item);
  t.b = ip.b;
  t.hg = ip.hg;
  t.L = __ldg(p.seq_lens + ip.b);
  t.pg0 = ip.split * C;
  t.pg1 = min(t.pg0 + C, seq_pages(p, ip.b));
  t.ntiles = (t.pg1 - t.pg0 + mla::kPagesPerTile - 1) / mla::kPagesPerTile;
  t.i = 0;
}

__device__ __forceinline__ void mla_first(MlaIter& t, const int32_t* tab, const KParams& p, int32_t C, int32_t n) {
  t.item = blockIdx.x;
  t.live = t.item < n;
  if (t.live) mla_load_item(t, tab, p, C);
}

__device__ __forceinline__ void mla_next(MlaIter& t, const int32_t* tab, const KParams& p, int32_t C, int32_t n) {
  if (!t.live) return;
  if (++t.i < t.ntiles) return;
  t.item += gridDim.x;
  t.live = t.item < n;
  if (t.live) mla_load_item(t, tab, p, C);
}

// Valid-token test of token slot (pi, off) of tile t: its page is mapped, in the pool, and the token
// is before the sequence end.  Returns the physical page or -1.
__device__ __forceinline__ int32_t mla_phys(const KParams& p, const MlaIter& t, int pi, int off) {
  if (!t.live) return -1;
  const int32_t pg = t.pg0 + t.i * mla::kPagesPerTile + pi;
  if (pg >= t.pg1 || pg * kPage + off >= t.L) return -1;
  const int32_t e = bt_entry(p, t.b, pg);
  return (e >= 0 && e < p.num_pages) ? e : -1;
}

template <int KIND>
__global__ void __launch_bounds__(mla::kThreads, 1) decode_mla_kernel(const KParams p,
                                                                     const __grid_constant__ CUtensorMap tmap) {
  using namespace mla;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sRing = smem + RING_OFF;
  uint8_t* sVt = smem + VT_OFF;
  uint8_t* sQ = smem + Q_OFF;
  uint8_t* sP = smem + P_OFF;
  uint8_t* sSc = smem + SC_OFF;
  float* sRed = reinterpret_cast<float*>(smem + RED_OFF);
  float* sM = reinterpret_cast<float*>(smem + M_OFF);
  float* sA = reinterpret_cast<float*>(smem + A_OFF);
  int32_t* sFlag = reinterpret_cast<int32_t*>(smem + FLAG_OFF);
  int32_t* sMeta = reinterpret_cast<int32_t*>(smem + META_OFF);
  uint8_t* sValid = smem + VAL_OFF;
  int32_t* sTab = reinterpret_cast<int32_t*>(smem + TAB_OFF);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + BAR_OFF);
  // Each barrier completes once per use of its buffer, so a waiter names an unambiguous phase.
  uint64_t* bar_k_full = bars + 0;     // [2] K slot s written (K warps)
  uint64_t* bar_k_free = bars + 2;     // [2] the QK reading K slot s completed (commit)
  uint64_t* bar_qk_done = bars + 4;    // [2] S buffer b complete for its tile (commit)
  uint64_t* bar_p_full = bars + 6;     // [2] P of tile parity b written, S buffer b read (softmax warps)
  uint64_t* bar_v_full = bars + 8;     // [2] V^T buffer v written (V warps)
  uint64_t* bar_v_free = bars + 10;    // [2] the PV reading V^T buffer v completed (commit)
  uint64_t* bar_pv_done = bars + 12;   // [2] every PV of tile parity b completed (commit)
  uint64_t* bar_sc_free = bars + 14;   // [2] scale buffer b read and token validity b written (K warps)
  uint64_t* bar_full = bars + 18;              // [kRing] ring slot landed (producer arrival + bytes)
  uint64_t* bar_empty = bars + 18 + kRing;     // [kRing] ring slot read (K warps)
  uint32_t* sTmem = reinterpret_cast<uint32_t*>(smem + BAR_OFF + NBARS * 8);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const Plan plan = make_plan(p, 0, -1);
  const int32_t C = plan.C;
  const int32_t n_items = plan.n_items;
  const int32_t groups = p.num_kv_heads * p.head_tiles;
  const int32_t HP = p.group / p.head_tiles;  // query heads per item, <= kHG (the rest of N is padding)
  if (tid == 0) {
    int32_t run = 0;
    for (int32_t b = 0; b < p.batch; ++b) {
      sTab[b] = run;
      run += groups * ((seq_pages(p, b) + C - 1) / C);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar_k_full[b], 8);
      mbar_init(&bar_k_free[b], 1);
      mbar_init(&bar_qk_done[b], 1);
      mbar_init(&bar_p_full[b], kSmWarps);
      mbar_init(&bar_v_full[b], 8);
      mbar_init(&bar_v_free[b], 1);
      mbar_init(&bar_pv_done[b], 1);
      mbar_init(&bar_sc_free[b], 8);
    }
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 8);
    }
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(sTmem)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  for (int h = tid; h < kHG; h += kThreads) sM[h] = h < HP ? kNoMax : INFINITY;
  for (int i = tid; i < kHG * kD * 2 / 16; i += kThreads) reinterpret_cast<uint4*>(sQ)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  mla_fence_before();
  __syncthreads();
  mla_fence_after();
  const uint32_t tmem = *sTmem;
  const uint32_t tS = tmem;         // S^T buffers: columns [64 b, 64 b + 64)
  const uint32_t tO = tmem + 128;   // O^T block c: columns [128 + 64 c, 192 + 64 c)
  const uint32_t tK = tmem + 384;   // K slots: columns [384 + 64 s, 448 + 64 s)
  const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
  // the merge kernel that follows may launch now; it waits for this grid to complete before it reads
  asm volatile("griddepcontrol.launch_dependents;");
  bool ok = true;

  if (warp == kProdWarp) {
    // ===================================================================== producer
    // Lane pi (< 8) owns page pi of the tile.  Slab j of tile n is the (5n + j)-th use of the ring.
    MlaIter t;
    mla_first(t, sTab, p, C, n_items);
    uint32_t n = 0;
    while (ok && t.live) {
      int32_t phys = -1, nvalid = 0;
      if (lane < kPagesPerTile) {
        const int32_t pg = t.pg0 + t.i * kPagesPerTile + lane;
        if (pg < t.pg1) {
          phys = bt_entry(p, t.b, pg);
          if (phys >= p.num_pages) {
            set_status(p.status, kStatusBadPage);
            phys = -1;
          }
          if (phys >= 0) nvalid = min(kPage, t.L - pg * kPage);  // >= 1: pg < the sequence's page count
        }
      }
      const uint32_t npg = __reduce_add_sync(0xffffffffu, phys >= 0 ? 1u : 0u);
      int32_t nv[kPagesPerTile];
#pragma unroll
      for (int i = 0; i < kPagesPerTile; ++i) nv[i] = __shfl_sync(0xffffffffu, nvalid, i);
      // the scale buffer of this tile parity was last read by the K warps two tiles ago
      if (n >= 2 && !mbar_wait_bounded(&bar_sc_free[n & 1], ((n >> 1) - 1) & 1)) { ok = false; break; }
#pragma unroll 1
      for (int j = 0; j < kSlabs; ++j) {
        const uint32_t u = n * kSlabs + j;  // ring use
        const int rs = u % kRing;
        if (u >= kRing && !mbar_wait_bounded(&bar_empty[rs], ((u / kRing) - 1) & 1)) { ok = false; break; }
        if (lane == 0) {
#pragma unroll
          for (int i = 0; i < kPagesPerTile; ++i) sMeta[rs * kPagesPerTile + i] = nv[i];
          mbar_arrive_expect_tx(&bar_full[rs], npg * (kBox + (j == 0 && KindTraits<KIND>::kScaled ? kScPage : 0)));
        }
        __syncwarp();
        if (phys >= 0) {
          mla_tma(smem_u32(sRing + rs * kSlab + lane * kBox), &tmap, j < 4 ? 128 * j : 448, phys, &bar_full[rs]);
          if (j == 0 && KindTraits<KIND>::kScaled)  // an unscaled pool has codes only
            bulk_g2s(sSc + (n & 1) * kScTile + lane * kScPage,
                     reinterpret_cast<const uint8_t*>(p.scales) + static_cast<int64_t>(phys) * kScPage, kScPage,
                     &bar_full[rs]);
        }
      }
      if (!ok) break;
      mla_next(t, sTab, p, C, n_items);
      ++n;
    }
    // no copy may still be in flight when the CTA exits
    const uint32_t uses = n * kSlabs;
    for (uint32_t j = 1; j <= uses && j <= static_cast<uint32_t>(kRing); ++j) {
      const uint32_t u = uses - j;
      (void)mbar_wait_bounded(&bar_full[u % kRing], (u / kRing) & 1);
    }
  } else if (warp >= kKWarp0 && warp < kKWarp0 + 8) {
    // ===================================================================== K dequant
    const int kt = tid - kKWarp0 * 32;  // 0 .. 255
    const int tt = kt & (kTile - 1);    // token slot = TMEM lane
    const int part = kt >> 7;           // which 64 dims of each slab
    const int pi = tt / kPage, off = tt % kPage, swz = off & 7;
    MlaIter t;
    mla_first(t, sTab, p, C, n_items);
    uint32_t n = 0;
    while (ok && t.live) {
      if (t.i == 0) {
        // this item's 64 query rows; every QK of the previous tile must have read the old ones
        if (n >= 1 && !mbar_wait_bounded(&bar_qk_done[(n - 1) & 1], ((n - 1) >> 1) & 1)) { ok = false; break; }
        const __nv_bfloat16* qb = p.q + (static_cast<int64_t>(t.b) * p.num_q_heads + t.hg * HP) * kD;
#pragma unroll 4
        for (int idx = kt; idx < kHG * (kD / 8); idx += 256) {
          const int h = idx % kHG, d8 = idx / kHG;
          if (h >= HP) continue;  // padding rows stay zero
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(qb + static_cast<int64_t>(h) * kD + d8 * 8));
          *reinterpret_cast<uint4*>(sQ + (h % 8) * 16 + (h / 8) * kQS + d8 * 128) = v;
        }
        fence_proxy_async_smem();
      }
      bool v_ok = false;
      const uint16_t* sc = reinterpret_cast<const uint16_t*>(sSc + (n & 1) * kScTile + pi * kScPage) + off * kNB;
#pragma unroll 1
      for (int j = 0; j < kSlabs; ++j) {
        const uint32_t u = n * kSlabs + j;  // ring use = K slot use
        const int rs = u % kRing, ks = u & 1;
        if (!mbar_wait_bounded(&bar_full[rs], (u / kRing) & 1)) { ok = false; break; }
        if (j == 0) {
          v_ok = off < sMeta[rs * kPagesPerTile + pi];
          // the validity slot of this tile parity was last read by the softmax of tile n - 2
          if (n >= 2 && !mbar_wait_bounded(&bar_p_full[n & 1], ((n >> 1) - 1) & 1)) { ok = false; break; }
          if (part == 0) sValid[(n & 1) * kTile + tt] = v_ok ? 1 : 0;  // published with sc_free (last slab)
        }
        if (u >= 2 && !mbar_wait_bounded(&bar_k_free[ks], ((u >> 1) - 1) & 1)) { ok = false; break; }
        const uint8_t* slot = sRing + rs * kSlab + pi * kBox + off * 128;
        // 32 codes (one scale) -> 16 TMEM columns; a part takes chunk pairs 2 part, 2 part + 1 of a latent
        // slab, and of the rope slab (whose upper half, d = 512..575, is all that is used) pair 2 + part
        const int c2a = (j < 4) ? 2 * part : 2 + part;
        const int c2b = (j < 4) ? 2 * part + 2 : 3 + part;
#pragma unroll 1
        for (int c2 = c2a; c2 < c2b; ++c2) {
          uint32_t w[16];
          const int blk = (j < 4 ? 4 * j : 14) + c2;  // scale block of these 32 dims
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int c = 2 * c2 + h;
            if (v_ok) {
              uint32_t ww[8];
              dequant16<KIND>(*reinterpret_cast<const uint4*>(slot + ((c ^ swz) * 16)),
                              KindTraits<KIND>::kScaled ? sc[blk] : kHalfOne, ww);
#pragma unroll
              for (int e = 0; e < 8; ++e) w[8 * h + e] = ww[e];
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e) w[8 * h + e] = 0u;
            }
          }
          mla_st16(tK + ks * 64 + lane_base + c2 * 16, w);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        mla_fence_before();
        __syncwarp();
        if (lane == 0) {
          mla_arrive(&bar_k_full[ks]);
          mla_arrive(&bar_empty[rs]);
          if (j == kSlabs - 1) mla_arrive(&bar_sc_free[n & 1]);
        }
      }
      if (!ok) break;
      mla_next(t, sTab, p, C, n_items);
      ++n;
    }
  } else if (warp >= kVWarp0 && warp < kVWarp0 + 8) {
    // ===================================================================== V dequant
    const int vt = tid - kVWarp0 * 32;  // 0 .. 255
    const int tt = vt & (kTile - 1);
    const int part = vt >> 7;           // which 64 dims of each V block
    const int pi = tt / kPage, off = tt % kPage;
    const uint32_t voff = (tt % 8) * 16 + (tt / 8) * kVRS + part * 8 * 128;
    MlaIter t;
    mla_first(t, sTab, p, C, n_items);
    // codes and the two scales of this part of V block c of the tile whose page for this token is
    // `phys` (-1: zeros)
    uint4 nxt[4];
    uint32_t nxt_s = 0;
    auto fetch = [&](int32_t phys, int c) {
      if (phys < 0) return;
      const int64_t row = static_cast<int64_t>(phys) * kPage + off;
      const uint4* src = reinterpret_cast<const uint4*>(p.codes + row * kD + c * 128 + part * 64);
#pragma unroll
      for (int k = 0; k < 4; ++k) nxt[k] = __ldg(src + k);
      // a row's scales start 36 bytes apart: a 4-byte load is always aligned
      if (KindTraits<KIND>::kScaled)
        nxt_s = __ldg(reinterpret_cast<const uint32_t*>(reinterpret_cast<const uint16_t*>(p.scales) + row * kNB + c * 4 +
                                                      part * 2));
    };
    int32_t phys = mla_phys(p, t, pi, off);
    fetch(phys, 0);
    uint32_t nb = 0;  // V blocks written
    while (ok && t.live) {
      MlaIter tn = t;
      mla_next(tn, sTab, p, C, n_items);
      const int32_t phys_n = mla_phys(p, tn, pi, off);
#pragma unroll 1
      for (int c = 0; c < kVBlocks; ++c, ++nb) {
        uint4 cur[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) cur[k] = nxt[k];
        const uint32_t cs = nxt_s;
        const bool v_ok = phys >= 0;
        if (c + 1 < kVBlocks) fetch(phys, c + 1);
        else fetch(phys_n, 0);
        const int vb = nb & 1;
        if (nb >= 2 && !mbar_wait_bounded(&bar_v_free[vb], ((nb >> 1) - 1) & 1)) { ok = false; break; }
        uint8_t* dst = sVt + vb * (kTile * 128 * 2) + voff;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint32_t w[8];
          if (v_ok) {
            dequant16<KIND>(cur[k], static_cast<uint16_t>((k & 2) ? (cs >> 16) : cs), w);
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) w[e] = 0u;
          }
          *reinterpret_cast<uint4*>(dst + (2 * k) * 128) = make_uint4(w[0], w[1], w[2], w[3]);
          *reinterpret_cast<uint4*>(dst + (2 * k + 1) * 128) = make_uint4(w[4], w[5], w[6], w[7]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mla_arrive(&bar_v_full[vb]);
      }
      if (!ok) break;
      t = tn;
      phys = phys_n;
    }
  } else if (warp == kMmaWarp) {
    // ===================================================================== MMA issue (elected lane)
    const uint32_t idesc_qk = mla_idesc(false, false);
    const uint32_t idesc_pv = mla_idesc(true, true);
    const uint64_t dQ = mla_desc(smem_u32(sQ), 128, kQS);
    const uint64_t dV0 = mla_desc(smem_u32(sVt), kVRS, 128);
    const uint64_t dP = mla_desc(smem_u32(sP), 128, kPS);
    MlaIter tq, tp;
    mla_first(tq, sTab, p, C, n_items);
    tp = tq;
    uint32_t nq = 0, jq = 0;  // QK: tiles completed, next slab
    uint32_t np = 0, cp = 0;  // PV: tiles completed, next block
    uint64_t idle_since = 0;
    while (tp.live) {
      bool progressed = false;
      if (np < nq) {  // PV block cp of tile np
        const uint32_t nb = np * kVBlocks + cp;
        const int vb = nb & 1;
        int ready = 0;
        if (lane == 0)
          ready = (cp > 0 || mbar_test_wait(&bar_p_full[np & 1], (np >> 1) & 1)) &&
                  mbar_test_wait(&bar_v_full[vb], (nb >> 1) & 1);
        if (__shfl_sync(0xffffffffu, ready, 0)) {
          mla_fence_after();
          const uint64_t dV = dV0 + static_cast<uint64_t>((vb * kTile * 128 * 2) >> 4);
          static_assert(kTile / 16 == 8, "one group of eight k-steps per V block");
          mma8_bf16(tO + cp * 64, dV, static_cast<uint64_t>((2 * kVRS) >> 4), dP, static_cast<uint64_t>((2 * 128) >> 4),
                    idesc_pv, tp.i > 0 ? 1u : 0u);
          mla_commit(&bar_v_free[vb]);
          if (cp == kVBlocks - 1) mla_commit(&bar_pv_done[np & 1]);
          __syncwarp();
          if (++cp == kVBlocks) {
            cp = 0;
            ++np;
            mla_next(tp, sTab, p, C, n_items);
          }
          progressed = true;
        }
      }
      if (tq.live && nq < np + 2) {  // QK slab jq of tile nq
        const uint32_t u = nq * kSlabs + jq;
        const int ks = u & 1;
        int ready = 0;
        if (lane == 0)
          ready = mbar_test_wait(&bar_k_full[ks], (u >> 1) & 1) &&
                  (jq > 0 || nq < 2 || mbar_test_wait(&bar_p_full[nq & 1], ((nq >> 1) - 1) & 1));
        if (__shfl_sync(0xffffffffu, ready, 0)) {
          mla_fence_after();
          const uint32_t d_s = tS + (nq & 1) * 64;
          const uint32_t a0 = tK + ks * 64;
          if (jq < 4) {
            mma8_bf16_tmem_a(d_s, a0, 8u, dQ + static_cast<uint64_t>(((16 * jq) * 128) >> 4),
                             static_cast<uint64_t>((2 * 128) >> 4), idesc_qk, jq > 0 ? 1u : 0u);
          } else {
#pragma unroll
            for (int k = 4; k < 8; ++k)  // dims 512..575 sit in the upper half of the slot
              mla_mma_ts(d_s, a0 + k * 8, dQ + static_cast<uint64_t>(((64 + 2 * (k - 4)) * 128) >> 4), idesc_qk, 1u);
          }
          mla_commit(&bar_k_free[ks]);
          if (jq == kSlabs - 1) mla_commit(&bar_qk_done[nq & 1]);
          __syncwarp();
          if (++jq == kSlabs) {
            jq = 0;
            ++nq;
            mla_next(tq, sTab, p, C, n_items);
          }
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
    // Warp w: TMEM lane quarter w % 4 (its tokens; in the epilogue, dims), heads h0 .. h0 + 31.
    const int tt = tid & (kTile - 1);
    const int h0 = (warp >> 2) * kHS;
    uint32_t n = 0;  // tiles
    for (int32_t item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
      MlaIter t;
      t.item = item;
      t.live = true;
      mla_load_item(t, sTab, p, C);
      float l_t[kHS];
#pragma unroll
      for (int h = 0; h < kHS; ++h) l_t[h] = 0.0f;
      bool o_live = false;
      for (; t.i < t.ntiles && ok; ++t.i, ++n) {
        const int b = n & 1;
        if (!mbar_wait_bounded(&bar_qk_done[b], (n >> 1) & 1)) { ok = false; break; }
        // token validity was written before sc_free of this tile completed (already complete: the K warps
        // arrive on it after the last slab, which this QK read)
        if (!mbar_wait_bounded(&bar_sc_free[b], (n >> 1) & 1)) { ok = false; break; }
        mla_fence_after();
        const bool valid = sValid[b * kTile + tt] != 0;
        const uint32_t s_base = tS + b * 64 + h0 + lane_base;
        // One pass over the scores: does any score move its head's running max (one vote per warp, one
        // barrier)?  P is formed with the current running maxima at the same time; it is final unless a
        // maximum moves, which the lazy rescale makes rare, and then it is formed again.
        uint32_t pw[kHS / 2];
        // d = s * scale - m per head: a max moves when d > 2^8 headroom; p = 2^d (2^-inf = 0 for invalid
        // tokens and padded heads; the +inf of a head without a max yet is never used: its vote fires)
        auto form_p = [&](bool& moved) {
#pragma unroll
          for (int g = 0; g < kHS / 16; ++g) {
            float s[16];
            mla_ld16(s_base + g * 16, s);
            float m[16];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const float4 m4 = *reinterpret_cast<const float4*>(sM + h0 + g * 16 + 4 * q4);
              m[4 * q4] = m4.x; m[4 * q4 + 1] = m4.y; m[4 * q4 + 2] = m4.z; m[4 * q4 + 3] = m4.w;
            }
            bool mv = false;
#pragma unroll
            for (int h2 = 0; h2 < 8; ++h2) {
              float pr[2];
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const float d = valid ? fmaf(s[2 * h2 + e], p.score_scale, -m[2 * h2 + e]) : -INFINITY;
                mv |= d > kLazyRescale;
                pr[e] = mla_ex2(d);
              }
              pw[g * 8 + h2] = pack_bf16x2(pr[0], pr[1]);
            }
            moved |= mv;
          }
        };
        bool moved = false;
        form_p(moved);
        const int wv = __any_sync(0xffffffffu, moved);
        if (lane == 0) sFlag[warp] = wv;
        mla_named_sync(1, kSmWarps * 32);
        int fl = 0;
#pragma unroll
        for (int w = 0; w < kSmWarps; ++w) fl |= sFlag[w];
        const bool any_moved = fl != 0;
        bool rescale = false;
        if (any_moved) {  // uniform branch: exact tile maxima, new running maxima, rescale factors
          mla_named_sync(1, kSmWarps * 32);  // sFlag has been read by every warp
#pragma unroll 1
          for (int g = 0; g < kHS / 16; ++g) {
            float s[16];
            mla_ld16(s_base + g * 16, s);
#pragma unroll
            for (int h = 0; h < 16; ++h) {
              float mx = (valid && h0 + g * 16 + h < HP) ? s[h] * p.score_scale : -INFINITY;
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
              if (lane == 0) sRed[warp * kHS + g * 16 + h] = mx;
            }
          }
          mla_named_sync(1, kSmWarps * 32);
          if (tid < kHG) {  // thread tid updates head tid: the four warps of its half hold its maxima
            const int half = tid / kHS, idx = tid % kHS;
            float mx = -INFINITY;
#pragma unroll
            for (int w = 0; w < 4; ++w) mx = fmaxf(mx, sRed[(half * 4 + w) * kHS + idx]);
            const float m = sM[tid];  // kNoMax before the head's first valid score; +inf for padded heads
            float a = 1.0f;
            if (mx > -INFINITY && mx > m + kLazyRescale) {
              if (m != kNoMax) a = exp2f(m - mx);
              sM[tid] = mx;
            }
            sA[tid] = a;
          }
          mla_named_sync(1, kSmWarps * 32);
#pragma unroll
          for (int h = 0; h < kHS; ++h) rescale |= sA[h0 + h] != 1.0f;
          bool unused = false;
          form_p(unused);  // P with the new running maxima
        }
        mla_named_sync(1, kSmWarps * 32);  // sFlag / sRed are rewritten next tile
        // P is single-buffered: the previous tile's PV must be complete before it is rewritten (and
        // before O is rescaled)
        if (n >= 1 && !mbar_wait_bounded(&bar_pv_done[(n - 1) & 1], ((n - 1) >> 1) & 1)) { ok = false; break; }
        mla_fence_after();
        if (rescale && o_live) {
#pragma unroll 1
          for (int c = 0; c < kVBlocks; ++c) {
#pragma unroll 1
            for (int g = 0; g < kHS / 16; ++g) {
              float o[16];
              mla_ld16(tO + c * 64 + h0 + g * 16 + lane_base, o);
              uint32_t r[16];
#pragma unroll
              for (int h = 0; h < 16; ++h) r[h] = __float_as_uint(o[h] * sA[h0 + g * 16 + h]);
              mla_st16(tO + c * 64 + h0 + g * 16 + lane_base, r);
            }
          }
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        }
        // P row of this token for heads h0 .. h0 + 31 (bf16) and the row sums of exactly those values
#pragma unroll
        for (int g = 0; g < kHS / 16; ++g) {
#pragma unroll
          for (int h2 = 0; h2 < 8; ++h2) {
            const float2 pb = unpack_bf16x2(pw[g * 8 + h2]);
            const int h = g * 16 + 2 * h2;
            const float a0 = any_moved ? sA[h0 + h] : 1.0f, a1 = any_moved ? sA[h0 + h + 1] : 1.0f;
            l_t[h] = fmaf(l_t[h], a0, pb.x);
            l_t[h + 1] = fmaf(l_t[h + 1], a1, pb.y);
          }
          const int hg8 = (h0 + g * 16) / 8;  // 8-head group of pw[8g .. 8g + 3]
          *reinterpret_cast<uint4*>(sP + (tt % 8) * 16 + (tt / 8) * 128 + hg8 * kPS) =
              make_uint4(pw[g * 8 + 0], pw[g * 8 + 1], pw[g * 8 + 2], pw[g * 8 + 3]);
          *reinterpret_cast<uint4*>(sP + (tt % 8) * 16 + (tt / 8) * 128 + (hg8 + 1) * kPS) =
              make_uint4(pw[g * 8 + 4], pw[g * 8 + 5], pw[g * 8 + 6], pw[g * 8 + 7]);
        }
        o_live = true;
        fence_proxy_async_smem();
        mla_fence_before();
        __syncwarp();
        if (lane == 0) mla_arrive(&bar_p_full[b]);
      }
      if (!ok) break;
      // ---- item end: O^T -> partials (thread = dim within each 128-dim block); (m, l) per head
      if (!mbar_wait_bounded(&bar_pv_done[(n - 1) & 1], ((n - 1) >> 1) & 1)) { ok = false; break; }
      mla_fence_after();
      float* acc = p.part_acc + static_cast<int64_t>(item) * HP * kDV;
#pragma unroll 1
      for (int c = 0; c < kVBlocks; ++c) {
#pragma unroll 1
        for (int g = 0; g < kHS / 16; ++g) {
          float o[16];
          mla_ld16(tO + c * 64 + h0 + g * 16 + lane_base, o);
#pragma unroll
          for (int h = 0; h < 16; ++h) {
            const int hd = h0 + g * 16 + h;
            if (hd < HP) acc[static_cast<int64_t>(hd) * kDV + c * 128 + tt] = o[h];
          }
        }
      }
#pragma unroll
      for (int h = 0; h < kHS; ++h) {
        float v = l_t[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) sRed[warp * kHS + h] = v;
      }
      mla_named_sync(1, kSmWarps * 32);
      if (tid < kHG) {
        if (tid < HP) {
          const int half = tid / kHS, idx = tid % kHS;
          float lsum = 0.0f;
#pragma unroll
          for (int w = 0; w < 4; ++w) lsum += sRed[(half * 4 + w) * kHS + idx];
          const float m = sM[tid];
          p.part_ml[(static_cast<int64_t>(item) * HP + tid) * 2 + 0] = m == kNoMax ? -INFINITY : m;
          p.part_ml[(static_cast<int64_t>(item) * HP + tid) * 2 + 1] = lsum;
        }
        sM[tid] = tid < HP ? kNoMax : INFINITY;  // the next item starts afresh
      }
      mla_fence_before();
      mla_named_sync(1, kSmWarps * 32);
    }
  }
  if (!ok) set_status(p.status, kStatusTimeout);
  mla_fence_before();
  __syncthreads();
  mla_fence_after();
  if (warp == kMmaWarp)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
}

using EncodeTiledFnMla = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                      const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                      CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFnMla mla_encoder() {
  static const EncodeTiledFnMla fn = []() -> EncodeTiledFnMla {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFnMla>(f);
  }();
  return fn;
}

// 2-D view of the latent code pool [page * 16 + token][576]; a box is 128 code bytes of 16 rows.
bool encode_mla_map(CUtensorMap* map, const DecodeArgs& a) {
  const EncodeTiledFnMla enc = mla_encoder();
  if (!enc) return false;
  const cuuint64_t rows = static_cast<cuuint64_t>(std::max<int64_t>(a.num_pages, 1)) * kPage;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(mla::kD), rows};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(mla::kD)};
  const cuuint32_t box[2] = {128, kPage};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(a.codes), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int32_t decode_mla_tc_heads_per_item(int32_t group) { return group <= mla::kHG ? group : mla::kHG; }

bool decode_mla_tc_supported(int32_t head_dim, int32_t v_dim, int32_t is_mla, int32_t group, int32_t batch) {
  return is_mla && head_dim == mla::kD && v_dim == mla::kDV && group > 0 &&
         (group <= mla::kHG || group % mla::kHG == 0) && batch <= mla::kMaxBatch;
}

kvq_status launch_decode_mla_tc(const DecodeArgs& a, cudaStream_t stream) {
  decltype(&decode_mla_kernel<KVQ_FP8_E4M3>) kern = nullptr;
  switch (a.kind) {
    case KVQ_FP8_E4M3: kern = decode_mla_kernel<KVQ_FP8_E4M3>; break;
    case KVQ_Q8_0: kern = decode_mla_kernel<KVQ_Q8_0>; break;
    case KVQ_FP8_E4M3_UNSCALED: kern = decode_mla_kernel<KVQ_FP8_E4M3_UNSCALED>; break;
    case KVQ_FP8_E5M2_UNSCALED: kern = decode_mla_kernel<KVQ_FP8_E5M2_UNSCALED>; break;
  }
  if (kern == nullptr) return KVQ_EKIND;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, mla::SMEM_BYTES) != cudaSuccess)
    return KVQ_ECUDA;
  CUtensorMap map;
  if (!encode_mla_map(&map, a)) return KVQ_ECUDA;
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const KParams p = make_kparams(a);
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(a.max_items, sms));
  kern<<<static_cast<unsigned>(grid), mla::kThreads, mla::SMEM_BYTES, stream>>>(p, map);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ECUDA;
}

}  // namespace kvq
