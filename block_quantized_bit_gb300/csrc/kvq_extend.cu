// kvq_extend.cu -- extend (prefill) attention over the 8-bit pool on the tcgen05 tensor cores.
//
// "feat(kvcache): 8-bit KV cache (q8_0 / fp8_e4m3) behind --kv-cache-dtype", section "What": the dequant
// sits inside every attention kernel, prefill included, and K and V are dequantized to bf16 before the dot
// (the scale runs along the reduction dim).  "feat(kvcache): 8-bit DSV4 window/compressed KV", section
// "Testing": quantized attention on the prefill kernel, masked -1 pages.
//
// The n_b new tokens of sequence b are the last n_b of its seq_len stored tokens; token i sits at position
// seq_len - n_b + i and attends to the unmasked positions up to and including its own.  The query side is
// wide, so the contraction takes the flash-attention shape.  A work item is (sequence, kv head g, block of
// 128 query rows); row r holds new token blk * (128 / G) + r / G and query head g * G + r % G, so the G
// heads of a kv head share every dequantized K and V tile:
//   S[128 rows][T keys]  = Q[128][D] . Kd[T][D]^T   (A = Q, B = the K tile; both K-major in shared memory)
//   O[128 rows][D]      += P[128][T] . Vd[T][D]     (A = P in tensor memory, B = the V tile read MN-major)
// with fp32 S and O in tensor memory.  Q, K and V use the canonical no-swizzle core-matrix layout
//   off(t, d) = (t % 8) * 16 + (t / 8) * RS + (d % 8) * 2 + (d / 8) * 128,   RS = D * 16,
// with t the row (query row or key): K-major descriptors take LBO = 128 and SBO = RS, the MN-major one
// LBO = RS and SBO = 128.  T = 128 keys per tile at D = 128 and 64 at D = 256 (shared memory).
// P enters the MMA as bf16.  The SPLIT instances feed it as two bf16 terms, P = hi + lo with hi = bf16(p)
// and lo = bf16(p - hi), through a second PV into the same O: the product then carries P to about 2^-17
// relative instead of 2^-9, for twice the PV MMAs.  (All their exponentials run on the MUFU unit: the FMA-
// pipe cubic's 1.5e-4 would otherwise dominate that error.)
//
// One persistent CTA per SM, 19 warps:
//   warps 17-18 producers, one for K and one for V: TMA copies of a tile's codes (128-byte swizzled boxes of
//               16 tokens x 128 code bytes) and bulk copies of their scales into that producer's staging ring,
//               with each page's number of valid tokens; the block table is read one tile ahead.
//   warps 8-15  dequant: a thread owns 64 codes of one token row, of K and then of V.  K of tile j + 1 is
//               written before V of tile j, so the next QK never waits for the V tile.
//   warp 16     allocates tensor memory and issues every MMA (one elected lane): QK of tile j, then PV of
//               tile j - 1, so the softmax of tile j overlaps the tensor pipe.
//   warps 0-7   softmax: warps q and q + 4 own the 32 query rows of tensor-memory lane quarter q (one row
//               per thread) and each takes half of a tile's keys and of O's columns; the two exchange
//               their half-tile maxima and, per item, their row sums through shared memory, meeting on
//               bounded mbarriers.  Causal and page masks (one warp-uniform branch per tile picks a
//               straight-line unmasked or masked variant), online softmax in the exp2 domain with lazy
//               rescaling (the running max moves only when a score passes it by more than 2^8), a quarter
//               of the exponentials on the FMA pipe, P as bf16 into tensor memory.  At an item's end they
//               write the next item's Q rows, then O / l to the output.
// Every wait is bounded (2 s) and reports a timeout in the status word instead of hanging.
#include <cuda.h>
#include <math.h>

#include <algorithm>
#include <type_traits>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_tc.cuh"

namespace kvq {
namespace {

constexpr int kM = 128;  // query rows per item (the MMA M)
constexpr int kSmWarps = 8;  // two per tensor-memory lane quarter, each on half of a tile's keys
constexpr int kDwWarps = 8;
constexpr int kMmaWarp = kSmWarps + kDwWarps;   // warp 16
constexpr int kProdWarp = kMmaWarp + 1;         // warps 17 (K ring) and 18 (V ring)
constexpr int kThreads = (kProdWarp + 2) * 32;  // 19 warps
constexpr int kDwThreads = kDwWarps * 32;
constexpr int kTmemCols = 512;
constexpr int kBox = kPage * 128;      // one TMA box: 16 tokens x 128 code bytes
constexpr float kLazyRescale = 8.0f;   // log2 headroom before the running max must move

template <int D>
struct XCfg {
  static constexpr int T = (D == 128) ? 128 : 64;  // keys per tile
  static constexpr int PPT = T / kPage;            // pages per tile
  static constexpr int RS = D * 16;                // bytes between 8-row groups of a tile
  static constexpr int KV_TILE = T * D * 2;        // one bf16 K or V tile
  static constexpr int Q_BYTES = kM * D * 2;
  static constexpr int PARTS = kDwThreads / T;     // dequant threads per token row
  static constexpr int SPAN = D / PARTS;           // codes per dequant thread (of K, and of V)
  static constexpr int NCH = SPAN / 16;            // 16-code chunks per dequant thread
  static constexpr int NBT = SPAN / 32;            // scale blocks per dequant thread
  static constexpr int NB = D / 32;
  static constexpr int NSL = D / 128;              // 128-byte slices of a code row
  static constexpr int SC_KV = kPage * NB * 2;     // scale bytes of one page of K or of V
  // a ring slot (of the K ring or of the V ring): codes [page][slice] boxes as TMA wrote them, then the
  // scales [page].  The K ring is freed as soon as K is dequantized, the V ring only after the previous PV,
  // so the two rings run at their own pace and the K ring runs deeper.
  static constexpr int CODE_BYTES = PPT * NSL * kBox;
  static constexpr int SLOT_BYTES = CODE_BYTES + PPT * SC_KV;
  static constexpr int KSTAGES = 3;
  static constexpr int VSTAGES = (D == 128) ? 3 : 2;
  static constexpr int NSLOTS = KSTAGES + VSTAGES;  // K ring slots, then V ring slots
  static constexpr int RING_OFF = 0;  // 1024-byte aligned: swizzle atoms
  static constexpr int K_OFF = RING_OFF + NSLOTS * SLOT_BYTES;
  static constexpr int V_OFF = K_OFF + KV_TILE;
  static constexpr int Q_OFF = V_OFF + KV_TILE;
  static constexpr int META_OFF = Q_OFF + Q_BYTES;              // [NSLOTS][PPT] valid tokens per page
  static constexpr int RED_OFF = META_OFF + NSLOTS * PPT * 4;   // [2 parities][2 halves][128 rows] row maxima
  static constexpr int SUM_OFF = RED_OFF + 2 * 2 * kM * 4;      // [2 item parities][2 halves][128 rows] row sums
  static constexpr int TAB_OFF = SUM_OFF + 2 * 2 * kM * 4;      // [batch + 1] first item of each sequence
  static constexpr int NBARS = 2 * NSLOTS + 10 + 12;
  static constexpr int BAR_OFF = (TAB_OFF + (kMaxExtendBatch + 1) * 4 + 15) / 16 * 16;  // mbarriers: 8-byte aligned
  static constexpr int SMEM_BYTES = BAR_OFF + NBARS * 8 + 16 + 1024;  // + slack to align the base
  // tensor-memory columns: O [0, D); S buffer b [D + b T, D + (b + 1) T); P buffer b [384 + b T / 2, ...)
  static constexpr int S_COL = D;
  static constexpr int P_COL = 384;
  // the low P terms of the SPLIT instances: buffer b at [PLO_COL + b T / 2, ...) where those columns are
  // free (D = 256); else (D = 128) inside S buffer b, which the softmax has read when it forms them: half hf
  // of the keys puts its T / 4 columns at the start of its own T / 2 columns of S.  Tensor-core operations
  // of different accumulators are not ordered among themselves, so then the QK that next writes S buffer b
  // waits for the PV that read those columns.
  static constexpr int PLO_COL = P_COL + T;
  static constexpr bool LO_IN_S = PLO_COL + T > kTmemCols;
  static_assert(D == 128 || D == 256, "extend needs head_dim 128 or 256");
  static_assert(D + 2 * T <= P_COL && P_COL + T <= kTmemCols, "tensor-memory columns");
  static_assert(PARTS * T == kDwThreads && NCH % 2 == 0 && NBT == 2, "dequant split");
  static_assert(SLOT_BYTES % 1024 == 0, "slots keep the boxes 1024-byte aligned");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
  static_assert(K_OFF % 16 == 0 && V_OFF % 16 == 0 && Q_OFF % 16 == 0 && BAR_OFF % 8 == 0, "alignment");
};

// kind::f16 instruction descriptor: fp32 accumulate, bf16 A and B, M = 128, the given N; A K-major.
__device__ __forceinline__ uint32_t x_idesc(int n, bool b_mn_major) {
  uint32_t d = 0;
  d |= 1u << 4;   // D: f32
  d |= 1u << 7;   // A: bf16
  d |= 1u << 10;  // B: bf16
  d |= static_cast<uint32_t>(b_mn_major) << 16;
  d |= static_cast<uint32_t>(n >> 3) << 17;
  d |= static_cast<uint32_t>(kM >> 4) << 24;
  return d;
}

__device__ __forceinline__ void bar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// The new tokens of sequence b after validation: 0 <= n <= seq_len and q_start[b + 1] <= total_q, else none
// (the status word then reports the bad sequence).
__device__ __forceinline__ int32_t new_tokens(const ExtendArgs& a, int32_t b, bool report) {
  const int32_t q0 = __ldg(a.q_start + b), q1 = __ldg(a.q_start + b + 1);
  const int32_t n = q1 - q0;
  if (q0 < 0 || n < 0 || q1 > a.total_q || n > __ldg(a.seq_lens + b)) {
    if (report) set_status(a.status, kStatusBadExtend);
    return 0;
  }
  return n;
}

// One work item: sequence b, kv head g, query block blk; its rows' positions end at pos_max.
struct XItem {
  int32_t b, g, blk, n, L, q0, pos_max, ntiles;
};

template <int D>
__device__ __forceinline__ XItem x_locate(const int32_t* tab, const ExtendArgs& a, int32_t G, int32_t item) {
  using Cfg = XCfg<D>;
  int lo = 0, hi = a.batch;  // first b with tab[b] > item
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (tab[mid] <= item) lo = mid + 1;
    else hi = mid;
  }
  XItem it;
  it.b = lo - 1;
  it.L = __ldg(a.seq_lens + it.b);
  it.q0 = __ldg(a.q_start + it.b);
  it.n = new_tokens(a, it.b, false);
  const int32_t tb = kM / G;                   // new tokens per block
  const int32_t nblk = (it.n + tb - 1) / tb;
  const int32_t k = item - tab[it.b];
  it.blk = nblk - 1 - k / a.num_kv_heads;      // the last blocks (the most keys) first
  it.g = k % a.num_kv_heads;
  const int32_t last_tok = min(it.n, (it.blk + 1) * tb) - 1;
  it.pos_max = it.L - it.n + last_tok;
  it.ntiles = it.pos_max / Cfg::T + 1;
  return it;
}

// The sequence of (item, tile) pairs a persistent CTA works through.
template <int D>
struct XIter {
  XItem it;
  int32_t item, i, n_items;
  bool live;
  __device__ __forceinline__ void first(const int32_t* tab, const ExtendArgs& a, int32_t G, int32_t total) {
    n_items = total;
    item = blockIdx.x;
    i = 0;
    live = item < n_items;
    if (live) it = x_locate<D>(tab, a, G, item);
  }
  __device__ __forceinline__ void next(const int32_t* tab, const ExtendArgs& a, int32_t G) {
    if (!live) return;
    if (++i < it.ntiles) return;
    i = 0;
    item += gridDim.x;
    live = item < n_items;
    if (live) it = x_locate<D>(tab, a, G, item);
  }
};

// Tensor-memory loads and stores of 32 consecutive columns of this warp's 32 lanes.  A load's registers are
// valid only after tcgen05.wait::ld; the waits below take them as operands, so no use moves above the wait.
__device__ __forceinline__ void tmem_ld32_issue(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {"
      "%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31"
      "}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  tmem_ld32_issue(taddr, r);
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                 "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
  tmem_ld32_issue(taddr, r);
  tmem_ld32_issue(taddr + 32, r + 32);
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                 "+r"(r[29]), "+r"(r[30]), "+r"(r[31]), "+r"(r[32]), "+r"(r[33]), "+r"(r[34]), "+r"(r[35]),
                 "+r"(r[36]), "+r"(r[37]), "+r"(r[38]), "+r"(r[39]), "+r"(r[40]), "+r"(r[41]), "+r"(r[42]),
                 "+r"(r[43]), "+r"(r[44]), "+r"(r[45]), "+r"(r[46]), "+r"(r[47]), "+r"(r[48]), "+r"(r[49]),
                 "+r"(r[50]), "+r"(r[51]), "+r"(r[52]), "+r"(r[53]), "+r"(r[54]), "+r"(r[55]), "+r"(r[56]),
                 "+r"(r[57]), "+r"(r[58]), "+r"(r[59]), "+r"(r[60]), "+r"(r[61]), "+r"(r[62]), "+r"(r[63])
               :
               : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {"
      "%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32"
      "};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
      "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]),
      "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// 2^x by the hardware approximation (relative error far below the bf16 rounding that follows); 2^-inf = 0.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 2^x on the FMA pipe, for a share of the probabilities (the MUFU unit alone would pace the softmax):
// x = j + f with j = round(x) by the 1.5 * 2^23 addition (the sum's low mantissa bits hold j) and f in
// [-0.5, 0.5]; 2^f by a cubic; j added to the exponent field.  The cubic's coefficients are a minimax fit of
// 2^f on [-0.5, 0.5] for relative error, computed by Lawson's iteratively reweighted least squares on
// Chebyshev nodes (the weights grow where the error is largest until it equioscillates), then rounded to
// fp32.  Relative error at most 1.5e-4 over [-126, 8] (kvq_exp2_probe exposes this routine so that a test
// checks the bound on the GPU), far below the bf16 rounding of P that follows.  x is clamped at -126 (the
// result is then about 2^-126, not 0: callers zero masked keys themselves).
__device__ __forceinline__ float ex2_fma(float x) {
  x = fmaxf(x, -126.0f);
  const float t = x + 12582912.0f;
  const int j = __float_as_int(t) - 0x4B400000;
  const float f = x - (t - 12582912.0f);
  const float p = fmaf(fmaf(fmaf(0.0551716685f, f, 0.2426111251f), f, 0.6932609677f), f, 0.9999280572f);
  return __int_as_float(__float_as_int(p) + (j << 23));
}

// A bounded wait that the whole warp agrees on: no lane runs ahead into a warp-collective tcgen05 instruction
// while another gave up.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity));
}

template <int D, int KIND, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1) extend_tc_kernel(const ExtendArgs a, const __grid_constant__ CUtensorMap tmap) {
  using Cfg = XCfg<D>;
  constexpr int T = Cfg::T;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);  // swizzle atoms are 1024 B
  uint8_t* sRing = smem + Cfg::RING_OFF;
  uint8_t* sK = smem + Cfg::K_OFF;
  uint8_t* sV = smem + Cfg::V_OFF;
  uint8_t* sQ = smem + Cfg::Q_OFF;
  int32_t* sMeta = reinterpret_cast<int32_t*>(smem + Cfg::META_OFF);
  int32_t* sTab = reinterpret_cast<int32_t*>(smem + Cfg::TAB_OFF);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::BAR_OFF);
  // Every barrier completes once per use of its buffer, so a waiter names an unambiguous phase.
  uint64_t* bar_full = bars;                      // [NSLOTS] ring slot landed (producer arrival + bytes)
  uint64_t* bar_empty = bars + Cfg::NSLOTS;       // [NSLOTS] ring slot read by every dequant warp
  uint64_t* bar_k_full = bars + 2 * Cfg::NSLOTS;  // K tile written (dequant warps), once per tile
  uint64_t* bar_v_full = bar_k_full + 1;          // V tile written (dequant warps), once per tile
  uint64_t* bar_qk_done = bar_k_full + 2;         // [2] QK into S buffer b completed (commit)
  uint64_t* bar_pv_done = bar_k_full + 4;         // [2] PV that read P buffer b completed (commit)
  uint64_t* bar_p_full = bar_k_full + 6;          // [2] P buffer b written, S buffer b read (softmax warps)
  uint64_t* bar_q_full = bar_k_full + 8;          // an item's Q rows written (softmax warps), once per item
  uint64_t* bar_o_free = bar_k_full + 9;          // an item's O read out (softmax warps), once per item
  uint64_t* bar_pair = bar_k_full + 10;           // [4 quarters][2 parities] both half-tile maxima written
  uint64_t* bar_sum = bar_k_full + 18;            // [4 quarters] both half row sums written, once per item
  uint32_t* sTmem = reinterpret_cast<uint32_t*>(smem + Cfg::BAR_OFF + Cfg::NBARS * 8);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t G = a.num_q_heads / a.num_kv_heads;

  // ---- plan: first item of every sequence (items of a sequence: query blocks x kv heads)
  if (tid == 0) {
    int32_t run = 0;
    for (int32_t b = 0; b < a.batch; ++b) {
      sTab[b] = run;
      const int32_t n = new_tokens(a, b, blockIdx.x == 0);
      run += ((n * G + kM - 1) / kM) * a.num_kv_heads;
    }
    sTab[a.batch] = run;
    for (int s = 0; s < Cfg::NSLOTS; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], kDwWarps);
    }
    mbar_init(bar_k_full, kDwWarps);
    mbar_init(bar_v_full, kDwWarps);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar_qk_done[b], 1);
      mbar_init(&bar_pv_done[b], 1);
      mbar_init(&bar_p_full[b], kSmWarps);
    }
    mbar_init(bar_q_full, kSmWarps);
    mbar_init(bar_o_free, kSmWarps);
    for (int i = 0; i < 12; ++i) mbar_init(&bar_pair[i], 2);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(sTmem)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sTmem;
  const int32_t n_items = sTab[a.batch];
  bool ok = true;

  if (warp >= kProdWarp) {
    // ===================================================================== producers
    // Warp 13 fills the K ring, warp 14 the V ring.  Lane pi (< PPT) owns page pi of a tile: its block-table
    // entry (read one tile ahead), valid tokens and copies.
    const int kv = warp - kProdWarp;
    const int stages = kv ? Cfg::VSTAGES : Cfg::KSTAGES;
    const int base = kv ? Cfg::KSTAGES : 0;
    auto page_entry = [&](const XIter<D>& ti) -> int32_t {
      if (!ti.live || lane >= Cfg::PPT) return -1;
      const int32_t pg = ti.i * Cfg::PPT + lane;
      if (pg >= a.max_pages || pg * kPage >= ti.it.L) return -1;
      return __ldg(a.block_table + static_cast<int64_t>(ti.it.b) * a.max_pages + pg);
    };
    XIter<D> t;
    t.first(sTab, a, G, n_items);
    int32_t bt = page_entry(t);
    uint32_t n = 0;  // tiles issued
    while (ok && t.live) {
      int32_t phys = bt, nvalid = 0;
      if (phys >= a.num_pages) {  // never dereferenced; reported in the status word
        set_status(a.status, kStatusBadPage);
        phys = -1;
      }
      if (phys >= 0) nvalid = min(kPage, t.it.L - (t.i * Cfg::PPT + lane) * kPage);
      XIter<D> nx = t;
      nx.next(sTab, a, G);
      bt = page_entry(nx);
      const int sl = base + static_cast<int>(n % stages);
      const uint32_t use = n / stages;
      if (use > 0 && !warp_wait(&bar_empty[sl], (use - 1) & 1)) { ok = false; break; }
      constexpr uint32_t kPageBytes = Cfg::NSL * kBox + (KindTraits<KIND>::kScaled ? Cfg::SC_KV : 0);
      const uint32_t bytes = __reduce_add_sync(0xffffffffu, phys >= 0 ? kPageBytes : 0u);
      int32_t nv[Cfg::PPT];
#pragma unroll
      for (int i = 0; i < Cfg::PPT; ++i) nv[i] = __shfl_sync(0xffffffffu, nvalid, i);
      if (lane == 0) {
#pragma unroll
        for (int i = 0; i < Cfg::PPT; ++i) sMeta[sl * Cfg::PPT + i] = nv[i];
        mbar_arrive_expect_tx(&bar_full[sl], bytes);  // releases the page counts with the slot
      }
      __syncwarp();
      if (phys >= 0) {
        uint8_t* slot = sRing + sl * Cfg::SLOT_BYTES;
#pragma unroll
        for (int c = 0; c < Cfg::NSL; ++c)
          tma_load_codes(smem_u32(slot + (lane * Cfg::NSL + c) * kBox), &tmap, c, t.it.g * kPage, kv, phys,
                         &bar_full[sl]);
        if (KindTraits<KIND>::kScaled) {  // an unscaled pool has codes only
          const uint8_t* src = reinterpret_cast<const uint8_t*>(a.scales) +
                               ((static_cast<int64_t>(phys) * 2 + kv) * a.num_kv_heads + t.it.g) * Cfg::SC_KV;
          bulk_g2s(slot + Cfg::CODE_BYTES + lane * Cfg::SC_KV, src, Cfg::SC_KV, &bar_full[sl]);
        }
      }
      t = nx;
      ++n;
    }
    // no copy may still be in flight when the CTA exits
    for (uint32_t j = 1; j <= n && j <= static_cast<uint32_t>(stages); ++j) {
      const uint32_t m = n - j;
      (void)mbar_wait_bounded(&bar_full[base + m % stages], (m / stages) & 1);
    }
  } else if (warp >= kSmWarps && warp < kMmaWarp) {
    // ===================================================================== dequant warps
    const int dw = tid - kSmWarps * 32;
    const int tt = dw % T;     // key of the tile (consecutive threads: consecutive keys)
    const int part = dw / T;   // which SPAN of the row
    const int pi = tt / kPage, off = tt % kPage;
    const int swz = off & 7;   // 128-byte swizzle phase of this token's staging rows
    const uint32_t toff = (tt % 8) * 16 + (tt / 8) * Cfg::RS;
    // dequantize this thread's codes of K or V from a ring slot into a bf16 tile
    auto write_tile = [&](uint8_t* dst, const uint8_t* slot, bool v_ok) {
      const uint8_t* rows = slot + pi * Cfg::NSL * kBox + off * 128;
      const uint32_t sc = KindTraits<KIND>::kScaled ? *reinterpret_cast<const uint32_t*>(
          slot + Cfg::CODE_BYTES + pi * Cfg::SC_KV + (off * Cfg::NB + part * Cfg::NBT) * 2) : 0u;
#pragma unroll
      for (int k = 0; k < Cfg::NCH; ++k) {
        uint32_t w[8];
        if (v_ok) {
          const int c = part * Cfg::NCH + k;  // 16-code chunk along the row
          const uint4 codes = *reinterpret_cast<const uint4*>(rows + (c / 8) * kBox + (((c % 8) ^ swz) * 16));
          dequant16<KIND>(codes, static_cast<uint16_t>(sc >> (16 * (k >> 1))), w);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) w[e] = 0u;
        }
        const int d8 = part * (Cfg::SPAN / 8) + 2 * k;
        *reinterpret_cast<uint4*>(dst + toff + d8 * 128) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(dst + toff + (d8 + 1) * 128) = make_uint4(w[4], w[5], w[6], w[7]);
      }
      fence_proxy_async_smem();
      __syncwarp();
    };
    XIter<D> tk;  // next tile whose K is dequantized
    tk.first(sTab, a, G, n_items);
    uint32_t nk = 0, nv = 0;  // tiles whose K / V have been written
    while (ok && (tk.live || nv < nk)) {
      if (tk.live) {
        const int ring = nk % Cfg::KSTAGES;
        if (!warp_wait(&bar_full[ring], (nk / Cfg::KSTAGES) & 1)) { ok = false; break; }
        const uint8_t* slot = sRing + ring * Cfg::SLOT_BYTES;
        const bool v_ok = off < sMeta[ring * Cfg::PPT + pi];
        // the K tile was last read by the QK of tile nk - 1
        if (nk >= 1 && !warp_wait(&bar_qk_done[(nk - 1) & 1], ((nk - 1) >> 1) & 1)) { ok = false; break; }
        write_tile(sK, slot, v_ok);
        if (lane == 0) {
          bar_arrive(bar_k_full);
          bar_arrive(&bar_empty[ring]);
        }
        tk.next(sTab, a, G);
        ++nk;
        if (nk == 1 && tk.live) continue;  // K runs one tile ahead of V
      }
      {
        const int ring = Cfg::KSTAGES + nv % Cfg::VSTAGES;
        if (!warp_wait(&bar_full[ring], (nv / Cfg::VSTAGES) & 1)) { ok = false; break; }
        const uint8_t* slot = sRing + ring * Cfg::SLOT_BYTES;
        const bool v_ok = off < sMeta[ring * Cfg::PPT + pi];
        // the V tile was last read by the PV of tile nv - 1
        if (nv >= 1 && !warp_wait(&bar_pv_done[(nv - 1) & 1], ((nv - 1) >> 1) & 1)) { ok = false; break; }
        write_tile(sV, slot, v_ok);
        if (lane == 0) {
          bar_arrive(bar_v_full);
          bar_arrive(&bar_empty[ring]);
        }
        ++nv;
      }
    }
  } else if (warp == kMmaWarp) {
    // ===================================================================== MMA issue (elected lane)
    const uint32_t idesc_qk = x_idesc(T, false);
    const uint32_t idesc_pv = x_idesc(D, true);
    // descriptors of the first K-step; later steps add their byte offset >> 4 to the address field
    const uint64_t dQ = smem_desc(smem_u32(sQ), 128, Cfg::RS);
    const uint64_t dK = smem_desc(smem_u32(sK), 128, Cfg::RS);
    const uint64_t dV = smem_desc(smem_u32(sV), Cfg::RS, 128);
    const uint32_t tS = tmem + Cfg::S_COL, tO = tmem, tP = tmem + Cfg::P_COL;
    // column of the low P terms of k-step ks (16 keys) of buffer bp (SPLIT)
    auto lo_col = [&](int bp, int ks) -> uint32_t {
      if constexpr (Cfg::LO_IN_S)
        return tmem + Cfg::S_COL + bp * T + (ks / (T / 32)) * (T / 2) + (ks % (T / 32)) * 8;
      else
        return tmem + Cfg::PLO_COL + bp * (T / 2) + ks * 8;
    };
    uint32_t n = 0, items = 0;  // tiles QK'd; items finished
    // PV of tile m; the first tile of an item overwrites O, once the previous item's O has been read out
    auto pv = [&](uint32_t m, bool first) -> bool {
      const int bp = m & 1;
      if (!warp_wait(bar_v_full, m & 1)) return false;
      if (!warp_wait(&bar_p_full[bp], (m >> 1) & 1)) return false;
      if (first && items >= 1 && !warp_wait(bar_o_free, (items - 1) & 1)) return false;
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < T / 16; ++ks)
        mma_bf16_tmem_a(tO, tP + bp * (T / 2) + ks * 8, dV + static_cast<uint64_t>((ks * 2 * Cfg::RS) >> 4),
                        idesc_pv, (!first || ks > 0) ? 1u : 0u);
      if constexpr (SPLIT) {
#pragma unroll
        for (int ks = 0; ks < T / 16; ++ks)
          mma_bf16_tmem_a(tO, lo_col(bp, ks), dV + static_cast<uint64_t>((ks * 2 * Cfg::RS) >> 4), idesc_pv, 1u);
      }
      mma_commit(&bar_pv_done[bp]);
      __syncwarp();
      return true;
    };
    for (int32_t item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
      const XItem it = x_locate<D>(sTab, a, G, item);
      if (!warp_wait(bar_q_full, items & 1)) { ok = false; break; }
      for (int32_t i = 0; i < it.ntiles; ++i, ++n) {
        const int b = n & 1;
        if (!warp_wait(bar_k_full, n & 1)) { ok = false; break; }
        // S buffer b was read by the softmax of tile n - 2 (and, holding low P terms, by the PV of tile n - 2)
        if (n >= 2 && !warp_wait(&bar_p_full[b], ((n >> 1) - 1) & 1)) { ok = false; break; }
        if constexpr (SPLIT && Cfg::LO_IN_S) {
          if (n >= 2 && !warp_wait(&bar_pv_done[b], ((n >> 1) - 1) & 1)) { ok = false; break; }
        }
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          mma_bf16(tS + b * T, dQ + static_cast<uint64_t>((ks * 256) >> 4), dK + static_cast<uint64_t>((ks * 256) >> 4),
                   idesc_qk, ks > 0 ? 1u : 0u);
        mma_commit(&bar_qk_done[b]);
        __syncwarp();
        if (i > 0 && !pv(n - 1, i == 1)) { ok = false; break; }
      }
      if (!ok) break;
      if (!pv(n - 1, it.ntiles == 1)) { ok = false; break; }
      ++items;
    }
    // before tensor memory is freed, every MMA issued must have completed (the last commit implies all)
    if (n > 0) (void)mbar_wait_bounded(&bar_pv_done[(n - 1) & 1], ((n - 1) >> 1) & 1);
    if (n > 0) (void)mbar_wait_bounded(&bar_qk_done[(n - 1) & 1], ((n - 1) >> 1) & 1);
  } else {
    // ===================================================================== softmax warps
    const int quarter = warp & 3, hf = warp >> 2;  // lane quarter; which half of the keys and of O
    const int r = quarter * 32 + lane;             // query row = tensor-memory lane
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + Cfg::S_COL + lane_base + hf * (T / 2);
    const uint32_t tO = tmem + lane_base + hf * (D / 2);
    const uint32_t tP = tmem + Cfg::P_COL + lane_base + hf * (T / 4);
    // this warp's low P terms of buffer b start at tPlo + b * PLO_STRIDE (SPLIT)
    const uint32_t tPlo = Cfg::LO_IN_S ? tS : tmem + Cfg::PLO_COL + lane_base + hf * (T / 4);
    constexpr int PLO_STRIDE = Cfg::LO_IN_S ? T : T / 2;
    float* sRed = reinterpret_cast<float*>(smem + Cfg::RED_OFF);
    float* sSum = reinterpret_cast<float*>(smem + Cfg::SUM_OFF);
    const int32_t tb = kM / G;  // new tokens per query block
    // this warp's half of the item's Q rows into the shared tile (rows past the new tokens are zero)
    auto write_q = [&](const XItem& it) {
      const int32_t tok = it.blk * tb + r / G;
      const bool valid = tok < it.n;
      const uint4* src = reinterpret_cast<const uint4*>(
          a.q + (static_cast<int64_t>(it.q0 + (valid ? tok : 0)) * a.num_q_heads + it.g * G + r % G) * D);
      uint8_t* dst = sQ + (r % 8) * 16 + (r / 8) * Cfg::RS;
#pragma unroll 4
      for (int j = hf * (D / 16); j < (hf + 1) * (D / 16); ++j)
        *reinterpret_cast<uint4*>(dst + j * 128) = valid ? __ldg(src + j) : make_uint4(0, 0, 0, 0);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) bar_arrive(bar_q_full);
    };
    // the two warps of a lane quarter meet on mbarriers (bounded waits: a warp that gave up cannot strand
    // the other)
    auto pair_meet = [&](uint64_t* bar, uint32_t parity) -> bool {
      __syncwarp();
      if (lane == 0) bar_arrive(bar);
      return warp_wait(bar, parity);
    };
    uint32_t n = 0, items = 0;  // tiles processed; items finished
    if (static_cast<int32_t>(blockIdx.x) < n_items) write_q(x_locate<D>(sTab, a, G, blockIdx.x));
    for (int32_t item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
      const XItem it = x_locate<D>(sTab, a, G, item);
      const int32_t tok = it.blk * tb + r / G;
      const bool row_ok = tok < it.n;
      const int32_t pos = row_ok ? it.L - it.n + tok : -1;  // last key position this row sees
      float m_used = -INFINITY, l = 0.0f;
      // lane pi (< PPT) holds the block-table entry of page pi of a tile, read one tile ahead of its use
      auto fetch = [&](int32_t i) -> int32_t {
        const int32_t pg = i * Cfg::PPT + lane;
        if (lane >= Cfg::PPT || i >= it.ntiles || pg >= a.max_pages || pg * kPage >= it.L) return -1;
        return __ldg(a.block_table + static_cast<int64_t>(it.b) * a.max_pages + pg);
      };
      int32_t ent = fetch(0);
      for (int32_t i = 0; i < it.ntiles; ++i, ++n) {
        const int b = n & 1;
        // mapped pages of the tile (chunk c of 16 keys is page c of the tile)
        const uint32_t pmask = __ballot_sync(0xffffffffu, ent >= 0 && ent < a.num_pages) & ((1u << Cfg::PPT) - 1u);
        ent = fetch(i + 1);
        const int32_t lim = pos - i * T - hf * (T / 2);  // keys k <= lim of this warp's half are visible
        const uint32_t hmask = pmask >> (hf * Cfg::PPT / 2);  // this half's pages
        if (!warp_wait(&bar_qk_done[b], (n >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
        // every row of the warp sees every key of its half (no causal edge, no masked page): no masking.  The
        // two variants of each pass are separate straight-line loops behind one warp-uniform branch.
        const bool full = __all_sync(0xffffffffu, lim >= T / 2 - 1) && (hmask & ((1u << (Cfg::PPT / 2)) - 1u)) ==
                                                                         (1u << (Cfg::PPT / 2)) - 1u;
        // pass 1: the row's max over the visible keys of this half (sm_scale > 0: scaling commutes with it)
        float mh = -INFINITY;
        auto pass1 = [&](auto masked) {
          float m[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
          for (int h = 0; h < T / 64; ++h) {
            uint32_t v[32];
            tmem_ld32(tS + b * T + h * 32, v);
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              float x = __uint_as_float(v[e]);
              if constexpr (decltype(masked)::value) {
                const int k = h * 32 + e;
                const bool vis = (((hmask >> (k / kPage)) & 1u) != 0u) & (k <= lim);
                x = vis ? x : -INFINITY;
              }
              m[e & 3] = fmaxf(m[e & 3], x);
            }
          }
          mh = fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
        };
        if (full) pass1(std::false_type{});
        else pass1(std::true_type{});
        // the row's max over the whole tile: exchange halves with the other warp of the lane quarter
        // (double-buffered by tile parity, so one barrier per tile suffices)
        sRed[(b * 2 + hf) * kM + r] = mh;
        if (!pair_meet(&bar_pair[quarter * 2 + b], (n >> 1) & 1)) { ok = false; break; }
        float mx = fmaxf(sRed[(b * 2) * kM + r], sRed[(b * 2 + 1) * kM + r]);
        if (mx > -INFINITY) mx *= a.score_scale;
        float alpha = 1.0f;
        bool resc = false;
        if (mx > -INFINITY && (m_used == -INFINITY || mx > m_used + kLazyRescale)) {
          if (m_used != -INFINITY) {
            alpha = ex2(m_used - mx);
            resc = true;
          }
          m_used = mx;
        }
        // P buffer b is free once the PV two tiles back has read it
        if (n >= 2 && !warp_wait(&bar_pv_done[b], ((n >> 1) - 1) & 1)) { ok = false; break; }
        if (__any_sync(0xffffffffu, resc)) {  // (only from the second tile of an item on)
          // O must hold the PV of the previous tile before it is scaled; this warp scales its half of O
          if (!warp_wait(&bar_pv_done[(n - 1) & 1], ((n - 1) >> 1) & 1)) { ok = false; break; }
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < D / 64; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + c * 32, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tO + c * 32, o);
          }
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
          l *= alpha;
        }
        // pass 2: P = 2^(s * scale - m) of this half as bf16 into tensor memory; the row sum in fp32
        auto pass2 = [&](auto masked) {
          float ls[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 1
          for (int h = 0; h < T / 64; ++h) {
            uint32_t v[32];
            tmem_ld32(tS + b * T + h * 32, v);
            uint32_t w[16], wl[SPLIT ? 16 : 1];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float x0 = fmaf(__uint_as_float(v[2 * e]), a.score_scale, -m_used);
              const float x1 = fmaf(__uint_as_float(v[2 * e + 1]), a.score_scale, -m_used);
              // every fourth pair on the FMA pipe, the rest on the MUFU unit
              const bool fma_pipe = !SPLIT && (e & 3) == 3;
              float p0 = fma_pipe ? ex2_fma(x0) : ex2(x0);
              float p1 = fma_pipe ? ex2_fma(x1) : ex2(x1);
              if constexpr (decltype(masked)::value) {
                const int k = h * 32 + 2 * e;  // k and k + 1 share a page
                const bool pg = ((hmask >> (k / kPage)) & 1u) != 0u;
                p0 = (pg & (k <= lim)) ? p0 : 0.0f;
                p1 = (pg & (k + 1 <= lim)) ? p1 : 0.0f;
              }
              ls[(2 * e) & 3] += p0;
              ls[(2 * e + 1) & 3] += p1;
              w[e] = pack_bf16x2(p0, p1);
              if constexpr (SPLIT) {
                const float2 hv = unpack_bf16x2(w[e]);  // p - bf16(p) is exact in fp32
                wl[e] = pack_bf16x2(p0 - hv.x, p1 - hv.y);
              }
            }
            tmem_st16u(tP + b * (T / 2) + h * 16, w);
            // (in S: columns [16 h, 16 h + 16) of this half, all loaded by now)
            if constexpr (SPLIT) tmem_st16u(tPlo + b * PLO_STRIDE + h * 16, wl);
          }
          l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        };
        if (full) pass2(std::false_type{});
        else pass2(std::true_type{});
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) bar_arrive(&bar_p_full[b]);
      }
      if (!ok) break;
      // the next item's Q rows (every QK of this item has completed: its last S was read above)
      const int32_t nxt = item + static_cast<int32_t>(gridDim.x);
      if (nxt < n_items) write_q(x_locate<D>(sTab, a, G, nxt));
      // the row sum over both halves (double-buffered by item parity)
      float* sum = sSum + (items & 1) * 2 * kM;
      sum[hf * kM + r] = l;
      if (!pair_meet(&bar_sum[quarter], items & 1)) { ok = false; break; }
      const float lt = sum[r] + sum[kM + r];
      ++items;
      // this warp's half of O / l, once the item's last PV has completed
      if (!warp_wait(&bar_pv_done[(n - 1) & 1], ((n - 1) >> 1) & 1)) { ok = false; break; }
      tc_fence_after();
      const float inv = lt > 0.0f ? 1.0f / lt : 0.0f;
      const int64_t orow =
          (static_cast<int64_t>(it.q0 + (row_ok ? tok : 0)) * a.num_q_heads + it.g * G + r % G) * D + hf * (D / 2);
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {
        uint32_t ov[32];
        tmem_ld32(tO + c * 32, ov);
        if (row_ok) {
          float o[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __uint_as_float(ov[e]) * inv;
          if (a.out_dtype == KVQ_OUT_F32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.out) + orow + c * 32);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) dst[q4] = make_float4(o[4 * q4], o[4 * q4 + 1], o[4 * q4 + 2], o[4 * q4 + 3]);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + orow + c * 32);
#pragma unroll
            for (int h8 = 0; h8 < 4; ++h8)
              dst[h8] = make_uint4(pack_bf16x2(o[8 * h8], o[8 * h8 + 1]), pack_bf16x2(o[8 * h8 + 2], o[8 * h8 + 3]),
                                   pack_bf16x2(o[8 * h8 + 4], o[8 * h8 + 5]), pack_bf16x2(o[8 * h8 + 6], o[8 * h8 + 7]));
          }
        }
      }
      tc_fence_before();  // the reads are ordered before the arrival that lets the next PV overwrite O
      __syncwarp();
      if (lane == 0) bar_arrive(bar_o_free);
    }
  }
  if (!ok) set_status(a.status, kStatusTimeout);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
}

__global__ void exp2_probe_kernel(const float* __restrict__ x, float* __restrict__ y, int64_t n) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    y[i] = ex2_fma(x[i]);
}

template <int D, bool SPLIT>
kvq_status launch_extend_d(const ExtendArgs& a, cudaStream_t stream) {
  using Cfg = XCfg<D>;
  decltype(&extend_tc_kernel<D, KVQ_FP8_E4M3, SPLIT>) kern = nullptr;
  switch (a.kind) {
    case KVQ_FP8_E4M3: kern = extend_tc_kernel<D, KVQ_FP8_E4M3, SPLIT>; break;
    case KVQ_Q8_0: kern = extend_tc_kernel<D, KVQ_Q8_0, SPLIT>; break;
    case KVQ_FP8_E4M3_UNSCALED: kern = extend_tc_kernel<D, KVQ_FP8_E4M3_UNSCALED, SPLIT>; break;
    case KVQ_FP8_E5M2_UNSCALED: kern = extend_tc_kernel<D, KVQ_FP8_E5M2_UNSCALED, SPLIT>; break;
  }
  if (kern == nullptr) return KVQ_EKIND;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) != cudaSuccess)
    return KVQ_ECUDA;
  CUtensorMap map;
  if (!encode_code_map(&map, a.codes, a.num_pages, a.num_kv_heads, D)) return KVQ_ECUDA;
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t G = a.num_q_heads / a.num_kv_heads;
  const int64_t bound = ((static_cast<int64_t>(a.total_q) * G + kM - 1) / kM + a.batch) * a.num_kv_heads;
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(bound, sms));
  kern<<<static_cast<unsigned>(grid), kThreads, Cfg::SMEM_BYTES, stream>>>(a, map);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ECUDA;
}

}  // namespace

bool extend_tc_supported(int32_t head_dim, int32_t v_dim, int32_t mla, int32_t group, int32_t batch) {
  if (mla || v_dim != head_dim) return false;
  if (head_dim != 128 && head_dim != 256) return false;
  return group >= 1 && group <= kM && kM % group == 0 && batch <= kMaxExtendBatch;
}

kvq_status launch_exp2_probe(const float* x, float* y, int64_t n, cudaStream_t stream) {
  if (n == 0) return KVQ_OK;
  const int threads = 256;
  const int64_t grid = std::min<int64_t>((n + threads - 1) / threads, 152 * 8);
  exp2_probe_kernel<<<static_cast<unsigned>(grid), threads, 0, stream>>>(x, y, n);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ECUDA;
}

namespace {
// One CTA per sequence: new token i of sequence b (query row q_start[b] + i) sits at position
// seq_lens[b] - n_b + i and attends to the prefix of seq_lens[b] - n_b + i + 1 positions.
__global__ void extend_expand_kernel(const int32_t* __restrict__ q_start, const int32_t* __restrict__ seq_lens,
                                     int32_t total_q, int32_t* __restrict__ vlens, int32_t* __restrict__ vrow,
                                     uint32_t* status) {
  const int32_t b = blockIdx.x;
  const int32_t q0 = __ldg(q_start + b), q1 = __ldg(q_start + b + 1), L = __ldg(seq_lens + b);
  const int32_t n = q1 - q0;
  if (q0 < 0 || n < 0 || n > L || q1 > total_q) {
    if (threadIdx.x == 0) set_status(status, kStatusBadExtend);
    return;
  }
  for (int32_t i = threadIdx.x; i < n; i += blockDim.x) {
    vlens[q0 + i] = L - n + i + 1;
    vrow[q0 + i] = b;
  }
}
}  // namespace

kvq_status launch_extend_expand(const int32_t* q_start, const int32_t* seq_lens, int32_t batch, int32_t total_q,
                                int32_t* vlens, int32_t* vrow, uint32_t* status, cudaStream_t stream) {
  if (batch == 0) return KVQ_OK;
  extend_expand_kernel<<<static_cast<unsigned>(batch), 256, 0, stream>>>(q_start, seq_lens, total_q, vlens, vrow,
                                                                         status);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ECUDA;
}

kvq_status launch_extend_tc(const ExtendArgs& a, cudaStream_t stream) {
  if (a.head_dim == 128) return a.split_p ? launch_extend_d<128, true>(a, stream) : launch_extend_d<128, false>(a, stream);
  if (a.head_dim == 256) return a.split_p ? launch_extend_d<256, true>(a, stream) : launch_extend_d<256, false>(a, stream);
  return KVQ_EUNSUPPORTED;
}

}  // namespace kvq
