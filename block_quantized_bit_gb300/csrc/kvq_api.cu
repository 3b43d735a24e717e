// kvq_api.cu -- the C ABI of libkvq: argument validation, the pool cost model, workspace sizing and
// kernel dispatch.  Every check runs on the host before any launch; a rejected call touches nothing.
//
// Cost model: "feat(kvcache): 8-bit KV cache (q8_0 / fp8_e4m3) behind --kv-cache-dtype", section "What"
// (1.0625 bytes per element: one code byte plus an fp16 scale per 32 elements) and its review comment's
// "End-to-end numbers" (the KV pool grows by 2 / 1.0625 at the same budget).  "feat(kvcache): 8-bit
// DSV4 window/compressed KV", section "One ordering trap": the budget must be priced with the same
// bytes-per-token the pool uses, which is why both come from this one function.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <limits>

#include "../../include/kvq.h"
#include "kvq_internal.h"

namespace kvq {

namespace {

constexpr size_t kAlign = 16;
constexpr uint32_t kStatusTimeoutWord = 0x7100u;  // written by a kernel that gave up a bounded wait

bool aligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) % kAlign) == 0; }

int n_kv_of(const kvq_layout& L) { return L.mla ? 1 : 2; }

kvq_status check_layout(const kvq_layout* L) {
  if (L == nullptr) return KVQ_EINVAL;
  if (L->num_pages < 0 || L->page_size <= 0 || L->num_kv_heads <= 0) return KVQ_EINVAL;
  if (L->mla != 0 && L->mla != 1) return KVQ_EINVAL;
  if (L->head_dim <= 0 || L->head_dim % 32 != 0) return KVQ_EHEADDIM;
  if (L->v_dim <= 0 || L->v_dim % 32 != 0) return KVQ_EHEADDIM;
  if (!L->mla && L->v_dim != L->head_dim) return KVQ_EINVAL;
  if (L->mla && L->v_dim > L->head_dim) return KVQ_EINVAL;
  // element count must fit comfortably in int64 / size_t
  const double elems = static_cast<double>(L->num_pages) * n_kv_of(*L) * L->num_kv_heads * L->page_size *
                       static_cast<double>(L->head_dim);
  if (elems > 4.0e18) return KVQ_EINVAL;
  return KVQ_OK;
}

bool kind_ok(int kind) { return kind == KVQ_FP8_E4M3 || kind == KVQ_Q8_0; }

// Kinds the attention entry points read: the block-scaled ones and the unscaled fp8 casts.
bool kind_read_ok(int kind) { return kind_ok(kind) || kind == KVQ_FP8_E4M3_UNSCALED || kind == KVQ_FP8_E5M2_UNSCALED; }

// The unscaled kinds have no scale array: their scales pointer is ignored (it may be NULL).
bool has_scales(int kind) { return kind_ok(kind); }

// SMs of the current device (the MLA tensor-core plan targets one work item per SM).
int32_t sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      sms <= 0)
    return kTargetItems;
  return sms;
}

size_t elems_of(const kvq_layout& L) {
  return static_cast<size_t>(L.num_pages) * n_kv_of(L) * L.num_kv_heads * L.page_size * L.head_dim;
}

struct WorkspacePlan {
  int32_t path;
  int32_t split_align;
  int32_t target_items;
  int32_t heads_per_item;
  int32_t query_groups;
  int64_t max_items;
  size_t cnt_offset, acc_offset, ml_offset, tab_offset, total;
};

// 1 = CUDA-core kernel, 2 = tensor-core kernel, -1 = the requested path has no kernel for this shape.
// Automatic: tensor cores where QK^T and PV are dense enough -- 8..16 query heads per kv head, or an MLA
// pool read by a multiple of 64 query heads whose block tables can hold at least kMlaTcMinTokens tokens
// in all (the MLA tensor-core kernel costs ~50 us however short the contexts: at batch 1 it measured 54
// us at 256 and 1024 tokens against 21 and 58 us on the CUDA cores); the GQA tensor-core kernel also
// runs 1..7 heads (padded), but measured slower there than the CUDA cores.
constexpr int64_t kMlaTcMinTokens = 1024;

int32_t choose_path(const kvq_layout& L, int32_t batch, int32_t num_q_heads, int32_t max_pages,
                    const kvq_decode_options* opt) {
  const int32_t group = num_q_heads / L.num_kv_heads;
  const bool tc = L.mla ? decode_mla_tc_supported(L.head_dim, L.v_dim, L.mla, group, batch)
                        : decode_tc_supported(L.head_dim, L.v_dim, L.mla, group, batch);
  const bool cc = decode_cc_supported(L.head_dim, L.v_dim, L.mla);
  const int32_t want = opt ? opt->path : 0;
  if (want == 2) return tc ? 2 : -1;
  if (want == 1) return cc ? 1 : -1;
  const bool long_mla = static_cast<int64_t>(batch) * max_pages * kPageTokens >= kMlaTcMinTokens;
  if (tc && (L.mla ? long_mla : group >= 8)) return 2;
  return cc ? 1 : -1;
}

bool plan_workspace(const kvq_layout& L, int32_t batch, int32_t num_q_heads, int32_t max_pages,
                    const kvq_decode_options* opt, WorkspacePlan* w) {
  if (batch < 0 || num_q_heads <= 0 || max_pages <= 0) return false;
  if (num_q_heads % L.num_kv_heads != 0) return false;
  const int32_t group = num_q_heads / L.num_kv_heads;
  const int32_t pps = opt ? opt->pages_per_split : 0;
  if (pps < 0) return false;
  const int32_t path = choose_path(L, batch, num_q_heads, max_pages, opt);
  w->path = path;
  if (path == 2 && L.mla) w->heads_per_item = decode_mla_tc_heads_per_item(group);
  else w->heads_per_item = (path == 2) ? group : cc_heads_per_item(group, L.head_dim, L.mla);
  w->split_align = (path == 2) ? 8 : 1;
  // Tensor-core items are expensive to start and finish (a pipeline fill, a q tile, an O readout, and
  // partials the merge must read): the GQA kernel aims at about two items per SM, the MLA kernel
  // (64 query rows of 576, 64 x 512 partial outputs) at one.
  // CUDA-core items: a little under two waves of the resident CTAs, because each sequence's last split
  // is partial and rounds the count up (qwen3_1p7b: 1240 items against 2 x 608 slots at the full two
  // waves).
  w->target_items = (path == 2) ? (L.mla ? sm_count() : 2 * sm_count())
                                : std::max<int32_t>(64, 19 * cc_ctas_per_sm(L.head_dim, L.mla, w->heads_per_item) *
                                                            sm_count() / 10);
  w->query_groups = L.num_kv_heads * (group / w->heads_per_item);
  w->max_items = max_work_items(batch, w->query_groups, max_pages, pps, w->target_items);
  const size_t acc = static_cast<size_t>(w->max_items) * w->heads_per_item * L.v_dim * sizeof(float);
  const size_t ml = static_cast<size_t>(w->max_items) * w->heads_per_item * 2 * sizeof(float);
  // split counters of the fused merge (CUDA-core path) follow the header: one memset clears both
  const size_t cnt = static_cast<size_t>(batch) * w->query_groups * sizeof(int32_t);
  w->cnt_offset = kWorkspaceHeader;
  w->acc_offset = w->cnt_offset + ((cnt + 255) / 256) * 256;
  w->ml_offset = w->acc_offset + ((acc + 255) / 256) * 256;
  w->tab_offset = w->ml_offset + ((ml + 255) / 256) * 256;
  const size_t tab = static_cast<size_t>(batch) * 2 * sizeof(int32_t);
  w->total = w->tab_offset + ((tab + 255) / 256) * 256;
  return true;
}

}  // namespace

int64_t max_work_items(int32_t batch, int32_t query_groups, int32_t max_pages, int32_t pages_per_split,
                       int32_t target_items) {
  const int64_t per_seq = static_cast<int64_t>(query_groups);
  if (pages_per_split > 0)
    return static_cast<int64_t>(batch) * per_seq * ((max_pages + pages_per_split - 1) / pages_per_split);
  const int64_t upper = static_cast<int64_t>(batch) * per_seq * ((max_pages + kMinPagesPerSplit - 1) / kMinPagesPerSplit);
  return std::min<int64_t>(upper, static_cast<int64_t>(target_items) + static_cast<int64_t>(batch) * per_seq);
}

}  // namespace kvq

using namespace kvq;

namespace {

kvq_status decode_common(const void* q, const void* pool, const void* scales, const int32_t* block_table,
                         int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                         float sm_scale, void* out, kvq_out_dtype out_dtype, void* workspace,
                         size_t workspace_bytes, const kvq_layout* layout, kvq_kind kind,
                         const kvq_decode_options* options, void* stream, bool clear_status,
                         const int32_t* bt_row = nullptr) {
  kvq_status st = check_layout(layout);
  if (st != KVQ_OK) return st;
  if (!kind_read_ok(kind)) return KVQ_EKIND;
  if (!has_scales(kind)) scales = nullptr;
  if (out_dtype != KVQ_OUT_BF16 && out_dtype != KVQ_OUT_F32) return KVQ_EINVAL;
  if (batch < 0 || num_q_heads <= 0 || max_pages_per_seq <= 0) return KVQ_EINVAL;
  if (num_q_heads % layout->num_kv_heads != 0) return KVQ_EINVAL;
  if (!(sm_scale == sm_scale) || sm_scale > std::numeric_limits<float>::max() ||
      sm_scale < -std::numeric_limits<float>::max())
    return KVQ_EINVAL;
  if (options && (options->pages_per_split < 0 || options->path < 0 || options->path > 2)) return KVQ_EINVAL;
  if (layout->page_size != kPageTokens) return KVQ_EUNSUPPORTED;
  WorkspacePlan w;
  if (!plan_workspace(*layout, batch, num_q_heads, max_pages_per_seq, options, &w)) return KVQ_EINVAL;
  if (w.path < 0) return KVQ_EUNSUPPORTED;
  if (batch == 0) return KVQ_OK;
  if (!q || !pool || (has_scales(kind) && !scales) || !block_table || !seq_lens || !out || !workspace)
    return KVQ_EINVAL;
  if (workspace_bytes < w.total) return KVQ_EWORKSPACE;
  if (!aligned(q) || !aligned(pool) || !aligned(scales) || !aligned(out) || !aligned(workspace) ||
      (reinterpret_cast<uintptr_t>(block_table) % 4) != 0 || (reinterpret_cast<uintptr_t>(seq_lens) % 4) != 0)
    return KVQ_EALIGN;
  st = kvq_device_check();
  if (st != KVQ_OK) return st;

  DecodeArgs a;
  a.q = q;
  a.codes = static_cast<const uint8_t*>(pool);
  a.scales = static_cast<const uint16_t*>(scales);
  a.block_table = block_table;
  a.bt_row = bt_row;
  a.num_pages = layout->num_pages;
  a.max_pages = max_pages_per_seq;
  a.seq_lens = seq_lens;
  a.batch = batch;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = layout->num_kv_heads;
  a.head_dim = layout->head_dim;
  a.v_dim = layout->v_dim;
  a.mla = layout->mla;
  a.sm_scale = sm_scale;
  a.out = out;
  a.out_dtype = out_dtype;
  a.kind = kind;
  a.pages_per_split = options ? options->pages_per_split : 0;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.status = reinterpret_cast<uint32_t*>(ws);
  a.part_acc = reinterpret_cast<float*>(ws + w.acc_offset);
  a.part_ml = reinterpret_cast<float*>(ws + w.ml_offset);
  a.plan_tab = reinterpret_cast<int32_t*>(ws + w.tab_offset);
  a.split_cnt = (w.path == 1) ? reinterpret_cast<int32_t*>(ws + w.cnt_offset) : nullptr;
  a.max_items = w.max_items;
  a.heads_per_item = w.heads_per_item;
  a.split_align = w.split_align;
  a.target_items = w.target_items;
  // the GQA tensor-core kernel: one item per SM when the splits come out even (no second pipeline fill
  // and O readout per SM, half the partials to merge), else about two
  a.one_wave_items = (w.path == 2 && !layout->mla) ? sm_count() : 0;
  a.min_one_split = (w.path == 1) ? 1 : 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // status word and split counters (the counters only on the CUDA-core path, which merges in-kernel)
  // (a caller that already recorded errors in the status word, the sparse decode, keeps it)
  const size_t clear = (w.path == 1) ? w.acc_offset : sizeof(uint32_t);
  const size_t from = clear_status ? 0 : kWorkspaceHeader;
  if (clear > from && cudaMemsetAsync(ws + from, 0, clear - from, s) != cudaSuccess) return KVQ_ECUDA;
  if (w.path == 2) st = a.mla ? launch_decode_mla_tc(a, s) : launch_decode_tc(a, s);
  else return launch_decode_cc(a, s);
  if (st != KVQ_OK) return st;
  return launch_merge(a, w.query_groups, s);
}

// Sparse decode: the dense decode's workspace first (its status word at offset 0 is the call's), then
// the compact pool, its block table and its sequence lengths.  cpages = ceil(topk / 16) pages per
// sequence hold every column a list can select.
struct SparsePlan {
  kvq_layout compact;
  int32_t cpages;
  size_t dense_bytes, codes_offset, scales_offset, table_offset, lens_offset, total;
};

bool plan_sparse(const kvq_layout* layout, int32_t batch, int32_t num_q_heads, int32_t topk, SparsePlan* sp) {
  if (check_layout(layout) != KVQ_OK) return false;
  if (batch < 0 || num_q_heads <= 0 || topk < 0 || topk > kMaxSparseTopk) return false;
  if (num_q_heads % layout->num_kv_heads != 0) return false;
  sp->cpages = std::max<int32_t>(1, (topk + kPageTokens - 1) / kPageTokens);
  sp->compact = *layout;
  sp->compact.num_pages = static_cast<int64_t>(std::max<int32_t>(batch, 1)) * sp->cpages;
  WorkspacePlan w;
  if (!plan_workspace(sp->compact, batch, num_q_heads, sp->cpages, nullptr, &w)) return false;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t n_kv = layout->mla ? 1 : 2;
  const size_t rows = static_cast<size_t>(sp->compact.num_pages) * kPageTokens * n_kv * layout->num_kv_heads;
  sp->dense_bytes = up(w.total);
  sp->codes_offset = sp->dense_bytes;
  sp->scales_offset = sp->codes_offset + up(rows * layout->head_dim);
  sp->table_offset = sp->scales_offset + up(rows * (layout->head_dim / 32) * sizeof(uint16_t));
  sp->lens_offset = sp->table_offset + up(static_cast<size_t>(sp->compact.num_pages) * sizeof(int32_t));
  sp->total = sp->lens_offset + up(static_cast<size_t>(std::max<int32_t>(batch, 1)) * sizeof(int32_t));
  return true;
}

// Extend by prefixes: every new token is a sequence of its own (its causal prefix, the block-table row of the
// sequence it belongs to), decoded in chunks of at most kExtendChunk tokens by the decode kernels.  This is
// how the MLA latent row is extended, and the GQA path when the flash kernel cannot serve the shape or the
// caller asks for fp32 probabilities.  Workspace: the decode workspace of one chunk (its status word at
// offset 0 is the call's), then the per-token prefix lengths and block-table rows.
constexpr int32_t kExtendChunk = 1024;

struct ExtendPlan {
  bool flash;              // the GQA flash-style tcgen05 kernel (else: prefixes through the decode kernels)
  bool split;              // the flash kernel feeds P as two bf16 terms
  kvq_decode_options dec;  // the decode kernel choice of the prefix path
  int32_t chunk;
  size_t dense_bytes, lens_offset, rows_offset, total;
};

// The extend's kernel choice and workspace.  False: invalid sizes or options, or no kernel for the shape.
bool plan_extend(const kvq_layout& L, int32_t total_q, int32_t num_q_heads, int32_t max_pages,
                 const kvq_extend_options* o, ExtendPlan* ep) {
  const int32_t path = o ? o->path : 0;
  const bool precise = o && o->precise_p != 0;
  if (path < 0 || path > 2 || total_q < 0 || num_q_heads <= 0 || max_pages <= 0) return false;
  if (num_q_heads % L.num_kv_heads != 0) return false;
  const int32_t group = num_q_heads / L.num_kv_heads;
  // the batch bound is checked per call; any batch up to it gives the same choice
  const bool flash_ok = extend_tc_supported(L.head_dim, L.v_dim, L.mla, group, 1);
  ep->flash = !L.mla && (path == 2 || (path == 0 && flash_ok));
  ep->split = ep->flash && precise;
  ep->dec.pages_per_split = 0;
  ep->dec.path = path == 1 ? 1 : (path == 2 ? 2 : 0);
  if (!ep->flash && precise) {
    if (path == 2) return false;  // the tensor-core decode keeps P in bf16
    ep->dec.path = 1;
  }
  if (ep->flash) {
    ep->chunk = 0;
    ep->dense_bytes = ep->lens_offset = ep->rows_offset = ep->total = kWorkspaceHeader;
    return flash_ok;
  }
  ep->chunk = std::max<int32_t>(1, std::min<int32_t>(total_q, kExtendChunk));
  WorkspacePlan w;
  if (!plan_workspace(L, ep->chunk, num_q_heads, max_pages, &ep->dec, &w) || w.path < 0) return false;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t n = static_cast<size_t>(std::max<int32_t>(total_q, 1)) * sizeof(int32_t);
  ep->dense_bytes = up(w.total);
  ep->lens_offset = ep->dense_bytes;
  ep->rows_offset = ep->lens_offset + up(n);
  ep->total = ep->rows_offset + up(n);
  return true;
}

kvq_status extend_prefixes(const ExtendPlan& ep, const void* q, const void* pool, const void* scales,
                           const int32_t* block_table, int32_t max_pages_per_seq, const int32_t* seq_lens,
                           const int32_t* q_start, int32_t total_q, int32_t batch, int32_t num_q_heads, float sm_scale,
                           void* out, kvq_out_dtype out_dtype, void* workspace, const kvq_layout* layout,
                           kvq_kind kind, cudaStream_t s) {
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* vlens = reinterpret_cast<int32_t*>(ws + ep.lens_offset);
  int32_t* vrow = reinterpret_cast<int32_t*>(ws + ep.rows_offset);
  // rows no sequence covers (an inconsistent q_start) keep length 0: zeros out
  if (cudaMemsetAsync(ws + ep.lens_offset, 0, ep.total - ep.lens_offset, s) != cudaSuccess) return KVQ_ECUDA;
  kvq_status st =
      launch_extend_expand(q_start, seq_lens, batch, total_q, vlens, vrow, reinterpret_cast<uint32_t*>(ws), s);
  if (st != KVQ_OK) return st;
  const size_t q_row = static_cast<size_t>(num_q_heads) * layout->head_dim * 2;
  const size_t o_row = static_cast<size_t>(num_q_heads) * layout->v_dim * (out_dtype == KVQ_OUT_F32 ? 4 : 2);
  for (int32_t c0 = 0; c0 < total_q; c0 += ep.chunk) {
    const int32_t n = std::min<int32_t>(ep.chunk, total_q - c0);
    st = decode_common(static_cast<const uint8_t*>(q) + c0 * q_row, pool, scales, block_table, max_pages_per_seq,
                       vlens + c0, n, num_q_heads, sm_scale, static_cast<uint8_t*>(out) + c0 * o_row, out_dtype,
                       workspace, ep.dense_bytes, layout, kind, &ep.dec, s, false, vrow + c0);
    if (st != KVQ_OK) return st;
  }
  return KVQ_OK;
}

}  // namespace


extern "C" {

const char* kvq_version(void) { return "0.1.0"; }

const char* kvq_strerror(kvq_status s) {
  switch (s) {
    case KVQ_OK: return "ok";
    case KVQ_EINVAL: return "invalid argument";
    case KVQ_EKIND:
      return "quantization kind not accepted by this call (the block-scaled stores take KVQ_FP8_E4M3 or KVQ_Q8_0; "
             "kvq_store_unscaled the unscaled kinds; the attention calls all four)";
    case KVQ_EHEADDIM: return "head_dim and v_dim must be positive multiples of 32 (the quantization block)";
    case KVQ_EALIGN: return "device pointers must be 16-byte aligned";
    case KVQ_EWORKSPACE: return "workspace smaller than kvq_decode_workspace_bytes()";
    case KVQ_EARCH: return "current device is not compute capability 10.3 (GB300, sm_103a)";
    case KVQ_ECUDA: return "a CUDA call or kernel launch failed";
    case KVQ_EUNSUPPORTED: return "no decode kernel for this page size / head_dim / path";
    case KVQ_ETIMEOUT: return "a kernel gave up a bounded wait; its output is not valid";
  }
  return "unknown status";
}

size_t kvq_pool_bytes(const kvq_layout* layout) {
  if (check_layout(layout) != KVQ_OK) return 0;
  return elems_of(*layout);
}

size_t kvq_scale_bytes(const kvq_layout* layout) {
  if (check_layout(layout) != KVQ_OK) return 0;
  return elems_of(*layout) / 32 * 2;
}

double kvq_bytes_per_token(const kvq_layout* layout) {
  if (check_layout(layout) != KVQ_OK) return -1.0;
  const double elems = static_cast<double>(n_kv_of(*layout)) * layout->num_kv_heads * layout->head_dim;
  return elems + elems / 32.0 * 2.0;
}

int64_t kvq_num_pages(const kvq_layout* layout, size_t budget_bytes) {
  if (check_layout(layout) != KVQ_OK) return -1;
  const uint64_t elems_per_page =
      static_cast<uint64_t>(n_kv_of(*layout)) * layout->num_kv_heads * layout->page_size * layout->head_dim;
  const uint64_t bytes_per_page = elems_per_page + elems_per_page / 32 * 2;
  return static_cast<int64_t>(budget_bytes / bytes_per_page);
}

double kvq_bytes_per_token_ex(const kvq_layout* layout, kvq_kind kind) {
  if (check_layout(layout) != KVQ_OK || !kind_read_ok(kind)) return -1.0;
  if (has_scales(kind)) return kvq_bytes_per_token(layout);
  return static_cast<double>(n_kv_of(*layout)) * layout->num_kv_heads * layout->head_dim;
}

int64_t kvq_num_pages_ex(const kvq_layout* layout, kvq_kind kind, size_t budget_bytes) {
  if (check_layout(layout) != KVQ_OK || !kind_read_ok(kind)) return -1;
  if (has_scales(kind)) return kvq_num_pages(layout, budget_bytes);
  const uint64_t bytes_per_page =
      static_cast<uint64_t>(n_kv_of(*layout)) * layout->num_kv_heads * layout->page_size * layout->head_dim;
  return static_cast<int64_t>(budget_bytes / bytes_per_page);
}

kvq_status kvq_device_check(void) {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ECUDA;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return KVQ_ECUDA;
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return KVQ_ECUDA;
  if (major != 10 || minor != 3) return KVQ_EARCH;
  return KVQ_OK;
}

kvq_status kvq_store(void* pool, void* scales, const void* k, const void* v, const int64_t* slot_mapping,
                     int64_t num_tokens, const kvq_layout* layout, kvq_kind kind, void* stream) {
  kvq_status st = check_layout(layout);
  if (st != KVQ_OK) return st;
  if (!kind_ok(kind)) return KVQ_EKIND;
  if (num_tokens < 0) return KVQ_EINVAL;
  if (layout->mla ? (v != nullptr) : false) return KVQ_EINVAL;
  if (num_tokens == 0) return KVQ_OK;
  if (!pool || !scales || !k || !slot_mapping || (!layout->mla && !v)) return KVQ_EINVAL;
  if (!aligned(pool) || !aligned(scales) || !aligned(k) || (v && !aligned(v)) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) % 8) != 0)
    return KVQ_EALIGN;
  st = kvq_device_check();
  if (st != KVQ_OK) return st;
  return launch_store(pool, scales, k, v, slot_mapping, num_tokens, *layout, kind,
                      static_cast<cudaStream_t>(stream));
}

int32_t kvq_decode_path(const kvq_layout* layout, int32_t batch, int32_t num_q_heads, int32_t max_pages_per_seq,
                        const kvq_decode_options* options) {
  if (check_layout(layout) != KVQ_OK) return KVQ_EINVAL;
  if (batch < 0 || num_q_heads <= 0 || num_q_heads % layout->num_kv_heads != 0) return KVQ_EINVAL;
  if (max_pages_per_seq <= 0) return KVQ_EINVAL;
  if (options && (options->pages_per_split < 0 || options->path < 0 || options->path > 2)) return KVQ_EINVAL;
  if (layout->page_size != kPageTokens) return KVQ_EUNSUPPORTED;
  const int32_t path = choose_path(*layout, batch, num_q_heads, max_pages_per_seq, options);
  return path < 0 ? static_cast<int32_t>(KVQ_EUNSUPPORTED) : path;
}

size_t kvq_decode_workspace_bytes_ex(const kvq_layout* layout, int32_t batch, int32_t num_q_heads,
                                     int32_t max_pages_per_seq, const kvq_decode_options* options) {
  if (check_layout(layout) != KVQ_OK) return 0;
  WorkspacePlan w;
  if (!plan_workspace(*layout, batch, num_q_heads, max_pages_per_seq, options, &w)) return 0;
  return w.total;
}

size_t kvq_decode_workspace_bytes(const kvq_layout* layout, int32_t batch, int32_t num_q_heads,
                                  int32_t max_pages_per_seq) {
  return kvq_decode_workspace_bytes_ex(layout, batch, num_q_heads, max_pages_per_seq, nullptr);
}

kvq_status kvq_decode_ex(const void* q, const void* pool, const void* scales, const int32_t* block_table,
                         int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                         float sm_scale, void* out, kvq_out_dtype out_dtype, void* workspace,
                         size_t workspace_bytes, const kvq_layout* layout, kvq_kind kind,
                         const kvq_decode_options* options, void* stream) {
  return decode_common(q, pool, scales, block_table, max_pages_per_seq, seq_lens, batch, num_q_heads, sm_scale, out,
                       out_dtype, workspace, workspace_bytes, layout, kind, options, stream, true);
}

kvq_status kvq_decode(const void* q, const void* pool, const void* scales, const int32_t* block_table,
                      int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                      float sm_scale, void* out, kvq_out_dtype out_dtype, void* workspace, size_t workspace_bytes,
                      const kvq_layout* layout, kvq_kind kind, void* stream) {
  return kvq_decode_ex(q, pool, scales, block_table, max_pages_per_seq, seq_lens, batch, num_q_heads, sm_scale, out,
                       out_dtype, workspace, workspace_bytes, layout, kind, nullptr, stream);
}

size_t kvq_decode_sparse_workspace_bytes(const kvq_layout* layout, int32_t batch, int32_t num_q_heads, int32_t topk) {
  SparsePlan sp;
  if (!plan_sparse(layout, batch, num_q_heads, topk, &sp)) return 0;
  return sp.total;
}

kvq_status kvq_decode_sparse(const void* q, const void* pool, const void* scales, const int32_t* block_table,
                             int32_t max_pages_per_seq, const int32_t* seq_lens, const int32_t* indices, int32_t topk,
                             int32_t batch, int32_t num_q_heads, float sm_scale, void* out, kvq_out_dtype out_dtype,
                             void* workspace, size_t workspace_bytes, const kvq_layout* layout, kvq_kind kind,
                             void* stream) {
  kvq_status st = check_layout(layout);
  if (st != KVQ_OK) return st;
  if (!kind_read_ok(kind)) return KVQ_EKIND;
  if (!has_scales(kind)) scales = nullptr;
  if (out_dtype != KVQ_OUT_BF16 && out_dtype != KVQ_OUT_F32) return KVQ_EINVAL;
  if (max_pages_per_seq <= 0) return KVQ_EINVAL;
  SparsePlan sp;
  if (!plan_sparse(layout, batch, num_q_heads, topk, &sp)) return KVQ_EINVAL;
  if (layout->page_size != kPageTokens || layout->head_dim % 64 != 0) return KVQ_EUNSUPPORTED;
  if (batch == 0) return KVQ_OK;
  if (!q || !pool || (has_scales(kind) && !scales) || !block_table || !seq_lens || (topk > 0 && !indices) || !out ||
      !workspace)
    return KVQ_EINVAL;
  if (workspace_bytes < sp.total) return KVQ_EWORKSPACE;
  if (!aligned(pool) || !aligned(scales) || !aligned(workspace) || (reinterpret_cast<uintptr_t>(block_table) % 4) != 0 ||
      (reinterpret_cast<uintptr_t>(seq_lens) % 4) != 0 || (reinterpret_cast<uintptr_t>(indices) % 4) != 0)
    return KVQ_EALIGN;
  st = kvq_device_check();
  if (st != KVQ_OK) return st;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, sizeof(uint32_t), s) != cudaSuccess) return KVQ_ECUDA;
  SparseGatherArgs g;
  g.codes = static_cast<const uint8_t*>(pool);
  g.scales = static_cast<const uint16_t*>(scales);
  g.block_table = block_table;
  g.seq_lens = seq_lens;
  g.indices = indices;
  g.dst_codes = ws + sp.codes_offset;
  g.dst_scales = has_scales(kind) ? reinterpret_cast<uint16_t*>(ws + sp.scales_offset) : nullptr;
  g.dst_table = reinterpret_cast<int32_t*>(ws + sp.table_offset);
  g.dst_lens = reinterpret_cast<int32_t*>(ws + sp.lens_offset);
  g.status = reinterpret_cast<uint32_t*>(ws);
  g.num_pages = layout->num_pages;
  g.max_pages = max_pages_per_seq;
  g.batch = batch;
  g.topk = topk;
  g.cpages = sp.cpages;
  g.n_kv = layout->mla ? 1 : 2;
  g.Hkv = layout->num_kv_heads;
  g.D = layout->head_dim;
  st = launch_sparse_gather(g, s);
  if (st != KVQ_OK) return st;
  return decode_common(q, g.dst_codes, g.dst_scales, g.dst_table, sp.cpages, g.dst_lens, batch, num_q_heads, sm_scale,
                       out, out_dtype, workspace, sp.dense_bytes, &sp.compact, kind, nullptr, stream, false);
}

size_t kvq_extend_workspace_bytes(void) { return kWorkspaceHeader; }

size_t kvq_extend_workspace_bytes_ex(const kvq_layout* layout, int32_t total_q, int32_t num_q_heads,
                                     int32_t max_pages_per_seq, const kvq_extend_options* options) {
  if (check_layout(layout) != KVQ_OK || layout->page_size != kPageTokens) return 0;
  ExtendPlan ep;
  if (!plan_extend(*layout, total_q, num_q_heads, max_pages_per_seq, options, &ep)) return 0;
  return ep.total;
}

int32_t kvq_extend_path(const kvq_layout* layout, int32_t total_q, int32_t num_q_heads, int32_t max_pages_per_seq,
                        const kvq_extend_options* options) {
  if (check_layout(layout) != KVQ_OK) return KVQ_EINVAL;
  if (total_q < 0 || num_q_heads <= 0 || max_pages_per_seq <= 0 || num_q_heads % layout->num_kv_heads != 0)
    return KVQ_EINVAL;
  if (options && (options->path < 0 || options->path > 2)) return KVQ_EINVAL;
  if (layout->page_size != kPageTokens) return KVQ_EUNSUPPORTED;
  ExtendPlan ep;
  if (!plan_extend(*layout, total_q, num_q_heads, max_pages_per_seq, options, &ep)) return KVQ_EUNSUPPORTED;
  if (ep.flash) return ep.split ? 4 : 3;
  WorkspacePlan w;
  plan_workspace(*layout, ep.chunk, num_q_heads, max_pages_per_seq, &ep.dec, &w);
  return w.path;
}

kvq_status kvq_extend(const void* q, const void* pool, const void* scales, const int32_t* block_table,
                      int32_t max_pages_per_seq, const int32_t* seq_lens, const int32_t* q_start, int32_t total_q,
                      int32_t batch, int32_t num_q_heads, float sm_scale, void* out, kvq_out_dtype out_dtype,
                      void* workspace, size_t workspace_bytes, const kvq_layout* layout, kvq_kind kind, void* stream) {
  return kvq_extend_ex(q, pool, scales, block_table, max_pages_per_seq, seq_lens, q_start, total_q, batch,
                       num_q_heads, sm_scale, out, out_dtype, workspace, workspace_bytes, layout, kind, nullptr,
                       stream);
}

kvq_status kvq_extend_ex(const void* q, const void* pool, const void* scales, const int32_t* block_table,
                         int32_t max_pages_per_seq, const int32_t* seq_lens, const int32_t* q_start,
                         int32_t total_q, int32_t batch, int32_t num_q_heads, float sm_scale, void* out,
                         kvq_out_dtype out_dtype, void* workspace, size_t workspace_bytes, const kvq_layout* layout,
                         kvq_kind kind, const kvq_extend_options* options, void* stream) {
  kvq_status st = check_layout(layout);
  if (st != KVQ_OK) return st;
  if (!kind_read_ok(kind)) return KVQ_EKIND;
  if (!has_scales(kind)) scales = nullptr;
  if (out_dtype != KVQ_OUT_BF16 && out_dtype != KVQ_OUT_F32) return KVQ_EINVAL;
  if (batch < 0 || total_q < 0 || num_q_heads <= 0 || max_pages_per_seq <= 0) return KVQ_EINVAL;
  if (num_q_heads % layout->num_kv_heads != 0) return KVQ_EINVAL;
  if (options && (options->path < 0 || options->path > 2)) return KVQ_EINVAL;
  if (static_cast<int64_t>(total_q) * (num_q_heads / layout->num_kv_heads) > std::numeric_limits<int32_t>::max() - 128)
    return KVQ_EINVAL;  // the kernel counts query rows per sequence in 32 bits
  if (!(sm_scale > 0.0f) || sm_scale > std::numeric_limits<float>::max()) return KVQ_EINVAL;  // finite, > 0
  if (layout->page_size != kPageTokens) return KVQ_EUNSUPPORTED;
  if (batch > kMaxExtendBatch) return KVQ_EUNSUPPORTED;
  ExtendPlan ep;
  if (!plan_extend(*layout, total_q, num_q_heads, max_pages_per_seq, options, &ep)) return KVQ_EUNSUPPORTED;
  if (!workspace) return KVQ_EINVAL;
  if (workspace_bytes < ep.total) return KVQ_EWORKSPACE;
  if (!aligned(workspace)) return KVQ_EALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(workspace, 0, sizeof(uint32_t), s) != cudaSuccess) return KVQ_ECUDA;
  if (batch == 0 || total_q == 0) return KVQ_OK;
  if (!q || !pool || (has_scales(kind) && !scales) || !block_table || !seq_lens || !q_start || !out)
    return KVQ_EINVAL;
  if (!aligned(q) || !aligned(pool) || !aligned(scales) || !aligned(out) ||
      (reinterpret_cast<uintptr_t>(block_table) % 4) != 0 || (reinterpret_cast<uintptr_t>(seq_lens) % 4) != 0 ||
      (reinterpret_cast<uintptr_t>(q_start) % 4) != 0)
    return KVQ_EALIGN;
  st = kvq_device_check();
  if (st != KVQ_OK) return st;
  if (!ep.flash)
    return extend_prefixes(ep, q, pool, scales, block_table, max_pages_per_seq, seq_lens, q_start, total_q, batch,
                           num_q_heads, sm_scale, out, out_dtype, workspace, layout, kind, s);
  ExtendArgs a;
  a.q = static_cast<const uint16_t*>(q);
  a.codes = static_cast<const uint8_t*>(pool);
  a.scales = static_cast<const uint16_t*>(scales);
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.q_start = q_start;
  a.out = out;
  a.status = static_cast<uint32_t*>(workspace);
  a.num_pages = layout->num_pages;
  a.max_pages = max_pages_per_seq;
  a.batch = batch;
  a.total_q = total_q;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = layout->num_kv_heads;
  a.head_dim = layout->head_dim;
  a.score_scale = sm_scale * 1.4426950408889634f;  // log2(e)
  a.out_dtype = out_dtype;
  a.kind = kind;
  a.split_p = ep.split ? 1 : 0;
  return launch_extend_tc(a, s);
}

kvq_status kvq_workspace_status(const void* workspace, void* stream) {
  if (!workspace) return KVQ_EINVAL;
  uint32_t word = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess) return KVQ_ECUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return KVQ_ECUDA;
  if (word == 0) return KVQ_OK;
  return word == kStatusTimeoutWord ? KVQ_ETIMEOUT : KVQ_EINVAL;
}

kvq_status kvq_encode_probe(kvq_kind kind, const float* y, uint8_t* codes, int64_t n, void* stream) {
  if (!kind_ok(kind)) return KVQ_EKIND;
  if (n < 0) return KVQ_EINVAL;
  if (n == 0) return KVQ_OK;
  if (!y || !codes) return KVQ_EINVAL;
  kvq_status st = kvq_device_check();
  if (st != KVQ_OK) return st;
  return launch_encode_probe(kind, y, codes, n, static_cast<cudaStream_t>(stream));
}

kvq_status kvq_quantize_probe(kvq_kind kind, const uint16_t* x, int64_t nx, const uint16_t* s, int64_t ns,
                              uint8_t* codes, void* stream) {
  if (!kind_ok(kind)) return KVQ_EKIND;
  if (nx < 0 || ns < 0) return KVQ_EINVAL;
  if (nx == 0 || ns == 0) return KVQ_OK;
  if (!x || !s || !codes) return KVQ_EINVAL;
  kvq_status st = kvq_device_check();
  if (st != KVQ_OK) return st;
  return launch_quantize_probe(kind, x, nx, s, ns, codes, static_cast<cudaStream_t>(stream));
}

kvq_status kvq_dequant_probe(kvq_kind kind, const uint8_t* codes, const uint16_t* scales, uint16_t* out, int64_t n,
                             void* stream) {
  if (!kind_read_ok(kind)) return KVQ_EKIND;
  if (!has_scales(kind)) scales = nullptr;
  if (n < 0 || n % 16 != 0) return KVQ_EINVAL;
  if (n == 0) return KVQ_OK;
  if (!codes || (has_scales(kind) && !scales) || !out) return KVQ_EINVAL;
  if (!aligned(codes) || !aligned(out)) return KVQ_EALIGN;
  kvq_status st = kvq_device_check();
  if (st != KVQ_OK) return st;
  return launch_dequant_probe(kind, codes, scales, out, n, static_cast<cudaStream_t>(stream));
}

kvq_status kvq_exp2_probe(const float* x, float* y, int64_t n, void* stream) {
  if (n < 0) return KVQ_EINVAL;
  if (n == 0) return KVQ_OK;
  if (!x || !y) return KVQ_EINVAL;
  if ((reinterpret_cast<uintptr_t>(x) % 4) != 0 || (reinterpret_cast<uintptr_t>(y) % 4) != 0) return KVQ_EALIGN;
  const kvq_status st = kvq_device_check();
  if (st != KVQ_OK) return st;
  return launch_exp2_probe(x, y, n, static_cast<cudaStream_t>(stream));
}

kvq_status kvq_wait_probe(void* workspace, void* stream) {
  if (!workspace) return KVQ_EINVAL;
  if (!aligned(workspace)) return KVQ_EALIGN;
  kvq_status st = kvq_device_check();
  if (st != KVQ_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(workspace, 0, sizeof(uint32_t), s) != cudaSuccess) return KVQ_ECUDA;
  return launch_wait_probe(static_cast<uint32_t*>(workspace), s);
}

}  // extern "C"
