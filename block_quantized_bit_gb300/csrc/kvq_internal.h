// kvq_internal.h -- launchers shared between the libkvq translation units (host side).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvq.h"

namespace kvq {

// Arguments of one decode call after host validation.
struct DecodeArgs {
  const void* q;
  const uint8_t* codes;
  const uint16_t* scales;
  const int32_t* block_table;
  const int32_t* bt_row;  // block-table row of each sequence, or null (row b); set by the MLA extend
  int64_t num_pages;
  int32_t max_pages;
  const int32_t* seq_lens;
  int32_t batch;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t v_dim;
  int32_t mla;
  float sm_scale;
  void* out;
  kvq_out_dtype out_dtype;
  kvq_kind kind;
  int32_t pages_per_split;  // 0 = automatic
  // workspace carve-up
  uint32_t* status;
  float* part_acc;   // [max_items][heads_per_item][v_dim]
  float* part_ml;    // [max_items][heads_per_item][2]
  int32_t* plan_tab; // [batch][2]: first item and split count of each sequence (written by the decode)
  int32_t* split_cnt; // [batch][query groups]: splits finished, zeroed per call; set when the decode
                      // kernel merges its own partials (the last split of a group merges), else null
  int64_t max_items;
  int32_t heads_per_item;  // query heads one work item covers (a tile of the group)
  int32_t split_align;     // automatic split sizes are a multiple of this many pages
  int32_t target_items;    // automatic split sizes aim at about this many work items
  int32_t one_wave_items;  // nonzero: first try splits sized for this many items (one per resident CTA),
                           // kept when the batch's items fit; else target_items
  int32_t min_one_split;   // nonzero: every (sequence, group) has at least one split (an empty one when
                           // the sequence has no page), as the kernel that merges in-kernel needs
};

// Tokens per page the decode kernels support, and the workspace's leading status block.
constexpr int kPageTokens = 16;
constexpr size_t kWorkspaceHeader = 256;

// Work-item planning constants shared by the host (workspace bound) and the kernels.
constexpr int kTargetItems = 1216;  // items when the host sets no target; also the SM count assumed without a device
constexpr int kMinPagesPerSplit = 4;

// Heads of one query group that a CUDA-core work item covers.
int32_t cc_heads_per_item(int32_t group, int32_t head_dim, int32_t mla);
// Upper bound on work items for the given sizes (used for workspace sizing and the grid).
int64_t max_work_items(int32_t batch, int32_t query_groups, int32_t max_pages, int32_t pages_per_split,
                       int32_t target_items);

kvq_status launch_store(void* pool, void* scales, const void* k, const void* v, const int64_t* slot_mapping,
                        int64_t num_tokens, const kvq_layout& L, kvq_kind kind, cudaStream_t stream);
kvq_status launch_encode_probe(kvq_kind kind, const float* y, uint8_t* codes, int64_t n, cudaStream_t stream);
kvq_status launch_quantize_probe(kvq_kind kind, const uint16_t* x, int64_t nx, const uint16_t* s, int64_t ns,
                                 uint8_t* codes, cudaStream_t stream);
kvq_status launch_dequant_probe(kvq_kind kind, const uint8_t* codes, const uint16_t* scales, uint16_t* out,
                                int64_t n, cudaStream_t stream);
kvq_status launch_wait_probe(uint32_t* status, cudaStream_t stream);
bool decode_cc_supported(int32_t head_dim, int32_t v_dim, int32_t mla);
int32_t cc_ctas_per_sm(int32_t head_dim, int32_t mla, int32_t heads_per_item);
bool decode_tc_supported(int32_t head_dim, int32_t v_dim, int32_t mla, int32_t group, int32_t batch);
bool decode_mla_tc_supported(int32_t head_dim, int32_t v_dim, int32_t mla, int32_t group, int32_t batch);
int32_t decode_mla_tc_heads_per_item(int32_t group);
kvq_status launch_decode_mla_tc(const DecodeArgs& a, cudaStream_t stream);
kvq_status launch_decode_tc(const DecodeArgs& a, cudaStream_t stream);
kvq_status launch_decode_cc(const DecodeArgs& a, cudaStream_t stream);
kvq_status launch_merge(const DecodeArgs& a, int32_t query_groups, cudaStream_t stream);

// Sparse decode: the gather of the selected columns into a compact pool (pages b * cpages ..).
struct SparseGatherArgs {
  const uint8_t* codes;
  const uint16_t* scales;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const int32_t* indices;   // [batch][topk]
  uint8_t* dst_codes;
  uint16_t* dst_scales;
  int32_t* dst_table;       // [batch][cpages]
  int32_t* dst_lens;        // [batch]
  uint32_t* status;
  int64_t num_pages;
  int32_t max_pages;
  int32_t batch;
  int32_t topk;
  int32_t cpages;
  int32_t n_kv, Hkv, D;
};
constexpr int32_t kMaxSparseTopk = 8192;
kvq_status launch_sparse_gather(const SparseGatherArgs& g, cudaStream_t stream);

// Extend (prefill) attention: the new tokens of every sequence attend causally over the pool.
struct ExtendArgs {
  const uint16_t* q;          // [total_q][num_q_heads][head_dim] bf16
  const uint8_t* codes;
  const uint16_t* scales;
  const int32_t* block_table; // [batch][max_pages]
  const int32_t* seq_lens;    // [batch]
  const int32_t* q_start;     // [batch + 1]
  void* out;                  // [total_q][num_q_heads][v_dim]
  uint32_t* status;
  int64_t num_pages;
  int32_t max_pages;
  int32_t batch;
  int32_t total_q;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  float score_scale;          // sm_scale * log2(e): the kernels work in the exp2 domain
  kvq_out_dtype out_dtype;
  kvq_kind kind;
  int32_t split_p;            // nonzero: P enters the PV MMA as two bf16 terms (hi + lo)
};
constexpr int32_t kMaxExtendBatch = 2048;  // sequences whose item bases fit the kernel's shared table
bool extend_tc_supported(int32_t head_dim, int32_t v_dim, int32_t mla, int32_t group, int32_t batch);
kvq_status launch_extend_tc(const ExtendArgs& a, cudaStream_t stream);
kvq_status launch_exp2_probe(const float* x, float* y, int64_t n, cudaStream_t stream);
// MLA extend: each new token's causal prefix length and block-table row (rows of inconsistent sequences
// are left as they are and flagged in the status word).
kvq_status launch_extend_expand(const int32_t* q_start, const int32_t* seq_lens, int32_t batch, int32_t total_q,
                                int32_t* vlens, int32_t* vrow, uint32_t* status, cudaStream_t stream);
}  // namespace kvq
