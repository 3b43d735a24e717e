/*
 * kvq.h -- C ABI of libkvq: an 8-bit block-scaled paged KV cache for one GB300 (sm_103a).
 *
 * Two operations, taken from the pull-request pages on the 8-bit KV cache:
 *
 *   kvq_store   quantize incoming bf16 K/V rows and scatter them into a page pool
 *               ("feat(kvcache): 8-bit KV cache (q8_0 / fp8_e4m3) behind --kv-cache-dtype",
 *               section "What": one fp16 scale per 32 elements along head_dim, s = max/448 for
 *               fp8_e4m3 and s = max/127 for q8_0, 1.0625 bytes per element; review comment
 *               "A bug on sm_89": int8 rounds half away from zero then clamps to +-127, fp8 is
 *               clamped to +-448 then rounded once to nearest-even).
 *   kvq_decode  split-K decode attention over that pool: bf16 queries, K and V dequantized to bf16
 *               before the dot (same page, "What": the scale varies along the reduction dim), an fp32
 *               online softmax, split partials merged at the end ("feat(kvcache): 8-bit DSV4
 *               window/compressed KV", section "Testing": split-k decode kernel, masked -1 columns).
 *               GQA pools keep separate K and V rows; MLA pools keep one latent row per token that
 *               serves as both (same page, "What this adds").
 *
 * Conventions for every entry point:
 *   - Pointers named as device pointers must point to device memory of the current device; host
 *     pointers (kvq_layout) are read during the call only.  The caller owns every buffer; the
 *     library allocates nothing and keeps no state between calls.  The one exception is
 *     kvq_decode_noalloc (with kvq_noalloc_status), whose scratch is a fixed array in the library's own
 *     device memory that keeps its contents from one call to the next.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls are asynchronous on it.
 *   - Arguments are validated on the host before anything is launched.  A failed validation returns
 *     a negative kvq_status and leaves every buffer untouched.  A launch failure returns KVQ_ECUDA.
 *   - Device pointers must be 16-byte aligned (KVQ_EALIGN otherwise).
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Code format.  The first two use one fp16 scale per 32 elements; the unscaled ones have no scale array
 * (written by kvq_store_unscaled; every attention entry point reads all four, ignoring `scales` for the
 * unscaled kinds, which may then be NULL). */
typedef enum {
    KVQ_FP8_E4M3 = 1,          /* OCP E4M3 "fn" codes, s = amax / 448 */
    KVQ_Q8_0 = 2,              /* int8 codes,          s = amax / 127 */
    KVQ_FP8_E4M3_UNSCALED = 3, /* the plain E4M3 cast, no scales, 1 byte per element (kvq_store_unscaled) */
    KVQ_FP8_E5M2_UNSCALED = 4  /* the plain E5M2 cast, no scales, 1 byte per element (kvq_store_unscaled) */
} kvq_kind;

/* Element type of kvq_decode's output. */
typedef enum {
    KVQ_OUT_BF16 = 0, /* round-to-nearest-even bf16 */
    KVQ_OUT_F32 = 1   /* fp32, no final rounding to bf16 */
} kvq_out_dtype;

typedef enum {
    KVQ_OK = 0,
    KVQ_EINVAL = -1,       /* null pointer, negative size, bad layout, Hq % Hkv != 0, ... */
    KVQ_EKIND = -2,        /* kind is not a kvq_kind this call accepts */
    KVQ_EHEADDIM = -3,     /* head_dim (or v_dim) not a positive multiple of 32 */
    KVQ_EALIGN = -4,       /* a device pointer is not 16-byte aligned */
    KVQ_EWORKSPACE = -5,   /* workspace smaller than kvq_decode_workspace_bytes() */
    KVQ_EARCH = -6,        /* current device is not compute capability 10.3 */
    KVQ_ECUDA = -7,        /* a CUDA call or launch failed */
    KVQ_EUNSUPPORTED = -8, /* valid, but no kernel for this shape (see kvq_decode) */
    KVQ_ETIMEOUT = -9      /* a kernel gave up a bounded wait (reported by kvq_workspace_status) */
} kvq_status;

/*
 * Pool layout (one layer).  With n_kv = 2 for GQA (K and V) and n_kv = 1 for MLA:
 *   codes : uint8  [num_pages][n_kv][num_kv_heads][page_size][head_dim]
 *   scales: fp16   [num_pages][n_kv][num_kv_heads][page_size][head_dim / 32]
 * Token slot s lives in page s / page_size at offset s % page_size.  Each (page, kv, head) chunk is
 * contiguous, so one page of one head is one bulk copy.
 */
typedef struct {
    int64_t num_pages;
    int32_t page_size;    /* tokens per page; kvq_decode supports 16 */
    int32_t num_kv_heads; /* Hkv (1 for MLA) */
    int32_t head_dim;     /* K row width D, a multiple of 32 (576 for the MLA latent row) */
    int32_t v_dim;        /* V width: == head_dim for GQA; <= head_dim for MLA (V = row[0:v_dim]) */
    int32_t mla;          /* 0: separate K and V rows; 1: one latent row serves as K and V */
} kvq_layout;

/* ---------------------------------------------------------------- cost model (host only) */
/* Bytes of the codes array / the scales array for `layout->num_pages` pages. 0 if the layout is invalid. */
size_t kvq_pool_bytes(const kvq_layout* layout);
size_t kvq_scale_bytes(const kvq_layout* layout);
/* Bytes one cached token costs: n_kv * Hkv * head_dim * 17/16 (codes + fp16 scales).  -1 if invalid.
 * ("What": 1.0625 bytes per element against bf16's 2; the review's +88% pool growth = 2 / 1.0625.) */
double kvq_bytes_per_token(const kvq_layout* layout);
/* Whole pages (codes + scales) that fit in `budget_bytes`; num_pages of `layout` is ignored.  -1 if invalid. */
int64_t kvq_num_pages(const kvq_layout* layout, size_t budget_bytes);
/* The same two for any kind: 17/16 bytes per element for the block-scaled kinds, 1 for the unscaled fp8 casts
 * ("Add fp8 KV-cache quantization (--kv-dtype)", section "Benchmark": twice the bf16 token budget).  -1 if the
 * layout or the kind is invalid. */
double kvq_bytes_per_token_ex(const kvq_layout* layout, kvq_kind kind);
int64_t kvq_num_pages_ex(const kvq_layout* layout, kvq_kind kind, size_t budget_bytes);

/* ---------------------------------------------------------------- store */
/*
 * Quantize and scatter `num_tokens` rows.
 *   pool, scales  device, the arrays described by kvq_layout (written in place)
 *   k             device bf16 [num_tokens][num_kv_heads][head_dim]
 *   v             device bf16, same shape as k; must be NULL when layout->mla (the latent row is k)
 *   slot_mapping  device int64 [num_tokens]; row t goes to slot slot_mapping[t]; -1 skips the row.
 *                 Slots must be unique within one call; a slot >= num_pages * page_size is skipped
 *                 (never written).
 * Per 32-element block: amax in fp32; s = fp16_RNE(min(amax / Q, 65504)) with IEEE fp32 division;
 * a block whose fp16 scale is 0 stores zero codes and a zero scale; otherwise every element is
 * y = x / s (IEEE fp32) and the code is E4M3 nearest-even of clamp(y, +-448) (fp8) or
 * clamp(round-half-away(y), +-127) (q8_0).
 */
kvq_status kvq_store(void* pool, void* scales, const void* k, const void* v, const int64_t* slot_mapping,
                     int64_t num_tokens, const kvq_layout* layout, kvq_kind kind, void* stream);

/* ---------------------------------------------------------------- decode */
/* Options for kvq_decode_ex.  Zero-initialise for the defaults. */
typedef struct {
    int32_t pages_per_split; /* 0 = automatic; else every split covers this many pages */
    int32_t path;            /* 0 = automatic; 1 = CUDA-core kernel; 2 = tensor-core (tcgen05) kernel */
} kvq_decode_options;

/* Workspace bytes kvq_decode needs for these sizes (an upper bound independent of seq_lens). 0 if invalid. */
size_t kvq_decode_workspace_bytes(const kvq_layout* layout, int32_t batch, int32_t num_q_heads,
                                  int32_t max_pages_per_seq);
size_t kvq_decode_workspace_bytes_ex(const kvq_layout* layout, int32_t batch, int32_t num_q_heads,
                                     int32_t max_pages_per_seq, const kvq_decode_options* options);

/*
 * Decode attention for one new query token per sequence.
 *   q            device bf16 [batch][num_q_heads][head_dim]
 *   pool, scales device, filled by kvq_store (or by kvq_store_unscaled: then scales is ignored)
 *   block_table  device int32 [batch][max_pages_per_seq]; entry j is the physical page of tokens
 *                [16j, 16j+16); -1 masks that whole page.  Entries at or beyond ceil(seq_len/16) are
 *                never read.  An entry >= layout->num_pages is treated as masked and makes
 *                kvq_workspace_status report KVQ_EINVAL.
 *   seq_lens     device int32 [batch], each in [0, max_pages_per_seq * page_size]
 *   sm_scale     multiplies q.k before the softmax
 *   out          device [batch][num_q_heads][v_dim], bf16 or fp32 per out_dtype
 *   workspace    device scratch of at least kvq_decode_workspace_bytes(); its content on entry is
 *                irrelevant; it holds the split partials and a status word after the call.
 * Query head h reads kv head h / (num_q_heads / num_kv_heads).  For every (b, h) the result is
 * softmax(sm_scale * q.K^T) V over the valid tokens t < seq_lens[b] whose page is not masked, with
 * K and V dequantized to bf16 (RNE of code * scale) and fp32 accumulation; a sequence without a
 * valid token outputs zeros.  Supported: page_size 16 and head_dim in {64, 128, 256} with v_dim ==
 * head_dim (GQA), or the MLA row head_dim 576 / v_dim 512; other shapes return KVQ_EUNSUPPORTED.
 * Kernels (kvq_decode_options.path): the CUDA-core kernel (1) runs every supported shape, keeps the
 * softmax probabilities P in fp32 and merges its split partials itself (one launch).  The tensor-core
 * kernels (2) run head_dim 128 or 256 with 1..16 query heads per kv head and batch <= 2048, and the
 * MLA row with at most 64 query heads (or a multiple of 64) and batch <= 1024; a merge kernel follows
 * them (two launches).  They feed P to the MMA as bf16, so their error relative to the exact result
 * grows with the magnitude of V (about 2^-9 of max |V|).  Automatic (0) picks 2 for 8..16 query heads
 * per kv head, and for the MLA row when batch * max_pages_per_seq * 16 >= 1024 (the MLA tensor-core
 * kernel has a fixed cost of ~50 us); 1 otherwise; kvq_decode_path tells which.
 */
kvq_status kvq_decode(const void* q, const void* pool, const void* scales, const int32_t* block_table,
                      int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                      float sm_scale, void* out, kvq_out_dtype out_dtype, void* workspace,
                      size_t workspace_bytes, const kvq_layout* layout, kvq_kind kind, void* stream);
kvq_status kvq_decode_ex(const void* q, const void* pool, const void* scales, const int32_t* block_table,
                         int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t batch,
                         int32_t num_q_heads, float sm_scale, void* out, kvq_out_dtype out_dtype,
                         void* workspace, size_t workspace_bytes, const kvq_layout* layout, kvq_kind kind,
                         const kvq_decode_options* options, void* stream);

/*
 * Sparse (top-K) decode ("Experimental FP8 KV Cache": a query reads the K selected tokens of a long
 * latent pool; "feat(kvcache): 8-bit DSV4 window/compressed KV", section "Testing": masked -1 columns).
 *   indices      device int32 [batch][topk]: token positions of sequence b.  A column is valid when its
 *                position p satisfies 0 <= p < seq_lens[b] and block_table[b][p / 16] is not -1; -1 and
 *                any other invalid column are skipped; a position listed twice counts twice.
 *   topk         columns per sequence, 0 .. 8192 (0: every output is zero)
 * Other arguments as kvq_decode; the workspace comes from kvq_decode_sparse_workspace_bytes.  For every
 * (b, h) the result is softmax(sm_scale * q.K^T) V over the valid columns (order does not matter), with
 * K and V dequantized to bf16; no valid column gives zeros.  The library gathers the valid columns of
 * each sequence into a compact pool in the workspace (a byte copy of codes and scales), then runs the
 * dense decode over it, so the kernel choice and precision are those of kvq_decode for a sequence of
 * that many tokens.  Supported: page_size 16 and head_dim a multiple of 64 (every kvq_decode shape).
 * A block-table entry >= layout->num_pages at a selected position is skipped and makes
 * kvq_workspace_status report KVQ_EINVAL.
 */
size_t kvq_decode_sparse_workspace_bytes(const kvq_layout* layout, int32_t batch, int32_t num_q_heads,
                                         int32_t topk);
kvq_status kvq_decode_sparse(const void* q, const void* pool, const void* scales, const int32_t* block_table,
                             int32_t max_pages_per_seq, const int32_t* seq_lens, const int32_t* indices,
                             int32_t topk, int32_t batch, int32_t num_q_heads, float sm_scale, void* out,
                             kvq_out_dtype out_dtype, void* workspace, size_t workspace_bytes,
                             const kvq_layout* layout, kvq_kind kind, void* stream);

/*
 * Store into an unscaled fp8 pool ("Add fp8 KV-cache quantization (--kv-dtype)", section "How it works": the
 * store casts the incoming bf16 k/v to the pool's fp8 type, scale 1.0; fp8_e5m2 is wired the same way).
 * kind is KVQ_FP8_E4M3_UNSCALED or KVQ_FP8_E5M2_UNSCALED; each bf16 element becomes one code by a single
 * nearest-even rounding that saturates at the largest finite value (448 / 57344): finite and infinite inputs
 * give finite codes.  NaN inputs are outside the domain (as for kvq_store) and give NaN codes.  The pool has
 * the codes layout of kvq_pool_bytes and no scale array.  Other arguments as kvq_store.  kvq_decode,
 * kvq_decode_sparse and kvq_extend read such a pool with the same kind: every E4M3 and E5M2 value is a bf16
 * value, so K and V enter the attention exactly as stored.
 */
kvq_status kvq_store_unscaled(void* pool, const void* k, const void* v, const int64_t* slot_mapping,
                              int64_t num_tokens, const kvq_layout* layout, kvq_kind kind, void* stream);

/*
 * The MLA store fused with its producer ("feat(kvcache): 8-bit DSV4 window/compressed KV", section "Why the
 * precision cost is small": the model rounds each latent row onto the E4M3 grid with one scale per 64
 * elements right before every store; the rope tail stays bf16).  kv holds bf16 rows [num_tokens, head_dim]
 * as they leave the producer.  Each row's first head_dim - rope_dim elements are rounded per 64:
 *   s = fp32(amax / 448);  value = bf16_RNE(E4M3_sat_RNE(x / s) * s)   (IEEE fp32 division and product;
 *   an all-zero unit stays as it is).
 * The row, so rounded, is then stored exactly as kvq_store stores it, in one pass.  Requirements:
 *   - layout->mla = 1 with one kv head;
 *   - head_dim and rope_dim multiples of 64, with rope_dim <= head_dim (else KVQ_EUNSUPPORTED);
 *   - 16-byte aligned pool, scales and kv, and an 8-byte aligned slot_mapping.
 * Slots of -1 are skipped.  Asynchronous on `stream`.
 */
kvq_status kvq_store_act_quant(void* pool, void* scales, const void* kv, const int64_t* slot_mapping,
                               int64_t num_tokens, int32_t rope_dim, const kvq_layout* layout, kvq_kind kind,
                               void* stream);

/*
 * Extend (prefill) attention ("feat(kvcache): 8-bit KV cache (q8_0 / fp8_e4m3) behind --kv-cache-dtype",
 * section "What": the dequant sits inside every attention kernel, prefill included; "feat(kvcache): 8-bit
 * DSV4 window/compressed KV", section "Testing": quantized attention on the prefill kernel).  Store the
 * step's new K/V rows with kvq_store first: every key, the new ones included, is read from the pool.
 *   q            [total_q, num_q_heads, head_dim] bf16, device; the rows of sequence b are
 *                q_start[b] .. q_start[b + 1] - 1
 *   q_start      [batch + 1] int32, device: q_start[0] = 0, non-decreasing, q_start[batch] = total_q
 *   seq_lens     stored tokens per sequence, the new ones included: the n_b = q_start[b + 1] - q_start[b]
 *                new tokens are the last n_b, so new token i sits at position seq_lens[b] - n_b + i
 *   out          [total_q, num_q_heads, v_dim], bf16 or f32 (out_dtype), device
 *   workspace    at least kvq_extend_workspace_bytes_ex() for the same sizes and options, 16-byte aligned,
 *                device
 * sm_scale must be finite and > 0 (else KVQ_EINVAL).  Other arguments as kvq_decode.
 * Query row (b, i, h) gets softmax(sm_scale * q.K^T) V over the positions
 * 0 .. seq_lens[b] - n_b + i of sequence b whose pages are not masked (causal), with K and V dequantized to
 * bf16 and fp32 accumulation; no valid position gives zeros.
 * Kernels (kvq_extend_options.path; kvq_extend passes none, i.e. automatic):
 *   flash (GQA with head_dim = v_dim in {128, 256} and query heads per kv head dividing 128): one
 *     flash-style tcgen05 kernel, each dequantized K/V tile shared by a block of 128 query rows.  It feeds
 *     the probabilities P to the MMA as bf16, so its error grows with the magnitude of V (about 2^-9 of
 *     sum p|V|), as the tensor-core decode's does.
 *   prefixes: every new token is decoded as a sequence of its own over its causal prefix, by the decode
 *     kernels of kvq_decode (the tokens run in chunks of 1024, each chunk one kvq_decode-like call with
 *     that many sequences), so its precision is the decode's.  It reads each prefix once per new token,
 *     so it costs about n_b times the flash kernel's K/V bytes; L2 absorbs much of it.
 * path 0 (automatic): flash where it supports the shape, else prefixes with the decode's automatic choice
 * (the MLA latent row, head_dim 576 / v_dim 512, "feat(kvcache): 8-bit DSV4 window/compressed KV", section
 * "What this adds", always takes prefixes); 1: prefixes on the CUDA-core decode (fp32 P, every
 * kvq_decode shape); 2: flash for GQA, prefixes on the tensor-core decode for MLA.  kvq_extend_path tells
 * which.  With precise_p (below) every path keeps P's rounding under 2^-16 relative, so the error no longer
 * grows with |V| beyond the decode bound.  The rows of a skipped sequence (below) are left as they are by the flash kernel and set to zero
 * by the prefixes.
 * Supported: page_size 16, batch <= 2048, and the shapes of the chosen kernels; otherwise KVQ_EUNSUPPORTED.
 * q_start and seq_lens are read on the device: a sequence with n_b < 0, n_b > seq_lens[b] or q_start[b + 1]
 * > total_q is skipped and makes kvq_workspace_status report KVQ_EINVAL, as does a block-table entry >=
 * layout->num_pages (that page is skipped).  Asynchronous on `stream`.
 */
typedef struct kvq_extend_options {
    int32_t path;       /* 0 = automatic; 1 = prefixes on the CUDA-core decode; 2 = flash (GQA) / tensor-core
                           decode (MLA) */
    int32_t precise_p;  /* nonzero: P reaches the PV product with at least 16 significant bits.  The flash
                           kernel feeds it as two bf16 terms, hi = bf16(p) and lo = bf16(p - hi), through a
                           second PV (about 2^-17 relative; its exponentials all on the MUFU unit); prefixes
                           run on the CUDA-core decode (fp32 P); path 2 on MLA is then KVQ_EUNSUPPORTED */
} kvq_extend_options;
/* The flash kernel's workspace: its status word (enough for the automatic choice on a supported GQA shape). */
size_t kvq_extend_workspace_bytes(void);
/* Workspace bytes kvq_extend_ex needs for these sizes and options (options may be NULL): the flash kernel's
 * status word, or the decode workspace of one chunk of prefixes plus two int32 per query row.  0 if
 * invalid or unsupported. */
size_t kvq_extend_workspace_bytes_ex(const kvq_layout* layout, int32_t total_q, int32_t num_q_heads,
                                     int32_t max_pages_per_seq, const kvq_extend_options* options);
/* The extend kernel kvq_extend_ex would run: 3 (flash), 4 (flash with P as two bf16 terms), or the decode
 * kernel of the prefixes, 1 (CUDA cores) or 2 (tensor cores).  Otherwise a negative kvq_status (KVQ_EINVAL for invalid sizes or options,
 * KVQ_EUNSUPPORTED when no kernel supports the shape).  Host only; options may be NULL. */
int32_t kvq_extend_path(const kvq_layout* layout, int32_t total_q, int32_t num_q_heads, int32_t max_pages_per_seq,
                        const kvq_extend_options* options);
kvq_status kvq_extend(const void* q, const void* pool, const void* scales, const int32_t* block_table,
                      int32_t max_pages_per_seq, const int32_t* seq_lens, const int32_t* q_start, int32_t total_q,
                      int32_t batch, int32_t num_q_heads, float sm_scale, void* out, kvq_out_dtype out_dtype,
                      void* workspace, size_t workspace_bytes, const kvq_layout* layout, kvq_kind kind,
                      void* stream);
kvq_status kvq_extend_ex(const void* q, const void* pool, const void* scales, const int32_t* block_table,
                         int32_t max_pages_per_seq, const int32_t* seq_lens, const int32_t* q_start,
                         int32_t total_q, int32_t batch, int32_t num_q_heads, float sm_scale, void* out,
                         kvq_out_dtype out_dtype, void* workspace, size_t workspace_bytes, const kvq_layout* layout,
                         kvq_kind kind, const kvq_extend_options* options, void* stream);

/*
 * The decode kernel kvq_decode_ex would run for these sizes and options: 1 (CUDA cores, one launch) or
 * 2 (tensor cores, two launches with the merge).  Otherwise a negative kvq_status: KVQ_EINVAL for an
 * invalid layout, size or option, KVQ_EUNSUPPORTED when no kernel supports the shape.  Host only, no
 * device call; options may be NULL.
 */
int32_t kvq_decode_path(const kvq_layout* layout, int32_t batch, int32_t num_q_heads, int32_t max_pages_per_seq,
                        const kvq_decode_options* options);

/*
 * kvq_decode for callers that cannot allocate device memory.  The pages have no counterpart to
 * this entry point.  It exists because some callers cannot call cudaMalloc when they decode: a
 * serving loop that reserved all of its memory up front, a plugin running under another
 * framework's allocator, or code that has no allocator at all.  Arguments and results are those of
 * kvq_decode without the workspace: the split-K scratch is a fixed array of
 * KVQ_NOALLOC_SCRATCH_BYTES in the library's own device memory, which every GPU that loads the
 * library keeps until the process exits.  Sizes whose kvq_decode_workspace_bytes() exceeds that
 * return KVQ_EWORKSPACE.  Nothing is allocated.
 * The first call on each device looks up the array's device address (cudaGetSymbolAddress) with
 * that device current; make that first call before capturing any stream.  Every call shares the
 * array and it keeps the previous call's contents (the call clears what must start at zero); calls
 * whose kernels overlap on the GPU -- different streams, or host threads without ordering -- race
 * on it and give wrong results.
 */
#define KVQ_NOALLOC_SCRATCH_BYTES (8u << 20)
kvq_status kvq_decode_noalloc(const void* q, const void* pool, const void* scales, const int32_t* block_table,
                              int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t batch,
                              int32_t num_q_heads, float sm_scale, void* out, kvq_out_dtype out_dtype,
                              const kvq_layout* layout, kvq_kind kind, void* stream);
/*
 * Status word the last kvq_decode_noalloc left in the library's scratch array, as kvq_workspace_status
 * reports it for a caller's workspace: KVQ_OK; KVQ_ETIMEOUT if a kernel gave up a bounded wait (the output
 * of that call is not valid); KVQ_EINVAL if a block-table entry pointed past the pool.  The caller has no
 * pointer to that array, so this is the only way to read it.  Synchronizes `stream`; call it on the stream
 * of the decode it checks, before another kvq_decode_noalloc is issued on any stream.  Like the decode,
 * it has no counterpart on the pages.
 */
kvq_status kvq_noalloc_status(void* stream);

/*
 * Status word a decode left in its workspace: KVQ_OK; KVQ_ETIMEOUT if a kernel gave up a bounded
 * wait (its output is then not valid); KVQ_EINVAL if a block-table entry pointed past the pool.
 * Synchronizes `stream`.
 */
kvq_status kvq_workspace_status(const void* workspace, void* stream);

/* ---------------------------------------------------------------- rounding probes */
/*
 * Elementwise code step of the store on already-scaled fp32 values (device arrays of n):
 * codes[i] = E4M3_RNE(clamp(y[i], +-448)) for fp8, or int8 clamp(round-half-away(y[i]), +-127) for
 * q8_0.  Exposes the store kernel's own conversion so that it can be checked exhaustively.
 */
kvq_status kvq_encode_probe(kvq_kind kind, const float* y, uint8_t* codes, int64_t n, void* stream);
/*
 * Division-and-rounding step of the store, by the store kernel's own routine, for every pairing of
 * nx bf16 elements with ns nonzero fp16 scales (device arrays of bit patterns):
 * codes[i * nx + j] = code of x[j] / s[i] (fp8_e4m3 or q8_0, as kvq_store computes it).  Exposes the
 * store's quotient so that its codes can be checked against IEEE division on every (x, s).
 */
kvq_status kvq_quantize_probe(kvq_kind kind, const uint16_t* x, int64_t nx, const uint16_t* s, int64_t ns,
                              uint8_t* codes, void* stream);
/*
 * Dequant step of the decode, by the decode kernels' own routine, on n codes (n a multiple of 16)
 * in chunks of 16 that share one scale: out[i] = bf16 bits of RNE_bf16(value(codes[i]) *
 * fp16(scales[i / 16])).  codes and out 16-byte aligned device arrays of n; scales a device array
 * of n / 16 fp16 bit patterns.
 */
kvq_status kvq_dequant_probe(kvq_kind kind, const uint8_t* codes, const uint16_t* scales, uint16_t* out,
                             int64_t n, void* stream);
/*
 * Exponential step of the extend's softmax, by the extend kernel's own routine: y[i] = 2^x[i] for fp32 device
 * arrays of n, as the FMA-pipe path computes a share of the probabilities (a cubic for 2^f on [-0.5, 0.5]
 * and the integer part added to the exponent; x clamped at -126).  Relative error at most 1.5e-4 for x in
 * [-126, 8].  Exposes the routine so that its bound can be checked on the GPU; the pages print no such
 * step (they exponentiate in Triton / FlashInfer kernels).  4-byte aligned pointers.
 */
kvq_status kvq_exp2_probe(const float* x, float* y, int64_t n, void* stream);
/*
 * Bounded-wait probe: one kernel waits, with the decode kernels' own bounded wait, on an mbarrier
 * that nothing completes.  The wait gives up after the library's limit (2 s) and the kernel records a
 * timeout in the status word of `workspace` (a device buffer of at least 256 bytes, cleared first), so
 * that kvq_workspace_status then reports KVQ_ETIMEOUT.  It shows on the GPU that a wait which never
 * completes ends in an error the host can read and leaves the context usable.
 */
kvq_status kvq_wait_probe(void* workspace, void* stream);

/* ---------------------------------------------------------------- misc */
/* Message for a status code (static string). */
const char* kvq_strerror(kvq_status status);
/* KVQ_OK if the current device is sm_103 and the library's kernels load on it, else KVQ_EARCH / KVQ_ECUDA. */
kvq_status kvq_device_check(void);
/* Library version, e.g. "0.1.0". */
const char* kvq_version(void);

#ifdef __cplusplus
}
#endif
#endif /* KVQ_H */
