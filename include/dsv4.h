/*
 * dsv4.h -- C ABI of libdsv4: the decode hot path of DeepSeek-V4 compressed
 * sparse attention on one GB300 (sm_103a).
 *
 * The path, per decode step and layer:
 *   (1) dsv4_compress_insert : token-level Compressor -> RMSNorm -> RoPE ->
 *       FP8 quantisation -> paged compressed-cache insert (main cache d = 576,
 *       and on c4a layers the indexer cache d = 128).
 *   (2) dsv4_indexer_topk    : lightning-indexer scores over the causal
 *       compressed slots and a per-query top-k (c4a layers that are not
 *       IndexCache reuse layers).  c128a layers pass precomputed indices.
 *   (3) dsv4_sparse_mla_decode : absorbed-MQA attention of every query head
 *       over (selected compressed slots) || (SWA window), one 576-dim latent
 *       KV head, value = the first 512 dims (or, with the V4-native layout,
 *       one 512-dim head that is key and value, and optionally the output's
 *       inverse RoPE + FP8 quantisation, dsv4_inv_rope_fp8_quant).
 *   (4) prefill: the same indexer and attention with one query row per
 *       prefill token (dsv4_sparse_mla_prefill), plus the pages' dense-buffer
 *       helpers (dsv4_dequant_gather, dsv4_combine_topk_swa_indices).
 *
 * Sources (page title, section):
 *   [vLLM-V4-attn]  "DeepSeek V4 attention in vLLM" (juejin): compress_ratio
 *                   table, attention_impl call order, Compressor ratio 4 vs
 *                   128, Indexer / C4A / C128A top-k branch, SWA cache.
 *   [IndexCache]    "DeepSeek-V4 IndexCache freq2 cross-layer TopK reuse",
 *                   sections 2-4.
 *   [vLLM-classes]  "DeepseekV4Attention" class walkthrough (devpress):
 *                   DeepseekV4Indexer, DeepseekCompressor.forward, "CSA layer
 *                   Compressor", SparseAttnIndexer formula, _forward_decode.
 *   [V4-internals]  "From compressed attention to executable inference"
 *                   (talk write-up), sections 2, 4, 6.
 *   [MLA-to-CSA]    "From MLA to CSA + HCA", sections 2.2, 5.1-5.5, 6.3.
 *
 * Conventions for every entry point:
 *   - Pointers named *_dev are device pointers; the caller owns every buffer
 *     (caches, state, outputs, workspace).  The library allocates nothing on
 *     the hot path; plans are small host objects.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  The return value reports host-side validation and
 *     launch errors only.
 *   - Device-side checks (an index or block-table entry out of range, a
 *     position that breaks the contiguity rule, a bounded wait that ran out)
 *     skip the offending access and OR a bit into the caller's device status
 *     word (int, may be NULL); dsv4_read_device_status() reads and clears it.
 *     No call traps, asserts or aborts; nothing throws across the ABI.
 *   - Geometry: latent 512 (nope) + 64 (rope) = 576 dims, value = 512 latent
 *     dims by default, or the V4-native 448 + 64 rows with K = V per plan
 *     (dsv4_plan_set_kv_layout); pages of 64 entries / tokens, indexer head
 *     dim 128 (FP8 or MXFP4 entries, dsv4_plan_set_indexer_format), SWA
 *     window 128.
 *
 * Cache layouts in HBM (all pages 64 entries; page id from a block table):
 *   compressed (main) cache page, 64 * 648 = 41472 bytes:
 *     [64 rows x 640 B: 512 FP8 E4M3 nope codes, 64 bf16 rope values]
 *     [64 rows x 8 B: UE8M0 exponent byte (e + 127) per 64 nope dims]
 *   indexer cache page, 64 * 132 = 8448 bytes:
 *     [64 rows x 128 FP8 E4M3 codes][64 fp32 scales]
 *   SWA cache page, 64 * 1152 = 73728 bytes: [64 tokens x 576 bf16].
 *   Logical compressed slot j of a sequence lives in page bt[j / 64], row
 *   j % 64; SWA token t in page bt[t / 64], row t % 64.
 *
 * V4-native geometry (plans set to DSV4_KV_V4, cache kind DSV4_CACHE_V4;
 * [MLA-to-CSA] 5.5 and 6.4, [V4-internals] section 6): head 512 = 448 nope
 * + 64 rope dims, one vector serving as key and value (K = V, the value
 * includes the rope dims), and both the compressed and the SWA cache in one
 * FP8 row format of 584 bytes:
 *   page, 64 * 584 = 37376 bytes:
 *     [64 rows x 576 B: 448 FP8 E4M3 nope codes, 64 bf16 rope values]
 *     [64 rows x 8 B: UE8M0 byte per 64 nope dims (7), one zero pad byte]
 * The attention output then carries the keys' rotation on dims 448..511;
 * dsv4_inv_rope_fp8_quant applies R(-position) and quantises it for the
 * output projection.
 */
#ifndef DSV4_H
#define DSV4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DSV4_VERSION 1

#define DSV4_NOPE_DIM 512
#define DSV4_ROPE_DIM 64
#define DSV4_HEAD_DIM 576
#define DSV4_V_DIM 512
#define DSV4_IDX_DIM 128
#define DSV4_PAGE 64
#define DSV4_WINDOW 128
#define DSV4_MLA_ENTRY_BYTES 648
#define DSV4_MLA_PAGE_BYTES (64 * 648)
#define DSV4_IDX_ENTRY_BYTES 132
#define DSV4_IDX_PAGE_BYTES (64 * 132)
#define DSV4_IDX_FP4_ENTRY_BYTES 68
#define DSV4_IDX_FP4_PAGE_BYTES (64 * 68)
#define DSV4_SWA_PAGE_BYTES (64 * 576 * 2)
#define DSV4_V4_NOPE_DIM 448
#define DSV4_V4_HEAD_DIM 512
#define DSV4_V4_ENTRY_BYTES 584
#define DSV4_V4_PAGE_BYTES (64 * 584)
#define DSV4_MAX_HEADS 128
#define DSV4_MAX_IDX_HEADS 64

typedef struct CUstream_st* dsv4_stream_t;   /* a cudaStream_t */

typedef enum dsv4_status {
    DSV4_OK = 0,
    DSV4_ERR_INVALID = 1,       /* null pointer, negative size, bad enum */
    DSV4_ERR_SHAPE = 2,         /* sizes inconsistent with each other or the plan */
    DSV4_ERR_UNSUPPORTED = 3,   /* a value outside what this build implements */
    DSV4_ERR_CUDA = 4,          /* a CUDA runtime error at launch */
    DSV4_ERR_DEVICE_CHECK = 5,  /* a device-side range / consistency check fired */
    DSV4_ERR_TIMEOUT = 6        /* a bounded device-side wait ran out */
} dsv4_status;

/* Device status word bits (OR-ed by kernels into the caller's int). */
#define DSV4_DEV_BAD_INDEX 0x1      /* a gathered slot / token index out of range */
#define DSV4_DEV_BAD_PAGE 0x2       /* a block-table lookup out of range */
#define DSV4_DEV_BAD_POSITION 0x4   /* positions not contiguous per sequence */
#define DSV4_DEV_TIMEOUT 0x8        /* a bounded wait ran out */

/* [vLLM-V4-attn] "compress_ratio: the three layer types". */
typedef enum dsv4_layer_type {
    DSV4_SWAONLY = 1,
    DSV4_C4A = 4,
    DSV4_C128A = 128
} dsv4_layer_type;

typedef enum dsv4_cache_kind {
    DSV4_CACHE_MLA = 0,     /* main compressed cache, d = 576, 648-byte entries */
    DSV4_CACHE_IDX = 1,     /* indexer cache, d = 128, 132-byte entries (FP8 + fp32 scale) */
    DSV4_CACHE_IDX_FP4 = 2, /* indexer cache in MXFP4, d = 128, 68-byte entries: 64 bytes of
                               E2M1 codes (two per byte, the low nibble the even dim) and one
                               UE8M0 exponent byte per 32 dims; page = 64 x 64 code bytes, then
                               64 x 4 exponent bytes.  [V4-attn] use_fp4_indexer_cache;
                               [V4-internals] section 4 (64 x 68 B); [MLA-to-CSA] 6.1 */
    DSV4_CACHE_V4 = 3       /* V4-native row, d = 512 (448 nope + 64 rope), 584-byte entries
                               (DSV4_V4_PAGE_BYTES pages): the main compressed cache of a
                               DSV4_KV_V4 plan, and its FP8 SWA cache ([MLA-to-CSA] 5.5) */
} dsv4_cache_kind;

/* ---- host utilities ------------------------------------------------------ */

/* Layer type of a layer's compress_ratio: max(1, r); 1 -> swaonly, 4 -> c4a,
 * 128 -> c128a ([vLLM-V4-attn] compress_ratio table; the Compressor asserts
 * r in {4, 128}).  Other ratios: DSV4_ERR_UNSUPPORTED. */
dsv4_status dsv4_layer_type_from_ratio(int compress_ratio, dsv4_layer_type* out);

/* IndexCache top-k reuse schedule ([IndexCache] section 2).  For each layer l
 * with ratio 4, rank = number of ratio-4 layers before l; with
 * use_index_cache, skip_topk_out[l] = (rank % freq != 0), or, when `pattern`
 * is non-NULL (it takes precedence), 1 iff pattern[rank] == 'S'; ranks past
 * the end of the pattern compute.  The pattern must match F[FS]*.  Other
 * layers get 0.  A skipped layer consumes the index buffer last written by a
 * computing c4a layer of the same step (indices only, never KV: the reuse
 * layer still runs its own compressor and reads its own caches).
 * skip_topk_out: host array of n_layers bytes.
 * Errors: DSV4_ERR_INVALID for a bad pattern, freq < 1 with use_index_cache,
 * or NULL arrays. */
dsv4_status dsv4_index_schedule(const int* ratios, int n_layers, int use_index_cache, int freq,
                                const char* pattern, unsigned char* skip_topk_out);

/* RoPE table, [max_pos][rope_dim] fp32 into host memory: first half cos,
 * second half sin of pos * theta^(-2i/rope_dim), computed in double and
 * rounded once ([vLLM-classes] DeepseekCompressor.forward, cos_sin_cache
 * comment).  The caller copies it to the device. */
dsv4_status dsv4_rope_table(float* host_out, int max_pos, int rope_dim, double theta);

/* Read the device status word (blocking: copies 4 bytes and synchronises
 * `stream`), store its bits in *bits_out (may be NULL) and reset it to 0.
 * Returns DSV4_OK, DSV4_ERR_TIMEOUT if DSV4_DEV_TIMEOUT is set, else
 * DSV4_ERR_DEVICE_CHECK if any other bit is set. */
dsv4_status dsv4_read_device_status(int* status_dev, dsv4_stream_t stream, int* bits_out);

const char* dsv4_status_string(dsv4_status s);
int dsv4_version(void);

/* ---- plans (per layer type, reused by every layer of that type) --------- */

/* [vLLM-V4-attn] "SWA cache and tile scheduler": one scheduling plan per
 * layer type, never shared across types; every layer of a type reuses it
 * within a step.  A plan fixes the batch, heads, top-k width and maximum
 * context, and from them the work split of the indexer and attention kernels
 * and the workspace layout. */
typedef struct dsv4_geom {
    int n_heads;          /* query heads sharing the latent KV head, 1..128 */
    int idx_heads;        /* indexer heads (c4a), 1..64; ignored otherwise */
    int window;           /* SWA window; this build: 128 */
    float softmax_scale;  /* attention logit scale, e.g. 1/sqrt(576) */
} dsv4_geom;

typedef struct dsv4_plan dsv4_plan;

typedef struct dsv4_plan_info {
    int layer_type;
    int batch, n_heads, idx_heads, topk, max_ctx;
    int max_slots;            /* max compressed slots per sequence (c4a: max_ctx / 4) */
    int idx_ctas_per_seq;     /* indexer work split */
    int mla_splits;           /* key splits per (sequence, head group) */
    int mla_head_groups;      /* 64-head groups */
    int mla_keys_per_split;
    size_t workspace_bytes;
    int launches_indexer;     /* kernels one dsv4_indexer_topk call launches */
    int launches_mla;         /* kernels one dsv4_sparse_mla_decode call launches */
} dsv4_plan_info;

/* topk: width of the index rows (c4a: the indexer's k; c128a: the metadata
 * width; swaonly: 0).  max_ctx: largest context (query position + 1). */
dsv4_status dsv4_plan_create(dsv4_layer_type type, const dsv4_geom* geom, int batch, int topk,
                             int max_ctx, dsv4_plan** out);
void dsv4_plan_destroy(dsv4_plan* plan);
/* Device workspace the plan's calls need (bytes, 256-byte aligned base). */
size_t dsv4_plan_workspace_bytes(const dsv4_plan* plan);
dsv4_status dsv4_plan_get_info(const dsv4_plan* plan, dsv4_plan_info* info);

/* Indexer cache format of a c4a plan ([V4-attn] eval note
 * use_fp4_indexer_cache: only the indexer's K cache changes format;
 * [V4-internals] section 4: the C4 indexer block as 64 x 68 B;
 * [MLA-to-CSA] 6.1: lightning-indexer K cache in FP4 / MXFP4).
 *   DSV4_IDX_FP8 (the default): 132-byte entries (DSV4_CACHE_IDX pages);
 *   DSV4_IDX_FP4: 68-byte MXFP4 entries (DSV4_CACHE_IDX_FP4 pages).
 * With FP4, dsv4_indexer_topk scores k[s][c] = E2M1(code) * 2^(exponent
 * byte of c's 32-dim block - 127) with the same FP8 query and the same top-k
 * rule; idx_cache_dev then holds DSV4_IDX_FP4_PAGE_BYTES pages and
 * num_pages counts those.  Set it after dsv4_plan_create, before the plan's
 * first call.  Errors: DSV4_ERR_INVALID (NULL plan or unknown format),
 * DSV4_ERR_UNSUPPORTED (not a c4a plan). */
typedef enum dsv4_idx_format { DSV4_IDX_FP8 = 0, DSV4_IDX_FP4 = 1 } dsv4_idx_format;
dsv4_status dsv4_plan_set_indexer_format(dsv4_plan* plan, dsv4_idx_format format);

/* KV geometry of a plan's attention ([MLA-to-CSA] 5.5: the V4 layout with
 * K = V sharing and the FP8 SWA cache; 6.4: the output keeps the keys'
 * rotation until the inverse RoPE).
 *   DSV4_KV_576 (the default): q 576 dims, value = the 512 latent dims,
 *     compressed cache DSV4_CACHE_MLA, SWA cache bf16 [576].
 *   DSV4_KV_V4: q_dev bf16 [batch][n_heads][512]; keys are 512-dim rows of
 *     DSV4_CACHE_V4 pages in BOTH caches (compressed slots and SWA tokens,
 *     swa_cache_dev / swa_num_pages then count DSV4_V4_PAGE_BYTES pages);
 *     key = FP8 * 2^(scale byte - 127) on dims 0..447, bf16 on 448..511;
 *     s = softmax_scale * q . key (512 dims), out[b][h] = sum P * key (all 512
 *     dims, bf16).  Everything else as for DSV4_KV_576.
 * Set it after dsv4_plan_create, before the plan's first call.  Errors:
 * DSV4_ERR_INVALID (NULL plan or unknown layout). */
typedef enum dsv4_kv_layout { DSV4_KV_576 = 0, DSV4_KV_V4 = 1 } dsv4_kv_layout;
dsv4_status dsv4_plan_set_kv_layout(dsv4_plan* plan, dsv4_kv_layout layout);

/* ---- (1) compressor insert ----------------------------------------------- */

/* [vLLM-classes] DeepseekCompressor.forward, save_partial_states and "CSA
 * layer Compressor"; [vLLM-V4-attn] "Compressor: ratio 4 vs 128";
 * [MLA-to-CSA] 5.1, 5.2 and 6.3 (compressed slot mapping).
 *
 * For every token t (position p, sequence b):
 *   state row = (kv = fp32(bf16 kv), score' = fp32(bf16 score + ape[p % r]))
 * and when (p + 1) % r == 0 the entry of logical slot j = p / r is built from
 * the window (r = 4: tokens p-7..p-4 with block a, p-3..p with block b;
 * r = 128: tokens p-127..p; tokens at negative positions left out):
 *   y_c = sum_t softmax_t(score'_{t,c}) * kv_{t,c}       (per channel c)
 *   z = RMSNorm(y) * rms_weight;  RoPE (GPT-J pairs) on the last 64 dims at
 *   position (p / r) * r;  quantise (main: FP8 E4M3 nope with a UE8M0 scale
 *   per 64 dims + bf16 rope; indexer: FP8 E4M3 of all 128 dims with scale
 *   amax / 448) and write it to page bt[b][j / 64], row j % 64.
 * The fp32 operation sequence (and the exp used by the softmax) is fixed so
 * the cache bytes are reproducible bit for bit.
 *
 * kv_score_dev: bf16 [num_tokens][2*coff*d] (row stride kv_score_stride
 *   elements): [kv block 0 | kv block 1 | score block 0 | score block 1],
 *   coff = 2 for r = 4, 1 for r = 128; d = 576 (main), 512 (DSV4_CACHE_V4:
 *   RMSNorm over 512 dims, RoPE on 448..511, FP8 on 0..447 with 7 UE8M0
 *   bytes and a zero pad byte) or 128 (indexer).
 * positions_dev, seq_dev: int32 [num_tokens].  The tokens of one sequence in
 *   one call are adjacent in the token array with contiguous increasing
 *   positions (checked: DSV4_DEV_BAD_POSITION).
 * ape_dev: fp32 [r][coff*d];  rms_weight_dev: fp32 [d];
 * cos_sin_dev: fp32 [max_pos][64] (dsv4_rope_table layout).
 * state_dev: fp32 [num_seqs][coff*r][2*coff*d], a per-sequence ring: the row
 *   of position p lives at p % (coff*r).  The caller zero-fills it once; the
 *   library keeps it (rows of positions before a call are read from it).
 *   16-byte aligned, as is cache_dev (else DSV4_ERR_SHAPE).
 * cache_dev: paged cache of `kind`, num_pages pages; block_table_dev: int32
 *   [num_seqs][bt_stride], bt_stride >= pages needed by the largest slot.
 * one_token_per_seq: 1 when every sequence has at most one token in this
 *   call (decode): one fused launch.  0 allows several (chunked prefill):
 *   two launches (entries first, then the state ring).
 * Errors: DSV4_ERR_INVALID (null pointers, sizes < 0), DSV4_ERR_UNSUPPORTED
 *   (r not in {4, 128}; indexer cache with r != 4). */
typedef struct dsv4_compress_args {
    int kind;                    /* dsv4_cache_kind */
    int ratio;                   /* 4 or 128 */
    int num_tokens;
    int num_seqs;
    int one_token_per_seq;
    const void* kv_score_dev;
    long long kv_score_stride;   /* elements between token rows */
    const int* positions_dev;
    const int* seq_dev;
    const float* ape_dev;
    const float* rms_weight_dev;
    float rms_eps;
    const float* cos_sin_dev;
    int max_pos;                 /* rows of cos_sin */
    float* state_dev;
    void* cache_dev;
    int num_pages;               /* physical pages in cache_dev */
    const int* block_table_dev;
    int bt_stride;
    int* status_dev;             /* optional device status word */
} dsv4_compress_args;

dsv4_status dsv4_compress_insert(const dsv4_compress_args* args, dsv4_stream_t stream);

/* Both compressor streams of a layer in one launch, for decode steps:
 * main_args (DSV4_CACHE_MLA or DSV4_CACHE_V4, ratio 4 or 128) and idx_args
 * (DSV4_CACHE_IDX or DSV4_CACHE_IDX_FP4, ratio 4), each with one_token_per_seq set.  Same effect, arguments and
 * errors as the two dsv4_compress_insert calls (DSV4_ERR_INVALID also for a
 * wrong kind or a call without one_token_per_seq); the two streams touch
 * disjoint state and caches, so their entries are computed side by side. */
dsv4_status dsv4_compress_insert_pair(const dsv4_compress_args* main_args, const dsv4_compress_args* idx_args,
                                      dsv4_stream_t stream);

/* Quantise already-final rows into the cache format and insert them: the
 * quantise-and-insert tail of dsv4_compress_insert on its own (no pooling,
 * normalisation or rotation), for filling caches with given entries.
 * rows_dev: fp32 [num_rows][d] (d = 576, 128 or 512 by kind; DSV4_CACHE_V4
 * rows also serve as the FP8 SWA tokens of a DSV4_KV_V4 plan, slot = token
 * position); seq_dev, slot_dev:
 * int32 [num_rows] (sequence and logical slot of each row). */
typedef struct dsv4_insert_rows_args {
    int kind;
    int num_rows;
    const float* rows_dev;
    const int* seq_dev;
    const int* slot_dev;
    void* cache_dev;
    int num_pages;
    const int* block_table_dev;
    int bt_stride;
    int num_seqs;
    int* status_dev;
} dsv4_insert_rows_args;

dsv4_status dsv4_cache_insert_rows(const dsv4_insert_rows_args* args, dsv4_stream_t stream);

/* ---- (2) lightning indexer + top-k ---------------------------------------- */

/* [vLLM-classes] SparseAttnIndexer: I_{t,s} = sum_j w_{t,j} ReLU(q_{t,j} .
 * k_s) with one key per slot shared by all indexer heads;
 * [vLLM-V4-attn] "Indexer, C4A and C128A top-k"; [V4-internals] section 6
 * (top-k indices and lengths).
 *
 * For each sequence b with context L = ctx_len[b] (query position L - 1),
 * the causal slots are s < n_c = L / 4 (the slot emitted at the query's own
 * position is visible).  k_s = FP8 row * its fp32 scale.  The k slots with
 * the largest I (ties: lower slot first) are written to out_idx[b][0..len)
 * in ascending slot order, len = min(k, n_c), the rest of the row -1.
 *
 * q_fp8_dev: FP8 E4M3 [batch][idx_heads][128]; weights_dev: fp32
 *   [batch][idx_heads] (any per-head q scale folded in by the caller);
 * idx_cache_dev: indexer cache pages; block_table_dev int32 [batch][bt_stride];
 * ctx_len_dev: int32 [batch], 1 <= L <= plan max_ctx;
 * out_idx_dev: int32 [batch][out_stride] (out_stride >= topk);
 * out_len_dev: int32 [batch].
 * workspace: dsv4_plan_workspace_bytes(plan) bytes of device memory,
 *   16-byte aligned.
 * Errors: DSV4_ERR_SHAPE if the plan is not a c4a plan, the workspace is
 *   too small or not 16-byte aligned, or idx_cache_dev is not 16-byte
 *   aligned; DSV4_ERR_INVALID for null pointers. */
typedef struct dsv4_indexer_args {
    const void* q_fp8_dev;
    const float* weights_dev;
    const void* idx_cache_dev;
    int num_pages;
    const int* block_table_dev;
    int bt_stride;
    const int* ctx_len_dev;
    int* out_idx_dev;
    int out_stride;
    int* out_len_dev;
    int* status_dev;
    /* Prefill (and any caller whose rows are not sequences): NULL for decode,
     * where row b is sequence b; else int32 [batch], the block-table row of
     * each query row (a prefill query token of position ctx_len[b] - 1 takes
     * its sequence's row).  bt_rows: the block table's row count, which every
     * row_seq value must stay below (checked: DSV4_DEV_BAD_INDEX, the row
     * then reads row 0). */
    const int* row_seq_dev;
    int bt_rows;
} dsv4_indexer_args;

dsv4_status dsv4_indexer_topk(const dsv4_plan* plan, const dsv4_indexer_args* args,
                              void* workspace_dev, size_t workspace_bytes, dsv4_stream_t stream);

/* Allocation-free variant of dsv4_indexer_topk.  The pages have no
 * counterpart: this entry point exists for callers that cannot allocate
 * device memory or own a workspace -- e.g. a plugin inside a serving engine
 * whose allocator owns every device allocation, or a restricted deployment
 * where cudaMalloc is not permitted.  It computes exactly what
 * dsv4_indexer_topk computes, but the per-query logits live in a file-scope
 * device array of 4 MiB that every GPU loading the library holds until the
 * process exits; no call allocates or frees memory.
 *   - Limit: the plan's workspace (batch x max_slots fp32 logits, 256-byte
 *     aligned) must fit in 4 MiB, e.g. batch 32 at context 131072 or batch 4
 *     at context 1,048,576; larger plans return DSV4_ERR_UNSUPPORTED and
 *     launch nothing.
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current); make that first call before any
 *     stream capture.
 *   - All calls share the one array: calls whose executions overlap on the
 *     GPU (other streams, other host threads) race on it.  Nothing in it has
 *     to start at zero; each call writes every logit it reads.
 *   - The looked-up address belongs to the device's current context.  After
 *     cudaDeviceReset (or any other end of that context) it is stale: do not
 *     call this entry point on that device again in the same process.
 * Arguments and errors otherwise as dsv4_indexer_topk. */
dsv4_status dsv4_indexer_topk_noalloc(const dsv4_plan* plan, const dsv4_indexer_args* args,
                                      dsv4_stream_t stream);

/* ---- (3) sparse MLA decode --------------------------------------------------- */

/* [vLLM-classes] _forward_decode (SWA indices plus the compressed top-k,
 * flash_mla_with_kvcache over both caches); [V4-internals] section 2
 * (KV_actual = selected history || recent window); [MLA-to-CSA] 2.2
 * (absorbed decode over the 576-dim latent, MQA-style) and 5.1.
 *
 * For each sequence b (query position p = ctx_len[b] - 1) and head h:
 *   keys = compressed slots topk_idx[b][0..topk_len[b]) (dequantised: FP8 *
 *          2^(scale byte - 127), bf16 rope) followed by the SWA tokens
 *          max(0, p - 127) .. p;
 *   s = softmax_scale * q[b][h] . key (576 dims), P = softmax(s),
 *   out[b][h] = sum P * key[0:512] (bf16), lse[b][h] = max s + ln sum e^(s - max).
 * swaonly plans ignore the compressed cache and indices (may be NULL).
 *
 * q_dev: bf16 [batch][n_heads][576]; out_dev: bf16 [batch][n_heads][512]
 * (q_dev, out_dev and both caches 16-byte aligned, else DSV4_ERR_SHAPE);
 * lse_dev: fp32 [batch][n_heads] or NULL.
 * swa_cache_dev / swa_block_table_dev: SWA pages; comp_cache_dev /
 * comp_block_table_dev: compressed pages; topk_idx_dev: int32
 * [batch][topk_stride] logical slots; topk_len_dev: int32 [batch].
 * Errors: DSV4_ERR_SHAPE on plan / workspace mismatch, DSV4_ERR_INVALID. */
typedef struct dsv4_mla_args {
    const void* q_dev;
    const void* swa_cache_dev;
    int swa_num_pages;
    const int* swa_block_table_dev;
    int swa_bt_stride;
    const void* comp_cache_dev;
    int comp_num_pages;
    const int* comp_block_table_dev;
    int comp_bt_stride;
    const int* topk_idx_dev;
    int topk_stride;
    const int* topk_len_dev;
    const int* ctx_len_dev;
    void* out_dev;
    float* lse_dev;
    int* status_dev;
    /* As in dsv4_indexer_args: NULL for decode; else the block-table row
     * (of both tables, bt_rows rows each) of each query row. */
    const int* row_seq_dev;
    int bt_rows;
    /* DSV4_KV_V4 plans only, optional (NULL: not produced): the attention
     * output's inverse RoPE + FP8 quantisation as dsv4_inv_rope_fp8_quant
     * defines it (rotation R(-p) at the row's query position p = ctx_len - 1,
     * 128-dim blocks with fp32 scales), computed from the bf16 output and
     * written to out_codes_dev (E4M3 [batch][n_heads][512]) and out_scales_dev
     * (fp32 [batch][n_heads][4]); cos_sin_dev: fp32 [max_pos][64].  The
     * call launches the quantisation kernel after the attention (stream
     * order); out_dev is written as well.  A position outside [0, max_pos)
     * sets DSV4_DEV_BAD_POSITION and leaves that row's codes unwritten. */
    void* out_codes_dev;
    float* out_scales_dev;
    const float* cos_sin_dev;
    int max_pos;
} dsv4_mla_args;

dsv4_status dsv4_sparse_mla_decode(const dsv4_plan* plan, const dsv4_mla_args* args,
                                   void* workspace_dev, size_t workspace_bytes,
                                   dsv4_stream_t stream);

/* Inverse RoPE and FP8 quantisation of the attention output of a DSV4_KV_V4
 * plan ([MLA-to-CSA] 6.4, fused_inv_rope_fp8_quant ahead of the FP8 output
 * projection; [V4-internals] section 6, "Inverse RoPE + FP8 Quant" fused so
 * the rotated output never reaches HBM).  For token t (position
 * positions_dev[t]) and head h, with x = fp32 of o[t][h][0:512]:
 *   dims 448..511, GPT-J pairs i: (x0, x1) -> (x0 c + x1 s, x1 c - x0 s),
 *     c = cos_sin[pos][i], s = cos_sin[pos][32 + i] (the rotation R(-pos);
 *     each product and the sum rounded to fp32), so that the value rotated
 *     by R(j) at key position j carries R(j - pos);
 *   then each 128-dim block k: scale = amax / 448 (fp32, 1 for an all-zero
 *     block), codes = E4M3(x / scale) (round to nearest even, saturating).
 * Reading: the pages name the operator and its inputs but not the scale
 * grain; 128-dim blocks with fp32 scales (the indexer cache's rule) are used.
 * o_dev: bf16 [num_tokens][n_heads][512]; positions_dev: int32 [num_tokens];
 * cos_sin_dev: fp32 [max_pos][64]; codes_dev: E4M3 [num_tokens][n_heads][512];
 * scales_dev: fp32 [num_tokens][n_heads][4].  A position outside
 * [0, max_pos) sets DSV4_DEV_BAD_POSITION and leaves that token's rows
 * unwritten.  Errors: DSV4_ERR_INVALID (NULL pointers, negative sizes),
 * DSV4_ERR_SHAPE (o_dev or codes_dev not 16-byte aligned). */
typedef struct dsv4_inv_rope_quant_args {
    int num_tokens;
    int n_heads;
    const void* o_dev;
    const int* positions_dev;
    const float* cos_sin_dev;
    int max_pos;
    void* codes_dev;
    float* scales_dev;
    int* status_dev;
} dsv4_inv_rope_quant_args;
dsv4_status dsv4_inv_rope_fp8_quant(const dsv4_inv_rope_quant_args* args, dsv4_stream_t stream);

/* ---- (4) sparse prefill -------------------------------------------------------- */

/* Sparse prefill attention ([vLLM-classes] _forward_prefill: each prefill
 * token attends over its top-k compressed slots and its causal SWA window,
 * flash_mla_sparse_fwd).  Computes, for each query row b (a prefill token at
 * position ctx_len[b] - 1 of sequence row_seq_dev[b]), exactly what
 * dsv4_sparse_mla_decode computes for a decode row, reading the paged caches
 * through the sequence's block-table rows: a plan whose batch is the number
 * of query rows serves a prefill chunk.  The top-k of each row comes from
 * dsv4_indexer_topk with the same row_seq_dev (c4a) or from caller metadata
 * (c128a); the SWA cache must hold every token of the windows.
 * Errors: as dsv4_sparse_mla_decode; DSV4_ERR_INVALID if row_seq_dev is NULL. */
dsv4_status dsv4_sparse_mla_prefill(const dsv4_plan* plan, const dsv4_mla_args* args, void* workspace_dev,
                                    size_t workspace_bytes, dsv4_stream_t stream);

/* Dequantise-and-gather of cache rows into a dense bf16 buffer
 * ([vLLM-classes] _forward_prefill, dequantize_and_gather_k_cache: the
 * compressed cache into kv[:, 0:N], the SWA cache into kv[:, N:N+gather_len]).
 * For each sequence s < num_seqs and i < count_dev[s] (<= max_count):
 *   out[s][out_offset + i][0:576] = row of slot / token first_dev[s] + i,
 * through block_table_dev[s][...].  DSV4_GATHER_COMP: a compressed entry
 * dequantised (FP8 * 2^(scale - 127) for dims 0..511, the bf16 rope dims);
 * DSV4_GATHER_SWA: the bf16 SWA row.  out_dev: bf16 [num_seqs][out_rows][576]
 * (16-byte aligned, out_rows >= out_offset + max_count).  A bad page sets
 * DSV4_DEV_BAD_PAGE and writes a zero row; a count past max_count sets
 * DSV4_DEV_BAD_INDEX and is clamped.  Errors: DSV4_ERR_INVALID, _SHAPE,
 * _UNSUPPORTED (max_count or num_seqs above 65535). */
typedef enum dsv4_gather_kind { DSV4_GATHER_COMP = 0, DSV4_GATHER_SWA = 1 } dsv4_gather_kind;
typedef struct dsv4_gather_args {
    int kind;                      /* dsv4_gather_kind */
    const void* cache_dev;         /* compressed pages (DSV4_MLA_PAGE_BYTES) or SWA pages */
    int num_pages;
    const int* block_table_dev;    /* int32 [num_seqs][bt_stride] */
    int bt_stride;
    int num_seqs;
    const int* first_dev;          /* int32 [num_seqs] */
    const int* count_dev;          /* int32 [num_seqs] */
    int max_count;
    void* out_dev;
    int out_rows;
    int out_offset;
    int* status_dev;
} dsv4_gather_args;
dsv4_status dsv4_dequant_gather(const dsv4_gather_args* args, dsv4_stream_t stream);

/* Each prefill token's key list over the gathered buffer ([vLLM-classes]
 * _forward_prefill, combine_topk_swa_indices): the valid (>= 0) entries of
 * topk_dev[t][0:topk_len_dev[t]] in order, then the window tokens
 * max(0, pos - window + 1) .. pos as rows n_comp + (token - (seq_len -
 * gather_len)) of its sequence row_seq_dev[t]; out_len_dev[t] is the count
 * and the rest of the row is -1.  A window token outside the gathered run, a
 * sequence out of range or an output row too short sets DSV4_DEV_BAD_INDEX
 * and out_len -1. */
typedef struct dsv4_combine_args {
    const int* topk_dev;           /* int32 [num_tokens][topk_stride] (logical slots, -1 padding) */
    int topk_stride;
    const int* topk_len_dev;       /* int32 [num_tokens] */
    const int* pos_dev;            /* int32 [num_tokens] query positions */
    const int* row_seq_dev;        /* int32 [num_tokens] sequence of each token */
    const int* seq_len_dev;        /* int32 [num_seqs] */
    const int* gather_len_dev;     /* int32 [num_seqs] SWA tokens gathered (the last of the sequence) */
    int num_tokens;
    int num_seqs;
    int window;
    int n_comp;                    /* N: buffer row of the first gathered SWA token */
    int* out_dev;                  /* int32 [num_tokens][out_stride] */
    int out_stride;
    int* out_len_dev;              /* int32 [num_tokens] */
    int* status_dev;
} dsv4_combine_args;
dsv4_status dsv4_combine_topk_swa_indices(const dsv4_combine_args* args, dsv4_stream_t stream);

/* ---- pipelined input staging ------------------------------------------------- */

/* Stream gate for a decode loop whose inputs arrive by host-to-device copies
 * on another stream.  Not a step of the method: serving support around it.
 * Launches one 32-thread CTA that waits (bounded) until every non-NULL
 * flags_dev[i] is nonzero, clears those flags to 0 and then lets the next
 * kernel on `stream` launch under programmatic dependent launch; the gate's
 * grid completes only after the kernel before it on `stream` has completed.
 * Usage: on the copy stream, copy a step's inputs, then write 1 into the
 * step's flag (a 4-byte copy, stream-ordered after the data); on the compute
 * stream, call the gate in front of the step's calls instead of waiting on an
 * event.  An event wait between two kernels breaks their programmatic launch
 * link; the gate keeps the link to the previous step's last kernel.  Only work
 * ordered after the kernels that read what a flag guards may set it again
 * (e.g. a copy stream waiting on an event recorded after those kernels).
 * flags_dev: up to 4 int flags (4-byte aligned; NULL entries ignored, at
 *   least one given).  timeout_us: bound of the wait (0: 2 s); a wait that
 *   runs out sets DSV4_DEV_TIMEOUT in *status_dev, clears no flag and lets
 *   the next kernel launch.
 * Errors: DSV4_ERR_INVALID (NULL args, no flag, negative timeout),
 * DSV4_ERR_SHAPE (a misaligned flag), DSV4_ERR_CUDA (launch). */
typedef struct dsv4_gate_args {
    int* flags_dev[4];
    int timeout_us;
    int* status_dev;
} dsv4_gate_args;
dsv4_status dsv4_stream_gate(const dsv4_gate_args* args, dsv4_stream_t stream);

/* ---- diagnostics ------------------------------------------------------------- */

/* Launch one CTA that waits on an mbarrier nothing arrives at, bounded by
 * `spin_limit` polls, so a test can see the bounded-wait path set
 * DSV4_DEV_TIMEOUT in *status_dev and return (the context stays usable). */
dsv4_status dsv4_selftest_bounded_wait(int* status_dev, int spin_limit, dsv4_stream_t stream);

/* Run the decode kernel's key conversion (FP8 E4M3 code times 2^(s - 127),
 * s a UE8M0 scale byte, to bf16) over every code c and scale byte s:
 * out_dev: uint16 [256 * 256], out[s * 256 + c] = the bf16 bits.  Lets a test
 * check the conversion exhaustively against the definition of the two formats
 * (section "FP8 Quant" of the compressor walkthrough: E4M3 codes with one
 * power-of-two scale per 64 dims).  Errors: DSV4_ERR_INVALID (NULL),
 * DSV4_ERR_SHAPE (misaligned), DSV4_ERR_CUDA (launch). */
dsv4_status dsv4_selftest_key_dequant(void* out_dev, dsv4_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* DSV4_H */
