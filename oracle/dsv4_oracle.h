/*
 * dsv4_oracle.h -- plain, slow CPU reference for DeepSeek-V4 compressed sparse
 * attention at decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library and
 * its Python binding) includes, links or calls this code; only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg do.  It shares no code,
 * header, table or helper with the CUDA path.
 *
 * Sources are cited as "page title, section" of the five web pages the method
 * is described on:
 *   [vLLM-V4-attn]   juejin.cn "DeepSeek V4 attention in vLLM" (compress_ratio
 *                    table; Compressor: ratio 4 vs 128; Indexer/C4A/C128A top-k)
 *   [IndexCache]     "DeepSeek-V4 IndexCache freq2 cross-layer TopK reuse"
 *                    (sections 2 and 4)
 *   [vLLM-classes]   devpress "DeepseekV4Attention" walkthrough (DeepseekV4Indexer,
 *                    DeepseekCompressor, "CSA layer Compressor", SparseAttnIndexer,
 *                    _forward_decode)
 *   [V4-internals]   "From compressed attention to executable inference" talk
 *                    write-up (sections 2, 4, 6)
 *   [MLA-to-CSA]     "From MLA to CSA + HCA" (sections 2.2, 5.1, 5.2, 5.5, 6.3,
 *                    appendix A.4)
 *
 * Precision: fp64 everywhere except where a floating-point value decides a
 * stored integer code (the compressor's FP8/bf16 cache bytes).  There the
 * oracle computes in fp32 with one fixed, stated operation sequence (IEEE
 * add/mul/div/sqrt, no fused multiply-add, its own exp), so that the cache
 * bytes are defined exactly.
 */
#ifndef DSV4_ORACLE_H
#define DSV4_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- number formats ---------------------------------------------------- */
float    or_bf16_to_f32(uint16_t h);
uint16_t or_f32_to_bf16(float x);            /* round to nearest even */
double   or_e4m3_to_f64(uint8_t code);       /* OCP E4M3 ("e4m3fn") */
uint8_t  or_f32_to_e4m3(float x);            /* nearest, ties to even, saturate to +-448 */
int      or_ue8m0_exponent(float amax);      /* smallest e with amax <= 448 * 2^e */
float    or_expf(float x);                   /* the compressor's exp (Cody-Waite + Taylor) */
void     or_f32_to_e4m3_n(long long n, const float* x, uint8_t* out);
void     or_f32_to_bf16_n(long long n, const float* x, uint16_t* out);

/* ---- layer type and IndexCache schedule -------------------------------- */
int or_layer_type(int compress_ratio);       /* 1 swaonly, 4 c4a, 128 c128a, -1 unsupported */
int or_index_schedule(const int* ratios, int n_layers, int use_index_cache, int freq,
                      const char* pattern, uint8_t* skip_topk);   /* 0 ok, -1 invalid */

/* ---- cache byte accounting --------------------------------------------- */
int or_mla_entry_bytes(int nope_dim, int rope_dim);   /* fp8 nope + bf16 rope + 8 scale bytes */
int or_idx_entry_bytes(int head_dim);                 /* fp8 + one fp32 scale per 128 */

/* ---- RoPE table ---------------------------------------------------------- */
void or_rope_table(int max_pos, int rope_dim, double theta, float* out);

/* ---- compressor ---------------------------------------------------------- */
int  or_compress_pool(int ratio, int d, const uint16_t* kv_score, long long row_stride,
                      const float* ape, int p, float* y);
void or_rmsnorm(const float* y, int d, const float* w, float eps, float* z);
void or_rope_gptj(float* x, int rope_dim, const float* cos_sin_row);
void or_quant_mla(const float* z, int nope_dim, int rope_dim, uint8_t* data, uint8_t* scales);
void or_quant_idx(const float* z, int d, uint8_t* data, float* scale);
void or_quant_mla_rows(long long n, const float* z, int nope_dim, int rope_dim, uint8_t* data,
                       uint8_t* scales);
void or_quant_idx_rows(long long n, const float* z, int d, uint8_t* data, float* scale);
/* ---- FP4 (MXFP4) indexer cache ------------------------------------------ */
double  or_e2m1_to_f64(uint8_t code);
uint8_t or_f32_to_e2m1(float x);
int     or_mxfp4_exponent(float amax);
void    or_quant_idx_fp4(const float* z, int d, uint8_t* data, uint8_t* scales);
void    or_quant_idx_fp4_rows(long long n, const float* z, int d, uint8_t* data, uint8_t* scales);
int     or_idx_fp4_entry_bytes(int head_dim);

int  or_compress_stream(int kind, int ratio, int n_tokens, const uint16_t* kv_score,
                        long long row_stride, const float* ape, const float* rms_w, float eps,
                        const float* cos_sin, int rope_dim, int nope_dim,
                        uint8_t* out_data, uint8_t* out_scale);
void or_page_write(int kind, int nope_dim, int rope_dim, int page, const int* block_table,
                   int n_entries, const uint8_t* data, const uint8_t* scale, uint8_t* cache);

/* ---- indexer and top-k --------------------------------------------------- */
void or_indexer_logits(const uint8_t* q_fp8, const float* w, int n_heads, int d,
                       const uint8_t* cache, const int* block_table, int page, int n_c,
                       double* out);
void or_indexer_logits_fp4(const uint8_t* q_fp8, const float* w, int n_heads, int d,
                           const uint8_t* cache, const int* block_table, int page, int n_c,
                           double* out);
int  or_topk(const double* logits, int n, int k, int* out_idx, int* out_len);

/* ---- attention ----------------------------------------------------------- */
void or_dense_attention(const double* q, int n_heads, const double* keys, int n_keys,
                        int dk, int dv, double scale, double* out, double* lse);
int  or_gather_keys(int nope_dim, int rope_dim, int page,
                    const uint8_t* comp_cache, const int* comp_bt, const int* idx, int len,
                    const uint16_t* swa_cache, const int* swa_bt, int p, int window,
                    double* keys);
int  or_sparse_mla_v4(const uint16_t* q, int n_heads, int page, const uint8_t* comp_cache,
                      const int* comp_bt, const int* idx, int len, const uint8_t* swa_cache,
                      const int* swa_bt, int p, int window, double scale, double* out, double* lse);
void or_inv_rope_fp8_quant(const uint16_t* o, int n_heads, int pos, const float* cos_sin, int rope_dim,
                           uint8_t* codes, float* scales);
void or_dequant_gather(int kind, int nope_dim, int rope_dim, int page, const uint8_t* cache,
                       const int* bt, int s0, int n, uint16_t* out);
int  or_combine_topk_swa_indices(const int* topk, int topk_len, int pos, int seq_len, int gather_len,
                                 int window, int n_comp, int* out);
int  or_sparse_mla(const uint16_t* q, int n_heads, int nope_dim, int rope_dim, int page,
                   const uint8_t* comp_cache, const int* comp_bt, const int* idx, int len,
                   const uint16_t* swa_cache, const int* swa_bt, int p, int window,
                   double scale, double* out, double* lse);

#ifdef __cplusplus
}
#endif
#endif
