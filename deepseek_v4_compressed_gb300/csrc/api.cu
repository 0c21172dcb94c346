// api.cu -- plans, host utilities, device status and the bounded-wait self-test.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <cudaTypedefs.h>

#include <mutex>

#include "dsv4_common.cuh"
#include "plan.h"
#include "tmap.h"

using namespace dsv4;

namespace dsv4 {

bool encode_tmap(CUtensorMap* map, CUtensorMapDataType type, int rank, const void* base, const uint64_t* dims,
                 const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swizzle)
{
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    if (fn == nullptr) return false;
    cuuint64_t d[5], s[4];
    cuuint32_t b[5], e[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        e[i] = 1;
        if (i + 1 < rank) s[i] = strides_bytes[i];
    }
    const CUresult r = fn(map, type, static_cast<cuuint32_t>(rank), const_cast<void*>(base), d, s, b, e,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return 152;
    }
    return n;
}

}  // namespace dsv4

extern "C" int dsv4_version(void) { return DSV4_VERSION; }

extern "C" const char* dsv4_status_string(dsv4_status s)
{
    switch (s) {
    case DSV4_OK: return "ok";
    case DSV4_ERR_INVALID: return "invalid argument";
    case DSV4_ERR_SHAPE: return "shape or workspace mismatch";
    case DSV4_ERR_UNSUPPORTED: return "unsupported value";
    case DSV4_ERR_CUDA: return "CUDA error";
    case DSV4_ERR_DEVICE_CHECK: return "device-side check failed";
    case DSV4_ERR_TIMEOUT: return "device-side bounded wait ran out";
    }
    return "unknown status";
}

// compress_ratio table of "DeepSeek V4 attention in vLLM": max(1, r).
extern "C" dsv4_status dsv4_layer_type_from_ratio(int compress_ratio, dsv4_layer_type* out)
{
    if (out == nullptr) return DSV4_ERR_INVALID;
    const int r = compress_ratio < 1 ? 1 : compress_ratio;
    if (r == 1) *out = DSV4_SWAONLY;
    else if (r == 4) *out = DSV4_C4A;
    else if (r == 128) *out = DSV4_C128A;
    else return DSV4_ERR_UNSUPPORTED;
    return DSV4_OK;
}

// Section 2 of "DeepSeek-V4 IndexCache freq2 cross-layer TopK reuse".
extern "C" dsv4_status dsv4_index_schedule(const int* ratios, int n_layers, int use_index_cache, int freq,
                                           const char* pattern, unsigned char* skip_topk_out)
{
    if (n_layers < 0 || (n_layers > 0 && (ratios == nullptr || skip_topk_out == nullptr)))
        return DSV4_ERR_INVALID;
    int plen = 0;
    if (pattern != nullptr) {
        plen = static_cast<int>(strlen(pattern));
        if (plen == 0 || pattern[0] != 'F') return DSV4_ERR_INVALID;
        for (int i = 0; i < plen; ++i)
            if (pattern[i] != 'F' && pattern[i] != 'S') return DSV4_ERR_INVALID;
    } else if (use_index_cache && freq < 1) {
        return DSV4_ERR_INVALID;
    }
    int rank = 0;   // number of ratio-4 layers seen so far
    for (int l = 0; l < n_layers; ++l) {
        const int r = ratios[l] < 1 ? 1 : ratios[l];
        unsigned char skip = 0;
        if (r == 4) {
            if (use_index_cache)
                skip = pattern ? (rank < plen && pattern[rank] == 'S') : (rank % freq != 0);
            ++rank;
        }
        skip_topk_out[l] = skip;
    }
    return DSV4_OK;
}

// cos_sin_cache layout of DeepseekCompressor.forward: [pos][cos half | sin half].
extern "C" dsv4_status dsv4_rope_table(float* host_out, int max_pos, int rope_dim, double theta)
{
    if (host_out == nullptr || max_pos < 0 || rope_dim <= 0 || (rope_dim & 1) || !(theta > 0.0))
        return DSV4_ERR_INVALID;
    const int half = rope_dim / 2;
    for (int i = 0; i < half; ++i) {
        const double inv_freq = pow(theta, -2.0 * static_cast<double>(i) / static_cast<double>(rope_dim));
        for (int pos = 0; pos < max_pos; ++pos) {
            const double angle = static_cast<double>(pos) * inv_freq;
            host_out[static_cast<size_t>(pos) * rope_dim + i] = static_cast<float>(cos(angle));
            host_out[static_cast<size_t>(pos) * rope_dim + half + i] = static_cast<float>(sin(angle));
        }
    }
    return DSV4_OK;
}

extern "C" dsv4_status dsv4_read_device_status(int* status_dev, dsv4_stream_t stream, int* bits_out)
{
    if (status_dev == nullptr) return DSV4_ERR_INVALID;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int bits = 0;
    if (cudaMemcpyAsync(&bits, status_dev, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return DSV4_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return DSV4_ERR_CUDA;
    if (bits != 0 && cudaMemsetAsync(status_dev, 0, sizeof(int), st) != cudaSuccess) return DSV4_ERR_CUDA;
    if (bits_out) *bits_out = bits;
    if (bits & DSV4_DEV_TIMEOUT) return DSV4_ERR_TIMEOUT;
    return bits ? DSV4_ERR_DEVICE_CHECK : DSV4_OK;
}

// ---------------------------------------------------------------------------
// Plans: one per layer type ("SWA cache and tile scheduler": one tile plan per
// type, reused by all layers of the type).
// ---------------------------------------------------------------------------
extern "C" dsv4_status dsv4_plan_create(dsv4_layer_type type, const dsv4_geom* g, int batch, int topk,
                                        int max_ctx, dsv4_plan** out)
{
    if (g == nullptr || out == nullptr) return DSV4_ERR_INVALID;
    *out = nullptr;
    if (type != DSV4_SWAONLY && type != DSV4_C4A && type != DSV4_C128A) return DSV4_ERR_INVALID;
    if (batch < 1 || max_ctx < 1 || topk < 0) return DSV4_ERR_INVALID;
    if (g->n_heads < 1 || g->n_heads > DSV4_MAX_HEADS) return DSV4_ERR_UNSUPPORTED;
    if (g->window != DSV4_WINDOW) return DSV4_ERR_UNSUPPORTED;
    if (!(g->softmax_scale > 0.0f)) return DSV4_ERR_INVALID;
    if (type == DSV4_C4A && (g->idx_heads < 1 || g->idx_heads > DSV4_MAX_IDX_HEADS)) return DSV4_ERR_UNSUPPORTED;
    if (type != DSV4_SWAONLY && topk < 1) return DSV4_ERR_INVALID;
    if (topk + g->window > 8 * 1024) return DSV4_ERR_UNSUPPORTED;   // 8 CTAs x 1024 keys
    dsv4_plan* p = static_cast<dsv4_plan*>(calloc(1, sizeof(dsv4_plan)));
    if (p == nullptr) return DSV4_ERR_INVALID;
    p->type = type;
    p->geom = *g;
    p->batch = batch;
    p->topk = (type == DSV4_SWAONLY) ? 0 : topk;
    p->max_ctx = max_ctx;
    p->max_slots = (type == DSV4_C4A) ? max_ctx / 4 : (type == DSV4_C128A ? max_ctx / 128 : 0);
    p->max_keys = p->topk + g->window;
    if (type == DSV4_C4A) {
        // indexer: 128-slot tiles; a sequence's tiles are split over at most
        // SMs / batch CTAs (one CTA per SM), each streaming its share
        const int tiles = (p->max_slots + 127) / 128;
        int per_seq = sm_count() / batch;
        per_seq = per_seq < 1 ? 1 : (per_seq > tiles ? tiles : per_seq);
        p->idx_tiles_per_cta = tiles > 0 ? (tiles + per_seq - 1) / per_seq : 1;
        p->idx_ctas_per_seq = tiles > 0 ? (tiles + p->idx_tiles_per_cta - 1) / p->idx_tiles_per_cta : 0;
        // the CTAs of a sequence form a cluster that also selects the top-k,
        // when they fit one (at most 8 CTAs of at most 16 tiles each)
        p->idx_fused_topk = p->idx_ctas_per_seq >= 1 && p->idx_ctas_per_seq <= 8 && p->idx_tiles_per_cta <= 16;
    }
    p->mla_head_groups = (g->n_heads + 63) / 64;
    // attention: the keys of a (sequence, head group) are split over a cluster
    // of 1, 2 or 4 CTAs, the largest that keeps every CTA on its own SM; 8
    // only when 4 would leave a CTA more than 256 keys (clusters of 8 cost
    // more to place behind the previous kernel and to merge: at batch 16, 640
    // keys, 8 splits measured 25.8 us a layer against 14.2 us for 4; at batch
    // 4, 2176 keys, 20.7 against 29.8 us)
    {
        const int units = batch * p->mla_head_groups;
        const int sms = sm_count();
        int c = 1;
        while (c < 4 && units * c * 2 <= sms) c <<= 1;
        if (c == 4 && units * 8 <= sms && (p->max_keys + 3) / 4 > 256) c = 8;
        while (c < 8 && (p->max_keys + c - 1) / c > 1024) c <<= 1;   // a CTA owns at most 1024 keys
        p->mla_splits = c;
        p->mla_keys_per_split = (p->max_keys + c - 1) / c;
    }
    size_t off = 0;
    p->ws_logits_off = off;
    p->logits_stride = (p->max_slots + 3) & ~3;
    if (type == DSV4_C4A) off += align256(static_cast<size_t>(batch) * p->logits_stride * sizeof(float));
    p->ws_partial_off = off;
    p->ws_partial_bytes = 0;
    off += p->ws_partial_bytes;
    p->ws_bytes = off;
    *out = p;
    return DSV4_OK;
}

// The indexer cache format of a c4a plan: FP8 (the default) or MXFP4
// ([V4-attn] use_fp4_indexer_cache; [V4-internals] section 4).
extern "C" dsv4_status dsv4_plan_set_indexer_format(dsv4_plan* plan, dsv4_idx_format format)
{
    if (plan == nullptr) return DSV4_ERR_INVALID;
    if (format != DSV4_IDX_FP8 && format != DSV4_IDX_FP4) return DSV4_ERR_INVALID;
    if (plan->type != DSV4_C4A) return DSV4_ERR_UNSUPPORTED;
    plan->idx_fp4 = format == DSV4_IDX_FP4;
    return DSV4_OK;
}

extern "C" dsv4_status dsv4_plan_set_kv_layout(dsv4_plan* plan, dsv4_kv_layout layout)
{
    if (plan == nullptr) return DSV4_ERR_INVALID;
    if (layout != DSV4_KV_576 && layout != DSV4_KV_V4) return DSV4_ERR_INVALID;
    plan->kv_v4 = layout == DSV4_KV_V4;
    return DSV4_OK;
}

extern "C" void dsv4_plan_destroy(dsv4_plan* plan) { free(plan); }

extern "C" size_t dsv4_plan_workspace_bytes(const dsv4_plan* plan) { return plan ? plan->ws_bytes : 0; }

extern "C" dsv4_status dsv4_plan_get_info(const dsv4_plan* p, dsv4_plan_info* info)
{
    if (p == nullptr || info == nullptr) return DSV4_ERR_INVALID;
    memset(info, 0, sizeof(*info));
    info->layer_type = p->type;
    info->batch = p->batch;
    info->n_heads = p->geom.n_heads;
    info->idx_heads = p->geom.idx_heads;
    info->topk = p->topk;
    info->max_ctx = p->max_ctx;
    info->max_slots = p->max_slots;
    info->idx_ctas_per_seq = p->idx_ctas_per_seq;
    info->mla_splits = p->mla_splits;
    info->mla_head_groups = p->mla_head_groups;
    info->mla_keys_per_split = p->mla_keys_per_split;
    info->workspace_bytes = p->ws_bytes;
    info->launches_indexer = (p->type == DSV4_C4A) ? (p->idx_fused_topk ? 1 : 2) : 0;
    info->launches_mla = 1;   // one cluster launch; partials merge through DSMEM
    return DSV4_OK;
}

// ---------------------------------------------------------------------------
// Bounded wait self-test: an mbarrier that nothing arrives at.
// ---------------------------------------------------------------------------
__global__ void bounded_wait_kernel(int* status, int spin_limit)
{
    __shared__ __align__(8) uint64_t bar;
    const uint32_t addr = static_cast<uint32_t>(__cvta_generic_to_shared(&bar));
    if (threadIdx.x == 0)
        asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(addr), "r"(1) : "memory");
    __syncthreads();
    uint32_t done = 0;
    for (int i = 0; i < spin_limit && !done; ++i) {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(addr), "r"(0)
            : "memory");
    }
    if (!done && threadIdx.x == 0) flag(status, DSV4_DEV_TIMEOUT);
}

extern "C" dsv4_status dsv4_selftest_bounded_wait(int* status_dev, int spin_limit, dsv4_stream_t stream)
{
    if (status_dev == nullptr || spin_limit < 0) return DSV4_ERR_INVALID;
    bounded_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(status_dev, spin_limit);
    return cudaGetLastError() == cudaSuccess ? DSV4_OK : DSV4_ERR_CUDA;
}
