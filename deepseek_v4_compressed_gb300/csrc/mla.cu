// mla.cu -- sparse absorbed-MQA decode over (selected compressed slots) ||
// (SWA window), one 576-dim latent KV head, value = the 512 latent dims.
//
// _forward_decode of the "DeepseekV4Attention" class walkthrough
// (flash_mla_with_kvcache over the SWA cache plus the compressed cache with
// their two index sets); KV_actual = selected history || recent window in
// section 2 of the V4 internals talk write-up; absorbed decode over the
// cached latent in section 2.2 of "From MLA to CSA + HCA".
#include "dsv4_common.cuh"
#include "plan.h"

namespace dsv4 {

struct MlaParams {
    const uint16_t* q;
    const uint8_t* swa;
    int swa_pages;
    const int* swa_bt;
    int swa_bt_stride;
    const uint8_t* comp;
    int comp_pages;
    const int* comp_bt;
    int comp_bt_stride;
    const int* idx;
    int idx_stride;
    const int* idx_len;
    const int* ctx_len;
    uint16_t* out;
    float* lse;
    int H;
    int window;
    float scale;
    int* status;
};

// Row pointer of key i of sequence b (compressed keys first, then the SWA
// window).  Returns false (and flags) for an out-of-range index or page.
struct KeyRef {
    const uint8_t* row;     // compressed: 640 data bytes; SWA: 576 bf16
    const uint8_t* scales;  // compressed only
    bool comp;
};

__device__ __forceinline__ bool key_ref(const MlaParams& P, int b, int i, int n_comp, int t0, KeyRef& k)
{
    if (i < n_comp) {
        const int slot = P.idx[static_cast<long long>(b) * P.idx_stride + i];
        const int pi = slot / kPage;
        if (slot < 0 || pi >= P.comp_bt_stride) {
            flag(P.status, DSV4_DEV_BAD_INDEX);
            return false;
        }
        const int pg = P.comp_bt[static_cast<long long>(b) * P.comp_bt_stride + pi];
        if (pg < 0 || pg >= P.comp_pages) {
            flag(P.status, DSV4_DEV_BAD_PAGE);
            return false;
        }
        const uint8_t* page = P.comp + static_cast<long long>(pg) * kMlaPage;
        const int r = slot % kPage;
        k.row = page + r * kMlaData;
        k.scales = page + kPage * kMlaData + r * 8;
        k.comp = true;
        return true;
    }
    const int t = t0 + (i - n_comp);
    const int pi = t / kPage;
    const int pg = (pi < P.swa_bt_stride) ? P.swa_bt[static_cast<long long>(b) * P.swa_bt_stride + pi] : -1;
    if (pg < 0 || pg >= P.swa_pages) {
        flag(P.status, DSV4_DEV_BAD_PAGE);
        return false;
    }
    k.row = P.swa + static_cast<long long>(pg) * kSwaPage + (t % kPage) * (kHead * 2);
    k.scales = nullptr;
    k.comp = false;
    return true;
}

// ---------------------------------------------------------------------------
// CUDA-core version: CTA = (head group of 8, sequence), 256 threads; keys in
// chunks of 32 dequantised into shared memory; online softmax per head.
// ---------------------------------------------------------------------------
constexpr int kSimtHeads = 8;
constexpr int kSimtKeys = 32;
constexpr int kSimtRow = kHead + 1;   // padded row (bank-conflict free column reads)

__global__ void __launch_bounds__(256) mla_decode_simt(MlaParams P)
{
    extern __shared__ float smem[];
    float* qs = smem;                              // [8][576]
    float* ks = qs + kSimtHeads * kHead;           // [32][577]
    float* ps = ks + kSimtKeys * kSimtRow;         // [8][32]
    __shared__ float s_m[kSimtHeads], s_l[kSimtHeads], s_alpha[kSimtHeads];

    const int b = blockIdx.y;
    const int h0 = blockIdx.x * kSimtHeads;
    const int nh = min(kSimtHeads, P.H - h0);
    const int tid = threadIdx.x;
    const int p = P.ctx_len[b] - 1;
    const int n_comp = P.idx_len ? max(0, P.idx_len[b]) : 0;
    const int t0 = max(0, p - P.window + 1);
    const int n_keys = n_comp + (p >= 0 ? p - t0 + 1 : 0);

    for (int i = tid; i < kSimtHeads * kHead; i += 256) {
        const int h = i / kHead;
        qs[i] = (h < nh) ? bf16_bits_to_f32(P.q[(static_cast<long long>(b) * P.H + h0 + h) * kHead + i % kHead]) : 0.f;
    }
    if (tid < kSimtHeads) {
        s_m[tid] = -INFINITY;
        s_l[tid] = 0.f;
    }
    // thread owns head hh = tid / 32 and dims v = lane + 32 * u (u < 16)
    const int hh = tid >> 5, lane = tid & 31;
    float acc[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) acc[u] = 0.f;
    __syncthreads();

    for (int base = 0; base < n_keys; base += kSimtKeys) {
        const int nk = min(kSimtKeys, n_keys - base);
        // stage keys: 32 rows x 576 values, 8 warps x 4 rows
        for (int kk = tid >> 5; kk < kSimtKeys; kk += 8) {
            float* dst = ks + kk * kSimtRow;
            KeyRef kr;
            const bool ok = kk < nk && key_ref(P, b, base + kk, n_comp, t0, kr);
            if (!ok) {
                for (int c = lane; c < kHead; c += 32) dst[c] = 0.f;
                continue;
            }
            if (kr.comp) {
                for (int c = lane; c < kNope; c += 32)
                    dst[c] = e4m3_to_f32(kr.row[c]) * exp2i(static_cast<int>(kr.scales[c >> 6]) - 127);
                const uint16_t* rope = reinterpret_cast<const uint16_t*>(kr.row + kNope);
                for (int c = lane; c < kRope; c += 32) dst[kNope + c] = bf16_bits_to_f32(rope[c]);
            } else {
                const uint16_t* row = reinterpret_cast<const uint16_t*>(kr.row);
                for (int c = lane; c < kHead; c += 32) dst[c] = bf16_bits_to_f32(row[c]);
            }
        }
        __syncthreads();
        // scores: thread (hh, key lane)
        float s = -INFINITY;
        if (lane < nk && hh < nh) {
            float dot = 0.f;
            const float* qr = qs + hh * kHead;
            const float* kr = ks + lane * kSimtRow;
            for (int c = 0; c < kHead; ++c) dot = fmaf(qr[c], kr[c], dot);
            s = dot * P.scale;
        }
        const float cmax = warp_max(s);
        const float m_old = s_m[hh];
        const float m_new = fmaxf(m_old, cmax);
        const float pexp = (s == -INFINITY) ? 0.f : __expf(s - m_new);
        const float csum = warp_sum(pexp);
        ps[hh * kSimtKeys + lane] = pexp;
        const float alpha = (m_old == -INFINITY) ? 0.f : __expf(m_old - m_new);
        __syncthreads();
        if (lane == 0) {
            s_m[hh] = m_new;
            s_l[hh] = s_l[hh] * alpha + csum;
        }
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int v = lane + 32 * u;
            float a = acc[u] * alpha;
            for (int kk = 0; kk < nk; ++kk) a = fmaf(ps[hh * kSimtKeys + kk], ks[kk * kSimtRow + v], a);
            acc[u] = a;
        }
        __syncthreads();
    }
    if (hh < nh) {
        const float l = s_l[hh];
        const float inv = (l > 0.f) ? 1.f / l : 0.f;
        uint16_t* o = P.out + (static_cast<long long>(b) * P.H + h0 + hh) * kV;
#pragma unroll
        for (int u = 0; u < 16; ++u) o[lane + 32 * u] = f32_to_bf16_bits(acc[u] * inv);
        if (P.lse && lane == 0)
            P.lse[static_cast<long long>(b) * P.H + h0 + hh] = (l > 0.f) ? s_m[hh] + logf(l) : -INFINITY;
    }
}

}  // namespace dsv4

using namespace dsv4;

extern "C" dsv4_status dsv4_sparse_mla_decode(const dsv4_plan* plan, const dsv4_mla_args* a,
                                              void* workspace, size_t workspace_bytes,
                                              dsv4_stream_t stream)
{
    if (plan == nullptr || a == nullptr) return DSV4_ERR_INVALID;
    if (workspace_bytes < plan->ws_bytes || (workspace == nullptr && plan->ws_bytes)) return DSV4_ERR_SHAPE;
    if (!a->q_dev || !a->swa_cache_dev || !a->swa_block_table_dev || !a->ctx_len_dev || !a->out_dev)
        return DSV4_ERR_INVALID;
    const bool sparse = plan->type != DSV4_SWAONLY;
    if (sparse && (!a->comp_cache_dev || !a->comp_block_table_dev || !a->topk_idx_dev || !a->topk_len_dev))
        return DSV4_ERR_INVALID;
    if (sparse && a->topk_stride < plan->topk) return DSV4_ERR_SHAPE;
    MlaParams P;
    P.q = static_cast<const uint16_t*>(a->q_dev);
    P.swa = static_cast<const uint8_t*>(a->swa_cache_dev);
    P.swa_pages = a->swa_num_pages;
    P.swa_bt = a->swa_block_table_dev;
    P.swa_bt_stride = a->swa_bt_stride;
    P.comp = sparse ? static_cast<const uint8_t*>(a->comp_cache_dev) : nullptr;
    P.comp_pages = a->comp_num_pages;
    P.comp_bt = sparse ? a->comp_block_table_dev : nullptr;
    P.comp_bt_stride = a->comp_bt_stride;
    P.idx = sparse ? a->topk_idx_dev : nullptr;
    P.idx_stride = a->topk_stride;
    P.idx_len = sparse ? a->topk_len_dev : nullptr;
    P.ctx_len = a->ctx_len_dev;
    P.out = static_cast<uint16_t*>(a->out_dev);
    P.lse = a->lse_dev;
    P.H = plan->geom.n_heads;
    P.window = plan->geom.window;
    P.scale = plan->geom.softmax_scale;
    P.status = a->status_dev;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const size_t smem = sizeof(float) * (kSimtHeads * kHead + kSimtKeys * kSimtRow + kSimtHeads * kSimtKeys);
    static bool attr_set = false;
    if (!attr_set) {
        cudaFuncSetAttribute(mla_decode_simt, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        attr_set = true;
    }
    dim3 grid((P.H + kSimtHeads - 1) / kSimtHeads, plan->batch);
    mla_decode_simt<<<grid, 256, smem, st>>>(P);
    return cudaGetLastError() == cudaSuccess ? DSV4_OK : DSV4_ERR_CUDA;
}
