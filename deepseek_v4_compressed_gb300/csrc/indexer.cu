// indexer.cu -- lightning indexer logits and per-query top-k.
//
// I_{t,s} = sum_j w_{t,j} ReLU(q_{t,j} . k_s) (SparseAttnIndexer formula in
// the "DeepseekV4Attention" class walkthrough; section 2 of the V4 internals
// talk write-up), with k_s = FP8 row * fp32 scale of the indexer cache, over
// the causal slots s < ctx_len / 4; then the k largest per query ("Indexer,
// C4A and C128A top-k", "DeepSeek V4 attention in vLLM").
#include "dsv4_common.cuh"
#include "plan.h"

namespace dsv4 {

// ---------------------------------------------------------------------------
// Logits on the CUDA cores: one thread per slot, q in shared memory.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) indexer_logits_simt(
    const uint8_t* __restrict__ q_fp8, const float* __restrict__ w, int H,
    const uint8_t* __restrict__ cache, int num_pages, const int* __restrict__ bt, int bt_stride,
    const int* __restrict__ ctx_len, float* __restrict__ logits, int max_slots, int* status)
{
    __shared__ float qs[DSV4_MAX_IDX_HEADS * kIdx];
    __shared__ float ws[DSV4_MAX_IDX_HEADS];
    const int b = blockIdx.y;
    int n_c = ctx_len[b] / 4;
    if (n_c > max_slots) n_c = max_slots;
    if (static_cast<int>(blockIdx.x) * 128 >= n_c) return;
    const uint8_t* qb = q_fp8 + static_cast<long long>(b) * H * kIdx;
    for (int i = threadIdx.x; i < H * kIdx; i += blockDim.x) qs[i] = e4m3_to_f32(qb[i]);
    for (int i = threadIdx.x; i < H; i += blockDim.x) ws[i] = w[static_cast<long long>(b) * H + i];
    __syncthreads();
    const int s = blockIdx.x * 128 + threadIdx.x;
    if (s >= n_c) return;
    const int pi = s / kPage;
    int pg = (pi < bt_stride) ? bt[static_cast<long long>(b) * bt_stride + pi] : -1;
    if (pg < 0 || pg >= num_pages) {
        flag(status, DSV4_DEV_BAD_PAGE);
        logits[static_cast<long long>(b) * max_slots + s] = -INFINITY;
        return;
    }
    const uint8_t* page = cache + static_cast<long long>(pg) * kIdxPage;
    const int r = s % kPage;
    float k[kIdx];
    const uint4* src = reinterpret_cast<const uint4*>(page + r * kIdx);
#pragma unroll
    for (int v = 0; v < kIdx / 16; ++v) {
        uint4 u = src[v];
        const uint32_t words[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) k[v * 16 + q * 4 + bb] = e4m3_to_f32((words[q] >> (8 * bb)) & 0xff);
    }
    const float scale = reinterpret_cast<const float*>(page + kPage * kIdx)[r];
    float acc = 0.f;
    for (int j = 0; j < H; ++j) {
        float dot = 0.f;
#pragma unroll
        for (int c = 0; c < kIdx; ++c) dot = fmaf(qs[j * kIdx + c], k[c], dot);
        acc = fmaf(ws[j], fmaxf(dot, 0.f), acc);
    }
    logits[static_cast<long long>(b) * max_slots + s] = scale * acc;
}

// ---------------------------------------------------------------------------
// Top-k by radix select: one CTA per query.  Keys are the order-preserving
// uint32 images of the logits; four 8-bit passes find the k-th largest key K*
// and how many of the keys equal to K* to take (lowest slots first); a final
// ordered compaction writes the selected slots in ascending order.
// ---------------------------------------------------------------------------
constexpr int kTopkThreads = 1024;
constexpr int kTopkSmemKeys = 32768;   // keys staged in shared memory up to this many

__device__ __forceinline__ int block_excl_scan(int v, int* warp_tot, int& total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int t = (lane < kTopkThreads / 32) ? warp_tot[lane] : 0;
        int u = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, u, o);
            if (lane >= o) u += y;
        }
        warp_tot[lane] = u - t;          // exclusive prefix of warp totals
        if (lane == 31) warp_tot[32] = u;
    }
    __syncthreads();
    total = warp_tot[32];
    const int r = warp_tot[warp] + x - v;
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(kTopkThreads) topk_radix_kernel(
    const float* __restrict__ logits, int max_slots, const int* __restrict__ ctx_len, int k,
    int* __restrict__ out_idx, int out_stride, int* __restrict__ out_len, int smem_keys)
{
    extern __shared__ uint32_t skeys[];
    __shared__ int hist[256];
    __shared__ int warp_tot[33];
    __shared__ uint32_t s_prefix, s_mask;
    __shared__ int s_remaining;

    const int b = blockIdx.x;
    int n = ctx_len[b] / 4;
    if (n > max_slots) n = max_slots;
    if (n < 0) n = 0;
    int* orow = out_idx + static_cast<long long>(b) * out_stride;
    const float* lrow = logits + static_cast<long long>(b) * max_slots;
    if (n <= k) {
        for (int i = threadIdx.x; i < k; i += blockDim.x) orow[i] = (i < n) ? i : -1;
        if (threadIdx.x == 0) out_len[b] = n;
        return;
    }
    const bool in_smem = n <= smem_keys;
    if (in_smem)
        for (int i = threadIdx.x; i < n; i += blockDim.x) skeys[i] = f32_order_key(lrow[i]);
    auto key_at = [&](int i) -> uint32_t { return in_smem ? skeys[i] : f32_order_key(lrow[i]); };
    if (threadIdx.x == 0) {
        s_prefix = 0;
        s_mask = 0;
        s_remaining = k;
    }
    __syncthreads();

    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
        __syncthreads();
        const uint32_t prefix = s_prefix, mask = s_mask;
        const int lane = threadIdx.x & 31;
        // warp-aggregated histogram (most keys share their top byte)
        for (int base = 0; base < n; base += blockDim.x) {
            const int i = base + threadIdx.x;
            int digit = -1;
            if (i < n) {
                const uint32_t key = key_at(i);
                if ((key & mask) == prefix) digit = (key >> shift) & 0xff;
            }
            const unsigned peers = __match_any_sync(0xffffffffu, digit);
            if (digit >= 0 && lane == __ffs(peers) - 1) atomicAdd(&hist[digit], __popc(peers));
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            // lane l scans bins 255-8l .. 248-8l (descending digits)
            int local = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) local += hist[255 - 8 * lane - q];
            int incl = local;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const int before = incl - local;
            const int rem = s_remaining;
            const bool mine = before < rem && rem <= incl;
            const unsigned who = __ballot_sync(0xffffffffu, mine);
            if (mine && lane == __ffs(who) - 1) {
                int cum = before;
                for (int q = 0; q < 8; ++q) {
                    const int d = 255 - 8 * lane - q;
                    if (cum + hist[d] >= rem) {
                        s_prefix = prefix | (static_cast<uint32_t>(d) << shift);
                        s_mask = mask | (0xffu << shift);
                        s_remaining = rem - cum;
                        break;
                    }
                    cum += hist[d];
                }
            }
        }
        __syncthreads();
    }
    const uint32_t kstar = s_prefix;
    const int take_eq = s_remaining;   // keys equal to K* to take, lowest slots first

    // Ordered compaction: thread i owns a contiguous chunk of slots.
    const int chunk = (n + blockDim.x - 1) / blockDim.x;
    const int lo = threadIdx.x * chunk;
    const int hi = min(n, lo + chunk);
    int gt = 0, eq = 0;
    for (int i = lo; i < hi; ++i) {
        const uint32_t key = key_at(i);
        gt += key > kstar;
        eq += key == kstar;
    }
    int tot;
    const int gt_before = block_excl_scan(gt, warp_tot, tot);
    const int eq_before = block_excl_scan(eq, warp_tot, tot);
    int g = gt_before, e = eq_before;
    for (int i = lo; i < hi; ++i) {
        const uint32_t key = key_at(i);
        bool sel = false;
        if (key > kstar) {
            sel = true;
        } else if (key == kstar) {
            sel = e < take_eq;
        }
        if (sel) orow[g + min(e, take_eq)] = i;
        g += key > kstar;
        e += key == kstar;
    }
    if (threadIdx.x == 0) out_len[b] = k;
}

}  // namespace dsv4

using namespace dsv4;

extern "C" dsv4_status dsv4_indexer_topk(const dsv4_plan* plan, const dsv4_indexer_args* a,
                                         void* workspace, size_t workspace_bytes, dsv4_stream_t stream)
{
    if (plan == nullptr || a == nullptr) return DSV4_ERR_INVALID;
    if (plan->type != DSV4_C4A) return DSV4_ERR_SHAPE;
    if (workspace_bytes < plan->ws_bytes || (workspace == nullptr && plan->ws_bytes)) return DSV4_ERR_SHAPE;
    if (!a->q_fp8_dev || !a->weights_dev || !a->idx_cache_dev || !a->block_table_dev ||
        !a->ctx_len_dev || !a->out_idx_dev || !a->out_len_dev)
        return DSV4_ERR_INVALID;
    if (a->out_stride < plan->topk || a->bt_stride < 1 || a->num_pages < 1) return DSV4_ERR_SHAPE;
    if (reinterpret_cast<uintptr_t>(a->idx_cache_dev) & 15) return DSV4_ERR_SHAPE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    float* logits = reinterpret_cast<float*>(static_cast<char*>(workspace) + plan->ws_logits_off);
    const int B = plan->batch, H = plan->geom.idx_heads;
    dim3 grid((plan->max_slots + 127) / 128, B);
    indexer_logits_simt<<<grid, 128, 0, st>>>(
        static_cast<const uint8_t*>(a->q_fp8_dev), a->weights_dev, H,
        static_cast<const uint8_t*>(a->idx_cache_dev), a->num_pages, a->block_table_dev, a->bt_stride,
        a->ctx_len_dev, logits, plan->max_slots, a->status_dev);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return DSV4_ERR_CUDA;
    const int smem_keys = plan->max_slots <= kTopkSmemKeys ? plan->max_slots : 0;
    const size_t smem = static_cast<size_t>(smem_keys) * 4;
    static bool attr_set = false;
    if (!attr_set) {
        cudaFuncSetAttribute(topk_radix_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kTopkSmemKeys * 4);
        attr_set = true;
    }
    topk_radix_kernel<<<B, kTopkThreads, smem, st>>>(logits, plan->max_slots, a->ctx_len_dev, plan->topk,
                                                      a->out_idx_dev, a->out_stride, a->out_len_dev,
                                                      smem_keys);
    e = cudaGetLastError();
    return e == cudaSuccess ? DSV4_OK : DSV4_ERR_CUDA;
}
